// launch.h -- host-side launchers shared between the translation units of
// libpagedkv (not part of the public ABI; see include/pagedkv.h for that).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pagedkv.h"

namespace pkv {

// Everything decode kernels need, by value (one __grid_constant__ struct).
struct DecodeParams {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  void* out;
  float* ws_o;   // [S][Hq][max_parts][D] un-normalised partition outputs (fp32)
  float* ws_ml;  // [S][Hq][max_parts][2] partition (max, sum) in the log2 domain
  int* err;      // device error flag
  int4* work_list;  // tensor-core path: items sorted longest first (work-list kernel)
  int* work_count;  // number of entries in work_list
  int* work_next;   // claims so far past the grid's first entries (reset by the work-list kernel)
  int32_t num_seqs, num_q_heads, num_kv_heads, group, max_blocks_per_seq;
  int32_t block_size, num_blocks, head_dim;
  int32_t part_tokens, max_parts;
  int32_t out_f32;   // 1: out is fp32, 0: out has the cache dtype
  float scale_log2;  // softmax scale * log2(e): scores live in the exp2 domain
  uint64_t wait_limit_ns;  // bound of every pipeline wait (kWaitLimitNs unless a test lowers it)
  int32_t heads_per_item;  // KV heads of one tensor-core work item: 1, or 2 (head_dim 64, paired heads)
};

// Multi-token causal (prefill) attention, tensor cores; f16/bf16, head_dim 64 or 128.
struct PrefillParams {
  const void* q;  // [T][Hq][head_dim]
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* query_start;  // [S+1]
  void* out;                   // [T][Hq][head_dim]
  int4* work_list;
  int* work_count;
  int* err;
  int32_t num_seqs, num_q_heads, num_kv_heads, group, max_blocks_per_seq;
  int32_t block_size, num_blocks, max_context_len, num_query_tokens, tile_tokens;
  int32_t head_dim;  // 64 or 128
  int32_t out_f32;
  float scale_log2;
  uint64_t wait_limit_ns;  // bound of every pipeline wait (kWaitLimitNs unless a test lowers it)
};
int prefill_tile_tokens(int group);
size_t prefill_max_items(int num_seqs, int num_query_tokens, int num_kv_heads, int group);
cudaError_t launch_prefill_tc(const PrefillParams& p, int dtype, cudaStream_t stream);

// CUDA-core split-K decode (any supported dtype, head_dim 64/128, group <= 8).
cudaError_t launch_decode_simt(const DecodeParams& p, int dtype, cudaStream_t stream);
// Tensor-core (tcgen05) decode: f16/bf16, head_dim 64/128, group <= 16, persistent CTAs
// fed by a work list that a one-CTA kernel builds first.  Partitions <= 4096 tokens.
constexpr int kTcMaxPartition = 4096;
bool tc_supported(int dtype, int head_dim, int group, int block_size);
// KV heads one work item of the 16-bit tensor-core decode covers (2: paired heads).
int tc_heads_per_item(int dtype, int head_dim, int num_kv_heads);
cudaError_t launch_decode_tc(const DecodeParams& p, int dtype, cudaStream_t stream);
// The f32 (tf32, split-operand) decode kernel over a work list already launched on the
// stream; head_dim 64/128, group <= 8.
cudaError_t launch_decode_tc32(const DecodeParams& p, int grid, cudaStream_t stream);
// Partition merge for sequences longer than one partition.
cudaError_t launch_merge(const DecodeParams& p, int dtype, cudaStream_t stream);

// Records a failure message for paged_kv_last_error() on this host thread.
pkv_status record_error(pkv_status status, const char* message);

// Swap whole blocks between the pools and a device-reachable staging buffer.
cudaError_t launch_swap(bool out, const int64_t* ids, int32_t n, void* k_cache, void* v_cache, void* stage_k,
                        void* stage_v, int64_t block_bytes, int32_t num_blocks, int* err, cudaStream_t stream);

// Diagnostic: one bounded wait that cannot complete (see paged_kv_selftest_wait_timeout).
cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, int* err, cudaStream_t stream);

cudaError_t launch_append(const void* k, const void* v, const int64_t* slots, int32_t num_tokens,
                          void* k_cache, void* v_cache, int32_t num_kv_heads, int32_t block_size,
                          int32_t row_bytes, int64_t num_slots, int* err, cudaStream_t stream);

cudaError_t launch_block_copy(const int64_t* pairs, int32_t num_pairs, void* k_cache,
                              void* v_cache, int64_t block_bytes, int32_t num_blocks, int* err,
                              cudaStream_t stream);

cudaError_t launch_gather(const void* k_cache, const void* v_cache, const int32_t* block_tables,
                          int32_t max_blocks_per_seq, const int32_t* context_lens,
                          int32_t num_seqs, int32_t max_len, void* k_out, void* v_out,
                          int32_t num_kv_heads, int32_t block_size, int32_t row_bytes,
                          int32_t num_blocks, int* err, cudaStream_t stream);

}  // namespace pkv
