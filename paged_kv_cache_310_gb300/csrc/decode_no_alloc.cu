// decode_no_alloc.cu -- paged_attention_decode for callers that cannot allocate
// device memory: the split-K / work-list workspace comes from a fixed array that the
// library itself places in device memory when it is loaded.
//
// Who needs it: code that runs where cudaMalloc is off limits -- inside a custom
// allocator or memory-pool callback, on a path that must never fail with
// out-of-memory once serving has started, or in a host runtime that only hands
// kernels pre-registered buffers.  Such callers still own q, the caches, the
// tables and out; only the scratch space is taken from this file's array.
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace {

// 32 MiB per GPU that loads the library, held until the process exits.
constexpr size_t kNoAllocWorkspaceBytes = size_t{32} << 20;

static __device__ __align__(256) unsigned char g_no_alloc_workspace[kNoAllocWorkspaceBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_workspace_ptr[kMaxDevices] = {};

// Device address of the array on the current device.  In host code the array's
// name is only a host-side stand-in, so the address is looked up once per device
// (this needs that device current) and cached.
pkv_status workspace_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return pkv::record_error(PKV_ERR_CUDA, "cudaGetDevice failed");
  if (dev < 0 || dev >= kMaxDevices) return pkv::record_error(PKV_ERR_UNSUPPORTED, "device index too large");
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_workspace_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_no_alloc_workspace);
    if (e != cudaSuccess || !p)
      return pkv::record_error(PKV_ERR_CUDA, "cudaGetSymbolAddress of the built-in workspace failed");
    g_workspace_ptr[dev] = p;
  }
  *out = g_workspace_ptr[dev];
  return PKV_OK;
}

}  // namespace

extern "C" {

size_t paged_attention_no_alloc_limit(void) { return kNoAllocWorkspaceBytes; }

pkv_status paged_attention_decode_no_alloc(const void* q, const void* k_cache, const void* v_cache,
                                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                                           const int32_t* context_lens, int32_t num_seqs,
                                           int32_t num_q_heads, int32_t max_context_len, float scale,
                                           void* out, int32_t out_dtype, const pkv_cache_desc* cache,
                                           const pkv_decode_config* config, void* stream) {
  const size_t need =
      paged_attention_workspace_bytes(num_seqs, num_q_heads, max_context_len, cache, config);
  if (need > kNoAllocWorkspaceBytes) {
    char msg[256];
    snprintf(msg, sizeof msg,
             "needs %zu bytes of workspace, more than the %zu-byte built-in array; use "
             "paged_attention_decode with a caller workspace or a larger partition_tokens",
             need, kNoAllocWorkspaceBytes);
    return pkv::record_error(PKV_ERR_WORKSPACE, msg);
  }
  void* ws = nullptr;
  if (need > 0) {
    if (pkv_status st = workspace_address(&ws)) return st;
  }
  // Every byte the decode kernels read from the workspace is written earlier in the
  // same call, so nothing needs clearing between calls.
  return paged_attention_decode(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                                num_seqs, num_q_heads, max_context_len, scale, out, out_dtype, ws,
                                need > 0 ? kNoAllocWorkspaceBytes : 0, cache, config, stream);
}

}  // extern "C"
