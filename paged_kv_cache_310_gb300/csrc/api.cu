// api.cu -- the extern "C" entry points of libpagedkv.so (declared in
// include/pagedkv.h): argument checks, launch configuration, the device error flag.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include "common.cuh"
#include "launch.h"

namespace pkv {
namespace {

// One error flag per device that loads the library.  Kernels OR bits into it
// instead of trapping; paged_kv_device_error() reads and clears it.
__device__ int g_device_error;

thread_local std::string t_last_error;

pkv_status fail(pkv_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return st;
}

pkv_status cuda_fail(cudaError_t e, const char* what) {
  return fail(PKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Bound of the decode and prefill kernels' pipeline waits (kWaitLimitNs unless a test
// lowers it with paged_kv_set_wait_limit); read once per launch.
std::atomic<uint64_t> g_wait_limit_ns{kWaitLimitNs};

constexpr int kMaxDevices = 64;
std::mutex g_flag_mutex;
int* g_flag_ptr[kMaxDevices] = {};

// Device address of g_device_error on the current device (looked up once per device).
pkv_status device_flag(int** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(PKV_ERR_UNSUPPORTED, "device %d", dev);
  std::lock_guard<std::mutex> lock(g_flag_mutex);
  if (!g_flag_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_error);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error flag)");
    g_flag_ptr[dev] = static_cast<int*>(p);
  }
  *out = g_flag_ptr[dev];
  return PKV_OK;
}

size_t elem_bytes(int dtype) { return dtype == PKV_F32 ? 4 : 2; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

pkv_status check_cache(const pkv_cache_desc* c) {
  if (!c) return fail(PKV_ERR_INVALID_ARG, "cache descriptor is NULL");
  if (c->dtype < PKV_F32 || c->dtype > PKV_BF16)
    return fail(PKV_ERR_UNSUPPORTED, "cache dtype %d", c->dtype);
  if (c->num_blocks <= 0 || c->num_kv_heads <= 0)
    return fail(PKV_ERR_INVALID_ARG, "num_blocks %d, num_kv_heads %d must be positive",
                c->num_blocks, c->num_kv_heads);
  if (c->block_size != 8 && c->block_size != 16 && c->block_size != 32 && c->block_size != 64)
    return fail(PKV_ERR_UNSUPPORTED, "block_size %d (supported: 8, 16, 32, 64)", c->block_size);
  if (c->head_dim != 64 && c->head_dim != 128)
    return fail(PKV_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", c->head_dim);
  if (c->num_kv_heads > 65535) return fail(PKV_ERR_UNSUPPORTED, "num_kv_heads %d", c->num_kv_heads);
  return PKV_OK;
}

struct DecodePlan {
  int path;         // PKV_PATH_CUDA_CORE or PKV_PATH_TENSOR_CORE
  int part_tokens;  // tokens per partition, multiple of 128
  int max_parts;    // partitions of the longest sequence
  size_t workspace; // bytes
  size_t list_bytes;  // work list (tensor-core path): 256-byte header + entries
  size_t ml_bytes;    // partition (max, sum) pairs
};

int round_up(int x, int m) { return (x + m - 1) / m * m; }

pkv_status plan_decode(int32_t num_seqs, int32_t num_q_heads, int32_t max_len,
                       const pkv_cache_desc* c, const pkv_decode_config* cfg, DecodePlan* plan) {
  if (pkv_status st = check_cache(c)) return st;
  if (num_seqs < 0 || num_seqs > 65535)
    return fail(PKV_ERR_INVALID_ARG, "num_seqs %d outside [0, 65535]", num_seqs);
  if (num_q_heads <= 0 || num_q_heads % c->num_kv_heads)
    return fail(PKV_ERR_INVALID_ARG, "num_q_heads %d is not a positive multiple of num_kv_heads %d",
                num_q_heads, c->num_kv_heads);
  const int group = num_q_heads / c->num_kv_heads;
  if (max_len < 0) return fail(PKV_ERR_INVALID_ARG, "max_context_len %d < 0", max_len);
  int path = cfg ? cfg->path : PKV_PATH_AUTO;
  if (path < PKV_PATH_AUTO || path > PKV_PATH_TENSOR_CORE)
    return fail(PKV_ERR_INVALID_ARG, "decode path %d", path);
  const bool tc_ok = tc_supported(c->dtype, c->head_dim, group, c->block_size);
  // Tensor cores wherever they apply to 16-bit caches: at G >= 2 QK and PV are real
  // contractions, and at G = 1 the persistent TMA/tcgen05 kernel still streams K/V
  // faster (1.00-1.02 against 0.92 of copy bandwidth on a 64 x 32-head bf16 batch; at
  // head_dim 64 0.91 with paired KV heads against 0.86).
  // f32 caches take the tf32 kernel at head_dim 128 from 5 query heads per KV head (at
  // 5 to 8: 0.82 of copy bandwidth against 0.36-0.37 on CUDA cores); up to 4 the CUDA-core
  // kernel streams faster (0.92 against 0.84 at 4) with no conversion work, and at head_dim
  // 64 it is as fast or a little faster at every group (0.53-0.54 against 0.53 at 5 to 8).
  if (path == PKV_PATH_AUTO)
    path = tc_ok && (c->dtype != PKV_F32 || (group >= 5 && c->head_dim == 128)) ? PKV_PATH_TENSOR_CORE
                                                                                : PKV_PATH_CUDA_CORE;
  if (path == PKV_PATH_TENSOR_CORE && !tc_ok)
    return fail(PKV_ERR_UNSUPPORTED,
                "tensor-core path needs head_dim 64 or 128 and group <= 16 (<= 8 for f32) (group %d)", group);
  if (path == PKV_PATH_CUDA_CORE && group > 8)
    return fail(PKV_ERR_UNSUPPORTED, "CUDA-core path supports query-head groups <= 8 (group %d)", group);
  if (static_cast<int64_t>(c->num_blocks) * c->num_kv_heads * c->block_size > (int64_t{1} << 30))
    return fail(PKV_ERR_UNSUPPORTED, "pool of %d blocks too large for 32-bit row coordinates", c->num_blocks);
  int part = cfg ? cfg->partition_tokens : 0;
  if (part < 0 || part % 128 || part > 16384)
    return fail(PKV_ERR_INVALID_ARG, "partition_tokens %d: need 0 or a multiple of 128 <= 16384", part);
  if (path == PKV_PATH_TENSOR_CORE && part > kTcMaxPartition)
    return fail(PKV_ERR_INVALID_ARG, "tensor-core partitions are at most %d tokens (%d asked)",
                kTcMaxPartition, part);
  if (part == 0) {
    int auto_part = 512;
    if (path == PKV_PATH_CUDA_CORE) {
      // one CTA per (partition, KV head, sequence): aim for about 12 CTAs per SM
      // (several waves of three resident CTAs), partitions of 512 to 2048 tokens
      const int64_t work = static_cast<int64_t>(num_seqs) * c->num_kv_heads * (max_len / 2 + 1);
      const int64_t per_cta = work / (12 * 152) + 1;
      auto_part = static_cast<int>(per_cta > 2048 ? 2048 : per_cta);
      auto_part = round_up(auto_part < 512 ? 512 : auto_part, 128);
    } else {
      // Persistent CTAs balance well with >= ~3 items per SM (GB300: 152 SMs): take
      // the largest partition (fewest items, no merge when a sequence fits) that
      // still leaves about that many, assuming lengths average half the maximum.
      const int64_t work = static_cast<int64_t>(num_seqs) * c->num_kv_heads * (max_len / 2 + 1);
      const int64_t per_item = work / (3 * 152) + 1;
      auto_part = static_cast<int>(per_item > kTcMaxPartition ? kTcMaxPartition : per_item);
      auto_part = round_up(auto_part < 512 ? 512 : auto_part, 128);
    }
    part = max_len <= auto_part ? (max_len < 128 ? 128 : round_up(max_len, 128)) : auto_part;
  }
  plan->path = path;
  plan->part_tokens = part;
  plan->max_parts = max_len == 0 ? 1 : (max_len + part - 1) / part;
  if (path == PKV_PATH_TENSOR_CORE && plan->max_parts >= 32768)
    return fail(PKV_ERR_UNSUPPORTED, "tensor-core path: %d partitions per sequence is too many", plan->max_parts);
  if (static_cast<int64_t>(plan->max_parts) * num_seqs * c->num_kv_heads > (int64_t{1} << 30))
    return fail(PKV_ERR_UNSUPPORTED, "too many (partition, sequence, kv head) items");
  // layout: [work list header + entries (tensor-core path)] [partition (max, sum)] [partition outputs]
  plan->list_bytes = 0;
  if (path == PKV_PATH_TENSOR_CORE) {
    const size_t entries = static_cast<size_t>(plan->max_parts) * num_seqs * c->num_kv_heads;
    plan->list_bytes = 256 + (entries * 16 + 255) / 256 * 256;
  }
  plan->ml_bytes = 0;
  plan->workspace = plan->list_bytes;
  if (plan->max_parts > 1) {
    const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads * plan->max_parts;
    plan->ml_bytes = (rows * 2 * sizeof(float) + 255) / 256 * 256;
    plan->workspace += plan->ml_bytes + rows * c->head_dim * sizeof(float);
  }
  return PKV_OK;
}

}  // namespace

pkv_status record_error(pkv_status status, const char* message) { return fail(status, "%s", message); }

}  // namespace pkv

using namespace pkv;

extern "C" {

const char* paged_kv_version(void) { return "0.1.0"; }

const char* paged_kv_last_error(void) { return t_last_error.c_str(); }

pkv_status paged_kv_device_error(void* stream) {
  int* flag = nullptr;
  if (pkv_status st = device_flag(&flag)) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int value = 0;
  e = cudaMemcpy(&value, flag, sizeof value, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error flag");
  if (value) {
    const int zero = 0;
    e = cudaMemcpy(flag, &zero, sizeof zero, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the device error flag");
  }
  if (value & kErrTimeout) return fail(PKV_ERR_DEVICE_TIMEOUT, "a kernel's bounded wait ran out (flag 0x%x)", value);
  if (value) return fail(PKV_ERR_DEVICE_INDEX, "a kernel met an out-of-range index or length (flag 0x%x)", value);
  return PKV_OK;
}

pkv_status paged_kv_set_wait_limit(uint64_t limit_ns) {
  if (limit_ns > 5000000000ull)
    return fail(PKV_ERR_INVALID_ARG, "limit_ns %llu above 5 s", (unsigned long long)limit_ns);
  g_wait_limit_ns.store(limit_ns == 0 ? kWaitLimitNs : limit_ns);
  return PKV_OK;
}

pkv_status paged_kv_selftest_wait_timeout(uint64_t limit_ns, void* stream) {
  if (limit_ns == 0 || limit_ns > 5000000000ull)
    return fail(PKV_ERR_INVALID_ARG, "limit_ns %llu outside (0, 5 s]", (unsigned long long)limit_ns);
  int* flag = nullptr;
  if (pkv_status st = device_flag(&flag)) return st;
  cudaError_t e = launch_wait_timeout_selftest(limit_ns, flag, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : cuda_fail(e, "self-test launch");
}

pkv_status paged_kv_append(const void* k, const void* v, const int64_t* slot_mapping,
                           int32_t num_tokens, void* k_cache, void* v_cache,
                           const pkv_cache_desc* cache, void* stream) {
  if (pkv_status st = check_cache(cache)) return st;
  if (num_tokens < 0) return fail(PKV_ERR_INVALID_ARG, "num_tokens %d < 0", num_tokens);
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache)
    return fail(PKV_ERR_INVALID_ARG, "NULL pointer argument");
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(PKV_ERR_INVALID_ARG, "k, v and the caches must be 16-byte aligned");
  int* flag = nullptr;
  if (pkv_status st = device_flag(&flag)) return st;
  const int row_bytes = static_cast<int>(cache->head_dim * elem_bytes(cache->dtype));
  cudaError_t e = launch_append(k, v, slot_mapping, num_tokens, k_cache, v_cache,
                                cache->num_kv_heads, cache->block_size, row_bytes,
                                static_cast<int64_t>(cache->num_blocks) * cache->block_size, flag,
                                static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : cuda_fail(e, "append launch");
}

pkv_status paged_block_copy(const int64_t* src_dst_pairs, const int64_t* host_pairs,
                            int32_t num_pairs, void* k_cache, void* v_cache,
                            const pkv_cache_desc* cache, void* stream) {
  if (pkv_status st = check_cache(cache)) return st;
  if (num_pairs < 0 || num_pairs > 65535)
    return fail(PKV_ERR_INVALID_ARG, "num_pairs %d outside [0, 65535]", num_pairs);
  if (num_pairs == 0) return PKV_OK;
  if (!src_dst_pairs || !k_cache || !v_cache) return fail(PKV_ERR_INVALID_ARG, "NULL pointer argument");
  if (!aligned16(k_cache) || !aligned16(v_cache))
    return fail(PKV_ERR_INVALID_ARG, "the caches must be 16-byte aligned");
  if (host_pairs) {
    // copy-on-write pairs: ids in range, src != dst, no dst twice, no dst also a src
    std::string seen_dst(static_cast<size_t>(cache->num_blocks), 0), seen_src(seen_dst);
    for (int32_t i = 0; i < num_pairs; ++i) {
      const int64_t a = host_pairs[2 * i], b = host_pairs[2 * i + 1];
      if (a < 0 || a >= cache->num_blocks || b < 0 || b >= cache->num_blocks)
        return fail(PKV_ERR_INVALID_ARG, "pair %d (%lld, %lld) outside [0, %d)", i, (long long)a,
                    (long long)b, cache->num_blocks);
      if (a == b) return fail(PKV_ERR_INVALID_ARG, "pair %d copies block %lld onto itself", i, (long long)a);
      if (seen_dst[b]) return fail(PKV_ERR_INVALID_ARG, "destination block %lld appears twice", (long long)b);
      seen_dst[b] = 1;
      seen_src[a] = 1;
    }
    for (int32_t i = 0; i < num_pairs; ++i)
      if (seen_src[host_pairs[2 * i + 1]])
        return fail(PKV_ERR_INVALID_ARG, "block %lld is both a source and a destination",
                    (long long)host_pairs[2 * i + 1]);
  }
  int* flag = nullptr;
  if (pkv_status st = device_flag(&flag)) return st;
  const int64_t block_bytes = static_cast<int64_t>(cache->num_kv_heads) * cache->block_size *
                              cache->head_dim * elem_bytes(cache->dtype);
  cudaError_t e = launch_block_copy(src_dst_pairs, num_pairs, k_cache, v_cache, block_bytes,
                                    cache->num_blocks, flag, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : cuda_fail(e, "block copy launch");
}

pkv_status paged_attention_plan(int32_t num_seqs, int32_t num_q_heads, int32_t max_context_len,
                                const pkv_cache_desc* cache, const pkv_decode_config* config,
                                pkv_decode_plan* out) {
  if (!out) return fail(PKV_ERR_INVALID_ARG, "plan output is NULL");
  DecodePlan plan;
  if (pkv_status st = plan_decode(num_seqs, num_q_heads, max_context_len, cache, config, &plan)) return st;
  out->path = plan.path;
  out->partition_tokens = plan.part_tokens;
  out->max_partitions = plan.max_parts;
  out->kernel_launches = num_seqs == 0 ? 0
                         : 1 + (plan.path == PKV_PATH_TENSOR_CORE ? 1 : 0) + (plan.max_parts > 1 ? 1 : 0);
  out->workspace_bytes = plan.workspace;
  out->kv_heads_per_item =
      plan.path == PKV_PATH_TENSOR_CORE ? tc_heads_per_item(cache->dtype, cache->head_dim, cache->num_kv_heads) : 1;
  return PKV_OK;
}

}  // extern "C"

namespace {

// A pointer the device can use for `host`: pinned or registered host memory (its
// device alias), device or managed memory (as is).  Pageable memory is refused.
pkv_status device_view(const void* host, void** out) {
  cudaPointerAttributes attr{};
  cudaError_t e = cudaPointerGetAttributes(&attr, host);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(PKV_ERR_INVALID_ARG, "swap buffer: not memory CUDA knows (%s)", cudaGetErrorString(e));
  }
  if (attr.type == cudaMemoryTypeUnregistered)
    return fail(PKV_ERR_INVALID_ARG, "swap buffer is pageable host memory: pin it (cudaHostAlloc / cudaHostRegister)");
  *out = attr.type == cudaMemoryTypeHost ? attr.devicePointer : const_cast<void*>(host);
  if (!*out) return fail(PKV_ERR_INVALID_ARG, "swap buffer has no device mapping");
  return PKV_OK;
}

pkv_status swap(bool out, const int64_t* ids, int32_t n, void* k_cache, void* v_cache, const void* stage_k,
                const void* stage_v, const pkv_cache_desc* cache, void* stream) {
  if (pkv_status st = check_cache(cache)) return st;
  if (n < 0 || n > 65535) return fail(PKV_ERR_INVALID_ARG, "num_ids %d outside [0, 65535]", n);
  if (n == 0) return PKV_OK;
  if (!ids || !k_cache || !v_cache || !stage_k || !stage_v) return fail(PKV_ERR_INVALID_ARG, "NULL pointer argument");
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(stage_k) || !aligned16(stage_v))
    return fail(PKV_ERR_INVALID_ARG, "caches and swap buffers must be 16-byte aligned");
  void *dk = nullptr, *dv = nullptr;
  if (pkv_status st = device_view(stage_k, &dk)) return st;
  if (pkv_status st = device_view(stage_v, &dv)) return st;
  int* flag = nullptr;
  if (pkv_status st = device_flag(&flag)) return st;
  const int64_t block_bytes = static_cast<int64_t>(cache->num_kv_heads) * cache->block_size *
                              cache->head_dim * elem_bytes(cache->dtype);
  cudaError_t e = launch_swap(out, ids, n, k_cache, v_cache, dk, dv, block_bytes, cache->num_blocks, flag,
                              static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : cuda_fail(e, "swap launch");
}

}  // namespace

extern "C" {

pkv_status paged_block_swap_out(const int64_t* block_ids, int32_t num_ids, const void* k_cache,
                                const void* v_cache, void* host_k, void* host_v,
                                const pkv_cache_desc* cache, void* stream) {
  return swap(true, block_ids, num_ids, const_cast<void*>(k_cache), const_cast<void*>(v_cache), host_k, host_v,
              cache, stream);
}

pkv_status paged_block_swap_in(const int64_t* block_ids, int32_t num_ids, const void* host_k,
                               const void* host_v, void* k_cache, void* v_cache,
                               const pkv_cache_desc* cache, void* stream) {
  return swap(false, block_ids, num_ids, k_cache, v_cache, host_k, host_v, cache, stream);
}

size_t paged_attention_workspace_bytes(int32_t num_seqs, int32_t num_q_heads,
                                       int32_t max_context_len, const pkv_cache_desc* cache,
                                       const pkv_decode_config* config) {
  DecodePlan plan;
  if (plan_decode(num_seqs, num_q_heads, max_context_len, cache, config, &plan) != PKV_OK) return 0;
  return plan.workspace;
}

pkv_status paged_attention_decode(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* block_tables, int32_t max_blocks_per_seq,
                                  const int32_t* context_lens, int32_t num_seqs,
                                  int32_t num_q_heads, int32_t max_context_len, float scale,
                                  void* out, int32_t out_dtype, void* workspace,
                                  size_t workspace_bytes, const pkv_cache_desc* cache,
                                  const pkv_decode_config* config, void* stream) {
  DecodePlan plan;
  if (pkv_status st = plan_decode(num_seqs, num_q_heads, max_context_len, cache, config, &plan))
    return st;
  if (num_seqs == 0) return PKV_OK;
  if (!q || !k_cache || !v_cache || !context_lens || !out)
    return fail(PKV_ERR_INVALID_ARG, "NULL pointer argument");
  if (max_context_len > 0 && !block_tables) return fail(PKV_ERR_INVALID_ARG, "block_tables is NULL");
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return fail(PKV_ERR_INVALID_ARG, "q, out and the caches must be 16-byte aligned");
  if (out_dtype != cache->dtype && out_dtype != PKV_F32)
    return fail(PKV_ERR_UNSUPPORTED, "out dtype %d (must be the cache dtype or f32)", out_dtype);
  if (!std::isfinite(scale)) return fail(PKV_ERR_INVALID_ARG, "scale is not finite");
  const int64_t need_blocks = (static_cast<int64_t>(max_context_len) + cache->block_size - 1) / cache->block_size;
  if (max_blocks_per_seq < need_blocks)
    return fail(PKV_ERR_INVALID_ARG, "max_blocks_per_seq %d < ceil(max_context_len / block_size) = %lld",
                max_blocks_per_seq, (long long)need_blocks);
  if (plan.workspace > 0) {
    if (!workspace || workspace_bytes < plan.workspace)
      return fail(PKV_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", plan.workspace,
                  workspace ? workspace_bytes : 0);
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
      return fail(PKV_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  }
  int* flag = nullptr;
  if (pkv_status st = device_flag(&flag)) return st;

  DecodeParams p{};
  p.q = q;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.out = out;
  if (plan.list_bytes > 0) {
    p.work_count = static_cast<int*>(workspace);
    p.work_next = reinterpret_cast<int*>(static_cast<char*>(workspace) + 128);
    p.work_list = reinterpret_cast<int4*>(static_cast<char*>(workspace) + 256);
  }
  if (plan.max_parts > 1) {
    char* base = static_cast<char*>(workspace) + plan.list_bytes;
    p.ws_ml = reinterpret_cast<float*>(base);
    p.ws_o = reinterpret_cast<float*>(base + plan.ml_bytes);
  }
  p.err = flag;
  p.num_seqs = num_seqs;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = cache->num_kv_heads;
  p.group = num_q_heads / cache->num_kv_heads;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.block_size = cache->block_size;
  p.num_blocks = cache->num_blocks;
  p.head_dim = cache->head_dim;
  p.part_tokens = plan.part_tokens;
  p.max_parts = plan.max_parts;
  p.heads_per_item = 1;  // the tensor-core launcher pairs heads where it can
  p.out_f32 = out_dtype == PKV_F32 ? 1 : 0;
  p.scale_log2 = scale * 1.4426950408889634f;  // log2(e): softmax is evaluated with exp2
  p.wait_limit_ns = g_wait_limit_ns.load();

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = plan.path == PKV_PATH_TENSOR_CORE ? launch_decode_tc(p, cache->dtype, s)
                                                    : launch_decode_simt(p, cache->dtype, s);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  e = launch_merge(p, cache->dtype, s);
  if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  return PKV_OK;
}

size_t paged_attention_prefill_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t num_query_tokens,
                                               const pkv_cache_desc* cache) {
  if (!cache || cache->num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % cache->num_kv_heads ||
      num_seqs < 0 || num_query_tokens < 0)
    return 0;
  const int group = num_q_heads / cache->num_kv_heads;
  if (group > 16) return 0;
  return 256 + (prefill_max_items(num_seqs, num_query_tokens, cache->num_kv_heads, group) * 16 + 255) / 256 * 256;
}

pkv_status paged_attention_prefill(const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_tables, int32_t max_blocks_per_seq,
                                   const int32_t* context_lens, const int32_t* query_start, int32_t num_seqs,
                                   int32_t num_q_heads, int32_t num_query_tokens, int32_t max_context_len,
                                   float scale, void* out, int32_t out_dtype, void* workspace,
                                   size_t workspace_bytes, const pkv_cache_desc* cache, void* stream) {
  if (pkv_status st = check_cache(cache)) return st;
  if (num_seqs < 0 || num_seqs > (1 << 20)) return fail(PKV_ERR_INVALID_ARG, "num_seqs %d", num_seqs);
  if (num_q_heads <= 0 || num_q_heads % cache->num_kv_heads)
    return fail(PKV_ERR_INVALID_ARG, "num_q_heads %d is not a positive multiple of num_kv_heads %d", num_q_heads,
                cache->num_kv_heads);
  const int group = num_q_heads / cache->num_kv_heads;
  if (cache->dtype == PKV_F32 || !tc_supported(cache->dtype, cache->head_dim, group, cache->block_size))
    return fail(PKV_ERR_UNSUPPORTED, "prefill needs f16/bf16, head_dim 64 or 128 and query-head groups <= 16");
  if (cache->num_kv_heads > 4095)  // a work-list entry packs the KV head into 12 bits
    return fail(PKV_ERR_UNSUPPORTED, "prefill supports at most 4095 KV heads (%d)", cache->num_kv_heads);
  if (num_query_tokens < 0 || max_context_len < 0) return fail(PKV_ERR_INVALID_ARG, "negative size");
  if (num_seqs == 0 || num_query_tokens == 0) return PKV_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !query_start || !out)
    return fail(PKV_ERR_INVALID_ARG, "NULL pointer argument");
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return fail(PKV_ERR_INVALID_ARG, "q, out and the caches must be 16-byte aligned");
  if (out_dtype != cache->dtype && out_dtype != PKV_F32)
    return fail(PKV_ERR_UNSUPPORTED, "out dtype %d (must be the cache dtype or f32)", out_dtype);
  if (!std::isfinite(scale)) return fail(PKV_ERR_INVALID_ARG, "scale is not finite");
  if (static_cast<int64_t>(cache->num_blocks) * cache->num_kv_heads * cache->block_size > (int64_t{1} << 30))
    return fail(PKV_ERR_UNSUPPORTED, "pool too large for 32-bit row coordinates");
  const int64_t need_blocks = (static_cast<int64_t>(max_context_len) + cache->block_size - 1) / cache->block_size;
  if (max_blocks_per_seq < need_blocks)
    return fail(PKV_ERR_INVALID_ARG, "max_blocks_per_seq %d < ceil(max_context_len / block_size)", max_blocks_per_seq);
  const size_t need = paged_attention_prefill_workspace_bytes(num_seqs, num_q_heads, num_query_tokens, cache);
  if (!workspace || workspace_bytes < need)
    return fail(PKV_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, workspace ? workspace_bytes : 0);
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return fail(PKV_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  int* flag = nullptr;
  if (pkv_status st = device_flag(&flag)) return st;
  PrefillParams p{};
  p.q = q;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.query_start = query_start;
  p.out = out;
  p.work_count = static_cast<int*>(workspace);
  p.work_list = reinterpret_cast<int4*>(static_cast<char*>(workspace) + 256);
  p.err = flag;
  p.num_seqs = num_seqs;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = cache->num_kv_heads;
  p.group = group;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.block_size = cache->block_size;
  p.num_blocks = cache->num_blocks;
  p.max_context_len = max_context_len;
  p.num_query_tokens = num_query_tokens;
  p.tile_tokens = prefill_tile_tokens(group);
  p.head_dim = cache->head_dim;
  p.out_f32 = out_dtype == PKV_F32 ? 1 : 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.wait_limit_ns = g_wait_limit_ns.load();
  cudaError_t e = launch_prefill_tc(p, cache->dtype, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : cuda_fail(e, "prefill launch");
}

pkv_status paged_kv_gather(const void* k_cache, const void* v_cache, const int32_t* block_tables,
                           int32_t max_blocks_per_seq, const int32_t* context_lens,
                           int32_t num_seqs, int32_t max_context_len, void* k_out, void* v_out,
                           const pkv_cache_desc* cache, void* stream) {
  if (pkv_status st = check_cache(cache)) return st;
  if (num_seqs < 0 || num_seqs > 65535) return fail(PKV_ERR_INVALID_ARG, "num_seqs %d", num_seqs);
  if (max_context_len < 0) return fail(PKV_ERR_INVALID_ARG, "max_context_len %d", max_context_len);
  if (num_seqs == 0 || max_context_len == 0) return PKV_OK;
  if (!k_cache || !v_cache || !block_tables || !context_lens || !k_out || !v_out)
    return fail(PKV_ERR_INVALID_ARG, "NULL pointer argument");
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_out) || !aligned16(v_out))
    return fail(PKV_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
  int* flag = nullptr;
  if (pkv_status st = device_flag(&flag)) return st;
  const int row_bytes = static_cast<int>(cache->head_dim * elem_bytes(cache->dtype));
  cudaError_t e = launch_gather(k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                                num_seqs, max_context_len, k_out, v_out, cache->num_kv_heads,
                                cache->block_size, row_bytes, cache->num_blocks, flag,
                                static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : cuda_fail(e, "gather launch");
}

}  // extern "C"
