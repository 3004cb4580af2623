// cache_ops.cu -- the data-movement kernels of the paged KV cache:
//  * append: scatter each new token's K/V row into its slot (a block row);
//  * block copy: copy-on-write duplication of whole blocks;
//  * gather: materialise each sequence's K/V through its block table (a test of the
//    indexing alone).
// All three move 16-byte vectors with coalesced accesses; they are bit-exact copies.
// Pages: "Efficient Memory Management ... with PagedAttention", How It Works (blocks
// filled as tokens are generated; copy when a sharer diverges); note-023, Method and
// Concepts (block table, copy-on-write).
#include "common.cuh"
#include "launch.h"

namespace pkv {
namespace {

constexpr int kThreads = 256;

int grid_for(int64_t work, int cap) {
  int64_t g = (work + kThreads - 1) / kThreads;
  return static_cast<int>(g < 1 ? 1 : (g > cap ? cap : g));
}

// One thread per 16-byte vector of one (token, kv head) row of K and of V.
__global__ void __launch_bounds__(kThreads)
append_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
              const int64_t* __restrict__ slots, int32_t num_tokens, uint4* __restrict__ kc,
              uint4* __restrict__ vc, int32_t num_kv_heads, int32_t block_size,
              int32_t row_vecs, int64_t num_slots, int* err) {
  // A kernel launched after this one as a programmatic dependent (the decode work
  // list, which reads only context lengths) may start now; it waits for this kernel
  // before it completes.
  grid_dependents_launch();
  const int64_t per_token = static_cast<int64_t>(num_kv_heads) * row_vecs;
  const int64_t total = per_token * num_tokens;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = i / per_token;
    const int64_t rem = i - t * per_token;  // = h * row_vecs + c
    const int64_t slot = slots[t];
    if (slot < 0) continue;  // padding
    if (slot >= num_slots) {
      set_error(err, kErrIndex);
      continue;
    }
    const int64_t b = slot / block_size;
    const int64_t r = slot - b * block_size;
    const int64_t h = rem / row_vecs;
    const int64_t c = rem - h * row_vecs;
    const int64_t dst = ((b * num_kv_heads + h) * block_size + r) * row_vecs + c;
    kc[dst] = k[i];
    vc[dst] = v[i];
  }
}

// blockIdx.y = pair; the CTAs along x split the block's vectors.
__global__ void __launch_bounds__(kThreads)
block_copy_kernel(const int64_t* __restrict__ pairs, uint4* __restrict__ kc,
                  uint4* __restrict__ vc, int64_t block_vecs, int32_t num_blocks, int* err) {
  const int64_t src = pairs[2 * static_cast<int64_t>(blockIdx.y)];
  const int64_t dst = pairs[2 * static_cast<int64_t>(blockIdx.y) + 1];
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_error(err, kErrIndex);
    return;
  }
  const uint4* ks = kc + src * block_vecs;
  const uint4* vs = vc + src * block_vecs;
  uint4* kd = kc + dst * block_vecs;
  uint4* vd = vc + dst * block_vecs;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < block_vecs;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint4 a = ks[i];
    const uint4 b = vs[i];
    kd[i] = a;
    vd[i] = b;
  }
}

// blockIdx.y = sequence, blockIdx.z = kv head; x strides over the sequence's rows.
__global__ void __launch_bounds__(kThreads)
gather_kernel(const uint4* __restrict__ kc, const uint4* __restrict__ vc,
              const int32_t* __restrict__ tables, int32_t max_blocks, const int32_t* __restrict__ lens,
              int32_t max_len, uint4* __restrict__ k_out, uint4* __restrict__ v_out,
              int32_t num_kv_heads, int32_t block_size, int32_t row_vecs, int32_t num_blocks,
              int* err) {
  const int s = blockIdx.y, h = blockIdx.z;
  const int n = lens[s];
  if (n > max_len) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_error(err, kErrLength);
    return;
  }
  const int64_t total = static_cast<int64_t>(n) * row_vecs;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int j = static_cast<int>(i / row_vecs);
    const int c = static_cast<int>(i - static_cast<int64_t>(j) * row_vecs);
    const int logical = j / block_size;
    if (logical >= max_blocks) {
      set_error(err, kErrIndex);
      continue;
    }
    const int b = tables[static_cast<int64_t>(s) * max_blocks + logical];
    if (b < 0 || b >= num_blocks) {
      set_error(err, kErrIndex);
      continue;
    }
    const int64_t src = ((static_cast<int64_t>(b) * num_kv_heads + h) * block_size + j % block_size) *
                            row_vecs + c;
    const int64_t dst = ((static_cast<int64_t>(s) * num_kv_heads + h) * max_len + j) * row_vecs + c;
    k_out[dst] = kc[src];
    v_out[dst] = vc[src];
  }
}

// Swap: whole blocks (all heads and rows of K and V) between the pools and a staging
// buffer of [n][block] in memory the device can reach (pinned host memory for a real
// swap).  blockIdx.y = listed block, x strides over its 16-byte vectors.
template <bool kOut>
__global__ void __launch_bounds__(kThreads)
swap_kernel(const int64_t* __restrict__ ids, uint4* kc, uint4* vc, uint4* hk, uint4* hv, int64_t block_vecs,
            int32_t num_blocks, int* err) {
  const int64_t b = ids[blockIdx.y];
  if (b < 0 || b >= num_blocks) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_error(err, kErrIndex);
    return;
  }
  uint4* pk = kc + b * block_vecs;
  uint4* pv = vc + b * block_vecs;
  uint4* sk = hk + static_cast<int64_t>(blockIdx.y) * block_vecs;
  uint4* sv = hv + static_cast<int64_t>(blockIdx.y) * block_vecs;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < block_vecs;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    if (kOut) {
      sk[i] = pk[i];
      sv[i] = pv[i];
    } else {
      pk[i] = sk[i];
      pv[i] = sv[i];
    }
  }
}

// Self-test of the bounded wait: an mbarrier that expects one arrival nobody makes.
// The wait gives up after limit_ns, sets the timeout flag and the kernel returns.
__global__ void wait_timeout_kernel(uint64_t limit_ns, int* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0, limit_ns)) set_error(err, kErrTimeout);
}

}  // namespace

cudaError_t launch_swap(bool out, const int64_t* ids, int32_t n, void* k_cache, void* v_cache, void* stage_k,
                        void* stage_v, int64_t block_bytes, int32_t num_blocks, int* err, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  const int64_t block_vecs = block_bytes / 16;
  dim3 grid(grid_for(block_vecs, 64), n);
  auto* kc = static_cast<uint4*>(k_cache);
  auto* vc = static_cast<uint4*>(v_cache);
  auto* sk = static_cast<uint4*>(stage_k);
  auto* sv = static_cast<uint4*>(stage_v);
  if (out)
    swap_kernel<true><<<grid, kThreads, 0, stream>>>(ids, kc, vc, sk, sv, block_vecs, num_blocks, err);
  else
    swap_kernel<false><<<grid, kThreads, 0, stream>>>(ids, kc, vc, sk, sv, block_vecs, num_blocks, err);
  return cudaGetLastError();
}

cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, int* err, cudaStream_t stream) {
  wait_timeout_kernel<<<1, 32, 0, stream>>>(limit_ns, err);
  return cudaGetLastError();
}

cudaError_t launch_append(const void* k, const void* v, const int64_t* slots, int32_t num_tokens,
                          void* k_cache, void* v_cache, int32_t num_kv_heads, int32_t block_size,
                          int32_t row_bytes, int64_t num_slots, int* err, cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const int32_t row_vecs = row_bytes / 16;
  const int64_t work = static_cast<int64_t>(num_tokens) * num_kv_heads * row_vecs;
  append_kernel<<<grid_for(work, 152 * 16), kThreads, 0, stream>>>(
      static_cast<const uint4*>(k), static_cast<const uint4*>(v), slots, num_tokens,
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), num_kv_heads, block_size,
      row_vecs, num_slots, err);
  return cudaGetLastError();
}

cudaError_t launch_block_copy(const int64_t* pairs, int32_t num_pairs, void* k_cache,
                              void* v_cache, int64_t block_bytes, int32_t num_blocks, int* err,
                              cudaStream_t stream) {
  if (num_pairs == 0) return cudaSuccess;
  const int64_t block_vecs = block_bytes / 16;
  dim3 grid(grid_for(block_vecs, 64), num_pairs);
  block_copy_kernel<<<grid, kThreads, 0, stream>>>(pairs, static_cast<uint4*>(k_cache),
                                                   static_cast<uint4*>(v_cache), block_vecs,
                                                   num_blocks, err);
  return cudaGetLastError();
}

cudaError_t launch_gather(const void* k_cache, const void* v_cache, const int32_t* block_tables,
                          int32_t max_blocks_per_seq, const int32_t* context_lens,
                          int32_t num_seqs, int32_t max_len, void* k_out, void* v_out,
                          int32_t num_kv_heads, int32_t block_size, int32_t row_bytes,
                          int32_t num_blocks, int* err, cudaStream_t stream) {
  if (num_seqs == 0 || max_len == 0) return cudaSuccess;
  const int32_t row_vecs = row_bytes / 16;
  dim3 grid(grid_for(static_cast<int64_t>(max_len) * row_vecs, 64), num_seqs, num_kv_heads);
  gather_kernel<<<grid, kThreads, 0, stream>>>(
      static_cast<const uint4*>(k_cache), static_cast<const uint4*>(v_cache), block_tables,
      max_blocks_per_seq, context_lens, max_len, static_cast<uint4*>(k_out),
      static_cast<uint4*>(v_out), num_kv_heads, block_size, row_vecs, num_blocks, err);
  return cudaGetLastError();
}

}  // namespace pkv
