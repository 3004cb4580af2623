// tc_util.cuh -- pieces shared by the persistent tensor-core kernels (decode and
// prefill): the work-list cursor, the role-aware bounded wait, 16-bit packing and
// output stores, and host helpers for tiled TMA maps of the block pool.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "common.cuh"

namespace pkv {
namespace {

// Walks this CTA's items: the list is sorted longest first and dealt out in snake
// order (round k goes left to right when k is even, right to left when odd), which
// evens out the CTAs' chunk counts to within a few percent (113-124 per CTA on the
// GQA-70B-like decode batch).  The next entry is always loaded one item ahead so its
// latency hides behind the current item.
struct ItemCursor {
  const int4* list;
  int count, k, idx, idx_next;
  int4 cur, nxt;

  __device__ __forceinline__ int snake(int r) const {
    return r * static_cast<int>(gridDim.x) +
           ((r & 1) ? static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x)
                    : static_cast<int>(blockIdx.x));
  }
  __device__ __forceinline__ void init(const int4* l, int n) {
    list = l;
    count = n;
    k = 0;
    idx = snake(0);
    cur = idx < count ? list[idx] : make_int4(0, 0, 0, 0);
    idx_next = snake(1);
    nxt = idx_next < count ? list[idx_next] : make_int4(0, 0, 0, 0);
  }
  __device__ __forceinline__ bool valid() const { return idx < count; }
  __device__ __forceinline__ void advance() {
    ++k;
    idx = idx_next;
    cur = nxt;
    idx_next = snake(k + 1);
    if (idx_next < count) nxt = list[idx_next];
  }
};

// Bounded wait that also gives up when another role has aborted; limit_ns is the
// launch's wait limit (normally kWaitLimitNs).
__device__ __forceinline__ bool wait_role(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          int* err, uint64_t limit_ns) {
  if (limit_ns < kPollBelowNs) {  // a short limit: probe without suspending, clock every round
    const uint64_t t0 = global_timer_ns();
    while (!mbar_test_wait(bar, parity)) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > limit_ns) {
        *abort_flag = 1;
        set_error(err, kErrTimeout);
        return false;
      }
    }
    return true;
  }
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      set_error(err, kErrTimeout);
      return false;
    }
  }
}

// The same for two barriers (b1 may be null): one round trip when both phases have
// already completed, else one wait after the other.
__device__ __forceinline__ bool wait_role2(uint64_t* b0, uint32_t p0, uint64_t* b1, uint32_t p1,
                                           volatile int* abort_flag, int* err, uint64_t limit_ns) {
  if (b1 == nullptr) return wait_role(b0, p0, abort_flag, err, limit_ns);
  if (mbar_test_wait2(b0, p0, b1, p1) == 3u) return true;
  return wait_role(b0, p0, abort_flag, err, limit_ns) && wait_role(b1, p1, abort_flag, err, limit_ns);
}

template <typename T>
__device__ __forceinline__ uint32_t pack2(float a, float b);
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float a, float b) {
  __half2 v = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}
// Round a pair to the 16-bit type (RNE) and also return the rounded values as floats.
template <typename T>
__device__ __forceinline__ uint32_t pack2_split(float a, float b, float& ra, float& rb);
template <>
__device__ __forceinline__ uint32_t pack2_split<__nv_bfloat16>(float a, float b, float& ra, float& rb) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  const uint32_t u = *reinterpret_cast<uint32_t*>(&v);
  ra = __uint_as_float(u << 16);
  rb = __uint_as_float(u & 0xffff0000u);
  return u;
}
template <>
__device__ __forceinline__ uint32_t pack2_split<__half>(float a, float b, float& ra, float& rb) {
  __half2 v = __floats2half2_rn(a, b);
  const float2 f = __half22float2(v);
  ra = f.x;
  rb = f.y;
  return *reinterpret_cast<uint32_t*>(&v);
}

// Maximum over the warp's 32 lanes in one instruction (sm_100 family); like fmaxf,
// NaN inputs are ignored.
__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

// Sums each of a lane's N values (N a power of two <= 32) over the warp's 32 lanes
// by a reduce-scatter: at each step a lane keeps half of its values and adds its
// partner's copy of that half, then a butterfly over the remaining lane bits.  Returns
// in every lane the total of value warp_sum_index<N>(lane), after N - 1 + 5 - log2 N
// shuffles instead of 5 N.
template <int N>
__device__ __forceinline__ float warp_sum_scatter(const float* v, int lane) {
  float a[N];
#pragma unroll
  for (int i = 0; i < N; ++i) a[i] = v[i];
  int off = 16;
#pragma unroll
  for (int n = N; n > 1; n >>= 1, off >>= 1) {
    const bool upper = lane & off;  // this lane keeps the upper half
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? a[i] : a[i + n / 2];
      const float keep = upper ? a[i + n / 2] : a[i];
      a[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  float r = a[0];
#pragma unroll
  for (; off > 0; off >>= 1) r += __shfl_xor_sync(0xffffffffu, r, off);
  return r;
}

// Which of the N values warp_sum_scatter<N> leaves in `lane`.
template <int N>
__device__ __forceinline__ int warp_sum_index(int lane) {
  int h = 0;
#pragma unroll
  for (int n = N, off = 16; n > 1; n >>= 1, off >>= 1) h = 2 * h + ((lane & off) ? 1 : 0);
  return h;
}

// 2^x with the hardware approximation (relative error about 2^-22; exp2(-inf) = 0).
__device__ __forceinline__ float exp2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Three-input maximum / minimum (one instruction on this architecture).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float fmin3(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

template <typename T>
__device__ __forceinline__ float round_to(float x) {
  return Elem<T>::to_float(Elem<T>::from_float(x));
}

template <typename T>
__device__ __forceinline__ void store_out(void* out, size_t i, float x, int out_f32) {
  if (out_f32)
    static_cast<float*>(out)[i] = x;
  else
    static_cast<T*>(out)[i] = Elem<T>::from_float(x);
}


typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  return fn;
}

// Encoding a tiled TMA map is host work a decode call repeated for each of its maps
// on every call.  A map depends only on what is in its key, so the last few encoded
// on this host thread are kept and handed out again (a serving loop reuses the same
// pools and a few q buffers).  `kind` tells the map layouts apart.
struct MapKey {
  const void* base;
  uint64_t rows;
  uint32_t box_rows;
  int kind, dtype, head_dim;
  bool operator==(const MapKey& o) const {
    return base == o.base && rows == o.rows && box_rows == o.box_rows && kind == o.kind && dtype == o.dtype &&
           head_dim == o.head_dim;
  }
};

template <typename Encode>
bool cached_map(CUtensorMap* m, const MapKey& key, Encode encode) {
  struct Entry {
    CUtensorMap map;
    MapKey key;
    bool used;
  };
  constexpr int kEntries = 16;
  thread_local Entry cache[kEntries] = {};
  thread_local int next = 0;
  for (int i = 0; i < kEntries; ++i)
    if (cache[i].used && cache[i].key == key) {
      *m = cache[i].map;
      return true;
    }
  if (!encode(m)) return false;
  cache[next].map = *m;
  cache[next].key = key;
  cache[next].used = true;
  next = (next + 1) % kEntries;
  return true;
}

// Pool of rows of head_dim (64 or 128) 16-bit elements seen as 4-D: (64 columns,
// 8 rows, 64-column blocks, 8-row groups) with byte strides (-, row, 128, 8 rows).  A
// box of (64, 8, head_dim/64, bs/8) is one block's tile for one KV head, landing as
// [group][column block][row][64 columns].
bool make_pool_map_uncached(CUtensorMap* m, const void* base, uint64_t rows, uint32_t block_size, bool bf16,
                            int head_dim) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || rows % 8 || (head_dim != 64 && head_dim != 128)) return false;
  const cuuint64_t row_bytes = static_cast<cuuint64_t>(head_dim) * 2, blocks = head_dim / 64;
  cuuint64_t dims[4] = {64, 8, blocks, rows / 8};
  cuuint64_t strides[3] = {row_bytes, 128, 8 * row_bytes};
  cuuint32_t box[4] = {64, 8, static_cast<cuuint32_t>(blocks), block_size / 8};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
            const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_pool_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t block_size, bool bf16,
                   int head_dim) {
  return cached_map(m, MapKey{base, rows, block_size, 1, bf16 ? 2 : 1, head_dim}, [&](CUtensorMap* out) {
    return make_pool_map_uncached(out, base, rows, block_size, bf16, head_dim);
  });
}

// Head_dim 64, two adjacent KV heads per box: their tiles of one block are
// consecutive (bs rows of 128 bytes each), and the box takes row r of both as one
// 256-byte operand row, head h's 64 columns as column block 0 and head h + 1's as
// column block 1: dims (64 columns, 8 rows, 2 heads, 8-row groups), so one box lands
// in shared memory exactly like a head_dim-128 tile.  The box at group w (w = the
// first row of head h's tile / 8, h even) covers the block's bs rows of both heads.
bool make_pair_pool_map_uncached(CUtensorMap* m, const void* base, uint64_t rows, uint32_t block_size, bool bf16) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || rows % 8 || block_size % 8) return false;
  cuuint64_t dims[4] = {64, 8, 2, rows / 8};
  cuuint64_t strides[3] = {128, static_cast<cuuint64_t>(block_size) * 128, 1024};
  cuuint32_t box[4] = {64, 8, 2, block_size / 8};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
            const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_pair_pool_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t block_size, bool bf16) {
  return cached_map(m, MapKey{base, rows, block_size, 5, bf16 ? 2 : 1, 64}, [&](CUtensorMap* out) {
    return make_pair_pool_map_uncached(out, base, rows, block_size, bf16);
  });
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

}  // namespace
}  // namespace pkv
