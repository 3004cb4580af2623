// common.cuh -- shared device helpers of libpagedkv: element traits, mbarrier and
// bulk-copy (TMA) wrappers written as inline PTX for sm_103a, bounded waits.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "pagedkv.h"

namespace pkv {

// Device error flag bits (OR-ed into the flag a kernel is given).
enum : int {
  kErrIndex = 1,    // block id, slot or pair outside the pool
  kErrLength = 2,   // a context length above the host's max_context_len bound
  kErrTimeout = 4,  // a bounded wait ran out
};

// A bounded wait gives up after this long (nanoseconds of %globaltimer).  A healthy
// wait here lasts microseconds; the limit only ever ends a wait that cannot finish.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// ---------------------------------------------------------------------------------
// element traits: 16-byte vectors of the cache dtype to and from fp32

template <typename T>
struct Elem;

template <>
struct Elem<float> {
  static constexpr int kVec = 4;  // elements per 16 bytes
  __device__ static inline void load16(const void* p, float* out) {
    float4 x = *reinterpret_cast<const float4*>(p);
    out[0] = x.x; out[1] = x.y; out[2] = x.z; out[3] = x.w;
  }
  __device__ static inline float to_float(float x) { return x; }
  __device__ static inline float from_float(float x) { return x; }
};

template <>
struct Elem<__half> {
  static constexpr int kVec = 8;
  __device__ static inline void load16(const void* p, float* out) {
    uint4 x = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
      float2 f = __half22float2(h);
      out[2 * i] = f.x;
      out[2 * i + 1] = f.y;
    }
  }
  __device__ static inline float to_float(__half x) { return __half2float(x); }
  __device__ static inline __half from_float(float x) { return __float2half_rn(x); }
};

template <>
struct Elem<__nv_bfloat16> {
  static constexpr int kVec = 8;
  // bf16 is the high half of an fp32: widening is a shift / mask, exact.
  __device__ static inline void load16(const void* p, float* out) {
    uint4 x = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      out[2 * i] = __uint_as_float(w[i] << 16);
      out[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ static inline float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }
  __device__ static inline __nv_bfloat16 from_float(float x) { return __float2bfloat16_rn(x); }
};

// ---------------------------------------------------------------------------------
// PTX wrappers

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Programmatic dependent launch: a kernel launched with launch_dependent() may start
// before the previous kernel on the stream has finished; grid_dependency_wait() blocks
// until that kernel has completed and its memory operations are visible (a no-op for
// an ordinary launch).  grid_dependents_launch() lets the next such kernel start early.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dependents_launch() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// Raises a kernel's dynamic shared-memory limit on the current device.  The attribute
// belongs to each device, so it is set on the first launch on every device; `done`
// holds one bit per device index that has it (indices >= 64 set it every time).
template <typename Kernel>
cudaError_t ensure_smem_limit(Kernel kernel, int bytes, std::atomic<unsigned long long>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev >= 0 && dev < 64 ? 1ull << dev : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

template <typename Kernel, typename Args>
cudaError_t launch_dependent(Kernel kernel, int grid, int threads, int smem_bytes, cudaStream_t stream,
                             const Args& args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args);
}

// Non-blocking probe of the same condition (for a thread polling several barriers).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Two non-blocking probes issued back to back; bit i set when barrier i's phase has completed.
__device__ __forceinline__ uint32_t mbar_test_wait2(uint64_t* b0, uint32_t p0, uint64_t* b1, uint32_t p1) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred q0, q1;\n\t.reg .b32 t0, t1;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 q0, [%1], %2;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 q1, [%3], %4;\n\t"
      "selp.b32 t0, 1, 0, q0;\n\tselp.b32 t1, 2, 0, q1;\n\tor.b32 %0, t0, t1;\n\t}"
      : "=r"(r)
      : "r"(smem_addr(b0)), "r"(p0), "r"(smem_addr(b1)), "r"(p1)
      : "memory");
  return r;
}

// Five non-blocking probes issued back to back; bit i set when barrier i's phase has completed.
__device__ __forceinline__ uint32_t mbar_test_wait5(uint64_t* b0, uint32_t p0, uint64_t* b1, uint32_t p1,
                                                    uint64_t* b2, uint32_t p2, uint64_t* b3, uint32_t p3,
                                                    uint64_t* b4, uint32_t p4) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred q0, q1, q2, q3, q4;\n\t.reg .b32 t0, t1, t2, t3, t4;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 q0, [%1], %2;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 q1, [%3], %4;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 q2, [%5], %6;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 q3, [%7], %8;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 q4, [%9], %10;\n\t"
      "selp.b32 t0, 1, 0, q0;\n\tselp.b32 t1, 2, 0, q1;\n\tselp.b32 t2, 4, 0, q2;\n\tselp.b32 t3, 8, 0, q3;\n\t"
      "selp.b32 t4, 16, 0, q4;\n\t"
      "or.b32 t0, t0, t1;\n\tor.b32 t2, t2, t3;\n\tor.b32 t0, t0, t4;\n\tor.b32 %0, t0, t2;\n\t}"
      : "=r"(r)
      : "r"(smem_addr(b0)), "r"(p0), "r"(smem_addr(b1)), "r"(p1), "r"(smem_addr(b2)), "r"(p2),
        "r"(smem_addr(b3)), "r"(p3), "r"(smem_addr(b4)), "r"(p4)
      : "memory");
  return r;
}

// Four non-blocking probes issued back to back (their latencies overlap); bit i of the
// result is set when barrier i's phase `parity_i` has completed.
__device__ __forceinline__ uint32_t mbar_test_wait4(uint64_t* b0, uint32_t p0, uint64_t* b1, uint32_t p1,
                                                    uint64_t* b2, uint32_t p2, uint64_t* b3, uint32_t p3) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred q0, q1, q2, q3;\n\t.reg .b32 t0, t1, t2, t3;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 q0, [%1], %2;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 q1, [%3], %4;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 q2, [%5], %6;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 q3, [%7], %8;\n\t"
      "selp.b32 t0, 1, 0, q0;\n\tselp.b32 t1, 2, 0, q1;\n\tselp.b32 t2, 4, 0, q2;\n\tselp.b32 t3, 8, 0, q3;\n\t"
      "or.b32 t0, t0, t1;\n\tor.b32 t2, t2, t3;\n\tor.b32 %0, t0, t2;\n\t}"
      : "=r"(r)
      : "r"(smem_addr(b0)), "r"(p0), "r"(smem_addr(b1)), "r"(p1), "r"(smem_addr(b2)), "r"(p2),
        "r"(smem_addr(b3)), "r"(p3)
      : "memory");
  return r;
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Below this limit a wait polls with the non-blocking probe and reads the clock every
// round: mbarrier.try_wait may suspend the thread for longer than such a limit, so a
// wait could otherwise never notice that it ran out.
constexpr uint64_t kPollBelowNs = 1000000ull;

// Wait for the phase of `bar` with the given parity to complete; false if the wait
// ran past limit_ns.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (limit_ns < kPollBelowNs) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_test_wait(bar, parity))
      if (global_timer_ns() - t0 > limit_ns) return false;
    return true;
  }
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

// 1-D bulk copy global -> shared (TMA engine), completion counted in bytes on `bar`.
// dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Same, with an L2 eviction-priority policy (created by createpolicy).
__device__ __forceinline__ void bulk_load_hint(void* dst, const void* src, uint32_t bytes,
                                               uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], "
      "%2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void set_error(int* flag, int bits) {
  if (flag) atomicOr(flag, bits);
}

template <int N>
__device__ __forceinline__ float group_sum(float x) {
  // butterfly sum across aligned groups of N lanes (N a power of two <= 32)
#pragma unroll
  for (int off = N / 2; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

// Sums each of N values over aligned groups of LANES lanes (N <= LANES, both powers of
// two) and leaves all N totals in every lane of the group: a reduce-scatter (each step
// a lane keeps half of its values and adds its partner's copy of that half), a
// butterfly over the remaining lane bits, then each total fetched from a lane that
// holds it.  N - 1 + log2(LANES / N) + N shuffles instead of N log2(LANES).
template <int N, int LANES>
__device__ __forceinline__ void group_sum_all(float (&v)[N]) {
  static_assert(N <= LANES && LANES <= 32, "at most one value per lane of the group");
  if (N == 1) {
    v[0] = group_sum<LANES>(v[0]);
    return;
  }
  const int lane = threadIdx.x & 31;
  float a[N];
#pragma unroll
  for (int i = 0; i < N; ++i) a[i] = v[i];
  int off = LANES / 2;
#pragma unroll
  for (int n = N; n > 1; n >>= 1, off >>= 1) {
    const bool upper = lane & off;
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
  // the lane of the group holding total j: j's binary digits, most significant first,
  // on the lane bits LANES/2, LANES/4, ... (a compile-time index within the group)
#pragma unroll
  for (int j = 0; j < N; ++j) {
    int src = 0;
#pragma unroll
    for (int b = N / 2, o = LANES / 2; b > 0; b >>= 1, o >>= 1) src += (j & b) ? o : 0;
    v[j] = __shfl_sync(0xffffffffu, r, src, LANES);
  }
}

}  // namespace pkv
