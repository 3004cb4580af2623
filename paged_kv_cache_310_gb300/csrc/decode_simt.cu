// decode_simt.cu -- CUDA-core paged decode attention with split-K partitions, and
// the partition merge.
//
// What it computes (note-023, Method/Concepts; "Paged Attention" glossary, paragraph 4
// and GQA paragraph): for sequence s, KV head g and each query head h of g's group,
// softmax(scale * q_h . K_j) weighted sum of V_j over the sequence's tokens, where
// token j lives in row j % bs of physical block block_tables[s][j / bs].
//
// Work decomposition: one CTA per (partition, kv head, sequence).  A partition is
// part_tokens consecutive logical tokens.  The CTA serves every query head of its KV
// head, so each K/V byte is read from HBM once per group (GQA reuse).
//
// Inside a CTA:
//  * warp 4 is the producer: it stages the partition's block ids in shared memory,
//    then one lane streams the partition through a 3- or 4-stage ring.  A stage holds
//    32 tokens: one 1-D bulk copy (TMA engine, cp.async.bulk) per (block, kv head) tile
//    for K and one for V (each tile is block_size*head_dim contiguous elements; a
//    64-token block spans two stages and is copied half per stage).  Completion is
//    counted in bytes on the stage's "full" mbarrier.
//  * warps 0-3 consume.  A row of head_dim elements is spread over head_dim/vec lanes
//    (16-byte vectors), so a warp covers 32/(lanes per row) rows at once; each such
//    lane group ("slot") owns the rows r == slot (mod slots) of every stage and keeps
//    its own running max / sum / output per query head (online softmax, exp2 domain).
//    A row's G dot products are all-reduced over its lanes together (warp shuffles);
//    after a stage the warp arrives on the stage's "empty" mbarrier so the producer
//    can refill it.
//  * at the end the slots are combined through shared memory in a fixed order, so
//    the result depends only on logical token positions (bit-identical under any
//    placement of the physical blocks).
//  A sequence that fits one partition writes `out` directly; otherwise each partition
//  writes (max, sum, un-normalised output) to the workspace and merge_kernel
//  combines them: M = max_p m_p, out = sum_p 2^(m_p-M) o_p / sum_p 2^(m_p-M) l_p.
#include <climits>

#include "common.cuh"
#include "launch.h"

namespace pkv {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;

template <typename T, int D, int GM>
struct Simt {
  static constexpr int kVec = Elem<T>::kVec;           // elements per 16-byte vector
  static constexpr int kLanesPerRow = D / kVec;        // lanes covering one token row
  static constexpr int kRowsPerWarp = 32 / kLanesPerRow;
  static constexpr int kSlots = kConsumerWarps * kRowsPerWarp;
  static constexpr int kRowBytes = D * static_cast<int>(sizeof(T));
  static constexpr int kChunk = 32;                    // tokens per pipeline stage
  static constexpr int kRowsPerSlot = kChunk / kSlots;  // rows a slot handles per stage
  static constexpr int kStageBytes = 2 * kChunk * kRowBytes;  // K rows then V rows
  // Four stages, or three of 32 KB (f32, head_dim 128): a 128 KB ring left room for one
  // CTA per SM, whose prologue and tail then idled the SM (0.74 of copy bandwidth on a
  // 64 x 32-head batch; 1.04 with two CTAs of three stages).
  static constexpr int kStages = kStageBytes >= 32768 ? 3 : 4;
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kReduceBytes = kSlots * GM * (D + 2) * 4;
  static constexpr int kMainBytes =
      ((kRingBytes > kReduceBytes ? kRingBytes : kReduceBytes) + 127) / 128 * 128;
  static constexpr int kBarrierBytes = 2 * kStages * 8 + 16;  // full, empty, 4 ints of flags
  static_assert(kChunk % kSlots == 0, "slots must tile a stage");
  static_assert(kLanesPerRow <= 32 && 32 % kLanesPerRow == 0, "row must fit a warp");

  static size_t smem_bytes(int part_tokens, int block_size) {
    return kMainBytes + kBarrierBytes + static_cast<size_t>(part_tokens / block_size) * 4;
  }
};

template <typename T>
__device__ __forceinline__ void store_out(void* out, size_t i, float x, int out_f32) {
  if (out_f32)
    static_cast<float*>(out)[i] = x;
  else
    static_cast<T*>(out)[i] = Elem<T>::from_float(x);
}

template <typename T, int D, int GM>
__global__ void __launch_bounds__(kThreads)
decode_simt_kernel(const __grid_constant__ DecodeParams p) {
  using C = Simt<T, D, GM>;
  using E = Elem<T>;
  extern __shared__ __align__(1024) unsigned char smem[];

  const int part = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int G = p.group;
  // with partitions the next kernel is this call's merge, which waits for this grid
  // before it reads anything: let it launch once every CTA here has started
  if (p.max_parts > 1) grid_dependents_launch();
  const int L = p.context_lens[s];
  if (L < 0 || L > p.max_parts * p.part_tokens) {
    if (part == 0 && threadIdx.x == 0) set_error(p.err, kErrLength);
    return;
  }
  if (L == 0) {  // empty context: the neutral output
    if (part == 0)
      for (int i = threadIdx.x; i < G * D; i += kThreads)
        store_out<T>(p.out, (static_cast<size_t>(s) * p.num_q_heads + g * G) * D + i, 0.f, p.out_f32);
    return;
  }
  const int t0 = part * p.part_tokens;
  if (t0 >= L) return;
  const int ntok = min(p.part_tokens, L - t0);
  const int nchunks = (ntok + C::kChunk - 1) / C::kChunk;
  const int nparts = (L + p.part_tokens - 1) / p.part_tokens;

  unsigned char* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kMainBytes);
  uint64_t* empty = full + C::kStages;
  int* flags = reinterpret_cast<int*>(empty + C::kStages);  // [0] first aborted chunk, [1] issued
  int* ids = flags + 4;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    flags[0] = INT_MAX;
    flags[1] = 0;
    fence_barrier_init();
  }
  __syncthreads();

  // per-slot online-softmax state (consumers only)
  float m[GM], l[GM], o[GM][C::kVec];
  const int sub = lane / C::kLanesPerRow, li = lane % C::kLanesPerRow;
  const int slot = warp * C::kRowsPerWarp + sub;

  if (warp == kConsumerWarps) {
    // ---------------- producer ----------------
    const int bs = p.block_size;
    const int first = t0 / bs;
    const int nblk = (ntok + bs - 1) / bs;
    const int32_t* row = p.block_tables + static_cast<size_t>(s) * p.max_blocks_per_seq;
    for (int i = lane; i < nblk; i += 32) {
      int b = first + i < p.max_blocks_per_seq ? row[first + i] : -1;
      if (b < 0 || b >= p.num_blocks) {
        set_error(p.err, kErrIndex);
        b = 0;  // keep the copy in bounds; the flag reports the bad table
      }
      ids[i] = b;
    }
    __syncwarp();
    if (lane == 0) {
      const size_t tile_elems = static_cast<size_t>(bs) * D;
      const size_t block_stride = static_cast<size_t>(p.num_kv_heads) * tile_elems;
      // one bulk copy per block of a stage, or per stage-sized piece of a block when a
      // block (64 tokens) spans several stages: its rows are contiguous either way
      const int copy_rows = bs < C::kChunk ? bs : C::kChunk;
      const uint32_t copy_bytes = static_cast<uint32_t>(copy_rows) * C::kRowBytes;
      const uint64_t policy = policy_evict_first();  // K/V are streamed once
      int issued = 0;
      for (int c = 0; c < nchunks; ++c) {
        const int st = c % C::kStages;
        if (c >= C::kStages && !mbar_wait(&empty[st], ((c / C::kStages) - 1) & 1, p.wait_limit_ns)) {
          set_error(p.err, kErrTimeout);
          atomicMin(&flags[0], c);
          break;
        }
        if (*reinterpret_cast<volatile int*>(&flags[0]) != INT_MAX) break;
        const int rows = min(C::kChunk, ntok - c * C::kChunk);
        const int ncopies = (rows + copy_rows - 1) / copy_rows;
        unsigned char* kdst = ring + st * C::kStageBytes;
        unsigned char* vdst = kdst + C::kChunk * C::kRowBytes;
        mbar_arrive_expect_tx(&full[st], 2u * ncopies * copy_bytes);
        for (int i = 0; i < ncopies; ++i) {
          const int tok = c * C::kChunk + i * copy_rows;  // first token of the piece, partition-relative
          const size_t off = ids[tok / bs] * block_stride + g * tile_elems + static_cast<size_t>(tok % bs) * D;
          bulk_load_hint(kdst + i * copy_bytes, static_cast<const T*>(p.k_cache) + off, copy_bytes,
                         &full[st], policy);
          bulk_load_hint(vdst + i * copy_bytes, static_cast<const T*>(p.v_cache) + off, copy_bytes,
                         &full[st], policy);
        }
        issued = c + 1;
      }
      flags[1] = issued;
    }
  } else {
    // ---------------- consumers ----------------
    float qf[GM][C::kVec];
#pragma unroll
    for (int h = 0; h < GM; ++h) {
      if (h < G) {
        const T* qp = static_cast<const T*>(p.q) +
                      (static_cast<size_t>(s) * p.num_q_heads + g * G + h) * D + li * C::kVec;
        E::load16(qp, qf[h]);
#pragma unroll
        for (int e = 0; e < C::kVec; ++e) qf[h][e] *= p.scale_log2;
      } else {
#pragma unroll
        for (int e = 0; e < C::kVec; ++e) qf[h][e] = 0.f;
      }
      m[h] = -INFINITY;
      l[h] = 0.f;
#pragma unroll
      for (int e = 0; e < C::kVec; ++e) o[h][e] = 0.f;
    }

    for (int c = 0; c < nchunks; ++c) {
      const int st = c % C::kStages;
      // warp-uniform: every lane must take the same branch before the shuffles below
      if (!__all_sync(0xffffffffu, mbar_wait(&full[st], (c / C::kStages) & 1, p.wait_limit_ns))) {
        if (lane == 0) {
          set_error(p.err, kErrTimeout);
          atomicMin(&flags[0], c);
        }
        break;
      }
      const unsigned char* ks = ring + st * C::kStageBytes;
      const unsigned char* vs = ks + C::kChunk * C::kRowBytes;
      const int rows = min(C::kChunk, ntok - c * C::kChunk);

      float sc[C::kRowsPerSlot][GM];
#pragma unroll
      for (int i = 0; i < C::kRowsPerSlot; ++i) {
        const int r = slot + i * C::kSlots;
        const bool valid = r < rows;
        float kf[C::kVec];
        if (valid) {
          E::load16(ks + r * C::kRowBytes + li * 16, kf);
        } else {
#pragma unroll
          for (int e = 0; e < C::kVec; ++e) kf[e] = 0.f;
        }
        float d[GM];
#pragma unroll
        for (int h = 0; h < GM; ++h) {
          float2 d2 = make_float2(0.f, 0.f);  // even and odd elements: two short chains
#pragma unroll
          for (int e = 0; e < C::kVec; e += 2)
            d2 = __ffma2_rn(make_float2(qf[h][e], qf[h][e + 1]), make_float2(kf[e], kf[e + 1]), d2);
          d[h] = d2.x + d2.y;
        }
        // the GM dot products over the row's lanes at once (fewer shuffles than one by one)
        group_sum_all<GM, C::kLanesPerRow>(d);
#pragma unroll
        for (int h = 0; h < GM; ++h) sc[i][h] = valid ? d[h] : -INFINITY;
      }
#pragma unroll
      for (int h = 0; h < GM; ++h) {
        float cm = sc[0][h];
#pragma unroll
        for (int i = 1; i < C::kRowsPerSlot; ++i) cm = fmaxf(cm, sc[i][h]);
        if (cm > m[h]) {  // new running max: rescale what was accumulated so far
          const float a = exp2f(m[h] - cm);
          l[h] *= a;
#pragma unroll
          for (int e = 0; e < C::kVec; ++e) o[h][e] *= a;
          m[h] = cm;
        }
      }
#pragma unroll
      for (int i = 0; i < C::kRowsPerSlot; ++i) {
        const int r = slot + i * C::kSlots;
        if (r < rows) {
          float vf[C::kVec];
          E::load16(vs + r * C::kRowBytes + li * 16, vf);
#pragma unroll
          for (int h = 0; h < GM; ++h) {
            const float w = exp2f(sc[i][h] - m[h]);
            l[h] += w;
#pragma unroll
            for (int e = 0; e < C::kVec; e += 2) {
              const float2 acc = __ffma2_rn(make_float2(w, w), make_float2(vf[e], vf[e + 1]),
                                            make_float2(o[h][e], o[h][e + 1]));
              o[h][e] = acc.x;
              o[h][e + 1] = acc.y;
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
  }

  __syncthreads();
  if (flags[0] != INT_MAX) {
    // A wait ran out: wait (bounded) for the copies still in flight, then leave.
    if (threadIdx.x == kConsumerWarps * 32) {
      for (int c = flags[0]; c < flags[1]; ++c)
        if (!mbar_wait(&full[c % C::kStages], (c / C::kStages) & 1)) break;
    }
    __syncthreads();
    return;
  }

  // ---------------- combine the slots (fixed order) ----------------
  float* red_m = reinterpret_cast<float*>(smem);  // [slots][GM]
  float* red_l = red_m + C::kSlots * GM;          // [slots][GM]
  float* red_o = red_l + C::kSlots * GM;          // [slots][GM][D]
  if (warp < kConsumerWarps) {
#pragma unroll
    for (int h = 0; h < GM; ++h) {
      if (li == 0) {
        red_m[slot * GM + h] = m[h];
        red_l[slot * GM + h] = l[h];
      }
      float* dst = red_o + (slot * GM + h) * D + li * C::kVec;
#pragma unroll
      for (int e = 0; e < C::kVec; e += 4)
        *reinterpret_cast<float4*>(dst + e) = make_float4(o[h][e], o[h][e + 1], o[h][e + 2], o[h][e + 3]);
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < G * D; i += kThreads) {
    const int h = i / D, d = i % D;
    float M = -INFINITY;
    for (int sl = 0; sl < C::kSlots; ++sl) M = fmaxf(M, red_m[sl * GM + h]);
    float lsum = 0.f, acc = 0.f;
    for (int sl = 0; sl < C::kSlots; ++sl) {
      const float ms = red_m[sl * GM + h];
      if (ms == -INFINITY) continue;  // slot saw no token of this partition
      const float cf = exp2f(ms - M);
      lsum = fmaf(cf, red_l[sl * GM + h], lsum);
      acc = fmaf(cf, red_o[(sl * GM + h) * D + d], acc);
    }
    const size_t row = static_cast<size_t>(s) * p.num_q_heads + g * G + h;
    if (nparts == 1) {
      store_out<T>(p.out, row * D + d, acc / lsum, p.out_f32);
    } else {
      const size_t k = row * p.max_parts + part;
      p.ws_o[k * D + d] = acc;
      if (d == 0) {
        p.ws_ml[2 * k] = M;
        p.ws_ml[2 * k + 1] = lsum;
      }
    }
  }
}

// One CTA per (query head, sequence), launched as a programmatic dependent of the
// partition kernel: it may be resident while that kernel runs and waits for it here.
template <typename T>
__global__ void __launch_bounds__(128) merge_kernel(const __grid_constant__ DecodeParams p) {
  grid_dependency_wait();
  const int h = blockIdx.x % p.num_q_heads, s = blockIdx.x / p.num_q_heads;
  const int L = p.context_lens[s];
  if (L < 0 || L > p.max_parts * p.part_tokens) return;
  const int np = (L + p.part_tokens - 1) / p.part_tokens;
  if (np <= 1) return;
  const size_t row = static_cast<size_t>(s) * p.num_q_heads + h;
  const float* ml = p.ws_ml + row * p.max_parts * 2;
  float M = -INFINITY;
  for (int i = 0; i < np; ++i) M = fmaxf(M, ml[2 * i]);
  const int D = p.head_dim;
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float lsum = 0.f, acc = 0.f;
    for (int i = 0; i < np; ++i) {
      const float cf = exp2f(ml[2 * i] - M);
      lsum = fmaf(cf, ml[2 * i + 1], lsum);
      acc = fmaf(cf, p.ws_o[(row * p.max_parts + i) * D + d], acc);
    }
    store_out<T>(p.out, row * D + d, acc / lsum, p.out_f32);
  }
}

template <typename T, int D, int GM>
cudaError_t launch_simt_t(const DecodeParams& p, cudaStream_t stream) {
  using C = Simt<T, D, GM>;
  const size_t smem = C::smem_bytes(p.part_tokens, p.block_size);
  static std::atomic<unsigned long long> configured{0};  // devices whose limit is raised
  cudaError_t e = ensure_smem_limit(decode_simt_kernel<T, D, GM>, 200 * 1024, configured);
  if (e != cudaSuccess) return e;
  dim3 grid(p.max_parts, p.num_kv_heads, p.num_seqs);
  decode_simt_kernel<T, D, GM><<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_simt_g(const DecodeParams& p, cudaStream_t stream) {
  if (p.group <= 1) return launch_simt_t<T, D, 1>(p, stream);
  if (p.group <= 2) return launch_simt_t<T, D, 2>(p, stream);
  if (p.group <= 4) return launch_simt_t<T, D, 4>(p, stream);
  return launch_simt_t<T, D, 8>(p, stream);
}

template <typename T>
cudaError_t launch_simt_d(const DecodeParams& p, cudaStream_t stream) {
  return p.head_dim == 64 ? launch_simt_g<T, 64>(p, stream) : launch_simt_g<T, 128>(p, stream);
}

}  // namespace

cudaError_t launch_decode_simt(const DecodeParams& p, int dtype, cudaStream_t stream) {
  switch (dtype) {
    case PKV_F32: return launch_simt_d<float>(p, stream);
    case PKV_F16: return launch_simt_d<__half>(p, stream);
    default: return launch_simt_d<__nv_bfloat16>(p, stream);
  }
}

cudaError_t launch_merge(const DecodeParams& p, int dtype, cudaStream_t stream) {
  if (p.max_parts <= 1) return cudaSuccess;
  const int grid = p.num_q_heads * p.num_seqs;  // (query head, sequence), head fastest
  switch (dtype) {
    case PKV_F32: return launch_dependent(merge_kernel<float>, grid, 128, 0, stream, p);
    case PKV_F16: return launch_dependent(merge_kernel<__half>, grid, 128, 0, stream, p);
    default: return launch_dependent(merge_kernel<__nv_bfloat16>, grid, 128, 0, stream, p);
  }
}

}  // namespace pkv
