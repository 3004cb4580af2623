// prefill_tc.cu -- multi-token paged attention with a causal mask (prefill and
// chunked prefill) on the tcgen05 tensor cores; f16/bf16, head_dim 128, up to 16
// query heads per KV head.
//
// What it computes ("anthology-of-the-sota note-023", Method: attention gathers K/V
// through the block table; the same arithmetic as attention over contiguous memory):
// sequence s brings n_s new tokens, the last n_s of its context_lens[s] tokens (their
// K/V already appended to the pool).  New token i sits at position
// p = context_lens[s] - n_s + i and attends to positions 0..p through the block table.
// One new token per sequence is exactly paged decode.
//
// Work item = (sequence, KV head, query tile).  A tile is 128 query rows: TQ =
// floor(128 / G) consecutive new tokens times the G query heads of the KV head, row
// r = token * G + head (rows past TQ * G are padding).  Per 64-key chunk:
//   S[128 rows x 64 keys] = Q . K^T            (M=128, N=64,  K=128 dims)
//   O[128 rows x 128 dims] = P . V             (M=128, N=128, K=64 keys), twice:
// the probabilities as hi = round(p) and lo = round(p - hi) in the cache dtype, so
// the 16-bit operand costs about 2^-17 relative per weight.  S (double-buffered) and
// O live in TMEM; the MMA accumulates O over the tile's chunks.  Softmax is row-local
// (no cross-thread reduction) with a lazy rescale: a row keeps the maximum it used
// for its probabilities until a chunk brings a score more than 8 (log2 units) above
// it -- probabilities stay <= 256 -- and only then is its O row rescaled in TMEM.
// O is double-buffered by tile and read out once, at the tile's end.
//
// Roles (192 threads, persistent CTAs over a longest-first work list dealt in snake
// order):
//  * warp 4, producer: loads the tile's 128 query rows (plain loads, written in the
//    128-byte swizzled operand layout), then per chunk one 4-D TMA box per block for
//    K and one for V into a 3-stage ring (blocks past the tile's last position are
//    loaded from outside the tensor: zero fill).
//  * warp 5, MMA: one lane polls and issues QK(c) once K/V and Q are in and an S
//    buffer is free, PV(c) once P(c) (and any rescale of O) is written.
//  * warps 0-3: thread t owns query row t.
#include <climits>
#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "tc_util.cuh"
#include "tcgen05.cuh"

namespace pkv {
namespace {

constexpr int kThreads = 192;
constexpr int kRows = 128;                 // query rows per tile (M)
constexpr int kKC = 64;                    // keys per chunk
constexpr int kStages = 3;
constexpr int kGroup = 2048;               // 8-row group of a 128-dim tile: two 64-column halves
constexpr int kKVTile = kKC * 256;         // K (or V) of one chunk: 16 KB
constexpr int kStageBytes = 2 * kKVTile;   // K then V
constexpr int kQBytes = kRows * 256;       // 32 KB: [16 groups][2 halves][8 rows][128 B]
constexpr int kPPart = kRows * kKC * 2;    // 16 KB: [16 groups][8 rows][128 B], one part
constexpr int kPBytes = 2 * kPPart;        // hi part then lo part
constexpr int kOffQ = kStages * kStageBytes;
constexpr int kOffP = kOffQ + 2 * kQBytes;
constexpr int kOffBar = kOffP + 2 * kPBytes;
constexpr int kNumBars = 2 * kStages + 7 * 2 + 1;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 64;
constexpr uint32_t kTmemCols = 512;        // S[2] at 0/64 (64 columns), O[2] at 128/256 (128 columns)
constexpr float kRescaleSlack = 8.f;       // log2 units a row's max may grow before O is rescaled
constexpr int kListThreads = 1024;
constexpr int kMaxBuckets = 1024;          // chunk-count buckets of the work list (last one open-ended)

struct Bars {
  uint64_t *full, *empty, *qfull, *qempty, *sfull, *sfree, *pfull, *ofull, *ofree, *drain;
};

__device__ __forceinline__ Bars carve(unsigned char* smem) {
  uint64_t* b = reinterpret_cast<uint64_t*>(smem + kOffBar);
  Bars r;
  r.full = b;
  r.empty = b + kStages;
  r.qfull = b + 2 * kStages;
  r.qempty = r.qfull + 2;
  r.sfull = r.qempty + 2;
  r.sfree = r.sfull + 2;
  r.pfull = r.sfree + 2;
  r.ofull = r.pfull + 2;
  r.ofree = r.ofull + 2;
  r.drain = r.ofree + 2;
  return r;
}

struct PrefillArgs {
  CUtensorMap tk;  // pool 4-D views: one box = one block's tile for one KV head
  CUtensorMap tv;
  PrefillParams p;
};

// {s, g | ntile << 16, first query row, position of the tile's first token}
struct Tile {
  int s, g, ntile, qrow0, pos0, nchunks;
};

__device__ __forceinline__ Tile unpack_tile(int4 e) {
  Tile t;
  t.s = e.x;
  t.g = e.y & 0xffff;
  t.ntile = static_cast<int>(static_cast<unsigned>(e.y) >> 16);
  t.qrow0 = e.z;
  t.pos0 = e.w;
  t.nchunks = (t.pos0 + t.ntile + kKC - 1) / kKC;
  return t;
}

// byte offset of 16-byte piece `c16` (0..15 over 128 dims) of row r in a
// [group][half][8 rows][128 B] tile with 128-byte swizzle
__device__ __forceinline__ int swz_dims(int r, int c16) {
  return (r >> 3) * kGroup + (c16 >> 3) * 1024 + (r & 7) * 128 + (((c16 & 7) ^ (r & 7)) << 4);
}
// same for a [group][8 rows][128 B] tile of 64 keys (one half)
__device__ __forceinline__ int swz_keys(int r, int c16) {
  return (r >> 3) * 1024 + (r & 7) * 128 + (((c16 & 7) ^ (r & 7)) << 4);
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(const __grid_constant__ PrefillArgs a) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const PrefillParams& p = a.p;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const Bars bars = carve(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  int* issued_slot = reinterpret_cast<int*>(smem + kOffMisc + 8);
  int* waited_slot = reinterpret_cast<int*>(smem + kOffMisc + 12);
  const int G = p.group;
  const int num_items = *p.work_count;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bars.full[i], 1);
      mbar_init(&bars.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.qfull[i], 1);
      mbar_init(&bars.qempty[i], 1);
      mbar_init(&bars.sfull[i], 1);
      mbar_init(&bars.sfree[i], 4);
      mbar_init(&bars.pfull[i], 4);
      mbar_init(&bars.ofull[i], 1);
      mbar_init(&bars.ofree[i], 4);
    }
    *abort_flag = 0;
    *issued_slot = 0;
    *waited_slot = 0;
    fence_barrier_init();
  }
  if (warp == 5) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ============================ producer ============================
    if (lane == 0) {
      prefetch_tensormap(&a.tk);
      prefetch_tensormap(&a.tv);
    }
    const uint64_t pol_stream = policy_evict_first();
    const int bs = p.block_size;
    const int blocks_per_chunk = kKC / bs;
    const int oob_group = p.num_blocks * p.num_kv_heads * bs / 8;  // first row group outside the pool
    int c = 0, j = 0;
    bool ok = true;
    ItemCursor cur;
    for (cur.init(p.work_list, num_items); cur.valid() && ok; cur.advance()) {
      const Tile it = unpack_tile(cur.cur);
      const int qb = j & 1;
      // ---- the tile's query rows, swizzled, zero past the tile ----
      ok = j < 2 || __shfl_sync(0xffffffffu, lane == 0 ? wait_role(&bars.qempty[qb], ((j >> 1) - 1) & 1,
                                                                   abort_flag, p.err)
                                                       : true, 0);
      if (!ok) break;
      unsigned char* qbuf = smem + kOffQ + qb * kQBytes;
      const int valid_rows = it.ntile * G;
#pragma unroll 1
      for (int r = lane; r < kRows; r += 32) {
        const bool valid = r < valid_rows;
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const T*>(p.q) +
            (static_cast<size_t>(it.qrow0 + r / G) * p.num_q_heads + it.g * G + r % G) * 128);
#pragma unroll
        for (int c16 = 0; c16 < 16; ++c16) {
          const uint4 v = valid ? src[c16] : make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(qbuf + swz_dims(r, c16)) = v;
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.qfull[qb]);
      // ---- K/V chunks ----
      const int pos_last = it.pos0 + it.ntile - 1;
      const int32_t* table = p.block_tables + static_cast<size_t>(it.s) * p.max_blocks_per_seq;
      for (int k = 0; k < it.nchunks && ok; ++k, ++c) {
        const int st = c % kStages;
        const int lb = k * blocks_per_chunk + lane;  // logical block of this lane
        const bool live = lane < blocks_per_chunk && lb * bs <= pos_last;
        int b = live ? (lb < p.max_blocks_per_seq ? table[lb] : -1) : 0;
        if (lane == 0) {
          ok = c < kStages || wait_role(&bars.empty[st], ((c / kStages) - 1) & 1, abort_flag, p.err);
          if (ok) mbar_arrive_expect_tx(&bars.full[st], kStageBytes);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        __syncwarp();
        if (lane < blocks_per_chunk) {
          int grp = oob_group;
          if (live) {
            if (b < 0 || b >= p.num_blocks) {
              set_error(p.err, kErrIndex);
              b = 0;
            }
            grp = (b * p.num_kv_heads + it.g) * bs / 8;
          }
          unsigned char* dst = smem + st * kStageBytes + lane * bs * 256;
          tma_load_4d(dst, &a.tk, grp, &bars.full[st], pol_stream);
          tma_load_4d(dst + kKVTile, &a.tv, grp, &bars.full[st], pol_stream);
        }
        if (lane == 0) *issued_slot = c + 1;
      }
      ++j;
    }
  } else if (warp == 5) {
    // ============================ MMA issuer ============================
    if (lane == 0) {
      constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
      constexpr uint32_t idesc_qk = instr_desc_f16(kBf16, false, false, kRows, kKC);
      constexpr uint32_t idesc_pv = instr_desc_f16(kBf16, false, true, kRows, 128);
      const uint32_t ring = smem_addr(smem);
      const uint32_t qbase = smem_addr(smem + kOffQ);
      const uint32_t pbase = smem_addr(smem + kOffP);
      ItemCursor qcur;
      qcur.init(p.work_list, num_items);
      int qk = 0, qj = 0;
      int qn = qcur.valid() ? unpack_tile(qcur.cur).nchunks : 0;
      // PV cursor: tile index (selects the O buffer), chunk within the tile
      ItemCursor pcur;
      pcur.init(p.work_list, num_items);
      int pk = 0, pj = 0;
      int pn = pcur.valid() ? unpack_tile(pcur.cur).nchunks : 0;
      int qc = 0, pc = 0;
      uint64_t idle_since = global_timer_ns();
      while (qcur.valid() || pc < qc) {
        bool progressed = false;
        if (qcur.valid()) {
          const int st = qc % kStages, sb = qc & 1, qb = qj & 1;
          if ((qk > 0 || mbar_try_wait(&bars.qfull[qb], (qj >> 1) & 1)) &&
              mbar_try_wait(&bars.full[st], (qc / kStages) & 1) &&
              (qc < 2 || mbar_try_wait(&bars.sfree[sb], ((qc >> 1) - 1) & 1))) {
            *waited_slot = qc + 1;
            tc_fence_after();
            const uint32_t kb = ring + st * kStageBytes;
            const uint32_t qa = qbase + qb * kQBytes;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t off = (kk >> 2) * 1024 + (kk & 3) * 32;
              mma_f16(tmem + sb * 64, smem_desc(qa + off, 16, kGroup, kLayoutSwizzle128),
                      smem_desc(kb + off, 16, kGroup, kLayoutSwizzle128), idesc_qk, kk > 0);
            }
            mma_commit(&bars.sfull[sb]);
            ++qc;
            if (++qk == qn) {  // the tile's last QK: its query buffer can be refilled
              mma_commit(&bars.qempty[qb]);
              qk = 0;
              ++qj;
              qcur.advance();
              qn = qcur.valid() ? unpack_tile(qcur.cur).nchunks : 0;
            }
            progressed = true;
          }
        }
        if (pc < qc) {
          const int pb = pc & 1, st = pc % kStages;
          if (mbar_try_wait(&bars.pfull[pb], (pc >> 1) & 1)) {
            tc_fence_after();
            const uint32_t vbase = ring + st * kStageBytes + kKVTile;
            const uint32_t pa = pbase + pb * kPBytes;
            const uint32_t od = tmem + 128 + (pj & 1) * 128;  // this tile's O buffer
#pragma unroll
            for (int kk = 0; kk < kKC / 16; ++kk) {
              const uint64_t bd = smem_desc(vbase + kk * 2 * kGroup, 1024, kGroup, kLayoutSwizzle128);
              mma_f16(od, smem_desc(pa + kk * 32, 16, 1024, kLayoutSwizzle128), bd, idesc_pv, pk > 0 || kk > 0);
              mma_f16(od, smem_desc(pa + kPPart + kk * 32, 16, 1024, kLayoutSwizzle128), bd, idesc_pv, true);
            }
            mma_commit(&bars.ofull[pb]);
            mma_commit(&bars.empty[st]);
            ++pc;
            if (++pk == pn) {
              pk = 0;
              ++pj;
              pcur.advance();
              pn = pcur.valid() ? unpack_tile(pcur.cur).nchunks : 0;
            }
            progressed = true;
          }
        }
        if (progressed) {
          idle_since = global_timer_ns();
        } else {
          if (*abort_flag) break;
          if (global_timer_ns() - idle_since > kWaitLimitNs) {
            *abort_flag = 1;
            set_error(p.err, kErrTimeout);
            break;
          }
        }
      }
    }
    __syncwarp();
  } else {
    // ============================ softmax warps ============================
    const int t = threadIdx.x;  // query row of the tile = TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    int c = 0, j = 0;
    bool ok = true;
    // the previous tile, read out once this tile's first chunk is under way
    int prev_row = -1, prev_c = -1;
    float prev_l = 1.f;

    // Warp-uniform: has PV of chunk cc completed?  Waited in chunk order per barrier.
    auto pv_done = [&](int cc) -> bool {
      return __all_sync(0xffffffffu, wait_role(&bars.ofull[cc & 1], (cc >> 1) & 1, abort_flag, p.err));
    };
    // The finished tile's output rows: O / l, once the tile's last PV has completed.
    auto finish = [&](int row, int last_c, float lsum, int buf) -> bool {
      if (!pv_done(last_c)) return false;
      tc_fence_after();
      const float inv = 1.f / lsum;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float o[16];
        tmem_load16(lane_base + 128 + buf * 128 + q * 16, o);
        if (row >= 0) {
          if (p.out_f32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + static_cast<size_t>(row) * 128 + q * 16);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv, o[4 * i + 3] * inv);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(p.out) + static_cast<size_t>(row) * 128 + q * 16);
#pragma unroll
            for (int i = 0; i < 2; ++i)
              dst[i] = make_uint4(pack2<T>(o[8 * i] * inv, o[8 * i + 1] * inv),
                                  pack2<T>(o[8 * i + 2] * inv, o[8 * i + 3] * inv),
                                  pack2<T>(o[8 * i + 4] * inv, o[8 * i + 5] * inv),
                                  pack2<T>(o[8 * i + 6] * inv, o[8 * i + 7] * inv));
          }
        }
      }
      tc_fence_before();
      return true;
    };

    ItemCursor cur;
    for (cur.init(p.work_list, num_items); cur.valid() && ok; cur.advance(), ++j) {
      const Tile it = unpack_tile(cur.cur);
      const int valid_rows = it.ntile * G;
      const bool row_valid = t < valid_rows;
      const int pos_last = it.pos0 + it.ntile - 1;
      const int qpos = row_valid ? it.pos0 + t / G : pos_last;  // padding rows act as the last token
      const int out_row = row_valid ? (it.qrow0 + t / G) * p.num_q_heads + it.g * G + t % G : -1;
      const uint32_t obuf = tmem + 128 + (j & 1) * 128;
      float m = 0.f, l = 0.f;  // max used for this row's probabilities, running row sum
      for (int k = 0; k < it.nchunks; ++k, ++c) {
        const int sb = c & 1;
        if (!__all_sync(0xffffffffu, wait_role(&bars.sfull[sb], (c >> 1) & 1, abort_flag, p.err))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int kbase = k * kKC;
        const bool diagonal = kbase + kKC - 1 > qpos;  // only then does the mask cut this row
        // pass 1: the row's chunk max under the causal mask (16-column pieces of S)
        float cm = -INFINITY;
#pragma unroll
        for (int q = 0; q < kKC / 16; ++q) {
          float sv[16];
          tmem_load16(lane_base + sb * 64 + q * 16, sv);
          if (diagonal) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (kbase + q * 16 + i <= qpos) cm = fmaxf(cm, sv[i] * p.scale_log2);
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) cm = fmaxf(cm, sv[i] * p.scale_log2);
          }
        }
        // lazy rescale: keep m unless the chunk brings a score more than the slack above
        float alpha = 1.f;
        if (k == 0) {
          m = cm;  // key 0 is never masked: finite
        } else if (cm > m + kRescaleSlack) {
          alpha = exp2f(m - cm);
          m = cm;
          l *= alpha;
        }
        const bool rescale = k > 0 && __any_sync(0xffffffffu, alpha != 1.f);
        // P(c) reuses the buffer P(c-2) filled: that PV must be done
        if (c >= 2 && !pv_done(c - 2)) {
          ok = false;
          break;
        }
        // pass 2: probabilities as hi + lo parts into P^T's swizzled rows
        float rowsum = 0.f;
        unsigned char* ph = smem + kOffP + sb * kPBytes;
        const float neg_m = -m;
#pragma unroll
        for (int q = 0; q < kKC / 16; ++q) {
          float sv[16];
          tmem_load16(lane_base + sb * 64 + q * 16, sv);
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int i = 0; i < 8; i += 2) {
              const int jj = q * 16 + half * 8 + i;
              float p0 = exp2_approx(fmaf(sv[half * 8 + i], p.scale_log2, neg_m));
              float p1 = exp2_approx(fmaf(sv[half * 8 + i + 1], p.scale_log2, neg_m));
              if (diagonal) {
                p0 = kbase + jj <= qpos ? p0 : 0.f;
                p1 = kbase + jj + 1 <= qpos ? p1 : 0.f;
              }
              rowsum += p0 + p1;
              float h0, h1;
              hw[i / 2] = pack2_split<T>(p0, p1, h0, h1);  // rounded pair, and its values
              lw[i / 2] = pack2<T>(p0 - h0, p1 - h1);      // exact remainders, rounded
            }
            const int off = swz_keys(t, q * 2 + half);
            *reinterpret_cast<uint4*>(ph + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4*>(ph + kPPart + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          }
        }
        l += rowsum;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.sfree[sb]);
        // a row whose max jumped: rescale its O row in TMEM once PV(c-1) is done
        if (rescale) {
          if (!pv_done(c - 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int q = 0; q < 8; ++q) {
            float o[16];
            tmem_load16(obuf + (static_cast<uint32_t>(warp * 32) << 16) + q * 16, o);
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] *= alpha;
            tmem_store16(obuf + (static_cast<uint32_t>(warp * 32) << 16) + q * 16, o);
          }
          tc_fence_before();
        }
        // V rows past the tile's last position inside loaded blocks: zero them (a NaN
        // there would survive a zero weight)
        const int rows_needed = pos_last + 1 - kbase;
        if (t < kKC && rows_needed < kKC) {
          const int rows_loaded = min(kKC, (rows_needed + p.block_size - 1) / p.block_size * p.block_size);
          if (t >= rows_needed && t < rows_loaded) {
            unsigned char* vrow = smem + (c % kStages) * kStageBytes + kKVTile + (t >> 3) * kGroup + (t & 7) * 128;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              reinterpret_cast<uint4*>(vrow)[q] = make_uint4(0, 0, 0, 0);
              reinterpret_cast<uint4*>(vrow + 1024)[q] = make_uint4(0, 0, 0, 0);
            }
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.pfull[sb]);
        // the previous tile's O can be read now that this tile's first chunk is queued
        if (k == 0 && prev_c >= 0) {
          if (!finish(prev_row, prev_c, prev_l, (j - 1) & 1)) {
            ok = false;
            break;
          }
          prev_c = -1;
        }
      }
      if (!ok) break;
      prev_row = out_row;
      prev_c = c - 1;
      prev_l = l;
    }
    if (ok && prev_c >= 0) finish(prev_row, prev_c, prev_l, (j - 1) & 1);
    __syncwarp();
  }

  // ---------------- teardown ----------------
  __syncthreads();
  if (*abort_flag) {
    if (warp == 4 && lane == 0) {
      for (int c = *waited_slot; c < *issued_slot; ++c)
        if (!mbar_wait(&bars.full[c % kStages], (c / kStages) & 1)) break;
    }
    if (warp == 5 && lane == 0) {
      mbar_init(bars.drain, 1);
      fence_barrier_init();
      mma_commit(bars.drain);
      mbar_wait(bars.drain, 0);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, kTmemCols);
}

// Work list: one entry per (sequence, KV head, query tile), sorted by chunk count,
// longest first (counting sort; order inside one count does not matter).
__global__ void __launch_bounds__(kListThreads) prefill_list_kernel(const __grid_constant__ PrefillParams p) {
  __shared__ int hist[kMaxBuckets];
  __shared__ int next[kMaxBuckets];
  const int H = p.num_kv_heads, TQ = p.tile_tokens;
  for (int i = threadIdx.x; i < kMaxBuckets; i += kListThreads) hist[i] = 0;
  __syncthreads();
  for (int s = threadIdx.x; s < p.num_seqs; s += kListThreads) {
    const int n = p.query_start[s + 1] - p.query_start[s], L = p.context_lens[s];
    if (n < 0 || L < n || L > p.max_context_len) {
      set_error(p.err, kErrLength);
      continue;
    }
    for (int t0 = 0; t0 < n; t0 += TQ) {
      const int ntile = min(TQ, n - t0), pos0 = L - n + t0;
      const int nch = (pos0 + ntile + kKC - 1) / kKC;
      atomicAdd(&hist[min(nch, kMaxBuckets - 1)], H);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int c = kMaxBuckets - 1; c >= 0; --c) {
      next[c] = run;
      run += hist[c];
    }
    *p.work_count = run;
  }
  __syncthreads();
  for (int s = threadIdx.x; s < p.num_seqs; s += kListThreads) {
    const int n = p.query_start[s + 1] - p.query_start[s], L = p.context_lens[s];
    if (n < 0 || L < n || L > p.max_context_len) continue;
    for (int t0 = 0; t0 < n; t0 += TQ) {
      const int ntile = min(TQ, n - t0), pos0 = L - n + t0;
      const int nch = (pos0 + ntile + kKC - 1) / kKC;
      const int pos = atomicAdd(&next[min(nch, kMaxBuckets - 1)], H);
      for (int g = 0; g < H; ++g)
        p.work_list[pos + g] = make_int4(s, g | (ntile << 16), p.query_start[s] + t0, pos0);
    }
  }
}

template <typename T>
cudaError_t launch_prefill_t(const PrefillArgs& args, int grid, cudaStream_t stream) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  prefill_tc_kernel<T><<<grid, kThreads, kSmemBytes, stream>>>(args);
  return cudaGetLastError();
}

}  // namespace

int prefill_tile_tokens(int group) { return kRows / group; }

size_t prefill_max_items(int num_seqs, int num_query_tokens, int num_kv_heads, int group) {
  const int TQ = kRows / group;
  return (static_cast<size_t>(num_query_tokens) / TQ + num_seqs) * num_kv_heads;
}

cudaError_t launch_prefill_tc(const PrefillParams& p, int dtype, cudaStream_t stream) {
  PrefillArgs args;
  args.p = p;
  const bool bf16 = dtype == PKV_BF16;
  const uint64_t pool_rows = static_cast<uint64_t>(p.num_blocks) * p.num_kv_heads * p.block_size;
  if (!make_pool_map(&args.tk, p.k_cache, pool_rows, p.block_size, bf16) ||
      !make_pool_map(&args.tv, p.v_cache, pool_rows, p.block_size, bf16))
    return cudaErrorInvalidValue;
  prefill_list_kernel<<<1, kListThreads, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const size_t items = prefill_max_items(p.num_seqs, p.num_query_tokens, p.num_kv_heads, p.group);
  const int grid = static_cast<int>(items < static_cast<size_t>(sms) ? items : sms);
  if (grid == 0) return cudaSuccess;
  return bf16 ? launch_prefill_t<__nv_bfloat16>(args, grid, stream) : launch_prefill_t<__half>(args, grid, stream);
}

}  // namespace pkv
