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
// A tile is 128 query rows: TQ = floor(128 / G) consecutive new tokens times the G
// query heads of one KV head, row r = token * G + head (rows past TQ * G are padding).
// A work item is a PAIR of consecutive tiles of one (sequence, KV head): both tiles
// consume the same K/V chunks, so each chunk is read once for 256 query rows.  Per
// 64-key chunk and tile:
//   S[128 rows x 64 keys] = Q . K^T            (M=128, N=64,  K=128 dims)
//   O[128 rows x 128 dims] += P . V            (M=128, N=128, K=64 keys), twice:
// the probabilities as hi = round(p) and lo = round(p - hi) in the cache dtype, so
// the 16-bit operand costs about 2^-17 relative per weight.  S (double-buffered) and
// O of each tile live in TMEM; the MMA accumulates O over the item's chunks.  Softmax
// is row-local (no cross-thread reduction) with a lazy rescale: a row keeps the
// maximum it used for its probabilities until a chunk brings a score more than 8
// (log2 units) above it -- probabilities stay <= 256 -- and only then is its O row
// rescaled in TMEM.
//
// Roles (320 threads, persistent CTAs over a longest-first work list dealt in snake
// order):
//  * warps 0-3 and 4-7: one softmax warpgroup per tile of the pair (thread = query
//    row = TMEM lane); while one group computes probabilities the tensor cores work
//    for the other.
//  * warp 8, producer: loads both tiles' query rows (plain loads, written in the
//    128-byte swizzled operand layout), then per chunk one 4-D TMA box per block for
//    K and one for V into a 3-stage ring (blocks past the pair's last position are
//    loaded from outside the tensor: zero fill).
//  * warp 9, MMA: one lane polls four streams -- QK and PV of each tile -- and issues
//    whatever is ready; a ring stage is released once both tiles' PVs of its chunk
//    are issued (their commit fires when they complete).
#include <climits>
#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "tc_util.cuh"
#include "tcgen05.cuh"

namespace pkv {
namespace {

constexpr int kGroups = 2;                 // tiles per item, one softmax warpgroup each
constexpr int kThreads = (4 * kGroups + 2) * 32;
constexpr int kProducerWarp = 4 * kGroups, kMmaWarp = 4 * kGroups + 1;
constexpr int kRows = 128;                 // query rows per tile (M)
constexpr int kKC = 64;                    // keys per chunk
constexpr int kStages = 3;
constexpr int kGroup = 2048;               // 8-row group of a 128-dim tile: two 64-column halves
constexpr int kKVTile = kKC * 256;         // K (or V) of one chunk: 16 KB
constexpr int kStageBytes = 2 * kKVTile;   // K then V
constexpr int kQBytes = kRows * 256;       // 32 KB per tile: [16 groups][2 halves][8 rows][128 B]
constexpr int kPPart = kRows * kKC * 2;    // 16 KB: [16 groups][8 rows][128 B], one part
constexpr int kPBytes = 2 * kPPart;        // per tile: hi part then lo part
constexpr int kOffQ = kStages * kStageBytes;
constexpr int kOffP = kOffQ + kGroups * kQBytes;
constexpr int kOffBar = kOffP + kGroups * kPBytes;
// ring full/empty, qfull, qempty, then per tile: sfull[2], sfree[2], pfull, pvdone[2]; drain
constexpr int kNumBars = 2 * kStages + 2 + kGroups * 7 + 1;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 64;
constexpr uint32_t kTmemCols = 512;        // per tile g: S[2] at 256g + 0/64, O at 256g + 128
constexpr float kRescaleSlack = 8.f;       // log2 units a row's max may grow before O is rescaled
constexpr int kListThreads = 1024;
constexpr int kMaxBuckets = 1024;          // chunk-count buckets of the work list (last one open-ended)

struct Bars {
  uint64_t *full, *empty, *qfull, *qempty, *drain, *grp;
  // per tile g: sfull[2], sfree[2], pfull, pvdone[2] (addresses computed, so a
  // runtime tile index needs no local-memory table)
  __device__ __forceinline__ uint64_t* sfull(int g, int i) const { return grp + 7 * g + i; }
  __device__ __forceinline__ uint64_t* sfree(int g, int i) const { return grp + 7 * g + 2 + i; }
  __device__ __forceinline__ uint64_t* pfull(int g) const { return grp + 7 * g + 4; }
  __device__ __forceinline__ uint64_t* pvdone(int g, int i) const { return grp + 7 * g + 5 + i; }
};

__device__ __forceinline__ Bars carve(unsigned char* smem) {
  uint64_t* b = reinterpret_cast<uint64_t*>(smem + kOffBar);
  Bars r;
  r.full = b;
  r.empty = b + kStages;
  r.qfull = b + 2 * kStages;
  r.qempty = r.qfull + 1;
  r.grp = r.qempty + 1;
  r.drain = r.grp + 7 * kGroups;
  return r;
}

struct PrefillArgs {
  CUtensorMap tk;  // pool 4-D views: one box = one block's tile for one KV head
  CUtensorMap tv;
  PrefillParams p;
};

// {s, g | ntile_a << 12 | ntile_b << 20, first query row of tile a, position of its first token}
struct Item {
  int s, g, na, nb, qrow0, pos0, last, nchunks;  // na, nb: tokens in tile a, tile b
  __device__ __forceinline__ int ntok(int tile) const { return tile ? nb : na; }
};

__device__ __forceinline__ Item unpack_item(int4 e, int tq) {
  Item t;
  t.s = e.x;
  t.g = e.y & 0xfff;
  t.na = (e.y >> 12) & 0xff;
  t.nb = (static_cast<unsigned>(e.y) >> 20) & 0xff;
  t.qrow0 = e.z;
  t.pos0 = e.w;
  t.last = t.pos0 + (t.nb ? tq + t.nb : t.na) - 1;  // position of the pair's last token
  t.nchunks = (t.last + kKC) / kKC;
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
  const int G = p.group, TQ = p.tile_tokens;
  const int num_items = *p.work_count;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bars.full[i], 1);
      mbar_init(&bars.empty[i], 1);
    }
    mbar_init(bars.qfull, 1);
    mbar_init(bars.qempty, 1);
    for (int g = 0; g < kGroups; ++g) {
      for (int i = 0; i < 2; ++i) {
        mbar_init(bars.sfull(g, i), 1);
        mbar_init(bars.sfree(g, i), 4);
        mbar_init(bars.pvdone(g, i), 1);
      }
      mbar_init(bars.pfull(g), 4);
    }
    *abort_flag = 0;
    *issued_slot = 0;
    *waited_slot = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kProducerWarp) {
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
    for (cur.init(p.work_list, num_items); cur.valid() && ok; cur.advance(), ++j) {
      const Item it = unpack_item(cur.cur, TQ);
      // ---- both tiles' query rows, swizzled, zero past each tile; the previous
      //      item's QKs must be done with the buffers ----
      ok = j < 1 || __shfl_sync(0xffffffffu, lane == 0 ? wait_role(bars.qempty, (j - 1) & 1, abort_flag, p.err)
                                                       : true, 0);
      if (!ok) break;
#pragma unroll 1
      for (int g = 0; g < kGroups; ++g) {
        unsigned char* qbuf = smem + kOffQ + g * kQBytes;
        const int valid_rows = it.ntok(g) * G;
#pragma unroll 1
        for (int r = lane; r < kRows; r += 32) {
          const bool valid = r < valid_rows;
          const uint4* src = reinterpret_cast<const uint4*>(static_cast<const T*>(p.q) +
              (static_cast<size_t>(it.qrow0 + g * TQ + r / G) * p.num_q_heads + it.g * G + r % G) * 128);
#pragma unroll
          for (int c16 = 0; c16 < 16; ++c16) {
            const uint4 v = valid ? src[c16] : make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(qbuf + swz_dims(r, c16)) = v;
          }
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.qfull);
      // ---- K/V chunks ----
      const int32_t* table = p.block_tables + static_cast<size_t>(it.s) * p.max_blocks_per_seq;
      for (int k = 0; k < it.nchunks && ok; ++k, ++c) {
        const int st = c % kStages;
        const int lb = k * blocks_per_chunk + lane;  // logical block of this lane
        const bool live = lane < blocks_per_chunk && lb * bs <= it.last;
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
    }
  } else if (warp == kMmaWarp) {
    // ============================ MMA issuer ============================
    if (lane == 0) {
      constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
      constexpr uint32_t idesc_qk = instr_desc_f16(kBf16, false, false, kRows, kKC);
      constexpr uint32_t idesc_pv = instr_desc_f16(kBf16, false, true, kRows, 128);
      const uint32_t ring = smem_addr(smem);
      const uint32_t qbase = smem_addr(smem + kOffQ);
      const uint32_t pbase = smem_addr(smem + kOffP);
      // one cursor per stream: QK and PV of each tile walk the same chunk sequence
      struct Stream {
        ItemCursor cur;
        int k, n, c;  // chunk within the item, chunks in the item, global chunk
      };
      Stream qs[kGroups], ps[kGroups];
#pragma unroll
      for (int g = 0; g < kGroups; ++g) {
        qs[g].cur.init(p.work_list, num_items);
        ps[g].cur.init(p.work_list, num_items);
        qs[g].k = ps[g].k = 0;
        qs[g].c = ps[g].c = 0;
        qs[g].n = ps[g].n = qs[g].cur.valid() ? unpack_item(qs[g].cur.cur, TQ).nchunks : 0;
      }
      auto step = [&](Stream& s) {
        ++s.c;
        if (++s.k == s.n) {
          s.k = 0;
          s.cur.advance();
          s.n = s.cur.valid() ? unpack_item(s.cur.cur, TQ).nchunks : 0;
        }
      };
      int q_items = 0;     // items whose query buffers both tiles are done with
      int q_last = 0;      // tiles that issued the current item's last QK
      uint64_t idle_since = global_timer_ns();
      while (true) {
        bool active = false, progressed = false;
#pragma unroll
        for (int g = 0; g < kGroups; ++g) {
          Stream& s = qs[g];
          if (!s.cur.valid()) continue;
          active = true;
          if (s.cur.k != q_items) continue;  // one query buffer per tile: no running ahead
          const int c = s.c, st = c % kStages, sb = c & 1;
          if ((s.k > 0 || mbar_try_wait(bars.qfull, q_items & 1)) &&
              mbar_try_wait(&bars.full[st], (c / kStages) & 1) &&
              (c < 2 || mbar_try_wait(bars.sfree(g, sb), ((c >> 1) - 1) & 1))) {
            if (g == 0) *waited_slot = c + 1;
            tc_fence_after();
            const uint32_t kb = ring + st * kStageBytes;
            const uint32_t qa = qbase + g * kQBytes;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t off = (kk >> 2) * 1024 + (kk & 3) * 32;
              mma_f16(tmem + g * 256 + sb * 64, smem_desc(qa + off, 16, kGroup, kLayoutSwizzle128),
                      smem_desc(kb + off, 16, kGroup, kLayoutSwizzle128), idesc_qk, kk > 0);
            }
            mma_commit(bars.sfull(g, sb));
            if (s.k == s.n - 1 && ++q_last == kGroups) {  // both tiles' queries consumed
              mma_commit(bars.qempty);
              q_last = 0;
              ++q_items;
            }
            step(s);
            progressed = true;
          }
        }
#pragma unroll
        for (int g = 0; g < kGroups; ++g) {
          Stream& s = ps[g];
          if (!s.cur.valid()) continue;
          active = true;
          if (s.c >= qs[g].c) continue;  // its QK comes first
          const int c = s.c, st = c % kStages;
          if (mbar_try_wait(bars.pfull(g), c & 1)) {
            tc_fence_after();
            const uint32_t vbase = ring + st * kStageBytes + kKVTile;
            const uint32_t pa = pbase + g * kPBytes;
            const uint32_t od = tmem + g * 256 + 128;
#pragma unroll
            for (int kk = 0; kk < kKC / 16; ++kk) {
              const uint64_t bd = smem_desc(vbase + kk * 2 * kGroup, 1024, kGroup, kLayoutSwizzle128);
              mma_f16(od, smem_desc(pa + kk * 32, 16, 1024, kLayoutSwizzle128), bd, idesc_pv, s.k > 0 || kk > 0);
              mma_f16(od, smem_desc(pa + kPPart + kk * 32, 16, 1024, kLayoutSwizzle128), bd, idesc_pv, true);
            }
            mma_commit(bars.pvdone(g, c & 1));
            // the stage is free once every tile's PV of this chunk has completed
            bool all = true;
#pragma unroll
            for (int h = 0; h < kGroups; ++h)
              if (h != g && ps[h].c <= c) all = false;
            if (all) mma_commit(&bars.empty[st]);
            step(s);
            progressed = true;
          }
        }
        if (!active) break;
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
    // ============================ softmax warpgroups ============================
    const int grp = warp / 4;                 // which tile of the pair
    const int t = threadIdx.x % 128;          // query row of the tile = TMEM lane
    const int wq = warp % 4;                  // lane quarter
    const uint32_t lane_base = tmem + grp * 256 + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t obuf = lane_base + 128;
    int c = 0;
    bool ok = true;
    int prev_row = -1, prev_c = -1;
    float prev_l = 1.f;

    // Warp-uniform: has this tile's PV of chunk cc completed?  (waited in chunk order)
    auto pv_done = [&](int cc) -> bool {
      return __all_sync(0xffffffffu, wait_role(bars.pvdone(grp, cc & 1), (cc >> 1) & 1, abort_flag, p.err));
    };
    // A finished item's output rows: O / l (O is final: its last PV was waited for).
    auto finish = [&](int row, float lsum) {
      tc_fence_after();
      const float inv = 1.f / lsum;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float o[16];
        tmem_load16(obuf + q * 16, o);
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
    };

    ItemCursor cur;
    for (cur.init(p.work_list, num_items); cur.valid() && ok; cur.advance()) {
      const Item it = unpack_item(cur.cur, TQ);
      const int valid_rows = it.ntok(grp) * G;
      const bool row_valid = t < valid_rows;
      const int qpos = row_valid ? it.pos0 + grp * TQ + t / G : it.last;  // padding rows act as the last token
      const int out_row = row_valid ? (it.qrow0 + grp * TQ + t / G) * p.num_q_heads + it.g * G + t % G : -1;
      float m = 0.f, l = 0.f;  // max used for this row's probabilities, running row sum
      for (int k = 0; k < it.nchunks; ++k, ++c) {
        const int sb = c & 1;
        if (!__all_sync(0xffffffffu, wait_role(bars.sfull(grp, sb), (c >> 1) & 1, abort_flag, p.err))) {
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
        // (a chunk entirely past this row's position gives cm = -inf and changes nothing)
        float alpha = 1.f;
        if (k == 0) {
          m = cm;  // key 0 is never masked: finite
        } else if (cm > m + kRescaleSlack) {
          alpha = exp2f(m - cm);
          m = cm;
          l *= alpha;
        }
        // the previous chunk's PV (reads P, accumulates O) must be done before P is
        // rewritten, O rescaled, or -- at an item's first chunk -- O read out
        if (c >= 1 && !pv_done(c - 1)) {
          ok = false;
          break;
        }
        if (k == 0 && prev_c >= 0) {
          finish(prev_row, prev_l);
          prev_c = -1;
        }
        if (k > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          tc_fence_after();
#pragma unroll 1
          for (int q = 0; q < 8; ++q) {
            float o[16];
            tmem_load16(obuf + q * 16, o);
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] *= alpha;
            tmem_store16(obuf + q * 16, o);
          }
          tc_fence_before();
        }
        // pass 2: probabilities as hi + lo parts into P's swizzled rows
        float rowsum = 0.f;
        unsigned char* ph = smem + kOffP + grp * kPBytes;
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
        if (lane == 0) mbar_arrive(bars.sfree(grp, sb));
        // V rows past the pair's last position inside loaded blocks: zero them (a NaN
        // there would survive a zero weight).  Both groups write the same zeros.
        const int rows_needed = it.last + 1 - kbase;
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
        if (lane == 0) mbar_arrive(bars.pfull(grp));
      }
      if (!ok) break;
      prev_row = out_row;
      prev_c = c - 1;
      prev_l = l;
    }
    if (ok && prev_c >= 0 && pv_done(prev_c)) finish(prev_row, prev_l);
    __syncwarp();
  }

  // ---------------- teardown ----------------
  __syncthreads();
  if (*abort_flag) {
    if (warp == kProducerWarp && lane == 0) {
      for (int c = *waited_slot; c < *issued_slot; ++c)
        if (!mbar_wait(&bars.full[c % kStages], (c / kStages) & 1)) break;
    }
    if (warp == kMmaWarp && lane == 0) {
      mbar_init(bars.drain, 1);
      fence_barrier_init();
      mma_commit(bars.drain);
      mbar_wait(bars.drain, 0);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

// Work list: one entry per (sequence, KV head, pair of query tiles), sorted by chunk
// count, longest first (counting sort; order inside one count does not matter).
__global__ void __launch_bounds__(kListThreads) prefill_list_kernel(const __grid_constant__ PrefillParams p) {
  __shared__ int hist[kMaxBuckets];
  __shared__ int next[kMaxBuckets];
  const int H = p.num_kv_heads, TQ = p.tile_tokens, span = kGroups * TQ;
  for (int i = threadIdx.x; i < kMaxBuckets; i += kListThreads) hist[i] = 0;
  __syncthreads();
  for (int s = threadIdx.x; s < p.num_seqs; s += kListThreads) {
    const int n = p.query_start[s + 1] - p.query_start[s], L = p.context_lens[s];
    if (n < 0 || L < n || L > p.max_context_len) {
      set_error(p.err, kErrLength);
      continue;
    }
    for (int t0 = 0; t0 < n; t0 += span) {
      const int nch = (L - n + t0 + min(span, n - t0) + kKC - 1) / kKC;
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
    for (int t0 = 0; t0 < n; t0 += span) {
      const int na = min(TQ, n - t0), nb = max(0, min(TQ, n - t0 - TQ));
      const int nch = (L - n + t0 + na + nb + kKC - 1) / kKC;
      const int pos = atomicAdd(&next[min(nch, kMaxBuckets - 1)], H);
      for (int g = 0; g < H; ++g)
        p.work_list[pos + g] = make_int4(s, g | (na << 12) | (nb << 20), p.query_start[s] + t0, L - n + t0);
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
  const int span = kGroups * (kRows / group);
  return (static_cast<size_t>(num_query_tokens) / span + num_seqs) * num_kv_heads;
}

cudaError_t launch_prefill_tc(const PrefillParams& p, int dtype, cudaStream_t stream) {
  if (p.num_kv_heads > 4095) return cudaErrorInvalidValue;  // packed into 12 bits of a list entry
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
