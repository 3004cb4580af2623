// prefill_tc.cu -- multi-token paged attention with a causal mask (prefill and
// chunked prefill) on the tcgen05 tensor cores; f16/bf16, head_dim 64 or 128, up to
// 16 query heads per KV head.
//
// What it computes ("anthology-of-the-sota note-023", Method: attention gathers K/V
// through the block table; the same arithmetic as attention over contiguous memory):
// sequence s brings n_s new tokens, the last n_s of its context_lens[s] tokens (their
// K/V already appended to the pool).  New token i sits at position
// p = context_lens[s] - n_s + i and attends to positions 0..p through the block table.
// One new token per sequence is exactly paged decode.
//
// A tile is 128 query rows of one KV head: its G query heads times TQ = 8 * floor(16 / G)
// consecutive new tokens, head-major (row r = head * TQ + token; rows past G * TQ are
// padding).  Every 8-row group is then 8 tokens of one head, which one TMA box loads in
// the 128-byte swizzled operand layout.  A work item is a PAIR of consecutive tiles of
// one (sequence, KV head): both consume the same K/V chunks, so each chunk is read once
// for 256 query rows.  Per 64-key chunk and tile:
//   S[128 rows x 64 keys] = Q . K^T             (M=128, N=64, K=D dims)
//   O[128 rows x D dims] += P . V               (M=128, N=D,  K=64 keys), twice:
// the probabilities as hi = round(p) and lo = round(p - hi) in the cache dtype, so the
// 16-bit operand costs about 2^-17 relative per weight.  S (double-buffered) and O of
// each tile live in TMEM; the probabilities are written back over the S columns they
// came from and the PV products read them from TMEM, so shared memory holds only K/V
// and Q.  Softmax is row-local (one thread per row, no cross-thread reduction) with a
// lazy rescale: a row keeps the maximum it used for its probabilities until a chunk
// brings a score more than 8 (log2 units) above it -- probabilities stay <= 256 -- and
// only then is its O row rescaled in TMEM.
//
// Roles (352 threads, persistent CTAs over a work list in which a sequence's items are
// adjacent -- they share K/V, which then stays in L2 -- and sequences come longest
// first, dealt in snake order):
//  * warps 0-3 and 4-7: one softmax warpgroup per tile of the pair (thread = query
//    row = TMEM lane); the two groups and the tensor cores work concurrently.
//  * warp 8, producer of Q and K: per item the query boxes of both tiles into a double
//    buffer, then per chunk one 4-D TMA box per block of K into a 48 KB ring (3 stages
//    at D = 128, 6 at D = 64; blocks past the pair's last position come from outside
//    the tensor: zero fill).  A K stage is free once both tiles' QKs of its chunk
//    completed.
//  * warp 10, producer of V: the same for V into its own ring, whose stage is free once
//    both tiles' PVs of its chunk completed.
//  * warp 9, MMA: a fixed schedule per chunk c -- PV of tile 0, PV of tile 1, then QK
//    of both tiles for chunk c + 2, whose S columns held the probabilities of chunk c
//    (tcgen05 MMAs of one thread run in issue order, so that QK may overwrite them
//    once PV(c) has been issued).  The whole warp runs it with warp-uniform control
//    flow; one batched barrier probe per chunk covers everything it needs, and one
//    elected lane issues.
#include <climits>
#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "tc_util.cuh"
#include "tcgen05.cuh"

namespace pkv {
namespace {

constexpr int kGroups = 2;                 // tiles per item, one softmax warpgroup each
constexpr int kThreads = (4 * kGroups + 3) * 32;
constexpr int kProducerWarp = 4 * kGroups, kMmaWarp = 4 * kGroups + 1, kVWarp = 4 * kGroups + 2;
constexpr int kRows = 128;                 // query rows per tile (M)
constexpr int kKC = 64;                    // keys per chunk
constexpr uint32_t kTmemCols = 512;        // per tile g: S[2] at 256g + 0/64, O at 256g + 128 (D columns)
constexpr float kRescaleSlack = 8.f;       // log2 units a row's max may grow before O is rescaled
constexpr int kListThreads = 1024;
constexpr int kMaxBuckets = 1024;          // chunk-count buckets of the work list (last one open-ended)

// Query buffers: items whose queries are resident.  Two, so an item's queries load
// while the previous item runs (one buffer with five-stage K/V rings instead of three
// measured 5 % slower).
constexpr int kQBufs = 2;

// Shared-memory layout for head_dim D (64 or 128): K, V and Q tiles as [8-row group]
// [64-column block][8 rows][128 B], 128-byte swizzled.
template <int D>
struct PfLayout {
  static constexpr int kBlocks = D / 64;                  // 64-column blocks of a row
  static constexpr int kGroup = 8 * D * 2;                // one 8-row group: all its blocks
  static constexpr int kKVTile = kKC * D * 2;             // K (or V) of one chunk: 8 or 16 KB
  static constexpr int kStages = (kQBufs == 2 ? 3 : 5) * 128 / D;  // per ring (K and V have one each)
  static constexpr int kQBytes = kRows * D * 2;           // one tile's queries: 16 or 32 KB
  static constexpr int kQItem = kGroups * kQBytes;        // both tiles of an item
  static constexpr int kOffV = kStages * kKVTile;
  static constexpr int kOffQ = 2 * kStages * kKVTile;
  static constexpr int kOffBar = kOffQ + kQBufs * kQItem;
  // K ring full/empty, V ring full/empty, qfull[2], qempty[2], then per tile: sfull[2],
  // pfull[2], pvdone[2]; drain
  static constexpr int kNumBars = 4 * kStages + 4 + kGroups * 6 + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 64;
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  static_assert(kOffQ % 1024 == 0 && kSmemBytes <= 232448, "shared memory");
};

struct Bars {
  uint64_t *kfull, *kempty, *vfull, *vempty, *qfull, *qempty, *grp, *drain;
  // per tile g (addresses computed, so a runtime tile index needs no local-memory table)
  __device__ __forceinline__ uint64_t* sfull(int g, int i) const { return grp + 6 * g + i; }
  __device__ __forceinline__ uint64_t* pfull(int g, int i) const { return grp + 6 * g + 2 + i; }
  __device__ __forceinline__ uint64_t* pvdone(int g, int i) const { return grp + 6 * g + 4 + i; }
};

template <int D>
__device__ __forceinline__ Bars carve(unsigned char* smem) {
  constexpr int kStages = PfLayout<D>::kStages;
  uint64_t* b = reinterpret_cast<uint64_t*>(smem + PfLayout<D>::kOffBar);
  Bars r;
  r.kfull = b;
  r.kempty = b + kStages;
  r.vfull = b + 2 * kStages;
  r.vempty = b + 3 * kStages;
  r.qfull = b + 4 * kStages;
  r.qempty = r.qfull + 2;
  r.grp = r.qempty + 2;
  r.drain = r.grp + 6 * kGroups;
  return r;
}

struct PrefillArgs {
  CUtensorMap tk;  // pool 4-D views: one box = one block's tile for one KV head
  CUtensorMap tv;
  CUtensorMap tq;  // queries (head_dim, heads, tokens): one box = 8 tokens x 64 dims of one head
  PrefillParams p;
};

// {s, g | ntile_a << 12 | ntile_b << 20, first query token of tile a, position of that token}
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

// Extreme of a row's 64 raw scores (maximum, or minimum when the scale is negative),
// keys past `lim` excluded when the chunk crosses the diagonal (overwritten in place
// with the neutral value).
template <bool kMin>
__device__ __forceinline__ float chunk_extreme(float* sv, bool diagonal, int lim) {
  constexpr float kNone = kMin ? INFINITY : -INFINITY;
  if (diagonal) {
#pragma unroll
    for (int i = 0; i < 64; ++i) sv[i] = i <= lim ? sv[i] : kNone;
  }
  float e0 = kNone, e1 = kNone;
#pragma unroll
  for (int i = 0; i < 64; i += 4) {
    e0 = kMin ? fmin3(e0, sv[i], sv[i + 1]) : fmax3(e0, sv[i], sv[i + 1]);
    e1 = kMin ? fmin3(e1, sv[i + 2], sv[i + 3]) : fmax3(e1, sv[i + 2], sv[i + 3]);
  }
  return kMin ? fminf(e0, e1) : fmaxf(e0, e1);
}

// One producer warp's copies of an item's chunks of K (or V) into its ring: per chunk
// one 4-D box per block (blocks past the pair's last position from outside the tensor:
// zero fill).  `c` counts the warp's chunks over all items.  Returns false on abort.
template <int D>
__device__ __forceinline__ bool load_chunks(const PrefillParams& p, const Item& it, const CUtensorMap* map,
                                            unsigned char* ring, uint64_t* full, uint64_t* empty, int& c,
                                            int* issued_slot, uint64_t policy, volatile int* abort_flag) {
  constexpr int kStages = PfLayout<D>::kStages, kKVTile = PfLayout<D>::kKVTile;
  const int lane = threadIdx.x % 32;
  const int bs = p.block_size;
  const int blocks_per_chunk = kKC / bs;
  const int oob_group = p.num_blocks * p.num_kv_heads * bs / 8;  // first row group outside the pool
  const int32_t* table = p.block_tables + static_cast<size_t>(it.s) * p.max_blocks_per_seq;
  for (int k = 0; k < it.nchunks; ++k, ++c) {
    const int st = c % kStages;
    const int lb = k * blocks_per_chunk + lane;  // logical block of this lane
    const bool live = lane < blocks_per_chunk && lb * bs <= it.last;
    int b = live ? (lb < p.max_blocks_per_seq ? table[lb] : -1) : 0;
    bool ok = true;
    if (lane == 0) {
      ok = c < kStages || wait_role(&empty[st], ((c / kStages) - 1) & 1, abort_flag, p.err, p.wait_limit_ns);
      if (ok) mbar_arrive_expect_tx(&full[st], kKVTile);
    }
    if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
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
      tma_load_4d(ring + st * kKVTile + lane * bs * (D * 2), map, grp, &full[st], policy);
    }
    if (lane == 0) *issued_slot = c + 1;
  }
  return true;
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(const __grid_constant__ PrefillArgs a) {
  using L = PfLayout<D>;
  constexpr int kStages = L::kStages, kGroup = L::kGroup, kKVTile = L::kKVTile;
  constexpr int kQBytes = L::kQBytes, kQItem = L::kQItem, kOffV = L::kOffV, kOffQ = L::kOffQ;
  constexpr int kOffMisc = L::kOffMisc;
  extern __shared__ __align__(1024) unsigned char smem[];
  const PrefillParams& p = a.p;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const Bars bars = carve<D>(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  int* kissued_slot = reinterpret_cast<int*>(smem + kOffMisc + 8);
  int* vissued_slot = reinterpret_cast<int*>(smem + kOffMisc + 12);
  int* qissued_slot = reinterpret_cast<int*>(smem + kOffMisc + 16);
  const int G = p.group, TQ = p.tile_tokens;
  const int num_items = *p.work_count;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bars.kfull[i], 1);
      mbar_init(&bars.kempty[i], 1);
      mbar_init(&bars.vfull[i], 1);
      mbar_init(&bars.vempty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.qfull[i], 1);
      mbar_init(&bars.qempty[i], 1);
    }
    for (int g = 0; g < kGroups; ++g) {
      for (int i = 0; i < 2; ++i) {
        mbar_init(bars.sfull(g, i), 1);
        mbar_init(bars.pfull(g, i), 4);
        mbar_init(bars.pvdone(g, i), 1);
      }
    }
    *abort_flag = 0;
    *kissued_slot = 0;
    *vissued_slot = 0;
    *qissued_slot = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kProducerWarp) {
    // ============================ producer: Q and K ============================
    if (lane == 0) {
      prefetch_tensormap(&a.tk);
      prefetch_tensormap(&a.tq);
    }
    const uint64_t pol_kv = policy_evict_normal();  // K/V: re-read by the sequence's other items
    const uint64_t pol_q = policy_evict_first();    // Q: read once
    // this lane's query box of a tile: 8-row group lane / kBlocks, 64-column block lane % kBlocks
    const int qrows = (lane / L::kBlocks) * 8, qhalf = lane % L::kBlocks;
    const int qhead = qrows / TQ, qtok = qrows % TQ;
    int c = 0, j = 0;
    bool ok = true;
    ItemCursor cur;
    for (cur.init(p.work_list, num_items); cur.valid() && ok; cur.advance(), ++j) {
      const Item it = unpack_item(cur.cur, TQ);
      // ---- both tiles' queries into buffer j % kQBufs (free once item j - kQBufs's QKs completed) ----
      const int qb = j % kQBufs;
      if (lane == 0) {
        ok = j < kQBufs || wait_role(&bars.qempty[qb], ((j / kQBufs) - 1) & 1, abort_flag, p.err, p.wait_limit_ns);
        if (ok) mbar_arrive_expect_tx(&bars.qfull[qb], kQItem);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      __syncwarp();
      if (lane < 16 * L::kBlocks) {
#pragma unroll
        for (int g = 0; g < kGroups; ++g) {
          // padding groups (past the G heads) read tokens outside the tensor: zeros
          const int tok = qhead < G ? it.qrow0 + g * TQ + qtok : p.num_query_tokens;
          const int head = it.g * G + min(qhead, G - 1);
          tma_load_3d(smem + kOffQ + qb * kQItem + g * kQBytes + (lane / L::kBlocks) * kGroup + qhalf * 1024, &a.tq,
                      qhalf * 64, head, tok, &bars.qfull[qb], pol_q);
        }
      }
      if (lane == 0) *qissued_slot = j + 1;
      // ---- K chunks (a stage is free once both tiles' QKs of its chunk completed) ----
      ok = load_chunks<D>(p, it, &a.tk, smem, bars.kfull, bars.kempty, c, kissued_slot, pol_kv, abort_flag);
    }
  } else if (warp == kVWarp) {
    // ============================ producer: V ============================
    if (lane == 0) prefetch_tensormap(&a.tv);
    const uint64_t pol_kv = policy_evict_normal();
    int c = 0;
    bool ok = true;
    ItemCursor cur;
    for (cur.init(p.work_list, num_items); cur.valid() && ok; cur.advance()) {
      // a stage is free once both tiles' PVs of its chunk completed
      ok = load_chunks<D>(p, unpack_item(cur.cur, TQ), &a.tv, smem + kOffV, bars.vfull, bars.vempty, c,
                          vissued_slot, pol_kv, abort_flag);
    }
  } else if (warp == kMmaWarp) {
    // ============================ MMA issuer ============================
    // A fixed schedule, per chunk c: PV of tile 0, PV of tile 1, then QK of both tiles
    // for chunk c + 2 (whose S buffers held the probabilities of chunk c).  The whole
    // warp runs it with warp-uniform control flow (descriptors and counters stay in
    // uniform registers); one elected lane issues.
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr uint32_t idesc_qk = instr_desc_f16(kBf16, false, false, kRows, kKC);
    constexpr uint32_t idesc_pv = instr_desc_f16(kBf16, false, true, kRows, D);
    // descriptor bases; adding (byte offset >> 4) moves a descriptor's start address
    const uint64_t dq0 = smem_desc(smem_addr(smem + kOffQ), 16, kGroup, kLayoutSwizzle128);
    const uint64_t dk0 = smem_desc(smem_addr(smem), 16, kGroup, kLayoutSwizzle128);
    const uint64_t dv0 = smem_desc(smem_addr(smem + kOffV), 1024, kGroup, kLayoutSwizzle128);
    auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, wait_role(bar, parity, abort_flag, p.err, p.wait_limit_ns));
    };
    // QK side: next chunk qc (global), its stage / phase, its place in the item
    ItemCursor qcur;
    qcur.init(p.work_list, num_items);
    int qc = 0, qst = 0, qph = 0, qk = 0, qn = qcur.valid() ? unpack_item(qcur.cur, TQ).nchunks : 0;
    // PV side
    ItemCursor pcur;
    pcur.init(p.work_list, num_items);
    int pc = 0, pst = 0, pph = 0, pk = 0, pn = qn;
    bool ok = true;
    // QK of chunk qc for both tiles (k_seen: its K stage was already seen landed)
    auto qk_pair = [&](bool k_seen) -> bool {
      const int qj = qcur.k, qb = qj % kQBufs, sb = qc & 1;
      if (qk == 0 && !wait_all(&bars.qfull[qb], (qj / kQBufs) & 1)) return false;
      if (!k_seen && !wait_all(&bars.kfull[qst], qph)) return false;
      const bool last = qk == qn - 1;
      const uint64_t dk = dk0 + ((qst * kKVTile) >> 4);
      const uint64_t dqb = dq0 + ((qb * kQItem) >> 4);
      tc_fence_after();
      if (elect_one()) {
#pragma unroll
        for (int g = 0; g < kGroups; ++g) {
          const uint64_t dq = dqb + ((g * kQBytes) >> 4);
          const uint32_t d = tmem + g * 256 + sb * 64;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * 1024 + (kk & 3) * 32) >> 4;
            mma_f16(d, dq + off, dk + off, idesc_qk, kk > 0);
          }
          mma_commit(bars.sfull(g, sb));
        }
        mma_commit(&bars.kempty[qst]);       // both tiles' QKs of this chunk
        if (last) mma_commit(&bars.qempty[qb]);  // both tiles are done with the item's queries
      }
      __syncwarp();
      ++qc;
      if (++qst == kStages) {
        qst = 0;
        qph ^= 1;
      }
      if (++qk == qn) {
        qk = 0;
        qcur.advance();
        qn = qcur.valid() ? unpack_item(qcur.cur, TQ).nchunks : 0;
      }
      return true;
    };
    for (int i = 0; i < 2 && ok && qcur.valid(); ++i) ok = qk_pair(false);
    while (ok && pcur.valid()) {
      const int sb = pc & 1;
      static_assert(kGroups == 2, "the probe below covers two tiles");
      // one round trip probes everything this iteration needs (V of chunk pc, both
      // tiles' probabilities, K of chunk pc + 2); only what is not ready yet is waited for
      const uint32_t seen = __shfl_sync(0xffffffffu,
          mbar_test_wait4(&bars.vfull[pst], pph, bars.pfull(0, sb), (pc >> 1) & 1, bars.pfull(1, sb),
                          (pc >> 1) & 1, &bars.kfull[qst], qph), 0);
      if (!(seen & 1) && !wait_all(&bars.vfull[pst], pph)) break;
      const uint64_t dv = dv0 + ((pst * kKVTile) >> 4);
      const bool acc0 = pk > 0;
#pragma unroll
      for (int g = 0; g < kGroups; ++g) {
        if (!(seen & (2u << g)) && !wait_all(bars.pfull(g, sb), (pc >> 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (elect_one()) {
          const uint32_t pa = tmem + g * 256 + sb * 64;  // probabilities: [hi 8 | lo 8] columns per 16 keys
          const uint32_t od = tmem + g * 256 + 128;
#pragma unroll
          for (int kk = 0; kk < kKC / 16; ++kk) {
            const uint64_t bd = dv + ((kk * 2 * kGroup) >> 4);
            mma_f16_tmem_a(od, pa + kk * 16, bd, idesc_pv, acc0 || kk > 0);
            mma_f16_tmem_a(od, pa + kk * 16 + 8, bd, idesc_pv, true);
          }
          mma_commit(bars.pvdone(g, sb));
          if (g == kGroups - 1) mma_commit(&bars.vempty[pst]);  // every tile's PV of this chunk
        }
        __syncwarp();
      }
      if (!ok) break;
      ++pc;
      if (++pst == kStages) {
        pst = 0;
        pph ^= 1;
      }
      if (++pk == pn) {
        pk = 0;
        pcur.advance();
        pn = pcur.valid() ? unpack_item(pcur.cur, TQ).nchunks : 0;
      }
      if (qcur.valid()) ok = qk_pair((seen & 8u) != 0);
    }
    __syncwarp();
  } else {
    // ============================ softmax warpgroups ============================
    const int grp = warp / 4;                 // which tile of the pair
    const int t = threadIdx.x % 128;          // query row of the tile = TMEM lane
    const int wq = warp % 4;                  // lane quarter
    const int head = t / TQ, tok = t % TQ;    // head-major rows
    const uint32_t lane_base = tmem + grp * 256 + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t obuf = lane_base + 128;
    const bool neg_scale = p.scale_log2 < 0.f;
    const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
    const float2 mone2 = make_float2(-1.f, -1.f);
    int c = 0;
    bool ok = true;
    int prev_row = -1, prev_c = -1;
    float prev_l = 1.f;

    // Warp-uniform: has this tile's PV of chunk cc completed?
    auto pv_done = [&](int cc) -> bool {
      return __all_sync(0xffffffffu, wait_role(bars.pvdone(grp, cc & 1), (cc >> 1) & 1, abort_flag, p.err, p.wait_limit_ns));
    };
    // A finished item's output rows: O / l (O is final: its last PV was waited for).
    auto finish = [&](int row, float lsum) {
      tc_fence_after();
      const float inv = 1.f / lsum;
#pragma unroll
      for (int q = 0; q < D / 32; ++q) {
        float o[32];
        tmem_load32(obuf + q * 32, o);
        if (row >= 0) {
          if (p.out_f32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + static_cast<size_t>(row) * D + q * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv, o[4 * i + 3] * inv);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(p.out) + static_cast<size_t>(row) * D + q * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i)
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
      const bool row_valid = head < G && tok < it.ntok(grp);
      const int qpos = row_valid ? it.pos0 + grp * TQ + tok : it.last;  // padding rows act as the last token
      const int out_row = row_valid ? (it.qrow0 + grp * TQ + tok) * p.num_q_heads + it.g * G + head : -1;
      float m = 0.f, l = 0.f;  // max used for this row's probabilities, running row sum
      for (int k = 0; k < it.nchunks; ++k, ++c) {
        const int sb = c & 1;
        const uint32_t sbuf = lane_base + sb * 64;
        if (!__all_sync(0xffffffffu, wait_role(bars.sfull(grp, sb), (c >> 1) & 1, abort_flag, p.err, p.wait_limit_ns))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int kbase = k * kKC;
        const int lim = qpos - kbase;            // keys of the chunk past lim are masked
        const bool diagonal = lim < kKC - 1;     // only then does the mask cut this row
        // the row's 64 scores, held in registers for both passes
        float sv[64];
        tmem_load64(sbuf, sv);
        // pass 1: the row's chunk maximum of scale * score under the mask
        const float cm = (neg_scale ? chunk_extreme<true>(sv, diagonal, lim)
                                    : chunk_extreme<false>(sv, diagonal, lim)) * p.scale_log2;
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
        // O is read out (at an item's first chunk) or rescaled only after the PVs that
        // accumulate it have completed
        if (k == 0 && prev_c >= 0) {
          if (!pv_done(prev_c)) {
            ok = false;
            break;
          }
          finish(prev_row, prev_l);
          prev_c = -1;
        }
        if (k > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          if (!pv_done(c - 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int q = 0; q < D / 16; ++q) {
            float o[16];
            tmem_load16(obuf + q * 16, o);
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] *= alpha;
            tmem_store16(obuf + q * 16, o);
          }
        }
        // pass 2: probabilities as hi + lo parts, written over the 16 S columns they
        // came from: [hi of 16 keys | lo of 16 keys]
        float2 acc = make_float2(0.f, 0.f);
        const float2 nm2 = make_float2(-m, -m);
#pragma unroll
        for (int q = 0; q < kKC / 16; ++q) {
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float2 x = __ffma2_rn(make_float2(sv[q * 16 + 2 * i], sv[q * 16 + 2 * i + 1]), sc2, nm2);
            float p0 = exp2_approx(x.x), p1 = exp2_approx(x.y);
            if (diagonal) {
              p0 = q * 16 + 2 * i <= lim ? p0 : 0.f;
              p1 = q * 16 + 2 * i + 1 <= lim ? p1 : 0.f;
            }
            const float2 pr = make_float2(p0, p1);
            float h0, h1;
            w[i] = pack2_split<T>(p0, p1, h0, h1);                               // rounded pair
            const float2 lo = __ffma2_rn(make_float2(h0, h1), mone2, pr);       // exact remainders
            w[8 + i] = pack2<T>(lo.x, lo.y);
            acc = __fadd2_rn(acc, pr);
          }
          tmem_store16_words(sbuf + q * 16, w);
        }
        l += acc.x + acc.y;
        tmem_store_wait();
        tc_fence_before();
        // V rows past the pair's last position inside loaded blocks: zero them (a NaN
        // there would survive a zero weight).  Both groups write the same zeros.
        const int rows_needed = it.last + 1 - kbase;
        if (rows_needed < kKC) {  // warp-uniform; V of this chunk must have landed first
          if (!__all_sync(0xffffffffu, wait_role(&bars.vfull[c % kStages], (c / kStages) & 1, abort_flag, p.err, p.wait_limit_ns))) {
            ok = false;
            break;
          }
        }
        if (t < kKC && rows_needed < kKC) {
          const int rows_loaded = min(kKC, (rows_needed + p.block_size - 1) / p.block_size * p.block_size);
          if (t >= rows_needed && t < rows_loaded) {
            unsigned char* vrow = smem + kOffV + (c % kStages) * kKVTile + (t >> 3) * kGroup + (t & 7) * 128;
#pragma unroll
            for (int q = 0; q < 8 * L::kBlocks; ++q)  // 128 bytes per 64-column block, 1 KB apart
              reinterpret_cast<uint4*>(vrow + (q >> 3) * 1024)[q & 7] = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.pfull(grp, sb));
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
    // copies still in flight land before the CTA exits: the last chunk issued on each
    // stage (and the last query buffers) -- a phase already completed returns at once
    if (warp == kProducerWarp && lane == 0) {
      for (int c = max(0, *kissued_slot - kStages); c < *kissued_slot; ++c)
        if (!mbar_wait(&bars.kfull[c % kStages], (c / kStages) & 1)) break;
      for (int jj = max(0, *qissued_slot - kQBufs); jj < *qissued_slot; ++jj)
        if (!mbar_wait(&bars.qfull[jj % kQBufs], (jj / kQBufs) & 1)) break;
    }
    if (warp == kVWarp && lane == 0) {
      for (int c = max(0, *vissued_slot - kStages); c < *vissued_slot; ++c)
        if (!mbar_wait(&bars.vfull[c % kStages], (c / kStages) & 1)) break;
    }
    if (warp == kMmaWarp) {
      // every lane commits (the MMAs went out from whichever lane was elected; a lane
      // that issued none arrives at once), so the barrier completes only when all of
      // the warp's MMAs have
      if (lane == 0) {
        mbar_init(bars.drain, 32);
        fence_barrier_init();
      }
      __syncwarp();
      mma_commit(bars.drain);
      mbar_wait(bars.drain, 0);
      __syncwarp();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

// Work list: one entry per (sequence, KV head, pair of query tiles).  A sequence's
// entries are adjacent (head by head, pairs in order) so the CTAs working on them at
// the same time share its K/V through L2; sequences are ordered by chunk count,
// longest first (counting sort over sequences).
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
    if (n > 0) atomicAdd(&hist[min((L + kKC - 1) / kKC, kMaxBuckets - 1)], (n + span - 1) / span * H);
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
    if (n <= 0 || L < n || L > p.max_context_len) continue;
    const int pairs = (n + span - 1) / span;
    int pos = atomicAdd(&next[min((L + kKC - 1) / kKC, kMaxBuckets - 1)], pairs * H);
    for (int g = 0; g < H; ++g)
      for (int i = pairs - 1; i >= 0; --i) {  // longest pair first
        const int t0 = i * span;
        const int na = min(TQ, n - t0), nb = max(0, min(TQ, n - t0 - TQ));
        p.work_list[pos++] = make_int4(s, g | (na << 12) | (nb << 20), p.query_start[s] + t0, L - n + t0);
      }
  }
}

// Queries [tokens][heads][head_dim] seen as 3-D (head_dim, heads, tokens); a box is 8
// tokens x 64 dims of one head, landing as one swizzled 64-column block of an 8-row group.
bool make_query_map_uncached(CUtensorMap* m, const void* q, uint32_t heads, uint32_t tokens, bool bf16,
                             int head_dim) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t row = static_cast<cuuint64_t>(head_dim) * 2;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim), heads, tokens};
  cuuint64_t strides[2] = {row, static_cast<cuuint64_t>(heads) * row};
  cuuint32_t box[3] = {64, 1, 8};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(q),
            dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_query_map(CUtensorMap* m, const void* q, uint32_t heads, uint32_t tokens, bool bf16, int head_dim) {
  return cached_map(m, MapKey{q, tokens, heads, 4, bf16 ? 2 : 1, head_dim}, [&](CUtensorMap* out) {
    return make_query_map_uncached(out, q, heads, tokens, bf16, head_dim);
  });
}

template <typename T, int D>
cudaError_t launch_prefill_t(const PrefillArgs& args, int grid, cudaStream_t stream) {
  constexpr int smem = PfLayout<D>::kSmemBytes;
  static std::atomic<unsigned long long> configured{0};  // devices whose limit is raised
  cudaError_t e = ensure_smem_limit(prefill_tc_kernel<T, D>, smem, configured);
  if (e != cudaSuccess) return e;
  prefill_tc_kernel<T, D><<<grid, kThreads, smem, stream>>>(args);
  return cudaGetLastError();
}

}  // namespace

int prefill_tile_tokens(int group) { return 8 * (kRows / 8 / group); }

size_t prefill_max_items(int num_seqs, int num_query_tokens, int num_kv_heads, int group) {
  const int span = kGroups * prefill_tile_tokens(group);
  return (static_cast<size_t>(num_query_tokens) / span + num_seqs) * num_kv_heads;
}

cudaError_t launch_prefill_tc(const PrefillParams& p, int dtype, cudaStream_t stream) {
  if (p.num_kv_heads > 4095) return cudaErrorInvalidValue;  // packed into 12 bits of a list entry
  if (p.group < 1 || p.group > 16 || p.num_query_tokens <= 0) return cudaErrorInvalidValue;
  PrefillArgs args;
  args.p = p;
  const bool bf16 = dtype == PKV_BF16;
  const uint64_t pool_rows = static_cast<uint64_t>(p.num_blocks) * p.num_kv_heads * p.block_size;
  if (p.head_dim != 64 && p.head_dim != 128) return cudaErrorInvalidValue;
  if (!make_pool_map(&args.tk, p.k_cache, pool_rows, p.block_size, bf16, p.head_dim) ||
      !make_pool_map(&args.tv, p.v_cache, pool_rows, p.block_size, bf16, p.head_dim) ||
      !make_query_map(&args.tq, p.q, p.num_q_heads, p.num_query_tokens, bf16, p.head_dim))
    return cudaErrorInvalidValue;
  prefill_list_kernel<<<1, kListThreads, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const size_t items = prefill_max_items(p.num_seqs, p.num_query_tokens, p.num_kv_heads, p.group);
  const int grid = static_cast<int>(items < static_cast<size_t>(sms) ? items : sms);
  if (grid == 0) return cudaSuccess;
  if (p.head_dim == 64)
    return bf16 ? launch_prefill_t<__nv_bfloat16, 64>(args, grid, stream) : launch_prefill_t<__half, 64>(args, grid, stream);
  return bf16 ? launch_prefill_t<__nv_bfloat16, 128>(args, grid, stream) : launch_prefill_t<__half, 128>(args, grid, stream);
}

}  // namespace pkv
