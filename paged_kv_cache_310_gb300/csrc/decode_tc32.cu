// decode_tc32.cu -- tensor-core (tcgen05, kind::tf32) paged decode attention for f32
// caches, head_dim 64 or 128, up to 8 query heads per KV head.
//
// It computes the same as the other decode paths (note-023, Method/Concepts; "Paged
// Attention" glossary, paragraph 4 and the GQA paragraph): per sequence s, KV head g
// and query head h of g's group, softmax(scale * q_h . K_j) weighted sum of V_j over
// the sequence's tokens, token j in row j % bs of block block_tables[s][j / bs].
//
// Why tensor cores for f32: with G query heads per KV head each K/V element feeds 2G
// multiply-adds; at G = 8 that is the whole fp32 CUDA-core rate at HBM speed, while
// the two contractions per 128-token chunk are a few percent of the tensor cores.
//   S^T[128 tokens x 16] = K[128 x D] . [q | q_lo]^T       (QK, M = 128, N = 16)
//   O^T[D x 16]          = V^T[D x 128] . [p | p_lo]^T     (PV, M = 128, N = 16)
// A tf32 operand keeps 10 of fp32's 23 fraction bits; the tensor core drops the other
// 13 (truncation, measured on this GPU).  So every operand x is used twice, as x
// itself (read as trunc(x)) and as x_lo = x - trunc(x) (exact in fp32), and the
// products are summed over both: columns [0, 8) of B hold q (or p), columns [8, 16)
// their low parts, and the MMAs run once with A = K (V^T) and once with A = K_lo
// (V_lo^T), accumulating into the same 16 columns.  Summing column h and column 8 + h
// gives x.y up to the truncation of the low parts, about 2^-20 relative per product.
//
// Operand placement (tf32 operands in shared memory must be K-major on this GPU, and
// V^T would be M-major): QK reads the raw K straight from its landing slot (K-major,
// 128-byte swizzle, as TMA wrote it) and K_lo from tensor memory ([token lane] x [D
// columns]); PV reads V^T and V_lo^T from tensor memory ([dimension lane] x [32-token
// columns], four piece buffers = one whole chunk, so a chunk's V is converted while
// its softmax runs).  q | q_lo and p | p_lo are the B operands in shared memory,
// K-major with 128-byte swizzle.
//
// Persistent CTAs (one per SM) over the decode work list (items = (sequence, KV head,
// partition), sorted longest first, taken in snake order), 480 threads (608 from 4
// query heads per KV head):
//  * warp 8, producer of K: per 128-token chunk and 64-dimension unit, one lane per
//    physical block issues one tiled TMA load (4-D box: 32 columns x 8 rows x 2
//    column blocks x bs/8 row groups, 128-byte swizzle) into a ring of three 32 KB
//    units; a unit is free once the chunk's QK completed.  Blocks past the item's end
//    are loaded from outside the tensor (zeros).  Warp 9, producer of V: the same per
//    64-token stage (all D / 32 column blocks) into a 96 KB ring; a stage is free once
//    converted.
//  * warps 4-7 and a second set of four, converters (thread = TMEM lane of the warp's
//    lane quarter; each set takes half of the columns): an item's q into the B buffer
//    (q | q_lo); a chunk's K_lo (lane = token) into tensor memory; the chunk's V
//    transposed (lane = dimension) into tensor memory as V^T and V_lo^T in 32-token
//    pieces, zeroing the rows past the context end.
//  * warp 10, MMA: polls and one elected lane issues QK of the next chunk whose K_lo is
//    in tensor memory, and PV piece by piece once the chunk's probabilities are written.
//  * warps 0-3 (and 11-14 from G = 4) softmax, as in the 16-bit kernel: thread t reads
//    S row t, lazy online-softmax rescale, writes p and p_lo for its heads into the B
//    buffer, and (thread = dimension) accumulates O of the previous chunk.
#include <climits>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"
#include "tc_util.cuh"

namespace pkv {
namespace {

constexpr int kChunk = 128;     // tokens per chunk: M of QK
constexpr int kStageTok = 64;   // tokens per landing stage
constexpr int kPiece = 32;      // tokens per V^T piece in tensor memory (K of one PV group)
constexpr int kN = 16;          // MMA N: [x 0-7 | x_lo 0-7]
constexpr int kMaxG = 8;
constexpr int kConvWarps = 8;  // two per TMEM lane quarter
constexpr uint32_t kTmemCols = 512;

template <int GM>
struct Roles32 {
  static constexpr int kSplit = GM >= 4 ? 2 : 1;  // softmax warps per lane quarter
  static constexpr int kHeads = GM / kSplit;
  static constexpr int kSoftmaxThreads = 128 * kSplit;
  static constexpr int kThreads = kSoftmaxThreads + 32 * (kConvWarps + 3);
  static constexpr int kConv2 = 11 + 4 * (kSplit - 1);  // first warp of the second converter set
};
// warps: 0-3 softmax, 4-7 converters (first set), 8 K producer, 9 V producer, 10 MMA,
// then 11-14 softmax (from G = 4), then four more converters (second set)
constexpr int kWarpKProd = 8, kWarpVProd = 9, kWarpMma = 10;
constexpr int kVBufs = kChunk / kPiece;  // V^T piece buffers in tensor memory: one whole chunk

template <int D>
struct Layout32 {
  static constexpr int kBlocks = D / 32;                 // 128-byte column blocks of a row
  static constexpr int kGroupBytes = 8 * D * 4;          // 8 token rows
  // K lands in units of 128 tokens x 64 dimensions (a chunk has D / 64 of them), each
  // the A operand of QK for its dimensions; three units in a ring (1.5 chunks at D =
  // 128, 3 at 64).  V lands in 64-token stages, 96 KB of them.
  static constexpr int kKUnitBytes = kChunk * 64 * 4;    // 32 KB
  static constexpr int kKUnitsPerChunk = D / 64;
  static constexpr int kKSlots = 3;
  static constexpr int kKUnitGroupBytes = 8 * 64 * 4;   // 8 token rows of a unit: 2 KB
  static constexpr int kVStageBytes = kStageTok * D * 4;  // 32 KB at D = 128
  static constexpr int kVStages = 3 * 128 / D;           // 96 KB
  static constexpr int kQBytes = kN * D * 4;             // [q | q_lo] of one item
  static constexpr int kPBytes = kN * kChunk * 4;        // [p | p_lo] of one chunk
  static constexpr int kOffV = kKSlots * kKUnitBytes;
  static constexpr int kOffQ = kOffV + kVStages * kVStageBytes;
  static constexpr int kOffP = kOffQ + 2 * kQBytes;
  static constexpr int kOffBar = kOffP + 2 * kPBytes;
  // kfull, kempty per K slot; vfull, vempty per V stage; qready, qfree, sfull, sfree,
  // pfull, ofull, ofree pairs; ktfull, ktfree, vtready, drain
  static constexpr int kNumBars = 2 * kKSlots + 2 * kVStages + 7 * 2 + 4;
  static constexpr int kOffRedMax = kOffBar + kNumBars * 8;
  static constexpr int kOffRedL = kOffRedMax + 2 * 4 * kN * 4;
  static constexpr int kOffMTot = kOffRedL + 2 * 4 * kN * 4;
  static constexpr int kOffMisc = kOffMTot + 2 * kN * 4;
  static constexpr int kSmemBytes = kOffMisc + 64;
  // tensor memory columns: K_lo, S[2], O[2], V^T buffers (b: V^T at +64b, V_lo^T at +64b+32)
  static constexpr uint32_t kColKLo = 0, kColS = D, kColO = D + 2 * kN, kColV = D + 4 * kN;
  static_assert(kColV + kVBufs * 2 * kPiece <= kTmemCols, "tensor memory");
  static_assert(kOffV % 1024 == 0 && kOffQ % 1024 == 0 && kOffP % 1024 == 0 && kSmemBytes <= 227 * 1024,
                "layout");
};

struct Bars32 {
  uint64_t *kfull, *kempty, *vfull, *vempty;
  uint64_t *qready, *qfree, *sfull, *sfree, *pfull, *ofull, *ofree;
  uint64_t *ktfull, *ktfree, *vtready, *drain;
};

template <int D>
__device__ __forceinline__ Bars32 carve32(unsigned char* smem) {
  using L = Layout32<D>;
  uint64_t* b = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  Bars32 r;
  r.kfull = b;
  r.kempty = r.kfull + L::kKSlots;
  r.vfull = r.kempty + L::kKSlots;
  r.vempty = r.vfull + L::kVStages;
  r.qready = r.vempty + L::kVStages;
  r.qfree = r.qready + 2;
  r.sfull = r.qfree + 2;
  r.sfree = r.sfull + 2;
  r.pfull = r.sfree + 2;
  r.ofull = r.pfull + 2;
  r.ofree = r.ofull + 2;
  r.ktfull = r.ofree + 2;
  r.ktfree = r.ktfull + 1;
  r.vtready = r.ktfree + 1;
  r.drain = r.vtready + 1;
  return r;
}

struct Tc32Args {
  CUtensorMap tk;  // K pool, 4-D view: one box = one block's tile of one KV head
  CUtensorMap tv;  // V pool, same
  DecodeParams p;
};

// work-list entry {s, g, t0, ntok | nparts << 16}
struct Item32 {
  int s, g, part, t0, ntok, nchunks, nparts;
};

__device__ __forceinline__ Item32 unpack32(int4 e, int part_tokens) {
  Item32 it;
  it.s = e.x;
  it.g = e.y;
  it.t0 = e.z;
  it.ntok = e.w & 0xffff;
  it.nparts = static_cast<int>(static_cast<unsigned>(e.w) >> 16);
  it.part = it.t0 / part_tokens;
  it.nchunks = (it.ntok + kChunk - 1) / kChunk;
  return it;
}

// tokens of chunk k of an item, 64-token V stages it loads, 32-token pieces it has
__device__ __forceinline__ int chunk_rows(const Item32& it, int k) { return min(kChunk, it.ntok - k * kChunk); }
__device__ __forceinline__ int chunk_stages(int rows) { return (rows + kStageTok - 1) / kStageTok; }
__device__ __forceinline__ int chunk_pieces(int rows) { return (rows + kPiece - 1) / kPiece; }

// Byte offset of 16-byte column chunk j (of 128-byte column block cb) of row r inside a
// landing buffer: rows in 8-row groups, each [block][8 rows][128 B], 128-byte swizzle
// (the K-major layout of a tf32 A operand with 8-row groups kGroupBytes apart).
template <int D>
__device__ __forceinline__ uint32_t stage_off(int r, int cb, int j) {
  return (r >> 3) * Layout32<D>::kGroupBytes + cb * 1024 + (r & 7) * 128 + ((j ^ (r & 7)) << 4);
}

// Byte offset of element (row n, column c) of a K-major B buffer of kN rows and `cols`
// columns, 128-byte swizzle: [8-row group][32-column block][8 rows][128 B].
__device__ __forceinline__ uint32_t bmat_off(int n, int c, int cols) {
  return (n >> 3) * (cols / 32) * 1024 + (c >> 5) * 1024 + (n & 7) * 128 + ((((c & 31) >> 2) ^ (n & 7)) << 4) +
         ((c & 3) << 2);
}

// the part of x a tf32 operand drops (x minus x truncated to 10 fraction bits): exact
__device__ __forceinline__ float tf32_low(float x) { return x - __uint_as_float(__float_as_uint(x) & 0xffffe000u); }

// D[tmem] (+)= A . B of kind::tf32, A in shared memory (descriptor) or in TMEM.
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
      : "memory");
}
__device__ __forceinline__ void mma_tf32_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
      : "memory");
}

// instruction descriptor of kind::tf32, fp32 accumulation, both operands K-major
constexpr uint32_t idesc_tf32(uint32_t m, uint32_t n) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

// 32 consecutive 32-bit columns of this thread's TMEM lane (not waited).
__device__ __forceinline__ void tmem_store32_nowait(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]), "f"(v[8]),
      "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15]), "f"(v[16]),
      "f"(v[17]), "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]), "f"(v[24]),
      "f"(v[25]), "f"(v[26]), "f"(v[27]), "f"(v[28]), "f"(v[29]), "f"(v[30]), "f"(v[31])
      : "memory");
}

template <int D, int GM>
__global__ void __launch_bounds__(Roles32<GM>::kThreads, 1) decode_tc32_kernel(const __grid_constant__ Tc32Args a) {
  using L = Layout32<D>;
  using R = Roles32<GM>;
  constexpr int kKS = L::kKSlots, kVS = L::kVStages;
  extern __shared__ __align__(1024) unsigned char smem[];
  const DecodeParams& p = a.p;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const Bars32 bars = carve32<D>(smem);
  float* red_max = reinterpret_cast<float*>(smem + L::kOffRedMax);  // [2][4 quarters][kN]
  float* red_l = reinterpret_cast<float*>(smem + L::kOffRedL);      // [2][4 quarters][kN]
  float* red_mtot = reinterpret_cast<float*>(smem + L::kOffMTot);   // [2][kN]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 4);
  int* kissued_slot = reinterpret_cast<int*>(smem + L::kOffMisc + 8);   // K chunks issued
  int* vissued_slot = reinterpret_cast<int*>(smem + L::kOffMisc + 12);  // V stages issued
  const int G = p.group;
  const uint64_t lim = p.wait_limit_ns;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kKS; ++i) {
      mbar_init(&bars.kfull[i], 1);
      mbar_init(&bars.kempty[i], 1);  // the QK of the unit's chunk completed
    }
    for (int i = 0; i < kVS; ++i) {
      mbar_init(&bars.vfull[i], 1);
      mbar_init(&bars.vempty[i], kConvWarps);  // converted into tensor memory
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.qready[i], kConvWarps);
      mbar_init(&bars.qfree[i], 1);
      mbar_init(&bars.sfull[i], 1);
      mbar_init(&bars.sfree[i], 4 * R::kSplit);
      mbar_init(&bars.pfull[i], 4 * R::kSplit);
      mbar_init(&bars.ofull[i], 1);
      mbar_init(&bars.ofree[i], 4 * R::kSplit);
    }
    mbar_init(bars.ktfull, kConvWarps);
    mbar_init(bars.ktfree, 1);
    mbar_init(bars.vtready, kConvWarps);
    *abort_flag = 0;
    *kissued_slot = 0;
    *vissued_slot = 0;
    fence_barrier_init();
  }
  if (warp == kWarpMma) tmem_alloc(tmem_slot, kTmemCols);
  // rows of P no softmax thread writes (heads past a group of fewer than 8) read as 0
  for (int i = threadIdx.x; i < 2 * L::kPBytes / 16; i += R::kThreads)
    reinterpret_cast<uint4*>(smem + L::kOffP)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // launched as a programmatic dependent of the work-list kernel: the list, the pool
  // and q are read only after it (and what ran before it) completed
  grid_dependency_wait();
  const int num_items = *p.work_count;

  if (warp == kWarpKProd || warp == kWarpVProd) {
    // ============================ TMA producers ============================
    // K: units of 128 tokens x 64 dimensions (the A operand of QK); V: 64-token stages.
    const bool is_k = warp == kWarpKProd;
    const CUtensorMap* map = is_k ? &a.tk : &a.tv;
    if (lane == 0) prefetch_tensormap(map);
    uint64_t* full = is_k ? bars.kfull : bars.vfull;
    uint64_t* empty = is_k ? bars.kempty : bars.vempty;
    unsigned char* ring = smem + (is_k ? 0 : L::kOffV);
    const int ring_n = is_k ? kKS : kVS;
    const int unit_tok = is_k ? kChunk : kStageTok;
    const uint32_t unit_bytes = is_k ? L::kKUnitBytes : L::kVStageBytes;
    const int row_bytes = is_k ? 64 * 4 : D * 4;  // bytes a token row of a unit holds
    int* issued_slot = is_k ? kissued_slot : vissued_slot;
    const uint64_t pol = policy_evict_first();
    const int bs = p.block_size;
    const int blocks_per_unit = unit_tok / bs;
    const int oob_row = p.num_blocks * p.num_kv_heads * bs;  // first row outside the pool
    int u = 0;  // units (K chunks or V stages) issued so far
    bool ok = true;
    ItemCursor cur;
    for (cur.init(p.work_list, num_items); cur.valid() && ok; cur.advance()) {
      const Item32 it = unpack32(cur.cur, p.part_tokens);
      const int32_t* table = p.block_tables + static_cast<size_t>(it.s) * p.max_blocks_per_seq;
      for (int k = 0; k < it.nchunks && ok; ++k) {
        const int nunits = is_k ? L::kKUnitsPerChunk : chunk_stages(chunk_rows(it, k));
        for (int h = 0; h < nunits; ++h, ++u) {
          const int slot = u % ring_n;
          // K unit h: the chunk's tokens, dimensions 64 h ..; V stage h: tokens 64 h ..
          const int lb = (it.t0 + k * kChunk + (is_k ? 0 : h * kStageTok)) / bs + lane;  // this lane's block
          const bool live = lane < blocks_per_unit && lb * bs < it.t0 + it.ntok;
          int b = live ? (lb < p.max_blocks_per_seq ? table[lb] : -1) : 0;
          if (lane == 0) {
            ok = u < ring_n || wait_role(&empty[slot], ((u / ring_n) - 1) & 1, abort_flag, p.err, lim);
            if (ok) mbar_arrive_expect_tx(&full[slot], unit_bytes);
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          __syncwarp();
          if (lane < blocks_per_unit) {
            int row = oob_row;  // blocks past the item's end: zero-filled by the TMA unit
            if (live) {
              if (b < 0 || b >= p.num_blocks) {
                if (is_k) set_error(p.err, kErrIndex);
                b = 0;
              }
              row = (b * p.num_kv_heads + it.g) * bs;
            }
            tma_load_4d_zw(ring + slot * unit_bytes + lane * bs * row_bytes, map, is_k ? 2 * h : 0, row / 8,
                           &full[slot], pol);
          }
          if (lane == 0) *issued_slot = u + 1;
        }
      }
    }
  } else if ((warp >= 4 && warp < 8) || warp >= R::kConv2) {
    // ============================ converters ============================
    // Two warps per TMEM lane quarter: set ch = 0 or 1 takes half of each piece's tokens,
    // half of K's column blocks and half of q.
    const int quarter = warp & 3;
    const int ch = warp >= R::kConv2 ? 1 : 0;
    const int r = quarter * 32 + lane;  // TMEM lane: token row (K_lo) or dimension (V^T)
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    int kc = 0;           // chunks whose K_lo was written
    int vst = 0;          // V stages consumed
    int j = 0;            // items whose q was converted
    bool ok = true;
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, wait_role(bar, parity, abort_flag, p.err, lim));
    };
    // q of item `it` -> B buffer j & 1 as rows [q_h | q_lo_h], zero rows past the group
    auto convert_q = [&](const Item32& it) -> bool {
      const int qb = j & 1;
      if (j >= 2 && !wait(&bars.qfree[qb], ((j >> 1) - 1) & 1)) return false;
      unsigned char* qbuf = smem + L::kOffQ + qb * L::kQBytes;
      const float* qg = static_cast<const float*>(p.q) + (static_cast<size_t>(it.s) * p.num_q_heads + it.g * G) * D;
      for (int e = r + 128 * ch; e < kMaxG * D; e += 256) {
        const int h = e / D, d = e % D;
        const float x = h < G ? qg[h * D + d] : 0.f;
        *reinterpret_cast<float*>(qbuf + bmat_off(h, d, D)) = x;
        *reinterpret_cast<float*>(qbuf + bmat_off(kMaxG + h, d, D)) = tf32_low(x);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.qready[qb]);
      ++j;
      return true;
    };
    // K_lo of one chunk -> tensor memory, lane = token (the raw K stays in its slot,
    // where QK reads it as the other A operand)
    auto convert_k = [&]() -> bool {
      const int u0 = kc * L::kKUnitsPerChunk;  // the chunk's first K unit
      if (kc >= 1 && !wait(bars.ktfree, (kc - 1) & 1)) return false;
      for (int h = 0; h < L::kKUnitsPerChunk; ++h)
        if (!wait(&bars.kfull[(u0 + h) % kKS], ((u0 + h) / kKS) & 1)) return false;
      tc_fence_after();
#pragma unroll
      for (int cb = ch * L::kBlocks / 2; cb < (ch + 1) * L::kBlocks / 2; ++cb) {
        // column block cb: block cb % 2 of unit cb / 2 ([8-row group][2 blocks][8 rows][128 B])
        const unsigned char* src = smem + ((u0 + cb / 2) % kKS) * L::kKUnitBytes + (r >> 3) * L::kKUnitGroupBytes +
                                   (cb & 1) * 1024 + (r & 7) * 128;
        float lo[32];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const float4 v = *reinterpret_cast<const float4*>(src + ((jj ^ (r & 7)) << 4));
          lo[4 * jj] = tf32_low(v.x);
          lo[4 * jj + 1] = tf32_low(v.y);
          lo[4 * jj + 2] = tf32_low(v.z);
          lo[4 * jj + 3] = tf32_low(v.w);
        }
        tmem_store32_nowait(lane_base + L::kColKLo + 32 * cb, lo);
      }
      tmem_store_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.ktfull);
      ++kc;
      return true;
    };
    // V of one chunk -> tensor memory, lane = dimension, in one pass: V^T of piece pp
    // (32 tokens) at kColV + 64 pp, V_lo^T at kColV + 64 pp + 32, rows past the context
    // end as 0.  The buffers are free once the previous chunk's PV completed (its O is
    // ready); set ch converts pieces 2 ch and 2 ch + 1, which sit in landing stage ch.
    int vc = 0;  // chunks of V converted
    auto convert_v = [&](int rows) -> bool {
      const int nst = chunk_stages(rows), np = chunk_pieces(rows);
      if (vc >= 1 && !wait(&bars.ofull[(vc - 1) & 1], ((vc - 1) >> 1) & 1)) return false;
      for (int h = 0; h < nst; ++h)
        if (!wait(&bars.vfull[(vst + h) % kVS], ((vst + h) / kVS) & 1)) return false;
      tc_fence_after();
      if (r < D && 2 * ch < np) {  // warp-uniform
        const unsigned char* src = smem + L::kOffV + ((vst + ch) % kVS) * L::kVStageBytes;
        const int cb = r >> 5, jj = (r & 31) >> 2, e = (r & 3) << 2;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int pp = 2 * ch + q;
          if (pp < np) {
            float x[kPiece], lo[kPiece];
#pragma unroll
            for (int i = 0; i < kPiece; ++i) {
              const int t = pp * kPiece + i;  // token within the chunk (row t % 64 of stage ch)
              x[i] = t < rows ? *reinterpret_cast<const float*>(src + stage_off<D>(t % kStageTok, cb, jj) + e) : 0.f;
              lo[i] = tf32_low(x[i]);
            }
            tmem_store32_nowait(lane_base + L::kColV + 64 * pp, x);
            tmem_store32_nowait(lane_base + L::kColV + 64 * pp + 32, lo);
          }
        }
        tmem_store_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bars.vtready);
        for (int h = 0; h < nst; ++h) mbar_arrive(&bars.vempty[(vst + h) % kVS]);
      }
      vst += nst;
      ++vc;
      return true;
    };

    // Order: the V pieces of chunk c, then K_lo of chunk c + 1 (and q of its item).  K_lo
    // of chunk 0 goes first, so K_lo(c) is always one step ahead and QK(c) overlaps the
    // softmax of chunk c - 1; V(c) is converted as soon as PV(c - 1) frees the V^T
    // buffers rather than after K(c + 1) has landed (1-3 % faster than K first).
    ItemCursor cur, nxt;
    cur.init(p.work_list, num_items);
    nxt.init(p.work_list, num_items);
    int nk = 0;  // chunk of the `nxt` item whose K_lo is converted next
    auto next_k = [&]() -> bool {
      if (!nxt.valid()) return true;
      const Item32 it = unpack32(nxt.cur, p.part_tokens);
      if (nk == 0 && !convert_q(it)) return false;
      if (!convert_k()) return false;
      if (++nk == it.nchunks) {
        nk = 0;
        nxt.advance();
      }
      return true;
    };
    ok = next_k();
    for (; cur.valid() && ok; cur.advance()) {
      const Item32 it = unpack32(cur.cur, p.part_tokens);
      for (int k = 0; k < it.nchunks && ok; ++k) {
        ok = convert_v(chunk_rows(it, k));
        if (ok) ok = next_k();
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ============================ MMA issuer ============================
    constexpr uint32_t idesc = idesc_tf32(128, kN);
    const uint64_t dk0 = smem_desc(smem_addr(smem), 16, L::kKUnitGroupBytes, kLayoutSwizzle128);
    const uint64_t dq0 = smem_desc(smem_addr(smem + L::kOffQ), 16, L::kBlocks * 1024, kLayoutSwizzle128);
    const uint64_t dp0 = smem_desc(smem_addr(smem + L::kOffP), 16, (kChunk / 32) * 1024, kLayoutSwizzle128);
    ItemCursor qcur, pcur;
    qcur.init(p.work_list, num_items);
    pcur.init(p.work_list, num_items);
    int qk = 0, qj = 0, qc = 0;
    int qn = qcur.valid() ? unpack32(qcur.cur, p.part_tokens).nchunks : 0;
    int pk = 0, pc = 0;  // PV: chunk within its item, global chunk
    int pn = qn;
    int prows = pcur.valid() ? chunk_rows(unpack32(pcur.cur, p.part_tokens), 0) : 0;
    uint64_t idle_since = global_timer_ns();
    while (qcur.valid() || pc < qc) {
      bool progressed = false;
      const int sb = qc & 1, pb = pc & 1;
      // bit 0: K_lo of chunk qc in tensor memory (its raw K landed before), 1: S[qc & 1]
      // free, 2: P of chunk pc written, 3: V^T of chunk pc in tensor memory
      const uint32_t seen = __shfl_sync(0xffffffffu,
          mbar_test_wait4(bars.ktfull, qc & 1, &bars.sfree[sb], ((qc >> 1) - 1) & 1, &bars.pfull[pb],
                          (pc >> 1) & 1, bars.vtready, pc & 1), 0);
      if (pc < qc && (seen & 4) && (seen & 8) &&
          (pc < 2 || __all_sync(0xffffffffu, mbar_test_wait(&bars.ofree[pb], ((pc >> 1) - 1) & 1)))) {
        const int np = chunk_pieces(prows);
        tc_fence_after();
        if (elect_one()) {
          for (int pp = 0; pp < np; ++pp) {
            const uint64_t dp = dp0 + ((pb * L::kPBytes + pp * 1024) >> 4);
            const uint32_t vcol = tmem + L::kColV + 64 * pp;
#pragma unroll
            for (int kk = 0; kk < kPiece / 8; ++kk)
              mma_tf32_tmem_a(tmem + L::kColO + pb * kN, vcol + 8 * kk, dp + ((kk * 32) >> 4), idesc,
                              pp > 0 || kk > 0);
#pragma unroll
            for (int kk = 0; kk < kPiece / 8; ++kk)
              mma_tf32_tmem_a(tmem + L::kColO + pb * kN, vcol + 32 + 8 * kk, dp + ((kk * 32) >> 4), idesc, true);
          }
          mma_commit(&bars.ofull[pb]);  // also frees the V^T buffers for the next chunk
        }
        __syncwarp();
        ++pc;
        if (++pk == pn) {
          pk = 0;
          pcur.advance();
          pn = pcur.valid() ? unpack32(pcur.cur, p.part_tokens).nchunks : 0;
        }
        prows = pcur.valid() ? chunk_rows(unpack32(pcur.cur, p.part_tokens), pk) : 0;
        progressed = true;
      }
      if (qcur.valid() && (seen & 1) && (qc < 2 || (seen & 2)) &&
          (qk > 0 || __all_sync(0xffffffffu, mbar_test_wait(&bars.qready[qj & 1], (qj >> 1) & 1)))) {
        const int u0 = qc * L::kKUnitsPerChunk;  // the chunk's first K unit
        const uint64_t dq = dq0 + (((qj & 1) * L::kQBytes) >> 4);
        const bool last = qk == qn - 1;
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 8; ++kk) {
            // dimensions 8 kk ..: unit kk / 8, its column block (kk / 4) % 2, 32 bytes per step
            const uint32_t ko = (((u0 + kk / 8) % kKS) * L::kKUnitBytes + ((kk >> 2) & 1) * 1024 + (kk & 3) * 32) >> 4;
            const uint32_t qo = ((kk >> 2) * 1024 + (kk & 3) * 32) >> 4;
            mma_tf32(tmem + L::kColS + sb * kN, dk0 + ko, dq + qo, idesc, kk > 0);
          }
#pragma unroll
          for (int kk = 0; kk < D / 8; ++kk) {
            const uint32_t qo = ((kk >> 2) * 1024 + (kk & 3) * 32) >> 4;
            mma_tf32_tmem_a(tmem + L::kColS + sb * kN, tmem + L::kColKLo + 8 * kk, dq + qo, idesc, true);
          }
          mma_commit(&bars.sfull[sb]);
          mma_commit(bars.ktfree);
          for (int h = 0; h < L::kKUnitsPerChunk; ++h) mma_commit(&bars.kempty[(u0 + h) % kKS]);
          if (last) mma_commit(&bars.qfree[qj & 1]);
        }
        __syncwarp();
        ++qc;
        if (++qk == qn) {
          qk = 0;
          ++qj;
          qcur.advance();
          qn = qcur.valid() ? unpack32(qcur.cur, p.part_tokens).nchunks : 0;
        }
        progressed = true;
      }
      if (progressed) {
        idle_since = global_timer_ns();
      } else {
        if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
        if (__any_sync(0xffffffffu, global_timer_ns() - idle_since > lim)) {
          if (lane == 0) {
            *abort_flag = 1;
            set_error(p.err, kErrTimeout);
          }
          break;
        }
      }
    }
    __syncwarp();
  } else {
    // ============================ softmax warps ============================
    constexpr int HG = R::kHeads;
    constexpr int NS = R::kSoftmaxThreads;
    const int quarter = warp & 3;
    const int h0 = warp >= 11 ? HG : 0;  // the second warp of a quarter takes the upper heads
    const int t = quarter * 32 + lane;   // TMEM lane: token of S, dimension of O
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    float m[HG], lp[HG], alpha[HG], alpha_pend[HG], acc[HG];
#pragma unroll
    for (int h = 0; h < HG; ++h) {
      m[h] = -INFINITY; lp[h] = 0.f; alpha[h] = 0.f; alpha_pend[h] = 0.f; acc[h] = 0.f;
    }
    int pend_s = 0, pend_g = 0, pend_part = 0, pend_nparts = 0;
    bool pend_first = false, pend_last = false, pend_keep = false;
    int c = 0;
    bool ok = true;

    // reads columns [col + h0, col + h0 + HG) and the same 8 further on (the low parts)
    auto load_pair = [&](uint32_t col, float* x, float* xlo) {
      if (HG <= 4) {
        float a4[4], b4[4];
        tmem_load4x2(lane_base + col + (h0 & ~3), lane_base + col + 8 + (h0 & ~3), a4, b4);
#pragma unroll
        for (int h = 0; h < HG; ++h) {
          x[h] = (h0 & 2) ? a4[(2 + h) & 3] : a4[h];
          xlo[h] = (h0 & 2) ? b4[(2 + h) & 3] : b4[h];
        }
      } else {
        tmem_load8x2(lane_base + col + h0, lane_base + col + 8 + h0, x, xlo);
      }
    };

    auto consume = [&](int cp) -> bool {
      const int pb = cp & 1;
      if (!__all_sync(0xffffffffu, wait_role(&bars.ofull[pb], (cp >> 1) & 1, abort_flag, p.err, lim)))
        return false;
      tc_fence_after();
      float o[HG], olo[HG];
      load_pair(L::kColO + pb * kN, o, olo);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.ofree[pb]);
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        const float v = o[h] + olo[h];
        acc[h] = pend_first ? v : pend_keep ? acc[h] + v : fmaf(acc[h], alpha_pend[h], v);
      }
      if (pend_last && t < D) {
        const float* rl = red_l + (cp & 1) * 4 * kN + h0;
        const size_t row0 = static_cast<size_t>(pend_s) * p.num_q_heads + pend_g * G + h0;
#pragma unroll
        for (int h = 0; h < HG; ++h) {
          if (h0 + h < G) {
            const float l = (rl[h] + rl[kN + h]) + (rl[2 * kN + h] + rl[3 * kN + h]);
            const size_t row = row0 + h;
            if (pend_nparts == 1) {
              static_cast<float*>(p.out)[row * D + t] = acc[h] / l;
            } else {
              const size_t k = row * p.max_parts + pend_part;
              p.ws_o[k * D + t] = acc[h];
              if (t == 0) {
                p.ws_ml[2 * k] = red_mtot[(cp & 1) * kN + h0 + h];
                p.ws_ml[2 * k + 1] = l;
              }
            }
          }
        }
      }
      return true;
    };

    bool prev_ok = true;
    ItemCursor cur;
    for (cur.init(p.work_list, num_items); cur.valid() && ok; cur.advance()) {
      const Item32 it = unpack32(cur.cur, p.part_tokens);
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        m[h] = h0 + h < G ? -INFINITY : INFINITY;  // padded heads: probabilities 0
        lp[h] = 0.f;
      }
      for (int k = 0; k < it.nchunks; ++k, ++c) {
        const int sb = c & 1;
        const bool wok = __all_sync(0xffffffffu, wait_role(&bars.sfull[sb], (c >> 1) & 1, abort_flag, p.err, lim));
        float sv[HG];
        if (wok) {
          tc_fence_after();
          float shi[HG], slo[HG];
          load_pair(L::kColS + sb * kN, shi, slo);
#pragma unroll
          for (int h = 0; h < HG; ++h) sv[h] = shi[h] + slo[h];
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars.sfree[sb]);
        }
        const int rows_valid = chunk_rows(it, k);
        const bool valid = wok && t < rows_valid;
        constexpr float kSlack = 8.f;  // lazy rescale: the running max moves only past 2^8
        float x[HG], pe[HG];
        float excess = -INFINITY;
#pragma unroll
        for (int h = 0; h < HG; ++h) {
          x[h] = valid ? fmaf(sv[h], p.scale_log2, -m[h]) : -INFINITY;
          excess = fmaxf(excess, x[h]);
        }
        const bool keep = named_barrier_and(1, NS, wok && prev_ok && !(excess > kSlack));
        if (keep) {
#pragma unroll
          for (int h = 0; h < HG; ++h) {
            pe[h] = exp2_approx(x[h]);
            lp[h] += pe[h];
          }
        } else {
#pragma unroll
          for (int h = 0; h < HG; ++h) {
            sv[h] = valid ? sv[h] * p.scale_log2 : -INFINITY;
            const float v = warp_max(sv[h]);
            if (lane == 0) red_max[(sb * 4 + quarter) * kN + h0 + h] = v;
          }
          if (!named_barrier_and(1, NS, wok && prev_ok)) {
            ok = false;
            break;
          }
#pragma unroll
          for (int h = 0; h < HG; ++h) {
            const float* rm = red_max + sb * 4 * kN + h0 + h;
            const float mn = fmaxf(m[h], fmaxf(fmaxf(rm[0], rm[kN]), fmaxf(rm[2 * kN], rm[3 * kN])));
            alpha[h] = exp2_approx(m[h] - mn);
            m[h] = mn;
            pe[h] = exp2_approx(sv[h] - mn);
            lp[h] = fmaf(lp[h], alpha[h], pe[h]);
          }
        }
        // B rows h (p) and 8 + h (p_lo) of token column t
        unsigned char* pbuf = smem + L::kOffP + sb * L::kPBytes;
#pragma unroll
        for (int h = 0; h < HG; ++h) {
          *reinterpret_cast<float*>(pbuf + bmat_off(h0 + h, t, kChunk)) = pe[h];
          *reinterpret_cast<float*>(pbuf + bmat_off(kMaxG + h0 + h, t, kChunk)) = tf32_low(pe[h]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.pfull[sb]);
        const bool last = k == it.nchunks - 1;
        if (last) {
          const float lsum = warp_sum_scatter<HG>(lp, lane);
          if ((lane & (32 / HG - 1)) == 0)
            red_l[((c & 1) * 4 + quarter) * kN + h0 + warp_sum_index<HG>(lane)] = lsum;
          if (t == 0) {
#pragma unroll
            for (int h = 0; h < HG; ++h) red_mtot[(c & 1) * kN + h0 + h] = m[h];
          }
          named_barrier_sync(1, NS);
        }
        if (c >= 1) prev_ok = consume(c - 1);
        if (!keep) {
#pragma unroll
          for (int h = 0; h < HG; ++h) alpha_pend[h] = alpha[h];
        }
        pend_keep = keep;
        pend_first = k == 0;
        pend_last = last;
        pend_s = it.s;
        pend_g = it.g;
        pend_part = it.part;
        pend_nparts = it.nparts;
      }
    }
    if (ok && prev_ok && c >= 1) consume(c - 1);
    __syncwarp();
  }

  // ---------------- teardown ----------------
  __syncthreads();
  if (*abort_flag) {
    // a wait ran out: copies and MMAs still in flight finish (bounded) before the CTA
    // leaves; the last stage issued on each ring slot is waited (a completed phase
    // returns at once)
    if ((warp == kWarpKProd || warp == kWarpVProd) && lane == 0) {
      uint64_t* full = warp == kWarpKProd ? bars.kfull : bars.vfull;
      const int n = warp == kWarpKProd ? kKS : kVS;
      const int issued = warp == kWarpKProd ? *kissued_slot : *vissued_slot;
      for (int s = max(0, issued - n); s < issued; ++s)
        if (!mbar_wait(&full[s % n], (s / n) & 1)) break;
    }
    if (warp == kWarpMma) {
      if (lane == 0) {
        mbar_init(bars.drain, 32);
        fence_barrier_init();
      }
      __syncwarp();
      mma_commit(bars.drain);  // every lane: whichever was elected issued the MMAs
      mbar_wait(bars.drain, 0);
      __syncwarp();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem, kTmemCols);
}

// f32 pool rows of head_dim elements seen as 4-D (32 columns, 8 rows, D/32 column
// blocks, 8-row groups), byte strides (row, 128, 8 rows); a box of (32, 8, D/32, bs/8)
// is one block's tile of one KV head, landing as [group][block][8 rows][128 B].
bool make_pool_map32_uncached(CUtensorMap* m, const void* base, uint64_t rows, uint32_t block_size,
                              int head_dim, uint32_t box_blocks) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || rows % 8 || (head_dim != 64 && head_dim != 128)) return false;
  const cuuint64_t row_bytes = static_cast<cuuint64_t>(head_dim) * 4, blocks = head_dim / 32;
  cuuint64_t dims[4] = {32, 8, blocks, rows / 8};
  cuuint64_t strides[3] = {row_bytes, 128, 8 * row_bytes};
  cuuint32_t box[4] = {32, 8, box_blocks, block_size / 8};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_pool_map32(CUtensorMap* m, const void* base, uint64_t rows, uint32_t block_size, int head_dim,
                     uint32_t box_blocks) {
  return cached_map(m, MapKey{base, rows, block_size, 3 + 16 * static_cast<int>(box_blocks), 0, head_dim},
                    [&](CUtensorMap* out) {
                      return make_pool_map32_uncached(out, base, rows, block_size, head_dim, box_blocks);
                    });
}

template <int D, int GM>
cudaError_t launch32_t(const Tc32Args& args, int grid, cudaStream_t stream) {
  constexpr int smem = Layout32<D>::kSmemBytes;
  static std::atomic<unsigned long long> configured{0};  // devices whose limit is raised
  cudaError_t e = ensure_smem_limit(decode_tc32_kernel<D, GM>, smem, configured);
  if (e != cudaSuccess) return e;
  return launch_dependent(decode_tc32_kernel<D, GM>, grid, Roles32<GM>::kThreads, smem, stream, args);
}

template <int D>
cudaError_t launch32_g(const Tc32Args& args, int grid, cudaStream_t stream) {
  const int G = args.p.group;
  if (G <= 1) return launch32_t<D, 1>(args, grid, stream);
  if (G <= 2) return launch32_t<D, 2>(args, grid, stream);
  if (G <= 4) return launch32_t<D, 4>(args, grid, stream);
  return launch32_t<D, 8>(args, grid, stream);
}

}  // namespace

cudaError_t launch_decode_tc32(const DecodeParams& p, int grid, cudaStream_t stream) {
  if (p.group > kMaxG) return cudaErrorInvalidValue;
  Tc32Args args;
  args.p = p;
  const uint64_t pool_rows = static_cast<uint64_t>(p.num_blocks) * p.num_kv_heads * p.block_size;
  if (!make_pool_map32(&args.tk, p.k_cache, pool_rows, p.block_size, p.head_dim, 2) ||
      !make_pool_map32(&args.tv, p.v_cache, pool_rows, p.block_size, p.head_dim, p.head_dim / 32))
    return cudaErrorInvalidValue;
  return p.head_dim == 64 ? launch32_g<64>(args, grid, stream) : launch32_g<128>(args, grid, stream);
}

}  // namespace pkv
