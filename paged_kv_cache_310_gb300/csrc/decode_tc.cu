// decode_tc.cu -- tensor-core (tcgen05) paged decode attention for f16/bf16 caches,
// head_dim 64 or 128, up to 16 query heads per KV head.
//
// What it computes is the same as the CUDA-core path (note-023, Method/Concepts;
// "Paged Attention" glossary, paragraph 4 and the GQA paragraph): per sequence s, KV
// head g and each query head h of g's group, softmax(scale * q_h . K_j) weighted sum
// of V_j over the tokens j of s, token j read from row j % bs of physical block
// block_tables[s][j / bs].
//
// Why tensor cores: with G query heads per KV head every K/V element feeds 2G
// multiply-adds.  At G = 8 streaming K/V at HBM speed needs ~64 TFLOP/s, the whole
// fp32 CUDA-core rate; as two small dense contractions per 128-token chunk it is a
// few percent of the tensor cores:
//   S^T[128 tokens x 16] = K[128 x D dims] . Q^T[D x 16]          (QK, M=128 N=16)
//   O^T[D dims x N]      = V^T[D dims x 128 tokens] . P^T[128 x N] (PV, M=128)
// The query heads of a group are the N dimension of QK (padded to 16; 32 for two
// paired heads' groups of 9 to 16).  PV's columns hold each head's probabilities twice,
// as a rounded part and its remainder (16 columns up to 8 heads, twice the S columns
// beyond).  At D = 64 two KV heads share an item where they pair up (see kPair);
// otherwise one PV tile of M = 128 rows covers the chunk's two 64-token halves (see
// PvGeom), so PV reads each V element once.
// PV accumulates an item's chunks in tensor memory (one O buffer per item, two
// buffers); the softmax warps read O once per item.
//
// Persistent CTAs (one per SM) over a work list of items = (partition, sequence, KV
// head, or at D = 64 a pair of KV heads where they pair up: see kPair) that
// work_list_kernel sorts longest first; with head_dim-128 operands each CTA claims its
// next item with a global atomic and hands it to its other roles through a
// shared-memory ring, at D = 64 unpaired the CTAs take the items in a fixed snake
// order (see kClaimItems).
// The kernel is launched as a programmatic dependent of the list kernel.  224 threads
// (352 from 4 query heads per KV head, 608 at 16) in five roles:
//  * warp 4, producer of Q and K (and, with head_dim-128 operands, the item claims):
//    per 128-token chunk, one lane per physical block reads the block id (before
//    waiting for a free stage, hiding its latency) and issues one tiled TMA load of the
//    block's K tile for this KV head (4-D box, 128-byte swizzle) into a K ring (3
//    stages of 32 KB at D = 128, 6 of 16 KB at D = 64; 2 of 32 KB with 32 S columns,
//    see TcLayout); blocks past the item's end are loaded from outside the tensor,
//    which the TMA unit fills with zeros.  It also loads the item's query rows.
//  * warp 6, producer of V: the same for V tiles into a 96 KB V ring.  The
//    rings are separate so that a K stage is reused as soon as its chunk's QK
//    completes, long before the chunk's V is done with: more of the rings stays in
//    flight, and the kernel is bound by bytes in flight.
//  * warp 5, MMA: the whole warp polls (one batched probe of five barriers per round)
//    and an elected lane issues PV for the oldest chunk whose probabilities are in
//    shared memory, or QK for the next chunk into S[c%2] (TMEM) once its K landed;
//    commits release the ring stages and the P buffers and signal the softmax warps.
//  * warps 0-3, and from G = 4 also warps 7-10 (from 16, 7-18), softmax (thread t = TMEM
//    lane t; a warp reads the lane quarter of its index mod 4, so with eight warps two
//    share each quarter and take half of the heads each): read S row t (token t, its
//    heads), vote on whether any score exceeds its head's running max by more than 2^8
//    (if so, chunk max across the 128 tokens by a warp reduction + shared memory and
//    an online-softmax rescale), probabilities split into two parts rounded to the
//    cache dtype (hi = round(p), lo = round(p - hi)) into P^T (shared memory).  When
//    the running max moves after an item's first chunk, the O accumulated so far is
//    multiplied by the factor before that chunk's PV: the MMA warp, seeing the
//    chunk's flag, waits for its earlier MMAs to complete and for the softmax warps'
//    rescale of O in tensor memory (rare: the max moves by more than 2^8).  After an
//    item's last PV the softmax warps read O row t (dimension t), add its hi and lo
//    columns and write the output (or the partition's unnormalised O, max and sum),
//    one chunk later so that the wait overlaps the next item's first chunk.
//  Rows of the last block past the context end hold real cache data; the softmax
//  warps zero those V rows in shared memory before PV (a NaN there would survive a
//  zero weight).
#include <climits>
#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"
#include "tc_util.cuh"

namespace pkv {
namespace {

constexpr int kChunk = 128;                    // tokens per MMA tile (M of QK)
constexpr int kMaxGroup = 16;                  // query heads per KV head on this path
// QK's N (S columns): 16, the query heads of a group padded; 32 for paired heads with
// 16 query heads per KV head (GM = 32: the two heads' groups side by side)
template <int GM>
constexpr int kNCols = GM <= 16 ? 16 : 32;
// P^T holds each probability as two rounded parts, hi = round(p) and
// lo = round(p - hi), as separate groups of 8 columns: the PV MMA then sums
// hi + lo in fp32, so rounding p to 16 bits costs about 2^-17 relative instead of
// 2^-9.  Up to 8 heads: [hi 0-7][lo 0-7] (16 columns, the columns are there anyway);
// up to 16: [hi 0-7][hi 8-15][lo 0-7][lo 8-15] (32 columns).

// PV geometry.  At D = 128, PV is O^T[128 dims x NP] = V^T . P^T over the chunk's
// 128 tokens (8 MMAs of K = 16) and P^T's column groups hold all 128 tokens.  At
// D = 64 the chunk's two 64-token halves share one M = 128 tile: rows 0-63 of A are
// dimensions 0-63 of tokens k..k+15 and rows 64-127 the same dimensions of tokens
// 64+k..64+k+15 (the descriptor's M-block offset is 64 tokens); P^T holds each half
// in its own column groups (64 tokens each), so N = 2 NP and 4 MMAs cover the chunk.
// Rows 0-63 x columns [0, NP) then hold the first half's sums, rows 64-127 x
// [NP, 2 NP) the second's, and the two other blocks cross terms that nobody reads.
// Without this, a 64-row V^T would be read twice per MMA (twice the shared-memory
// operand traffic, which is what paces the tensor pipe at these small N).
template <int D, int GM>
struct PvGeom {
  static constexpr bool kHalves = D == 64;
  static constexpr int kN = kNCols<GM>;
  static constexpr int kNP = GM <= 8 ? 16 : 2 * kN;      // P columns: heads' hi, then lo parts
  static constexpr int kNO = kHalves ? 2 * kNP : kNP;    // N of PV: O columns per buffer
  static constexpr int kPTok = kHalves ? 64 : kChunk;    // tokens per P column group
  static constexpr int kPGroupBytes = kPTok * 16;
  static constexpr int kSteps = kPTok / 16;              // PV MMAs per chunk
  // one P buffer: up to 2 kN / 8 groups of 8 columns x 128 tokens (8 or 16 KB)
  static constexpr int kPBytes = 4 * kChunk * kN;
  // tensor memory: S[2] at 0 and kN, O[2] at 2 kN and 2 kN + kNO
  static constexpr uint32_t kTmemCols = 2 * kN + 2 * kNO <= 128 ? 128 : 256;
  static_assert(kNP / 8 * (kHalves ? 2 : 1) * kPGroupBytes <= kPBytes, "P buffer");
  static_assert(2 * kN + 2 * kNO <= 256, "tensor memory");
};

// Roles: warps 0-3 softmax, 4 producer of Q and K, 5 MMA, 6 producer of V, and from
// 4 query heads per KV head warps 7-10 softmax too (from 16, warps 7-18): a warp
// reads the TMEM lane quarter of its index mod 4, so two (four) warps share each
// quarter (each 32 tokens) and take half (a quarter) of the heads each, which divides
// the softmax work per thread.
template <int GM>
struct TcRoles {
  // softmax warps per lane quarter (four at 16 heads: +2.5 % at head_dim 64 over two)
  static constexpr int kSplit = GM >= 16 ? 4 : GM >= 4 ? 2 : 1;  // 32 columns: 8 heads a thread
  static constexpr int kHeads = GM / kSplit;          // query heads per softmax thread
  static constexpr int kSoftmaxThreads = 128 * kSplit;
  static constexpr int kThreads = kSoftmaxThreads + 96;
};

// Claimed items (head_dim-128 operands: head_dim 128, and paired heads at 64): the Q/K
// producer of a CTA takes the next entry of the sorted list with a global atomic as it
// runs out of its current item, so the longest items go first and whichever CTA gets
// free takes the next (measured with a fixed snake order: per-CTA chunk counts 113-124
// and per-SM speeds within about 5 % left the last CTA 15-22 us behind the first).  The
// claimed entries reach the other roles through a ring of kItemRing slots in shared
// memory.
constexpr int kItemRing = 8;
// At head_dim 128 claiming measured 3-4 % faster than the fixed snake order on the
// 7B-like, GQA-70B-like and long-context workloads and 1-2 % on the shared-prefix one.
// At head_dim 64 with one head per item it measured slower in every form tried (claims
// early or late, items read ahead, block ids read ahead, head-major list order:
// 0.73-0.80 against 0.76-0.83 of the copy bandwidth), so the fixed order stays there.
// The template argument is the operand width (128 for paired heads).
template <int D>
constexpr bool kClaimItems = D == 128;

// Paired heads (head_dim 64, an even number of KV heads): a work item covers KV heads
// 2i and 2i + 1.  In the pool their tiles of a block are adjacent, so one TMA box lands
// row r of both as one 256-byte operand row (head 2i's 64 dimensions as column block 0,
// head 2i + 1's as block 1), the head_dim-128 shared-memory layout, and the item runs
// the head_dim-128 pipeline with 32 KB chunks.  QK's query operand is block diagonal:
// the first half of the S columns (8 up to 8 query heads per KV head, else 16: GM = 16
// or 32) holds the first head's query rows in dimension block 0 (zeros in block 1), the
// second half the second head's in block 1, so each S column sees its own head's K
// only.  PV computes O^T = V^T . P^T over all 128 rows; rows 0-63 (the first head's
// dimensions) are read in the first half of the columns and rows 64-127 in the second,
// the other two blocks are cross terms nobody reads.  With 16 KB chunks of one head the
// per-chunk costs (barrier round trips, the softmax pass, item changes) weigh twice as
// much per byte.

__device__ __forceinline__ bool item_valid(int4 e) { return (e.w & 0xffff) != 0; }  // ntok 0 = end

// Shared-memory layout for head_dim D (64 or 128).  A chunk's K (and V) sits as
// [8-row group][64-column block][8 rows] of 128-byte rows, 128-byte swizzled: the
// canonical K-major layout for the QK A operand (8-row groups kGroupBytes apart,
// column blocks 1 KB apart) and the MN-major layout for the PV A operand V^T (8-token
// groups kGroupBytes apart, 64-dimension blocks 1 KB apart), and one 4-D TMA box fills
// a whole block.  K and V have separate rings: a K stage is free once the chunk's QK
// completed, long before its V (needed until PV completes), so more of the rings stays
// in flight; each ring holds 96 KB whatever D is, except that with 32 S columns the
// doubled query and probability buffers take one K stage's room (64 KB of K: a K stage
// is held only until its QK completes, a V stage until PV; two V stages measured 1-3 %
// slower at 16 query heads per KV head).
template <int D, int GM>
struct TcLayout {
  static constexpr int kN = kNCols<GM>;
  static constexpr int kQHalfBytes = kN * 128;           // the query rows x one 64-dimension block
  static constexpr int kBlocks = D / 64;                 // 64-column blocks of a row
  static constexpr int kGroupBytes = 8 * D * 2;          // one 8-row group: all its blocks
  static constexpr int kTileBytes = kChunk * D * 2;      // K or V of one chunk: 16 or 32 KB
  static constexpr int kKStages = (kN == 32 ? 2 : 3) * 128 / D;  // K ring
  static constexpr int kVStages = 3 * 128 / D;                   // V ring
  static constexpr int kQBytes = kBlocks * kQHalfBytes;  // the item's query rows
  static constexpr int kPBytes = PvGeom<D, GM>::kPBytes;
  static constexpr int kOffV = kKStages * kTileBytes;
  static constexpr int kOffQ = kOffV + kVStages * kTileBytes;
  static constexpr int kOffP = kOffQ + 2 * kQBytes;
  static constexpr int kOffBar = kOffP + 2 * kPBytes;
  // rings (K, V: full, empty), 8 pairs, rescale handshake (2), drain, item ring
  static constexpr int kNumBars = 2 * kKStages + 2 * kVStages + 8 * 2 + 3 + 2 * kItemRing;
  static constexpr int kOffRedMax = kOffBar + kNumBars * 8;
  static constexpr int kOffRedL = kOffRedMax + 2 * 4 * kN * 4;  // [2 item slots][4 warps][kN]
  static constexpr int kOffMTot = kOffRedL + 2 * 4 * kN * 4;    // [2 item slots][kN]
  static constexpr int kOffAlpha = kOffMTot + 2 * kN * 4;       // [kN] rescale factors
  // D = 64: the second half's O sums, handed to the threads of the first half's rows
  static constexpr int kOffXfer = kOffAlpha + kN * 4;           // [64 dims][kN]
  static constexpr int kOffMisc = kOffXfer + (D == 64 ? 64 * kN * 4 : 0);
  static constexpr int kOffRing = (kOffMisc + 64 + 15) / 16 * 16;  // [kItemRing] work-list entries
  static constexpr int kSmemBytes = kOffRing + kItemRing * 16;
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  static_assert(kOffQ % 1024 == 0 && kSmemBytes <= 227 * 1024, "layout");
};

struct Bars {
  uint64_t* kfull;  // [stages] K of a chunk landed (TMA tx)
  uint64_t* kempty; // [stages] the chunk's QK done
  uint64_t* vfull;  // [stages] V of a chunk landed
  uint64_t* vempty; // [stages] the chunk's PV done
  uint64_t* qfull;  // [2] query tile landed
  uint64_t* qempty; // [2] QK MMAs of that item done
  uint64_t* sfull;  // [2] S ready
  uint64_t* sfree;  // [2] S read by the softmax warps
  uint64_t* pfull;  // [2] P written
  uint64_t* pfree;  // [2] the chunk's PV done: P buffer free
  uint64_t* ofull;  // [2] an item's O complete (its last PV done)
  uint64_t* ofree;  // [2] an item's O written out
  uint64_t* cdrain; // every MMA issued before a rescale completed
  uint64_t* cdone;  // O rescaled by the softmax warps
  uint64_t* drain;  // teardown after an abort
  uint64_t* ifull;  // [kItemRing] slot written by the producer
  uint64_t* iempty; // [kItemRing] slot read by every other role
};

template <int D, int GM>
__device__ __forceinline__ Bars carve_bars(unsigned char* smem) {
  using L = TcLayout<D, GM>;
  uint64_t* b = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  Bars r;
  r.kfull = b;
  r.kempty = b + L::kKStages;
  r.vfull = b + 2 * L::kKStages;
  r.vempty = r.vfull + L::kVStages;
  r.qfull = r.vempty + L::kVStages;
  r.qempty = r.qfull + 2;
  r.sfull = r.qempty + 2;
  r.sfree = r.sfull + 2;
  r.pfull = r.sfree + 2;
  r.pfree = r.pfull + 2;
  r.ofull = r.pfree + 2;
  r.ofree = r.ofull + 2;
  r.cdrain = r.ofree + 2;
  r.cdone = r.cdrain + 1;
  r.drain = r.cdone + 1;
  r.ifull = r.drain + 1;
  r.iempty = r.ifull + kItemRing;
  return r;
}

struct TcArgs {
  CUtensorMap tk;  // K pool, 4-D view (see make_pool_map): one box = one block's tile
  CUtensorMap tv;  // V pool, same
  CUtensorMap tq;  // q as [S*Hq rows, head_dim], box 64 x 16
  DecodeParams p;
};

// One work item = (sequence, KV head, partition) with at least one token, packed by
// the work-list kernel as {s, g, t0, ntok | nparts << 16}.
struct Item {
  int s, g, part, t0, ntok, nchunks, nparts;
};

__device__ __forceinline__ Item unpack_item(int4 e, int part_tokens) {
  Item it;
  it.s = e.x;
  it.g = e.y;
  it.t0 = e.z;
  it.ntok = e.w & 0xffff;
  it.nparts = static_cast<int>(static_cast<unsigned>(e.w) >> 16);
  it.part = it.t0 / part_tokens;
  it.nchunks = (it.ntok + kChunk - 1) / kChunk;
  return it;
}

// kPair (head_dim D = 64, an even number of KV heads): an item covers two adjacent KV
// heads and runs with head_dim-128 operands (see the paired-heads note above).
template <typename T, int D, int GM, bool kPair>
__global__ void __launch_bounds__(TcRoles<GM>::kThreads, 1) decode_tc_kernel(const __grid_constant__ TcArgs a) {
  static_assert(kPair ? D == 64 && (GM == 16 || GM == 32) : GM <= 16, "paired heads: head_dim 64");
  constexpr int DL = kPair ? 128 : D;  // operand width: dimensions of a K/V row in shared memory
  using L = TcLayout<DL, GM>;
  using R = TcRoles<GM>;
  constexpr int kKStages = L::kKStages, kVStages = L::kVStages;
  constexpr int kN = L::kN, kQHalfBytes = L::kQHalfBytes, kPBytes = L::kPBytes;
  constexpr int kHalfCols = kN / 2;  // paired: the columns of each head's group
  constexpr int kGroupBytes = L::kGroupBytes, kTileBytes = L::kTileBytes, kQBytes = L::kQBytes;
  constexpr int kOffV = L::kOffV, kOffQ = L::kOffQ, kOffP = L::kOffP;
  using PG = PvGeom<DL, GM>;
  constexpr uint32_t kTmemCols = PG::kTmemCols;
  constexpr bool kDyn = kClaimItems<DL>;
  constexpr int kNO = PG::kNO;
  extern __shared__ __align__(1024) unsigned char smem[];
  const DecodeParams& p = a.p;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const Bars bars = carve_bars<DL, GM>(smem);
  float* red_max = reinterpret_cast<float*>(smem + L::kOffRedMax);  // [2][4 warps][kN]
  float* red_l = reinterpret_cast<float*>(smem + L::kOffRedL);      // [2 item slots][4 warps][kN]
  float* red_mtot = reinterpret_cast<float*>(smem + L::kOffMTot);   // [2 item slots][kN]
  float* alpha_s = reinterpret_cast<float*>(smem + L::kOffAlpha);   // [kN]
  float* xfer = reinterpret_cast<float*>(smem + L::kOffXfer);       // [64][kN] (D = 64)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 4);
  int* kissued_slot = reinterpret_cast<int*>(smem + L::kOffMisc + 8);   // K chunks issued
  int* vissued_slot = reinterpret_cast<int*>(smem + L::kOffMisc + 12);  // V chunks issued
  int* qissued_slot = reinterpret_cast<int*>(smem + L::kOffMisc + 16);  // query tiles issued
  volatile int* cflag = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 20);  // [2] rescale before PV
  int4* ring = reinterpret_cast<int4*>(smem + L::kOffRing);
  const int G = p.group;
  // S/O column n holds a query head of the item: n < G; paired, n % (kN / 2) < G (the
  // first head's group in the first half of the columns, the second's in the second)
  auto col_ok = [G](int n) { return kPair ? n % kHalfCols < G : n < G; };

  if (threadIdx.x == 0) {
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(&bars.kfull[i], 1);
      mbar_init(&bars.kempty[i], 1);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(&bars.vfull[i], 1);
      mbar_init(&bars.vempty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.qfull[i], 1);
      mbar_init(&bars.qempty[i], 1);
      mbar_init(&bars.sfull[i], 1);
      mbar_init(&bars.sfree[i], 4 * R::kSplit);
      mbar_init(&bars.pfull[i], 4 * R::kSplit);
      mbar_init(&bars.pfree[i], 1);
      mbar_init(&bars.ofull[i], 1);
      mbar_init(&bars.ofree[i], 4 * R::kSplit);
      cflag[i] = 0;
    }
    mbar_init(bars.cdrain, 1);
    mbar_init(bars.cdone, 4 * R::kSplit);
    for (int h = 0; h < kN; ++h) alpha_s[h] = 0.f;  // factors of heads past the group stay 0
    for (int i = 0; i < kItemRing; ++i) {
      mbar_init(&bars.ifull[i], 1);
      mbar_init(&bars.iempty[i], 2 + 4 * R::kSplit);  // V producer, MMA warp, softmax warps
    }
    *abort_flag = 0;
    *kissued_slot = 0;
    *vissued_slot = 0;
    *qissued_slot = 0;
    fence_barrier_init();
  }
  if (warp == 5) tmem_alloc(tmem_slot, kTmemCols);
  // P's columns of heads a thread never writes (past the group, when two warps share
  // a group of 8 columns) must read as zero
  for (int i = threadIdx.x; i < 2 * kPBytes / 16; i += R::kThreads)
    reinterpret_cast<uint4*>(smem + kOffP)[i] = make_uint4(0, 0, 0, 0);
  // paired heads: the query operand's off-diagonal blocks (the first head's rows in the
  // second head's dimensions and back) are never loaded and must read as zero
  if constexpr (kPair) {
    for (int i = threadIdx.x; i < 2 * kQBytes / 16; i += R::kThreads)
      reinterpret_cast<uint4*>(smem + kOffQ)[i] = make_uint4(0, 0, 0, 0);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Launched while the work-list kernel may still run (programmatic dependent launch):
  // everything above touches only this CTA; the list, the pool and q are read after
  // the preceding kernels on the stream have completed and their writes are visible.
  grid_dependency_wait();
  // with partitions the next kernel is this call's merge, which waits for this grid
  // before it reads anything: let it launch now, so its start overlaps this kernel
  if (p.max_parts > 1) grid_dependents_launch();
  const int num_items = *p.work_count;

  if (warp == 4) {
    // ============================ TMA producer ============================
    if (lane == 0) {
      prefetch_tensormap(&a.tk);
      prefetch_tensormap(&a.tv);
      prefetch_tensormap(&a.tq);
    }
    const uint64_t pol_stream = policy_evict_first();
    const uint64_t pol_keep = policy_evict_last();
    const int bs = p.block_size;
    const int blocks_per_chunk = kChunk / bs;
    const int oob_row = p.num_blocks * p.num_kv_heads * bs;  // first row outside the pool
    int c = 0, j = 0;
    bool ok = true;
    // Claiming (head_dim-128 operands): item j + 1's list index is claimed four chunks
    // before item j's last chunk is issued (about when this CTA's rings run out of item
    // j), its entry read two chunks before, and it is published in the ring with that
    // last chunk, so neither latency stalls the issue.  Claiming that late keeps the
    // CTAs that run at the same time on neighbouring entries of the list: the
    // shared-prefix workload's L2 reuse depends on it (claims at the start of each item
    // measured 0.95 there against 1.01-1.02).  Lane 0 does all of it.
    auto publish = [&](int jj, int4 e) -> bool {
      const int r = jj % kItemRing;
      if (jj >= kItemRing &&
          !wait_role(&bars.iempty[r], ((jj / kItemRing) - 1) & 1, abort_flag, p.err, p.wait_limit_ns))
        return false;
      ring[r] = e;
      mbar_arrive(&bars.ifull[r]);
      return true;
    };
    int idx = 0;                        // lane 0: list index of the next item
    int4 e = make_int4(0, 0, 0, 0);     // claimed: the current item (then the next one, lane 0)
    ItemCursor sc;                      // fixed order (no claiming): this CTA's items
    if constexpr (!kDyn) {
      sc.init(p.work_list, num_items);
    } else if (lane == 0) {
      // the first item is list entry blockIdx.x (the grid takes the longest ones at once,
      // without waiting for an atomic's round trip); later claims start past the grid
      idx = blockIdx.x;
      if (idx < num_items) e = p.work_list[idx];
      ok = publish(0, e);
    }
    for (;; ++j) {
      if constexpr (!kDyn) {
        if (!(sc.valid() && ok)) break;
        e = sc.cur;
      } else {
        ok = __shfl_sync(0xffffffffu, ok, 0);
        e.x = __shfl_sync(0xffffffffu, e.x, 0);
        e.y = __shfl_sync(0xffffffffu, e.y, 0);
        e.z = __shfl_sync(0xffffffffu, e.z, 0);
        e.w = __shfl_sync(0xffffffffu, e.w, 0);
        if (!ok || !item_valid(e)) break;
      }
      const Item it = unpack_item(e, p.part_tokens);
      int4 nxt = make_int4(0, 0, 0, 0);  // lane 0: the entry of item j + 1
      const int qb = j & 1;
      if (lane == 0) {
        ok = j < 2 || wait_role(&bars.qempty[qb], ((j >> 1) - 1) & 1, abort_flag, p.err, p.wait_limit_ns);
        if (ok) {
          unsigned char* qdst = smem + kOffQ + qb * kQBytes;
          if constexpr (kPair) {
            // kN / 2 query rows from the first head's group into the first rows of
            // dimension block 0, kN / 2 from the second's into the rows after them in
            // block 1 (box 64 x kN / 2; rows past a group belong to no column that is read)
            const int qrow = it.s * p.num_q_heads + it.g * 2 * G;
            mbar_arrive_expect_tx(&bars.qfull[qb], 2 * kHalfCols * 128);
            tma_load_2d(qdst, &a.tq, 0, qrow, &bars.qfull[qb], pol_keep);
            tma_load_2d(qdst + kQHalfBytes + kHalfCols * 128, &a.tq, 0, qrow + G, &bars.qfull[qb], pol_keep);
          } else {
            const int qrow = it.s * p.num_q_heads + it.g * G;
            mbar_arrive_expect_tx(&bars.qfull[qb], kQBytes);
#pragma unroll
            for (int cb = 0; cb < L::kBlocks; ++cb)
              tma_load_2d(qdst + cb * kQHalfBytes, &a.tq, 64 * cb, qrow, &bars.qfull[qb], pol_keep);
          }
          *qissued_slot = j + 1;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      const int32_t* table = p.block_tables + static_cast<size_t>(it.s) * p.max_blocks_per_seq;
      for (int k = 0; k < it.nchunks && ok; ++k, ++c) {
        const int st = c % kKStages;
        // block ids first: their latency overlaps the wait for a free stage
        const int lb = it.t0 / bs + k * blocks_per_chunk + lane;  // logical block of this lane
        const bool live = lane < blocks_per_chunk && lb * bs < it.t0 + it.ntok;
        int b = live ? (lb < p.max_blocks_per_seq ? table[lb] : -1) : 0;
        if (lane == 0) {
          ok = c < kKStages || wait_role(&bars.kempty[st], ((c / kKStages) - 1) & 1, abort_flag, p.err, p.wait_limit_ns);
          if (ok) mbar_arrive_expect_tx(&bars.kfull[st], kTileBytes);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        __syncwarp();
        if (lane < blocks_per_chunk) {
          int row = oob_row;  // blocks past the item's end: zero-filled by the TMA unit
          if (live) {
            if (b < 0 || b >= p.num_blocks) {
              set_error(p.err, kErrIndex);
              b = 0;
            }
            row = (b * p.num_kv_heads + it.g * p.heads_per_item) * bs;
          }
          tma_load_4d(smem + st * kTileBytes + lane * bs * (DL * 2), &a.tk, row / 8, &bars.kfull[st], pol_stream);
        }
        if (lane == 0) {
          *kissued_slot = c + 1;
          if constexpr (kDyn) {
            if (k == max(0, it.nchunks - 4)) idx = static_cast<int>(gridDim.x) + atomicAdd(p.work_next, 1);
            if (k == max(0, it.nchunks - 2)) nxt = idx < num_items ? p.work_list[idx] : make_int4(0, 0, 0, 0);
            if (k == it.nchunks - 1) ok = publish(j + 1, nxt);
          }
        }
      }
      if constexpr (kDyn) e = nxt;  // lane 0's copy is the one broadcast
      else sc.advance();
    }
  } else if (warp == 6) {
    // ============================ TMA producer of V ============================
    if (lane == 0) prefetch_tensormap(&a.tv);
    const uint64_t pol_stream = policy_evict_first();
    const int bs = p.block_size;
    const int blocks_per_chunk = kChunk / bs;
    const int oob_row = p.num_blocks * p.num_kv_heads * bs;
    int c = 0;
    bool ok = true;
    ItemCursor vcur;  // fixed order (no claiming)
    if constexpr (!kDyn) vcur.init(p.work_list, num_items);
    for (int j = 0;; ++j) {
      int4 e = make_int4(0, 0, 0, 0);
      if constexpr (!kDyn) {
        if (!(vcur.valid() && ok)) break;
        e = vcur.cur;
      } else {
        if (!ok) break;
        const int r = j % kItemRing;
        ok = __all_sync(0xffffffffu, wait_role(&bars.ifull[r], (j / kItemRing) & 1, abort_flag, p.err, p.wait_limit_ns));
        if (!ok) break;
        e = ring[r];
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.iempty[r]);
        if (!item_valid(e)) break;
      }
      const Item it = unpack_item(e, p.part_tokens);
      const int32_t* table = p.block_tables + static_cast<size_t>(it.s) * p.max_blocks_per_seq;
      for (int k = 0; k < it.nchunks && ok; ++k, ++c) {
        const int st = c % kVStages;
        const int lb = it.t0 / bs + k * blocks_per_chunk + lane;
        const bool live = lane < blocks_per_chunk && lb * bs < it.t0 + it.ntok;
        int b = live ? (lb < p.max_blocks_per_seq ? table[lb] : -1) : 0;
        if (lane == 0) {
          ok = c < kVStages || wait_role(&bars.vempty[st], ((c / kVStages) - 1) & 1, abort_flag, p.err, p.wait_limit_ns);
          if (ok) mbar_arrive_expect_tx(&bars.vfull[st], kTileBytes);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        __syncwarp();
        if (lane < blocks_per_chunk) {
          int row = oob_row;
          if (live) {
            if (b < 0 || b >= p.num_blocks) b = 0;  // the K producer flags it
            row = (b * p.num_kv_heads + it.g * p.heads_per_item) * bs;
          }
          tma_load_4d(smem + kOffV + st * kTileBytes + lane * bs * (DL * 2), &a.tv, row / 8, &bars.vfull[st],
                      pol_stream);
        }
        if (lane == 0) *vissued_slot = c + 1;
      }
      if constexpr (!kDyn) vcur.advance();
    }
  } else if (warp == 5) {
    // ============================ MMA issuer ============================
    // The whole warp polls with warp-uniform control flow (descriptors and counters
    // stay in uniform registers) and one elected lane issues whichever is ready: PV of
    // the oldest chunk whose probabilities are written (first: its completion frees a
    // V stage and a P buffer) or QK of the next chunk (its K landed, its S buffer free).
    // Neither waits behind the other.  One round trip probes the five barriers both need.
    // PV accumulates into the item's O buffer (item j: O[j & 1]), overwriting it on the
    // item's first chunk; the item's last PV also signals O full.
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr uint32_t idesc_qk = instr_desc_f16(kBf16, false, false, kChunk, kN);
    constexpr uint32_t idesc_pv = instr_desc_f16(kBf16, true, true, 128, kNO);
    // descriptor bases; adding (byte offset >> 4) moves a descriptor's start address
    const uint64_t dk0 = smem_desc(smem_addr(smem), 16, kGroupBytes, kLayoutSwizzle128);
    const uint64_t dq0 = smem_desc(smem_addr(smem + kOffQ), 16, 1024, kLayoutSwizzle128);
    // rows 64-127 of V^T: the second 64-dimension block (1 KB on) at D = 128, the same
    // dimensions of the tokens 64 on (8 row groups on) at D = 64
    const uint64_t dv0 = smem_desc(smem_addr(smem + kOffV), DL == 128 ? 1024 : 8 * kGroupBytes, kGroupBytes,
                                   kLayoutSwizzle128);
    const uint64_t dp0 = smem_desc(smem_addr(smem + kOffP), 128, PG::kPGroupBytes, kLayoutNone);
    // QK cursor: items walked, chunk within the item, chunks in the item (0: the item
    // is not read from the ring yet); PV likewise.  QK reads an item's ring slot first
    // (as soon as it is published); PV reads the same slot when it starts the item and
    // then releases it.
    int qk = 0, qj = 0, pk = 0, pj = 0, qn = 0, pn = 0;
    bool qdone = false;  // QK read the end of the list
    ItemCursor qcur, pcur;  // fixed order (no claiming): each item's count is known at once
    if constexpr (!kDyn) {
      qcur.init(p.work_list, num_items);
      pcur.init(p.work_list, num_items);
      qn = qcur.valid() ? unpack_item(qcur.cur, p.part_tokens).nchunks : 0;
      pn = pcur.valid() ? unpack_item(pcur.cur, p.part_tokens).nchunks : 0;
      qdone = !qcur.valid();
    }
    int qc = 0, pc = 0;           // next chunk to QK, next chunk to PV
    int qst = 0, qph = 0;         // ring stage and phase of chunk qc
    int pst = 0, pph = 0;         // ring stage and phase of chunk pc
    int ncorr = 0;                // O rescales handed over so far
    uint64_t idle_since = global_timer_ns();
    while (!qdone || pc < qc) {
      bool progressed = false;
      if constexpr (kDyn) {
        if (qn == 0 && !qdone &&
            __all_sync(0xffffffffu, mbar_test_wait(&bars.ifull[qj % kItemRing], (qj / kItemRing) & 1))) {
          const int4 e = ring[qj % kItemRing];
          if (item_valid(e)) qn = unpack_item(e, p.part_tokens).nchunks;
          else qdone = true;
          progressed = true;
        }
      }
      const int sb = qc & 1, qb = qj & 1, pb = pc & 1, ob = pj & 1;
      // bit 0: chunk qc landed, 1: S[qc & 1] free, 2: P of chunk pc written, 3: O[pj & 1]
      // written out (matters on an item's first chunk only), 4: V of chunk pc landed
      const uint32_t seen = __shfl_sync(0xffffffffu,
          mbar_test_wait5(&bars.kfull[qst], qph, &bars.sfree[sb], ((qc >> 1) - 1) & 1, &bars.pfull[pb],
                          (pc >> 1) & 1, &bars.ofree[ob], ((pj >> 1) - 1) & 1, &bars.vfull[pst], pph), 0);
      if (pc < qc && (seen & 4) && (pk > 0 || pj < 2 || (seen & 8)) && (seen & 16)) {
        if constexpr (kDyn) {
          if (pk == 0) {  // PV starts item pj: its chunk count, then the slot is free
            pn = unpack_item(ring[pj % kItemRing], p.part_tokens).nchunks;
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.iempty[pj % kItemRing]);
          }
        }
        tc_fence_after();
        // the running max rose mid-item (rare): O must be rescaled before this PV adds
        // to it.  Signal when every MMA issued so far has completed, then wait for the
        // softmax warps to hand the rescaled buffer back.
        if (cflag[pb]) {
          if (elect_one()) mma_commit(bars.cdrain);
          __syncwarp();
          if (!__all_sync(0xffffffffu, wait_role(bars.cdone, ncorr & 1, abort_flag, p.err, p.wait_limit_ns))) break;
          ++ncorr;
          tc_fence_after();
        }
        const uint64_t dv = dv0 + ((pst * kTileBytes) >> 4);
        const uint64_t dp = dp0 + ((pb * kPBytes) >> 4);
        const bool last = pk == pn - 1;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < PG::kSteps; ++kk)
            mma_f16(tmem + 2 * kN + ob * kNO, dv + ((kk * 2 * kGroupBytes) >> 4), dp + ((kk * 256) >> 4), idesc_pv,
                    kk > 0 || pk > 0);
          mma_commit(&bars.pfree[pb]);
          mma_commit(&bars.vempty[pst]);
          if (last) mma_commit(&bars.ofull[ob]);
        }
        __syncwarp();
        ++pc;
        if (++pst == kVStages) {
          pst = 0;
          pph ^= 1;
        }
        if (++pk == pn) {
          pk = 0;
          ++pj;
          if constexpr (!kDyn) {
            pcur.advance();
            pn = pcur.valid() ? unpack_item(pcur.cur, p.part_tokens).nchunks : 0;
          }
        }
        progressed = true;
      }
      if (qn > 0 && (seen & 1) && (qc < 2 || (seen & 2)) &&
          (qk > 0 || __all_sync(0xffffffffu, mbar_test_wait(&bars.qfull[qb], (qj >> 1) & 1)))) {
        const uint64_t dk = dk0 + ((qst * kTileBytes) >> 4);
        const uint64_t dq = dq0 + ((qb * kQBytes) >> 4);
        const bool last = qk == qn - 1;
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < DL / 16; ++kk) {
            const uint32_t ko = ((kk >> 2) * 1024 + (kk & 3) * 32) >> 4;
            const uint32_t qo = ((kk >> 2) * kQHalfBytes + (kk & 3) * 32) >> 4;
            mma_f16(tmem + sb * kN, dk + ko, dq + qo, idesc_qk, kk > 0);
          }
          mma_commit(&bars.sfull[sb]);
          mma_commit(&bars.kempty[qst]);           // the K stage is free once this QK completed
          if (last) mma_commit(&bars.qempty[qb]);  // the item's last QK: its query buffer can be refilled
        }
        __syncwarp();
        ++qc;
        if (++qst == kKStages) {
          qst = 0;
          qph ^= 1;
        }
        if (++qk == qn) {
          qk = 0;
          ++qj;
          if constexpr (kDyn) {
            qn = 0;
          } else {
            qcur.advance();
            qn = qcur.valid() ? unpack_item(qcur.cur, p.part_tokens).nchunks : 0;
            qdone = !qcur.valid();
          }
        }
        progressed = true;
      }
      if (progressed) {
        idle_since = global_timer_ns();
      } else {
        if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
        if (__any_sync(0xffffffffu, global_timer_ns() - idle_since > p.wait_limit_ns)) {
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
    constexpr int HG = R::kHeads;              // heads of this thread: h0 .. h0 + HG - 1
    constexpr int NS = R::kSoftmaxThreads;     // threads in the softmax barriers
    const int quarter = warp & 3;              // TMEM lane quarter this warp may read
    // first head: warps 0-3 take the lowest HG heads of their quarter, each further set
    // of four warps (7-10, 11-14, ...) the next HG
    const int h0 = warp < 4 ? 0 : ((warp - 7) / 4 + 1) * HG;
    const int t = quarter * 32 + lane;         // TMEM lane: token row of S, dimension row of O (a copy at t >= D)
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    float m[HG], lp[HG], alpha[HG];
#pragma unroll
    for (int h = 0; h < HG; ++h) {
      m[h] = -INFINITY; lp[h] = 0.f; alpha[h] = 0.f;
    }
    // the last finished item, not yet written out (pend_j < 0: none)
    int pend_s = 0, pend_g = 0, pend_part = 0, pend_nparts = 0, pend_j = -1;
    int c = 0, j = 0, ncorr = 0;
    bool ok = true;

    // Writes out item pend_j once its last PV completed: its O buffer's hi and lo
    // columns summed, divided by the row sum (a partition instead leaves O unnormalised
    // with its max and sum for the merge).  Returns false (warp-uniform) when the wait
    // ran out or another role aborted.
    auto finalize = [&]() -> bool {
      const int ob = pend_j & 1;
      const bool w =
          __all_sync(0xffffffffu, wait_role(&bars.ofull[ob], (pend_j >> 1) & 1, abort_flag, p.err, p.wait_limit_ns));
      float o[HG];
      if (w) {
        tc_fence_after();
        // O columns: [hi 0-7][lo 0-7] up to 8 heads, [hi][lo] of kN columns each beyond;
        // with the 64-token halves (head_dim 64, one head per item) rows 64-127 hold the
        // chunks' second halves in the next NP columns
        const uint32_t oaddr = lane_base + 2 * kN + ob * kNO + (PG::kHalves && quarter >= 2 ? PG::kNP : 0) + h0;
        float olo[HG];
        if (GM <= 8) {  // 4-column aligned loads; a pair at column 2 is picked from them
          float a4[4], b4[4];
          tmem_load4x2(oaddr - (h0 & 3), oaddr - (h0 & 3) + 8, a4, b4);
#pragma unroll
          for (int h = 0; h < HG; ++h) {
            o[h] = (h0 & 2) ? a4[(2 + h) & 3] : a4[h];
            olo[h] = (h0 & 2) ? b4[(2 + h) & 3] : b4[h];
          }
        } else if (HG == 4) {
          tmem_load4x2(oaddr, oaddr + PG::kNP / 2, o, olo);
        } else {
          tmem_load8x2(oaddr, oaddr + PG::kNP / 2, o, olo);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.ofree[ob]);
#pragma unroll
        for (int h = 0; h < HG; ++h) o[h] += olo[h];  // hi part + lo part
      }
      if (PG::kHalves) {
        // the second half's sums (rows 64-127) move to the threads of rows 0-63; every
        // softmax thread takes the barrier, whether its wait succeeded or not
        if (w && quarter >= 2) {
#pragma unroll
          for (int h = 0; h < HG; ++h) xfer[(t - 64) * kN + h0 + h] = o[h];
        }
        if (!named_barrier_and(1, NS, w)) return false;
        if (quarter < 2) {
#pragma unroll
          for (int h = 0; h < HG; ++h) o[h] += xfer[t * kN + h0 + h];
        }
      } else if (!w) {
        return false;
      }
      // paired: rows 0-63 are the first head's dimensions, rows 64-127 the second's;
      // a thread writes the columns of its own head only
      if (kPair || t < D) {
        const int dim = kPair ? (t & 63) : t;
        // the item's totals, left in slot ob at its last chunk
        const float* rl = red_l + ob * 4 * kN + h0;
#pragma unroll
        for (int h = 0; h < HG; ++h) {
          const int n = h0 + h;
          if (col_ok(n) && (!kPair || n / kHalfCols == (t >> 6))) {
            const float acc = o[h];
            const float l = (rl[h] + rl[kN + h]) + (rl[2 * kN + h] + rl[3 * kN + h]);
            const size_t row = static_cast<size_t>(pend_s) * p.num_q_heads +
                               (kPair ? pend_g * 2 * G + (n / kHalfCols) * G + n % kHalfCols : pend_g * G + n);
            if (pend_nparts == 1) {
              store_out<T>(p.out, row * D + dim, acc / l, p.out_f32);
            } else {
              const size_t k = row * p.max_parts + pend_part;
              p.ws_o[k * D + dim] = acc;
              if (dim == 0) {
                p.ws_ml[2 * k] = red_mtot[ob * kN + h0 + h];
                p.ws_ml[2 * k + 1] = l;
              }
            }
          }
        }
      }
      return true;
    };

    // Rescales the O accumulator of buffer ob by each head's factor before the PV of a
    // chunk whose scores raised the running max: wait until every MMA issued before
    // that PV completed, multiply this warp's share of O's columns, hand it back.  All
    // softmax threads call it (the decision is CTA-uniform).
    auto rescale = [&](int ob) -> bool {
      if (quarter == 0 && lane == 0) {
#pragma unroll
        for (int h = 0; h < HG; ++h) alpha_s[h0 + h] = col_ok(h0 + h) ? alpha[h] : 0.f;
      }
      named_barrier_sync(1, NS);
      if (!__all_sync(0xffffffffu, wait_role(bars.cdrain, ncorr & 1, abort_flag, p.err, p.wait_limit_ns)))
        return false;
      ++ncorr;
      tc_fence_after();
      // O columns: per half, the heads' hi parts then their lo parts
      constexpr int kCols = kNO / R::kSplit;   // this warp's share of its lane quarter: 8 to 32
      const int c0 = (h0 / HG) * kCols;
      const uint32_t oaddr = lane_base + 2 * kN + ob * kNO + c0;
#pragma unroll
      for (int q = 0; q < kCols / 8; ++q) {
        float v[8];
        tmem_load8(oaddr + 8 * q, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] *= alpha_s[(c0 + 8 * q + i) % (PG::kNP / 2)];
        tmem_store8_nowait(oaddr + 8 * q, v);
      }
      tmem_store_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.cdone);
      return true;
    };

    bool prev_ok = true;  // outcome of the last rescale and write-out (warp-uniform)
    ItemCursor scur;  // fixed order (no claiming)
    if constexpr (!kDyn) scur.init(p.work_list, num_items);
    for (;; ++j) {
      int4 e = make_int4(0, 0, 0, 0);
      if constexpr (!kDyn) {
        if (!(scur.valid() && ok)) break;
        e = scur.cur;
      } else {
        if (!ok) break;
        const int r = j % kItemRing;
        const bool w =
            __all_sync(0xffffffffu, wait_role(&bars.ifull[r], (j / kItemRing) & 1, abort_flag, p.err, p.wait_limit_ns));
        if (w) e = ring[r];
        __syncwarp();
        if (lane == 0 && w) mbar_arrive(&bars.iempty[r]);
        // every softmax thread takes this barrier: after an abort some warps may have
        // given up on the slot while others read it, and all must leave together
        if (!named_barrier_and(1, NS, w)) {
          prev_ok = false;
          break;
        }
        if (!item_valid(e)) break;
      }
      const Item it = unpack_item(e, p.part_tokens);
      // padded heads (columns past the group) get m = +inf: their scores then come out as -inf and
      // their probabilities as 0 without a test (their l and O are never stored)
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        m[h] = col_ok(h0 + h) ? -INFINITY : INFINITY;
        lp[h] = 0.f;
      }
      for (int k = 0; k < it.nchunks; ++k, ++c) {
        const int sb = c & 1;
        // S of chunk c, and its P buffer free again (the PV of chunk c - 2 completed)
        const bool wok = __all_sync(0xffffffffu,
            wait_role2(&bars.sfull[sb], (c >> 1) & 1, c >= 2 ? &bars.pfree[sb] : nullptr, ((c >> 1) - 1) & 1,
                       abort_flag, p.err, p.wait_limit_ns));
        float sv[HG];
        if (wok) {
          tc_fence_after();
          if (HG <= 4) {  // 4-column aligned load; a pair at column 2 is picked from it
            float s4[4];
            tmem_load4(lane_base + sb * kN + (h0 & ~3), s4);
#pragma unroll
            for (int h = 0; h < HG; ++h) sv[h] = (h0 & 2) ? s4[(2 + h) & 3] : s4[h];
          } else {
            tmem_load8(lane_base + sb * kN + h0, sv);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars.sfree[sb]);
        }
        const int rows_valid = min(kChunk, it.ntok - k * kChunk);
        const bool valid = wok && t < rows_valid;
        // Lazy rescale: the running max m of a head only has to bound its scores
        // loosely (probabilities up to 2^kSlack stay exact enough in hi + lo and
        // in fp32 sums), so it moves only when some score of the chunk exceeds it
        // by more than kSlack (always on an item's first chunk, m = -inf).  One
        // barrier vote decides it for the chunk; most chunks then skip the max
        // reduction and the rescale.
        constexpr float kSlack = 8.f;
        float x[HG], pe[HG];  // x = score - running max (log2 domain), -inf past the context end
        float excess = -INFINITY;
#pragma unroll
        for (int h = 0; h < HG; ++h) {
          x[h] = valid ? fmaf(sv[h], p.scale_log2, -m[h]) : -INFINITY;
          excess = fmaxf(excess, x[h]);
        }
        // every softmax warp learns whether all got here normally, and whether any
        // head needs a new running max
        const bool keep = named_barrier_and(1, NS, wok && prev_ok && !(excess > kSlack));
        if (keep) {
#pragma unroll
          for (int h = 0; h < HG; ++h) {
            pe[h] = exp2_approx(x[h]);
            lp[h] += pe[h];
          }
        } else {
          // chunk max over the 128 tokens, per head
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
            const float* r = red_max + sb * 4 * kN + h0 + h;
            const float mn = fmaxf(m[h], fmaxf(fmaxf(r[0], r[kN]), fmaxf(r[2 * kN], r[3 * kN])));
            alpha[h] = exp2_approx(m[h] - mn);  // 0 on the item's first chunk (m = -inf)
            m[h] = mn;
            pe[h] = exp2_approx(sv[h] - mn);
            lp[h] = fmaf(lp[h], alpha[h], pe[h]);
          }
        }
        // O already holds earlier chunks of this item: it must be rescaled before this
        // chunk's PV (the MMA warp reads the flag once P is full)
        const bool corr = !keep && k > 0;
        if (warp == 0 && lane == 0) cflag[sb] = corr ? 1 : 0;
        // hi = round(p) and lo = round(p - hi) (p - hi is exact in fp32), two heads a
        // word; words past this thread's heads are zero
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (2 * i < HG) {
            const float a = pe[2 * i], b = 2 * i + 1 < HG ? pe[2 * i + 1] : 0.f;
            float ha, hb;
            hw[i] = pack2_split<T>(a, b, ha, hb);
            lw[i] = pack2<T>(a - ha, b - hb);
          } else {
            hw[i] = lw[i] = 0u;
          }
        }
        // P^T for PV: token t's head weights, MN-major without swizzle, 8 columns (16
        // bytes) a group: [hi 0-7][lo 0-7] up to 8 heads, then the hi groups of all kN
        // columns followed by their lo groups; with the 64-token halves (head_dim 64, one
        // head per item) those groups once per half
        const int tt = PG::kHalves ? (t & 63) : t;  // token within its column group
        unsigned char* pdst = smem + kOffP + sb * kPBytes + (tt >> 3) * 128 + (tt & 7) * 16 +
                              (PG::kHalves ? (t >> 6) * (PG::kNP / 8) * PG::kPGroupBytes : 0);
        constexpr int kGB = PG::kPGroupBytes;
        if (R::kSplit == 1) {
          *reinterpret_cast<uint4*>(pdst) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(pdst + kGB) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        } else if (GM == 4) {  // each of the two warps writes its two heads of a group
          *reinterpret_cast<uint32_t*>(pdst + h0 * 2) = hw[0];
          *reinterpret_cast<uint32_t*>(pdst + kGB + h0 * 2) = lw[0];
        } else if (GM == 8) {  // each of the two warps writes its four heads' half of a group
          *reinterpret_cast<uint2*>(pdst + h0 * 2) = make_uint2(hw[0], hw[1]);
          *reinterpret_cast<uint2*>(pdst + kGB + h0 * 2) = make_uint2(lw[0], lw[1]);
        } else if (HG == 4) {  // 16 heads over four warps: each writes half of a column group
          const int gh = h0 / 8, off = (h0 & 7) * 2;
          *reinterpret_cast<uint2*>(pdst + gh * kGB + off) = make_uint2(hw[0], hw[1]);
          *reinterpret_cast<uint2*>(pdst + (PG::kNP / 16 + gh) * kGB + off) = make_uint2(lw[0], lw[1]);
        } else {
          const int gh = h0 / 8;  // this warp's column group of hi parts
          *reinterpret_cast<uint4*>(pdst + gh * kGB) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(pdst + (PG::kNP / 16 + gh) * kGB) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
        // rows of the last loaded block past the context end: zero their V rows (only an
        // item's last chunk can have them; the first warp of each quarter does it)
        const bool last = k == it.nchunks - 1;
        if (last && rows_valid < kChunk && h0 == 0) {
          const int rows_loaded = min(kChunk, (rows_valid + p.block_size - 1) / p.block_size * p.block_size);
          // (warp-uniform) the chunk's V must have landed before its tail rows are zeroed
          const bool v_ok = rows_valid >= rows_loaded ||
                            __all_sync(0xffffffffu, wait_role(&bars.vfull[c % kVStages], (c / kVStages) & 1,
                                                              abort_flag, p.err, p.wait_limit_ns));
          if (v_ok && t >= rows_valid && t < rows_loaded) {
            unsigned char* vrow = smem + kOffV + (c % kVStages) * kTileBytes + (t >> 3) * kGroupBytes + (t & 7) * 128;
#pragma unroll
            for (int q = 0; q < 8 * L::kBlocks; ++q)  // 128 bytes per 64-column block, 1 KB apart
              reinterpret_cast<uint4*>(vrow + (q >> 3) * 1024)[q & 7] = make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.pfull[sb]);
        prev_ok = true;
        if (corr) prev_ok = rescale(j & 1);

        if (last) {  // this item's totals (row sums per lane quarter, running max) into slot j & 1
          const float lsum = warp_sum_scatter<HG>(lp, lane);  // head warp_sum_index<HG>(lane)
          if ((lane & (32 / HG - 1)) == 0)
            red_l[((j & 1) * 4 + quarter) * kN + h0 + warp_sum_index<HG>(lane)] = lsum;
          if (t == 0) {
#pragma unroll
            for (int h = 0; h < HG; ++h) red_mtot[(j & 1) * kN + h0 + h] = m[h];
          }
        }
        // the previous item is written out once this item's first P is on its way (the
        // vote barrier above made its totals visible)
        if (k == 0 && pend_j >= 0) {
          prev_ok = finalize() && prev_ok;
          pend_j = -1;
        }
        if (last) {
          pend_s = it.s;
          pend_g = it.g;
          pend_part = it.part;
          pend_nparts = it.nparts;
          pend_j = j;
        }
      }
      if constexpr (!kDyn) scur.advance();
    }
    // the last item: one barrier makes its totals visible (and every thread takes it,
    // aborted or not)
    if (named_barrier_and(1, NS, ok && prev_ok) && pend_j >= 0) finalize();
    __syncwarp();
  }

  // ---------------- teardown ----------------
  __syncthreads();
  if (*abort_flag) {
    // a wait ran out: let in-flight copies and MMAs finish (bounded) before leaving
    // copies still in flight land first: the last chunk issued on each stage (a
    // phase already completed returns at once)
    if (warp == 4 && lane == 0) {
      for (int c = max(0, *kissued_slot - kKStages); c < *kissued_slot; ++c)
        if (!mbar_wait(&bars.kfull[c % kKStages], (c / kKStages) & 1)) break;
      // the query tiles of the last two items (each has its own buffer and barrier)
      for (int jj = max(0, *qissued_slot - 2); jj < *qissued_slot; ++jj)
        if (!mbar_wait(&bars.qfull[jj & 1], (jj >> 1) & 1)) break;
    }
    if (warp == 6 && lane == 0) {
      for (int c = max(0, *vissued_slot - kVStages); c < *vissued_slot; ++c)
        if (!mbar_wait(&bars.vfull[c % kVStages], (c / kVStages) & 1)) break;
    }
    if (warp == 5) {
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
  if (warp == 5) tmem_dealloc(tmem, kTmemCols);
}

// Work list for the persistent kernel: one entry per (sequence, KV head, partition)
// holding at least one token, sorted by chunk count, longest first (a counting sort
// over at most 32 chunk counts; order inside one count does not matter, every item
// is computed the same way wherever it runs).  Sequences of length 0 get their
// all-zero output here; lengths outside [0, max_parts * part_tokens] set the flag.
constexpr int kListThreads = 1024;
constexpr int kMaxChunkCounts = kTcMaxPartition / kChunk;

template <typename T>
__global__ void __launch_bounds__(kListThreads) work_list_kernel(const __grid_constant__ DecodeParams p) {
  grid_dependents_launch();  // the decode kernel may start its prologue now
  if (threadIdx.x == 0) *p.work_next = 0;  // claims past the decode grid's first items
  __shared__ int hist[kMaxChunkCounts + 1];
  __shared__ int next[kMaxChunkCounts + 1];
  const int full_chunks = p.part_tokens / kChunk;
  const int H = p.num_kv_heads / p.heads_per_item;  // items per (sequence, partition)
  for (int i = threadIdx.x; i <= kMaxChunkCounts; i += kListThreads) hist[i] = 0;
  __syncthreads();
  for (int s = threadIdx.x; s < p.num_seqs; s += kListThreads) {
    const int L = p.context_lens[s];
    if (L < 0 || L > p.max_parts * p.part_tokens) {
      set_error(p.err, kErrLength);
      continue;
    }
    const int nfull = L / p.part_tokens, rem = L - nfull * p.part_tokens;
    if (nfull) atomicAdd(&hist[full_chunks], nfull * H);
    if (rem) atomicAdd(&hist[(rem + kChunk - 1) / kChunk], H);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int c = kMaxChunkCounts; c >= 1; --c) {
      next[c] = run;
      run += hist[c];
    }
    *p.work_count = run;
  }
  __syncthreads();
  for (int s = threadIdx.x; s < p.num_seqs; s += kListThreads) {
    const int L = p.context_lens[s];
    if (L <= 0 || L > p.max_parts * p.part_tokens) continue;
    const int nparts = (L + p.part_tokens - 1) / p.part_tokens;
    for (int part = 0; part < nparts; ++part) {
      const int t0 = part * p.part_tokens;
      const int ntok = min(p.part_tokens, L - t0);
      const int pos = atomicAdd(&next[(ntok + kChunk - 1) / kChunk], H);
      for (int g = 0; g < H; ++g) p.work_list[pos + g] = make_int4(s, g, t0, ntok | (nparts << 16));
    }
  }
  // empty contexts: the neutral output, one warp per sequence
  const int row = p.num_q_heads * p.head_dim;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  for (int s = warp; s < p.num_seqs; s += kListThreads / 32) {
    if (p.context_lens[s] != 0) continue;
    for (int i = lane; i < row; i += 32) store_out<T>(p.out, static_cast<size_t>(s) * row + i, 0.f, p.out_f32);
  }
  // Launched as a programmatic dependent of the previous kernel (the append, whose
  // writes this kernel does not read): finish only after it, so the decode kernel's
  // wait on this one also covers the append.
  grid_dependency_wait();
}

// 2-D map over rows of head_dim 16-bit elements, box 64 x box_rows, 128-byte swizzle.
bool make_map_uncached(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows, bool bf16,
                       int head_dim) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(head_dim), rows};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(head_dim) * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
            const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows, bool bf16, int head_dim) {
  return cached_map(m, MapKey{base, rows, box_rows, 2, bf16 ? 2 : 1, head_dim}, [&](CUtensorMap* out) {
    return make_map_uncached(out, base, rows, box_rows, bf16, head_dim);
  });
}

template <typename T, int D, int GM, bool kPair = false>
cudaError_t launch_tc_t(const TcArgs& args, int grid, cudaStream_t stream) {
  constexpr int smem = TcLayout<kPair ? 128 : D, GM>::kSmemBytes;
  static std::atomic<unsigned long long> configured{0};  // devices whose limit is raised
  cudaError_t e = ensure_smem_limit(decode_tc_kernel<T, D, GM, kPair>, smem, configured);
  if (e != cudaSuccess) return e;
  return launch_dependent(decode_tc_kernel<T, D, GM, kPair>, grid, TcRoles<GM>::kThreads, smem, stream, args);
}

template <typename T, int D>
cudaError_t launch_tc_g(const TcArgs& args, int grid, cudaStream_t stream) {
  const int G = args.p.group;
  if (G <= 1) return launch_tc_t<T, D, 1>(args, grid, stream);
  if (G <= 2) return launch_tc_t<T, D, 2>(args, grid, stream);
  if (G <= 4) return launch_tc_t<T, D, 4>(args, grid, stream);
  if (G <= 8) return launch_tc_t<T, D, 8>(args, grid, stream);
  return launch_tc_t<T, D, 16>(args, grid, stream);
}

template <typename T>
cudaError_t launch_tc_d(const TcArgs& args, int grid, cudaStream_t stream) {
  if (args.p.heads_per_item == 2)
    return args.p.group <= 8 ? launch_tc_t<T, 64, 16, true>(args, grid, stream)
                             : launch_tc_t<T, 64, 32, true>(args, grid, stream);
  return args.p.head_dim == 64 ? launch_tc_g<T, 64>(args, grid, stream) : launch_tc_g<T, 128>(args, grid, stream);
}

}  // namespace

bool tc_supported(int dtype, int head_dim, int group, int block_size) {
  const int max_group = dtype == PKV_F32 ? 8 : kMaxGroup;  // f32: the tf32 kernel's N holds 8 heads twice
  return (dtype == PKV_F16 || dtype == PKV_BF16 || dtype == PKV_F32) && (head_dim == 64 || head_dim == 128) &&
         group >= 1 && group <= max_group &&
         (block_size == 8 || block_size == 16 || block_size == 32 || block_size == 64);
}

// head_dim 64 on the 16-bit kernel: pairs of KV heads per item wherever the KV heads pair
// up (16 S columns up to 8 query heads per KV head, 32 beyond)
int tc_heads_per_item(int dtype, int head_dim, int num_kv_heads) {
  return dtype != PKV_F32 && head_dim == 64 && num_kv_heads % 2 == 0 ? 2 : 1;
}

cudaError_t launch_decode_tc(const DecodeParams& p, int dtype, cudaStream_t stream) {
  if (dtype == PKV_F32) {  // the tf32 kernel (decode_tc32.cu) over the same work list
    const int items = p.max_parts * p.num_seqs * p.num_kv_heads;
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const int grid = items < sms ? items : sms;
    cudaError_t e = launch_dependent(work_list_kernel<float>, 1, kListThreads, 0, stream, p);
    if (e != cudaSuccess || grid == 0) return e;
    return launch_decode_tc32(p, grid, stream);
  }
  TcArgs args;
  args.p = p;
  const bool pair = tc_heads_per_item(dtype, p.head_dim, p.num_kv_heads) == 2;
  args.p.heads_per_item = pair ? 2 : 1;
  const bool bf16 = dtype == PKV_BF16;
  const uint64_t pool_rows = static_cast<uint64_t>(p.num_blocks) * p.num_kv_heads * p.block_size;
  const uint64_t q_rows = static_cast<uint64_t>(p.num_seqs) * p.num_q_heads;
  const bool maps_ok =
      pair ? make_pair_pool_map(&args.tk, p.k_cache, pool_rows, p.block_size, bf16) &&
                 make_pair_pool_map(&args.tv, p.v_cache, pool_rows, p.block_size, bf16) &&
                 make_map(&args.tq, p.q, q_rows, p.group <= 8 ? 8 : 16, bf16, p.head_dim)
           : make_pool_map(&args.tk, p.k_cache, pool_rows, p.block_size, bf16, p.head_dim) &&
                 make_pool_map(&args.tv, p.v_cache, pool_rows, p.block_size, bf16, p.head_dim) &&
                 make_map(&args.tq, p.q, q_rows, kNCols<16>, bf16, p.head_dim);
  if (!maps_ok) return cudaErrorInvalidValue;
  const int items = p.max_parts * p.num_seqs * (p.num_kv_heads / args.p.heads_per_item);  // upper bound on the list
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const int grid = items < sms ? items : sms;
  cudaError_t e = bf16 ? launch_dependent(work_list_kernel<__nv_bfloat16>, 1, kListThreads, 0, stream, args.p)
                       : launch_dependent(work_list_kernel<__half>, 1, kListThreads, 0, stream, args.p);
  if (e != cudaSuccess || grid == 0) return e;
  return bf16 ? launch_tc_d<__nv_bfloat16>(args, grid, stream) : launch_tc_d<__half>(args, grid, stream);
}

}  // namespace pkv
