/*
 * pagedkv.h -- C ABI of libpagedkv.so: the data-parallel hot path of PagedAttention
 * on one GB300 (sm_103a).
 *
 * The method (four web pages on PagedAttention / vLLM):
 *  - "anthology-of-the-sota note-023", Method: a sequence's KV cache is cut into
 *    fixed-size blocks of a fixed number of tokens; a per-sequence block table maps
 *    logical block i to a physical block; attention gathers K/V from those
 *    non-contiguous blocks; blocks are allocated as the sequence grows and shared
 *    between sequences, with copy-on-write when one of them diverges.
 *  - "Efficient Memory Management for Large Language Model Serving with
 *    PagedAttention", How It Works: blocks of e.g. 16 tokens; the block table plays
 *    the part of an OS page table; copy-on-write for parallel sampling / beam search.
 *  - "Paged Attention" glossary, paragraph 4: attention's arithmetic is unchanged,
 *    only the storage of K/V moves; GQA paragraph: several query heads share one
 *    key/value head (Llama 2 70B: 64 query heads, 8 KV heads).
 *
 * Layouts (the pages fix none; this library's reading):
 *  - k_cache, v_cache: [num_blocks][num_kv_heads][block_size][head_dim], row-major.
 *    One (block, kv head) tile is block_size*head_dim contiguous elements.
 *  - q, out: [num_seqs][num_q_heads][head_dim].  Query head h reads KV head
 *    h / (num_q_heads / num_kv_heads).
 *  - k, v of new tokens: [num_tokens][num_kv_heads][head_dim].
 *  - block_tables: int32 [num_seqs][max_blocks_per_seq]; entry i of row s is the
 *    physical block of logical block i of sequence s.  Entries at or past
 *    ceil(context_lens[s] / block_size) are never read.
 *  - context_lens: int32 [num_seqs], tokens each sequence attends over (>= 0).
 *  - slot_mapping: int64 [num_tokens]; slot = physical_block * block_size + row;
 *    a negative slot is padding and is skipped.
 *  - src_dst_pairs: int64 [num_pairs][2] of (source block, destination block).
 *
 * Conventions:
 *  - Ownership: the caller owns every buffer.  Apart from arguments documented as
 *    host memory, every pointer is device memory of the current device.  The
 *    library allocates no device memory and keeps no pointer after a call returns.
 *    Caller-provided workspace holds the tensor-core decode work list, split-K
 *    partials and the prefill work list (the *_workspace_bytes calls size it).
 *  - Streams: `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *    call only enqueues work and returns; results are ready when the stream is.
 *    The calls can be captured in a CUDA graph once each kind has run once outside
 *    the capture (the first call sets its kernels' shared-memory limits).
 *  - Early start: the tensor-core decode's first kernel (its work list) is launched
 *    as a programmatic dependent of the kernel before it on the stream, so that it
 *    overlaps paged_kv_append.  Before it waits for that kernel it reads
 *    context_lens and writes its workspace and the zero rows of out for empty
 *    sequences.  A kernel that only ends, or one of this library's kernels, is
 *    always safe before it.  A caller's own kernel that releases its dependents
 *    early (griddepcontrol.launch_dependents) must do so only after its last write
 *    to context_lens, and must not touch out or the workspace after that point.
 *  - Alignment: q, k, v, out, k_cache, v_cache must be 16-byte aligned, and
 *    head_dim * element size must be a multiple of 16 bytes.
 *  - Errors: a call returns PKV_OK or an error status and records a message that
 *    paged_kv_last_error() returns (per host thread).  Host checks cover shapes,
 *    scalars, pointers and alignment.  Device-side index faults never trap: a
 *    kernel that meets an out-of-range block id or slot, or a bounded wait that
 *    runs out, sets a device flag, skips the access and completes;
 *    paged_kv_device_error() reports and clears that flag.
 *  - Supported set: dtype f32, f16, bf16 (q, k, v, caches share it); out dtype
 *    either that dtype or f32; head_dim 64 or 128; block_size 8, 16, 32 or 64;
 *    num_q_heads a multiple of num_kv_heads.  Group size (query heads per KV head)
 *    up to 8 on the CUDA-core decode path; on the tensor-core decode path up to 16
 *    for f16/bf16 and up to 8 for f32 (tf32 MMAs on split operands: scores to about
 *    2^-21 relative, within the f32 tolerance for logits of a few units; for logits
 *    of tens of units choose PKV_PATH_CUDA_CORE, fp32 throughout); prefill on tensor
 *    cores for f16/bf16, groups up to 16.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { PKV_F32 = 0, PKV_F16 = 1, PKV_BF16 = 2 } pkv_dtype;

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1,    /* bad pointer, shape, scalar or alignment */
  PKV_ERR_UNSUPPORTED = 2,    /* outside the supported set above */
  PKV_ERR_WORKSPACE = 3,      /* workspace missing or smaller than required */
  PKV_ERR_CUDA = 4,           /* a CUDA runtime call or launch failed */
  PKV_ERR_DEVICE_INDEX = 5,   /* a kernel met an out-of-range block id, slot or length */
  PKV_ERR_DEVICE_TIMEOUT = 6, /* a kernel's bounded wait ran out (copy never landed) */
  PKV_ERR_OUT_OF_BLOCKS = 7   /* block manager: not enough free physical blocks */
} pkv_status;

/* Geometry of one layer's block pool (both k_cache and v_cache). */
typedef struct {
  int32_t num_blocks;   /* physical blocks in the pool */
  int32_t block_size;   /* tokens per block: 8, 16, 32 or 64 */
  int32_t num_kv_heads;
  int32_t head_dim;     /* 64 or 128 */
  int32_t dtype;        /* pkv_dtype of the caches, q, k and v */
} pkv_cache_desc;

/* Decode path selection and split-K partition size (NULL config = automatic: tensor
 * cores for f16/bf16 with groups <= 16 and for f32 at head_dim 128 with groups 5 to 8,
 * CUDA cores otherwise). */
typedef enum { PKV_PATH_AUTO = 0, PKV_PATH_CUDA_CORE = 1, PKV_PATH_TENSOR_CORE = 2 } pkv_path;

typedef struct {
  int32_t path;              /* pkv_path */
  int32_t partition_tokens;  /* 0 = automatic, else a positive multiple of 128 */
} pkv_decode_config;

/*
 * paged_kv_append -- write new tokens' K and V into their cache slots.
 * Pages: "Efficient Memory Management ... with PagedAttention", How It Works (blocks
 * filled as tokens are generated, allocated on demand); note-023, Method.
 *
 * For each token t with slot_mapping[t] >= 0 and every KV head h:
 *   k_cache[slot / block_size][h][slot % block_size][:] = k[t][h][:], same for v.
 * Bit-exact copies.  Slots must be distinct (duplicates race).  A slot
 * >= num_blocks * block_size sets the device index flag and is skipped.
 * k, v: device [num_tokens][num_kv_heads][head_dim]; slot_mapping: device int64.
 */
pkv_status paged_kv_append(const void* k, const void* v, const int64_t* slot_mapping,
                           int32_t num_tokens, void* k_cache, void* v_cache,
                           const pkv_cache_desc* cache, void* stream);

/*
 * paged_block_copy -- copy-on-write divergence: block dst becomes a copy of block
 * src in both pools (all KV heads and rows).
 * Pages: note-023, Concepts (copy-on-write gives the writer its own copy of a shared
 * block); "Paged Attention" glossary, paragraph 2; "Efficient Memory Management ...",
 * How It Works (copy when a sequence sharing a prefix diverges).
 *
 * src_dst_pairs: device int64 [num_pairs][2].  host_pairs: optional host copy of the
 * same pairs; when given, the call checks every id is in [0, num_blocks), src != dst,
 * no dst repeats and no dst is also a src (PKV_ERR_INVALID_ARG otherwise).  Without
 * it, out-of-range ids set the device index flag and are skipped; overlapping pairs
 * are the caller's responsibility.  Bit-exact.
 */
pkv_status paged_block_copy(const int64_t* src_dst_pairs, const int64_t* host_pairs,
                            int32_t num_pairs, void* k_cache, void* v_cache,
                            const pkv_cache_desc* cache, void* stream);

/* What paged_attention_decode will do for these sizes and config. */
typedef struct {
  int32_t path;              /* pkv_path actually taken (never PKV_PATH_AUTO) */
  int32_t partition_tokens;  /* tokens per split-K partition */
  int32_t max_partitions;    /* partitions of the longest sequence (1 = no merge) */
  int32_t kernel_launches;   /* kernels one call enqueues */
  size_t workspace_bytes;    /* as paged_attention_workspace_bytes */
  int32_t kv_heads_per_item; /* tensor-core path: KV heads one work item covers; 2 for f16/bf16
                                at head_dim 64 with an even number of KV heads (their tiles of a
                                block are adjacent and load as one head_dim-128 tile), else 1 */
} pkv_decode_plan;

/*
 * paged_attention_plan -- fill *out with the plan paged_attention_decode follows for
 * these arguments (host only, no device work).  Automatic partitions: on CUDA cores
 * 512 to 2048 tokens, aiming at about 12 CTAs per SM; on tensor cores the largest
 * size up to 4096 that leaves about three (sequence, KV head, partition) items per SM
 * (lengths assumed to average half of max_context_len).  Errors as
 * paged_attention_decode's argument checks.
 */
pkv_status paged_attention_plan(int32_t num_seqs, int32_t num_q_heads, int32_t max_context_len,
                                const pkv_cache_desc* cache, const pkv_decode_config* config,
                                pkv_decode_plan* out);

/*
 * paged_block_swap_out / paged_block_swap_in -- preemption under memory pressure: move
 * whole blocks (all KV heads and rows of K and V) between the pools and CPU memory, so
 * a preempted sequence can be restored later and continue exactly where it stopped.
 * Pages: "Paged Attention" glossary, paragraphs 3 and 5 (blocks of preempted sequences
 * are evicted to CPU RAM and swapped back, generation resumes where it left off);
 * "Efficient Memory Management ...", How It Works (preemption and swapping).
 *
 * block_ids: device int64 [num_ids].  host_k, host_v: [num_ids][num_kv_heads]
 * [block_size][head_dim] in the cache dtype, in pinned (cudaHostAlloc /
 * cudaHostRegister) host memory, or device memory; pageable memory is refused with
 * PKV_ERR_INVALID_ARG.  swap_out copies pool block block_ids[i] to entry i; swap_in
 * copies entry i into pool block block_ids[i].  Bit-exact.  Out-of-range ids set the
 * device index flag and are skipped.  Stream-ordered like every other call: issue the
 * swap-out before anything reuses the blocks.
 */
pkv_status paged_block_swap_out(const int64_t* block_ids, int32_t num_ids, const void* k_cache,
                                const void* v_cache, void* host_k, void* host_v,
                                const pkv_cache_desc* cache, void* stream);
pkv_status paged_block_swap_in(const int64_t* block_ids, int32_t num_ids, const void* host_k,
                               const void* host_v, void* k_cache, void* v_cache,
                               const pkv_cache_desc* cache, void* stream);

/*
 * Bytes of workspace paged_attention_decode needs for these sizes and config.  The
 * CUDA-core path needs none when every sequence fits one partition; the tensor-core
 * path always needs room for its work list (16 bytes per (sequence, KV head,
 * partition) plus a 256-byte header holding the entry count and the counter from
 * which the CTAs claim entries) and, past one partition, the partition partials.
 * Two calls in flight at once (on different streams) need separate workspaces.
 * max_context_len: host upper bound on context_lens.  Returns 0 for invalid
 * arguments as well (then the decode call itself reports the error).
 */
size_t paged_attention_workspace_bytes(int32_t num_seqs, int32_t num_q_heads,
                                       int32_t max_context_len, const pkv_cache_desc* cache,
                                       const pkv_decode_config* config);

/*
 * paged_attention_decode -- single-token decode attention through block tables.
 * Pages: note-023, Method and Concepts (attention gathers K/V through the block
 * table from non-contiguous blocks); "Paged Attention" glossary, paragraph 4
 * (arithmetic unchanged) and GQA paragraph.
 *
 * For every sequence s and query head h, with n = context_lens[s], kv = h / G,
 * K_j / V_j = row j % block_size of physical block block_tables[s][j / block_size]:
 *   out[s][h][:] = sum_j softmax_j(scale * q[s][h] . K_j) V_j,   j < n;
 *   n == 0 gives zeros.  Accumulation in fp32; out rounded to out_dtype (RNE).
 * Sequences longer than the partition size are split into partitions whose
 * (max, sum, unnormalised output) go to the workspace and are merged by a second
 * kernel.  max_context_len: host upper bound on context_lens (a longer sequence
 * sets the device index flag).  workspace: device, at least
 * paged_attention_workspace_bytes(...) bytes, 256-byte aligned; NULL allowed when
 * that is 0.  out must not alias any input.
 */
pkv_status paged_attention_decode(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* block_tables, int32_t max_blocks_per_seq,
                                  const int32_t* context_lens, int32_t num_seqs,
                                  int32_t num_q_heads, int32_t max_context_len, float scale,
                                  void* out, int32_t out_dtype, void* workspace,
                                  size_t workspace_bytes, const pkv_cache_desc* cache,
                                  const pkv_decode_config* config, void* stream);

/*
 * paged_attention_decode_no_alloc -- paged_attention_decode for callers that must not
 * allocate device memory (allocator or memory-pool callbacks, serving paths that may
 * not fail with out-of-memory once running, runtimes that only pass pre-registered
 * buffers).  The pages have no counterpart: this is a packaging of the same decode.
 *
 * Same arguments and result as paged_attention_decode, minus the workspace: the
 * scratch comes from a fixed array of paged_attention_no_alloc_limit() bytes
 * (32 MiB) that every GPU loading the library holds until the process exits.  The
 * call allocates nothing.  Sizes whose workspace would exceed the array return
 * PKV_ERR_WORKSPACE (pass a larger partition_tokens, or use paged_attention_decode).
 * The first call on a device looks up the array's device address (with that device
 * current) and caches it; make that first call before any stream capture.  All calls
 * share the one array: calls that overlap on the GPU (other streams, other threads)
 * race on it and must be serialised by the caller.  Nothing in the array needs to
 * start at zero; each call writes what it reads.
 */
pkv_status paged_attention_decode_no_alloc(const void* q, const void* k_cache, const void* v_cache,
                                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                                           const int32_t* context_lens, int32_t num_seqs,
                                           int32_t num_q_heads, int32_t max_context_len, float scale,
                                           void* out, int32_t out_dtype, const pkv_cache_desc* cache,
                                           const pkv_decode_config* config, void* stream);

/* Bytes of the built-in array paged_attention_decode_no_alloc uses. */
size_t paged_attention_no_alloc_limit(void);

/*
 * paged_attention_prefill -- several new tokens per sequence (prefill, chunked prefill)
 * attending through block tables with a causal mask.
 * Pages: note-023, Method (attention gathers K/V through the block table) and Open
 * questions (chunked prefill); attention arithmetic unchanged ("Paged Attention"
 * glossary, paragraph 4).
 *
 * Sequence s brings n_s = query_start[s+1] - query_start[s] new tokens: rows
 * query_start[s] .. query_start[s+1]-1 of q and out ([num_query_tokens][Hq][D]),
 * the last n_s of its context_lens[s] tokens, whose K/V are already in the pool
 * (paged_kv_append first).  New token i at position p = context_lens[s] - n_s + i:
 *   out[row][h] = sum_{j <= p} softmax_j(scale * q[row][h] . K_j) V_j.
 * query_start: device int32 [num_seqs + 1], non-decreasing, query_start[0] = 0 and
 * query_start[num_seqs] = num_query_tokens.  A sequence with n_s > context_lens[s]
 * or context_lens[s] > max_context_len sets the device index flag and is skipped.
 * Tensor cores only: f16/bf16, head_dim 64 or 128, query-head groups <= 16, block size 8,
 * 16, 32 or 64, at most 4095 KV heads (else PKV_ERR_UNSUPPORTED); q, out and the pools
 * 16-byte aligned.  workspace: at least paged_attention_prefill_workspace_bytes(...)
 * bytes, 256-byte aligned.
 */
size_t paged_attention_prefill_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t num_query_tokens,
                                               const pkv_cache_desc* cache);
pkv_status paged_attention_prefill(const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_tables, int32_t max_blocks_per_seq,
                                   const int32_t* context_lens, const int32_t* query_start, int32_t num_seqs,
                                   int32_t num_q_heads, int32_t num_query_tokens, int32_t max_context_len,
                                   float scale, void* out, int32_t out_dtype, void* workspace,
                                   size_t workspace_bytes, const pkv_cache_desc* cache, void* stream);

/*
 * paged_kv_gather -- the block-table lookup alone (testing the indexing bit-exactly):
 * k_out[s][h][j][:] = k_cache[block_tables[s][j / bs]][h][j % bs][:] for j < n_s,
 * same for v.  Rows j >= context_lens[s] are not written.
 * k_out, v_out: device [num_seqs][num_kv_heads][max_context_len][head_dim].
 */
pkv_status paged_kv_gather(const void* k_cache, const void* v_cache, const int32_t* block_tables,
                           int32_t max_blocks_per_seq, const int32_t* context_lens,
                           int32_t num_seqs, int32_t max_context_len, void* k_out, void* v_out,
                           const pkv_cache_desc* cache, void* stream);

/* ----------------------------------------------------------------------------------
 * Host block manager: which physical block every token lives in.
 * Pages: note-023, Method (allocate on demand as a sequence grows, free when it
 * finishes, share blocks between sequences with identical prefixes, copy on write when
 * one diverges) and Concepts (internal fragmentation = unused tail of the last block);
 * "Paged Attention" glossary, paragraphs 1-3; "PagedAttention & Continuous Batching",
 * shared-system-prompt paragraph (blocks of a finished request go to the next one).
 *
 * Host memory only; not thread-safe (one manager per host thread, or a caller lock).
 * Policy: free blocks form a LIFO stack (first hands out 0, 1, 2, ...; freed blocks are
 * reused first).  Every call either succeeds as a whole or changes nothing.
 * ---------------------------------------------------------------------------------- */
typedef struct pkv_block_manager pkv_block_manager;

typedef struct {
  int32_t num_blocks, free_blocks, used_blocks, num_sequences;
  int32_t shared_blocks;   /* blocks referenced by more than one sequence */
  int64_t stored_tokens;   /* valid rows held in used blocks (shared rows counted once) */
  int64_t logical_tokens;  /* sum of sequence lengths (shared rows counted per sharer) */
  int64_t allocated_slots; /* used_blocks * block_size */
  int64_t max_len;         /* longest sequence */
  int64_t copies;          /* copy-on-write copies made so far */
  int64_t swapped;         /* sequences swapped out (holding no blocks) */
} pkv_block_stats;

/* A manager for a pool of num_blocks blocks of block_size tokens.  Free with destroy. */
pkv_status pkv_bm_create(int32_t num_blocks, int32_t block_size, pkv_block_manager** out);
void pkv_bm_destroy(pkv_block_manager* manager);

/* A new sequence with a prompt of num_tokens tokens: ceil(num_tokens / block_size)
 * fresh blocks.  PKV_ERR_OUT_OF_BLOCKS if the pool cannot hold them. */
pkv_status pkv_bm_add_sequence(pkv_block_manager* manager, int64_t seq_id, int64_t num_tokens);

/* child shares every block of parent by reference (parallel sampling, beam search). */
pkv_status pkv_bm_fork(pkv_block_manager* manager, int64_t parent, int64_t child);

/*
 * Reserve the slot of one new token for each of n distinct sequences, in order.  A
 * sequence at a block boundary takes a fresh block; one whose last block is shared
 * gets a fresh copy of it first (copy-on-write) and the pair (old, fresh) is appended
 * to cow_pairs ([n][2] capacity, *num_cow set).  slots[i] = block * block_size + row,
 * ready for paged_kv_append; apply the pairs with paged_block_copy before the append.
 */
pkv_status pkv_bm_append(pkv_block_manager* manager, const int64_t* seq_ids, int32_t n, int64_t* slots,
                         int64_t* cow_pairs, int32_t* num_cow);

/* The sequence finished: drop its references; blocks no longer referenced are freed. */
pkv_status pkv_bm_free_sequence(pkv_block_manager* manager, int64_t seq_id);

/*
 * Preemption: *num_out = the sequence's blocks in logical order, copied to blocks_out
 * (capacity entries), and the sequence drops its references (blocks nobody else
 * holds become free).  The sequence stays known, with its length, as swapped out:
 * copy those blocks out with paged_block_swap_out before anything reuses them.
 */
pkv_status pkv_bm_swap_out(pkv_block_manager* manager, int64_t seq_id, int32_t* blocks_out, int32_t capacity,
                           int32_t* num_out);

/* Restore a swapped-out sequence into fresh private blocks, listed in logical order;
 * copy its data back into them with paged_block_swap_in.  PKV_ERR_OUT_OF_BLOCKS if
 * the pool cannot hold it (nothing changes). */
pkv_status pkv_bm_swap_in(pkv_block_manager* manager, int64_t seq_id, int32_t* blocks_out, int32_t capacity,
                          int32_t* num_out);

/* Rows of block_tables ([n][max_blocks], -1 padded) and context_lens for n sequences. */
pkv_status pkv_bm_block_tables(const pkv_block_manager* manager, const int64_t* seq_ids, int32_t n,
                               int32_t max_blocks, int32_t* tables, int32_t* lens);

pkv_status pkv_bm_stats(const pkv_block_manager* manager, pkv_block_stats* out);

/* Message of the last failed call on this host thread ("" if none). */
const char* paged_kv_last_error(void);

/*
 * Synchronise `stream`, then read and clear the device error flag of the current
 * device: PKV_OK, PKV_ERR_DEVICE_INDEX or PKV_ERR_DEVICE_TIMEOUT (PKV_ERR_CUDA if
 * the synchronisation itself fails).
 */
pkv_status paged_kv_device_error(void* stream);

/*
 * Diagnostic (no counterpart on the pages): enqueue one kernel whose bounded wait can
 * never complete -- an mbarrier expecting an arrival nobody makes -- so that the wait
 * gives up after limit_ns (at most 5 s), records PKV_ERR_DEVICE_TIMEOUT in the device
 * flag and returns.  Shows that a stuck wait ends with a status the host reads and
 * leaves the context usable; every wait in the library's kernels ends the same way
 * (their limit is 2 s).
 */
pkv_status paged_kv_selftest_wait_timeout(uint64_t limit_ns, void* stream);

/*
 * Diagnostic (no counterpart on the pages): set the bound of the pipeline waits in
 * the decode and prefill kernels launched from now on, process-wide (0 restores the
 * default of 2 s; at most 5 s, else PKV_ERR_INVALID_ARG).  A bound far below a
 * healthy wait (say 1 us) makes a normal call give up part-way: its kernels then take
 * their abort path -- they wait (each up to 2 s) for the copies and MMAs they have in
 * flight, free their tensor memory, record PKV_ERR_DEVICE_TIMEOUT in the device flag
 * and return -- so that path can be exercised without any real fault.  The output of
 * such a call is undefined.  Not for production use.
 */
pkv_status paged_kv_set_wait_limit(uint64_t limit_ns);

/* Library version, e.g. "0.1.0". */
const char* paged_kv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
