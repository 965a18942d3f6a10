/*
 * pa.h -- C ABI of libpa, the paged KV-cache hot path for NVIDIA GB300 (sm_103a).
 *
 * Device entry points enqueue work on the caller's CUDA stream and return as
 * soon as the work is queued. They never allocate device memory, never
 * synchronise, and check their host arguments before any launch: a call that
 * returns anything but PA_OK has enqueued nothing. Faults inside a kernel
 * surface at the caller's next synchronisation, as usual in CUDA.
 * State the library keeps (nothing else): one device status word per device
 * (pa_device_status) and the fixed scratch of pa_decode_static_scratch. Every
 * kernel runs on the caller's stream; the library creates no stream or event.
 *
 * Conventions shared by every entry point
 *  - Pointers named *_cache, query, key, value, new_key, new_value, out,
 *    block_tables, context_lens, slot_mapping, block_mapping, tmp_out,
 *    max_logits, exp_sums and workspace are caller-owned DEVICE memory, contiguous,
 *    row-major, 16-byte aligned. The library keeps no reference after the
 *    call returns.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream), so that this header needs no CUDA include.
 *  - KV cache layout: k_cache and v_cache are [num_blocks, block_size,
 *    num_kv_heads, head_dim]; slot s = block * block_size + offset addresses
 *    row s of the cache viewed as [num_blocks * block_size, num_kv_heads,
 *    head_dim].
 *  - Block tables: [num_seqs, max_blocks_per_seq] int32; entry j of row b is
 *    the physical block that holds tokens [j*block_size, (j+1)*block_size) of
 *    sequence b. Entries at or past cdiv(context_lens[b], block_size) are
 *    never read.
 *
 * The source pages this follows are cited by title and section:
 *  [P1] "PagedAttention: KV cache virtual memory" (news.ainew.jp, Arc 6)
 *  [P3] "PagedAttention, explained." (vibeengines.com)
 *  [P4] "What Does PagedAttention Actually Optimize?" (hrletsgo.me)
 *  [P5] "Paged Attention: Virtual Memory for the KV Cache" (theservingstack.com)
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, inconsistent shapes */
    PA_ERR_UNSUPPORTED = 2,   /* a shape / dtype combination no kernel handles */
    PA_ERR_OUT_OF_BLOCKS = 3, /* block manager: the free list cannot satisfy the request */
    PA_ERR_WORKSPACE = 4,     /* workspace missing or smaller than pa_decode_workspace_size() */
    PA_ERR_TIMEOUT = 5,       /* a kernel gave up waiting on an async copy (see pa_device_status) */
    PA_ERR_CUDA = 6,          /* a CUDA runtime call failed (launch or attribute error) */
    PA_ERR_NOT_FOUND = 7      /* block manager: unknown sequence id */
} pa_status;

/* Element types. The KV-size estimate of [P4] section 2 counts fp16 and bf16
 * alike, two bytes a value; both run the same tensor-core kernels here, fp32
 * the CUDA-core one. */
typedef enum pa_dtype {
    PA_F32 = 0,
    PA_BF16 = 1,
    PA_F16 = 2
} pa_dtype;

/* Human-readable text of a status code (static storage, never NULL). */
PA_API const char *pa_status_string(pa_status status);

/* ABI version of this header (increases on any incompatible change). */
#define PA_ABI_VERSION 2
PA_API int pa_abi_version(void);

/* ------------------------------------------------------------------------
 * Slot scatter ("reshape_and_cache").
 * [P3] procedure step 4 (each generated token's key and value go into the
 * next free slot of the sequence's last block) and "Across GPUs" (fused
 * kernels that write new keys and values into blocks); [P5] "Finding a
 * token: position, block, slot" (slot = block number * block size + offset).
 *
 *   key, value    [num_tokens, num_kv_heads, head_dim], dtype kv_dtype
 *   slot_mapping  [num_tokens] int64; token i is written to slot
 *                 slot_mapping[i] of both caches (all heads, all dims).
 *                 A negative slot skips the token (padding). A slot at or
 *                 past num_blocks * block_size is skipped too (never written).
 *   Distinct tokens must map to distinct slots; if two share a slot, which
 *   one lands is unspecified.
 *   Requires (num_kv_heads * head_dim * element size) % 16 == 0.
 *   num_tokens == 0 is a no-op returning PA_OK.
 * ---------------------------------------------------------------------- */
PA_API pa_status pa_reshape_and_cache(const void *key, const void *value, void *k_cache,
                                      void *v_cache, const int64_t *slot_mapping, int num_tokens,
                                      int num_blocks, int block_size, int num_kv_heads,
                                      int head_dim, pa_dtype kv_dtype, void *stream);

/* ------------------------------------------------------------------------
 * Copy-on-write block copy ("copy_blocks").
 * [P1] "Copy-on-write: when two requests share a prefix" (clone the one block
 * being written); [P3] procedure step 6 and "Across GPUs" (the block copies
 * copy-on-write needs).
 *
 *   block_mapping [num_pairs, 2] int64 (src, dst): block dst of k_cache and of
 *                 v_cache becomes a byte copy of block src.
 *   Preconditions: dst ids distinct and disjoint from src ids (otherwise
 *   the result depends on copy order). They are not checked: the mapping is
 *   device memory, and checking it would cost a copy to the host and a
 *   synchronisation. pa_bm_append_slot only ever produces such pairs (each
 *   dst is a block just taken from the free queue). Pairs with an id outside
 *   [0, num_blocks) are skipped. num_pairs == 0 is a no-op.
 * ---------------------------------------------------------------------- */
PA_API pa_status pa_copy_blocks(void *k_cache, void *v_cache, const int64_t *block_mapping,
                                int num_pairs, int num_blocks, int block_size, int num_kv_heads,
                                int head_dim, pa_dtype kv_dtype, void *stream);

/* ------------------------------------------------------------------------
 * Block swap between two pools ("swap_blocks"), e.g. GPU cache <-> CPU pool.
 * [P3] procedure steps 7-8 (a preempted request's blocks are copied to CPU
 * memory and back) and the ablations (small blocks make swapping slow: many
 * small transfers); [P4] section 12 (moving KV blocks of lower-priority
 * requests to CPU memory, at block granularity).
 *
 *   src_k, src_v  [src_num_blocks, block_size, num_kv_heads, head_dim] pools
 *   dst_k, dst_v  [dst_num_blocks, block_size, num_kv_heads, head_dim] pools
 *                 Each may be device memory or page-locked host memory
 *                 (cudaHostAlloc / cudaHostRegister, e.g. a pinned tensor);
 *                 pageable host memory returns PA_ERR_INVALID_ARG.
 *   block_mapping [num_pairs, 2] int64 (src id, dst id), device or
 *                 page-locked host memory: block dst of dst_k / dst_v becomes
 *                 a byte copy of block src of src_k / src_v. Pairs with an id
 *                 outside its pool are skipped.
 *   One kernel moves every pair (no per-block copy call). Destination
 *   blocks must be distinct and must not overlap the sources.
 *   num_pairs == 0 is a no-op. Asynchronous on `stream`.
 * ---------------------------------------------------------------------- */
PA_API pa_status pa_swap_blocks(void *dst_k, void *dst_v, const void *src_k, const void *src_v,
                                const int64_t *block_mapping, int num_pairs, int src_num_blocks,
                                int dst_num_blocks, int block_size, int num_kv_heads, int head_dim,
                                pa_dtype kv_dtype, void *stream);

/* ------------------------------------------------------------------------
 * Paged single-query (decode) attention.
 * [P4] section 8 (Attention(Q,K,V) = softmax(QK^T / sqrt(d)) V, unchanged by
 * paging) and section 14 (per step: read the block table, find each
 * position's logical block, translate to the physical block, add the
 * offset, read K and V, compute scores and the weighted sum); [P3] step 5
 * (fetch key and value blocks wherever the table says, block by block).
 * Grouped-query attention: query head h reads KV head h / (num_heads /
 * num_kv_heads) ([P3], legend of the KV-size formula).
 *
 *   out          [num_seqs, num_heads, head_dim], out_dtype (F32, BF16 or F16)
 *   query        [num_seqs, num_heads, head_dim], q_dtype
 *   context_lens [num_seqs] int32: tokens attended by each sequence (the
 *                token written this step included). 0 gives an all-zero row.
 *   max_context_len  host-side upper bound of context_lens (sizes the grid;
 *                tokens past it are not attended).
 *   scale        multiplies q.k (normally 1/sqrt(head_dim)).
 *   workspace    scratch for a wide context split: at least
 *                pa_decode_workspace_size() bytes (0 when the plan needs
 *                none), or NULL / 0 bytes. Splits of up to 8 partitions are
 *                merged inside a thread-block cluster and need no workspace;
 *                wider ones need it (without it the split is capped at 8,
 *                or, on the CUDA-core kernel, not split at all). Its
 *                contents need no initialisation. Calls that share a
 *                workspace must not overlap on the GPU.
 *   Supported: head_dim 64 or 128; num_heads % num_kv_heads == 0;
 *   (q, kv) dtypes (F32, F32), (BF16, BF16) or (F16, F16); block_size
 *   1..256. bf16 and fp16 caches whose block_size is a power of two (1 to
 *   256) run the tensor-core kernel, the rest the CUDA-core kernel.
 *   Ragged batches: with a workspace, blocks of 16 or more and so many
 *   sequences (2 to 2,048) that the per-partition plan would cut each
 *   context at most twice, the tensor-core path cuts the whole batch's
 *   16-token tiles, sequence after sequence, into equal ranges per CTA on
 *   the device (where the lengths are) and merges the pieces of sequences
 *   that straddle two ranges: every CTA gets the same work however ragged
 *   the lengths. PA_DECODE_BALANCE=0 / 1 turns it off / on wherever it
 *   applies.
 * ---------------------------------------------------------------------- */
PA_API size_t pa_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads,
                                       int head_dim, int block_size, int max_context_len);

/* How pa_decode will run a problem on the current device (host only, no
 * launch): which kernel, how the context is split and merged, and how many
 * kernels one call launches. with_workspace: 1 if the call will pass a
 * workspace of pa_decode_workspace_size() bytes, 0 if it passes none. */
typedef struct pa_decode_plan_t {
    int tensor_cores;       /* 1: tensor-core kernel; 0: CUDA-core kernel */
    int heads_per_cta;      /* KV heads one CTA serves */
    int num_splits;         /* partitions per context (1: not split) */
    int partition_tokens;   /* tokens per partition */
    int cluster_merge;      /* 1: partitions merged inside a thread-block cluster */
    int kernel_launches;    /* kernels one call launches: 1, or 2 (decode + merge) */
    size_t workspace_bytes; /* workspace the plan uses (0: none) */
    int balanced;           /* 1: ragged-balanced decode (num_splits = CTAs per KV-head
                               group, partition_tokens 0: ranges are cut on the device) */
} pa_decode_plan_t;

PA_API pa_status pa_decode_plan(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                int block_size, int max_context_len, pa_dtype kv_dtype,
                                int with_workspace, pa_decode_plan_t *plan);

PA_API pa_status pa_decode(void *out, pa_dtype out_dtype, const void *query, pa_dtype q_dtype,
                           const void *k_cache, const void *v_cache, pa_dtype kv_dtype,
                           const int32_t *block_tables, const int32_t *context_lens,
                           int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                           int block_size, int max_blocks_per_seq, int num_blocks,
                           int max_context_len, float scale, void *workspace,
                           size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * One decode step ([P3] steps 4 and 5): each sequence's new token is written
 * into the next slot of its last block -- position context_lens[b] - 1,
 * its slot found through block_tables -- and then attention runs over the
 * whole context, new token included. Same result as pa_reshape_and_cache
 * with those slots followed by pa_decode. The per-partition tensor-core
 * kernel writes the new tokens itself: the CTA that reads a token's tile
 * stores the token first (no scatter launch). Other plans launch a small
 * scatter ahead of the decode.
 *   new_key, new_value  [num_seqs, num_kv_heads, head_dim], the cache's dtype
 *   every other argument as pa_decode
 * A sequence with context_len 0 writes nothing; so does one whose length
 * the decode cuts short (past the table's reach; a length past
 * max_context_len breaks the call's contract, as for pa_decode). All
 * arguments are checked before anything is launched, so a refused call
 * writes nothing.
 * ---------------------------------------------------------------------- */
PA_API pa_status pa_decode_append(void *out, pa_dtype out_dtype, const void *query, pa_dtype q_dtype,
                                  const void *new_key, const void *new_value, void *k_cache,
                                  void *v_cache, pa_dtype kv_dtype, const int32_t *block_tables,
                                  const int32_t *context_lens, int num_seqs, int num_heads,
                                  int num_kv_heads, int head_dim, int block_size,
                                  int max_blocks_per_seq, int num_blocks, int max_context_len,
                                  float scale, void *workspace, size_t workspace_bytes,
                                  void *stream);

/* ------------------------------------------------------------------------
 * Decode attention for a batch whose sequences share their leading blocks.
 * [P1] "Copy-on-write: when two requests share a prefix" (several block
 * tables point at the same physical blocks, reference-counted); [P5]
 * "Sharing a prefix: one copy for many requests" (the prefix is stored
 * once). pa_decode reads a shared block once per sequence; this entry point
 * reads it once for the whole batch: the shared tokens are attended for
 * every (sequence, query head) row by one pass, the rest of each context by
 * the paged decode kernel, and the two are merged by log-sum-exp. The result
 * is pa_decode's (the same softmax over the same tokens).
 *
 *   shared_blocks  the number of leading block-table entries that are the
 *                  same physical blocks in every row of block_tables, and
 *                  full: every context_len >= shared_blocks * block_size.
 *                  (Not checked on the device. Rows that differ give that
 *                  row's wrong answer, never an out-of-bounds access.)
 *                  Shared tokens are taken in whole 16-token tiles (blocks
 *                  of 8: an odd last shared block is attended with the rest).
 *   workspace      at least pa_decode_shared_prefix_workspace_size() bytes
 *                  (required: the two passes meet there). Its contents need
 *                  no initialisation; calls sharing it must not overlap.
 *   Other arguments as pa_decode. Supported: bf16 or fp16 query and cache, head_dim
 *   64 or 128, block_size 8, 16, 32, 64, 128 or 256. With no whole tile
 *   shared this is pa_decode.
 *   Launches: three kernels on `stream` (capturable into a CUDA graph): the
 *   prefix pass, the rest-of-context decode, the merge. The decode is
 *   launched as a programmatic dependent of the prefix pass and runs beside
 *   it, on the SMs the pass's plan leaves free; neither reads the other's
 *   output, and the decode completes only after the pass has, so the merge
 *   sees both. PA_PREFIX_ORDER=rest puts the decode first (the pass then
 *   fills the SMs it frees); PA_PREFIX_OVERLAP=0 runs the two one after the
 *   other. With PA_PREFIX_KERNEL=mma the decode goes first.
 * ---------------------------------------------------------------------- */
PA_API size_t pa_decode_shared_prefix_workspace_size(int num_seqs, int num_heads, int num_kv_heads,
                                                     int head_dim, int block_size,
                                                     int max_context_len, int shared_blocks);

PA_API pa_status pa_decode_shared_prefix(void *out, pa_dtype out_dtype, const void *query,
                                         pa_dtype q_dtype, const void *k_cache,
                                         const void *v_cache, pa_dtype kv_dtype,
                                         const int32_t *block_tables, const int32_t *context_lens,
                                         int num_seqs, int num_heads, int num_kv_heads,
                                         int head_dim, int block_size, int max_blocks_per_seq,
                                         int num_blocks, int max_context_len, int shared_blocks,
                                         float scale, void *workspace, size_t workspace_bytes,
                                         void *stream);

/* ------------------------------------------------------------------------
 * Decode attention over a contiguous (unpaged) cache: the baseline that
 * paging is measured against.
 * [P5] "The problem: reserving the maximum" (one buffer per request, sized
 * for its maximum length) and "What paging costs" (indirection: attention
 * reads through the block table, 20-26 % slower than a contiguous kernel of
 * the time); [P1] "Why the attention kernel works at all" (the lookup cost
 * is amortised over a block, single-digit percent).
 *
 *   k, v         [num_seqs, max_seq_len, num_kv_heads, head_dim] bf16 or fp16:
 *                sequence b's token t at row b * max_seq_len + t. No block
 *                table: the same kernel as pa_decode, with the block id
 *                lookup replaced by the token offset.
 *   max_seq_len  the reservation per sequence (rows per sequence).
 *   context_lens [num_seqs] int32, each in [0, max_seq_len] (larger values
 *                are clamped to max_seq_len).
 *   max_context_len  host upper bound of context_lens, <= max_seq_len.
 *   workspace    as pa_decode, sized by pa_decode_workspace_size() with
 *                block_size 16.
 *   Other arguments as pa_decode. Supported: bf16 or fp16 query and cache (F32
 *   returns PA_ERR_UNSUPPORTED), head_dim 64 or 128,
 *   num_seqs * max_seq_len < 2^31.
 * ---------------------------------------------------------------------- */
PA_API pa_status pa_decode_contiguous(void *out, pa_dtype out_dtype, const void *query,
                                      pa_dtype q_dtype, const void *k, const void *v,
                                      pa_dtype kv_dtype, const int32_t *context_lens,
                                      int num_seqs, int num_heads, int num_kv_heads,
                                      int head_dim, int max_seq_len, int max_context_len,
                                      float scale, void *workspace, size_t workspace_bytes,
                                      void *stream);

/* ------------------------------------------------------------------------
 * Decode for callers that cannot allocate device memory. (The source pages
 * have no counterpart: this is a library convenience.)
 *
 * Some callers cannot provide the scratch pa_decode may need: an engine whose
 * device memory is reserved up front by another allocator (cudaMalloc would
 * fail there or bypass its accounting), or a plugin interface that passes only
 * the operation's inputs and outputs. This entry point computes what pa_decode
 * computes, with the same arguments minus the workspace, and allocates
 * nothing. It splits a context as pa_decode given a workspace does (the
 * ragged-balanced path aside): a split of up to 8 partitions is merged inside
 * a thread-block cluster, in shared memory, and uses no scratch; a wider split
 * writes its partial outputs, maxima and sums into a fixed scratch array built
 * into the library, PA_STATIC_SCRATCH_BYTES bytes of device memory that every
 * GPU loading the library holds until the process exits, and a merge kernel
 * reads them back.
 *  - A problem whose wider split needs more scratch than that returns
 *    PA_ERR_WORKSPACE before anything is launched (use pa_decode with a
 *    workspace of pa_decode_workspace_size() bytes instead).
 *    pa_decode_plan(..., with_workspace = 1) reports the split and its
 *    workspace_bytes for every shape it does not run ragged-balanced.
 *  - The first call on a device looks up the scratch's device address (with
 *    that device current); make that first call before any stream capture.
 *  - Every call writes its partials into the one shared array (nothing in it
 *    needs clearing: each call writes every entry it reads). Calls that
 *    overlap on the GPU (other streams, other threads) therefore overwrite
 *    each other's partials and give wrong results. Serialise them.
 * ---------------------------------------------------------------------- */
#define PA_STATIC_SCRATCH_BYTES (8u << 20)
PA_API pa_status pa_decode_static_scratch(void *out, pa_dtype out_dtype, const void *query,
                                          pa_dtype q_dtype, const void *k_cache,
                                          const void *v_cache, pa_dtype kv_dtype,
                                          const int32_t *block_tables,
                                          const int32_t *context_lens, int num_seqs,
                                          int num_heads, int num_kv_heads, int head_dim,
                                          int block_size, int max_blocks_per_seq, int num_blocks,
                                          int max_context_len, float scale, void *stream);

/* ------------------------------------------------------------------------
 * Split-K decode: attention over fixed partitions of partition_size tokens
 * (a multiple of block_size), to be combined by pa_lse_merge. The pages
 * describe no split; its definition is the plain one: partition p of
 * sequence b is softmax attention over tokens [p*partition_size,
 * min(len, (p+1)*partition_size)), and long contexts still cost reads of
 * every token ([P4] section 15).
 *
 *   tmp_out    [num_seqs, num_heads, max_partitions, head_dim] f32: the
 *              partition's normalised output
 *   max_logits [num_seqs, num_heads, max_partitions] f32: max of scale*q.k
 *   exp_sums   [num_seqs, num_heads, max_partitions] f32: sum of exp(s - max)
 *   with max_partitions = cdiv(max_context_len, partition_size). Partitions
 *   past a sequence's length are written as (0, -inf, 0).
 *   Other arguments as pa_decode.
 * ---------------------------------------------------------------------- */
PA_API pa_status pa_decode_splitk(float *tmp_out, float *max_logits, float *exp_sums,
                                  int partition_size, const void *query, pa_dtype q_dtype,
                                  const void *k_cache, const void *v_cache, pa_dtype kv_dtype,
                                  const int32_t *block_tables, const int32_t *context_lens,
                                  int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                  int block_size, int max_blocks_per_seq, int num_blocks,
                                  int max_context_len, float scale, void *stream);

/* Log-sum-exp merge of pa_decode_splitk's partitions:
 *   M = max_p max_logits[p],  w_p = exp_sums[p] * exp(max_logits[p] - M),
 *   out = sum_p w_p * tmp_out[p] / sum_p w_p   (0 if every w_p is 0).
 * Only partitions p < cdiv(context_lens[b], partition_size) are read. */
PA_API pa_status pa_lse_merge(void *out, pa_dtype out_dtype, const float *tmp_out,
                              const float *max_logits, const float *exp_sums,
                              const int32_t *context_lens, int num_seqs, int num_heads,
                              int head_dim, int max_partitions, int partition_size,
                              void *stream);

/* Device status word: the kernels never spin without a bound. A wait on an
 * asynchronous copy that exceeds its time limit makes the kernel record
 * PA_ERR_TIMEOUT here, drain its own copies and return. This call copies the
 * word to *status (after synchronising `stream`) and, if `clear`, resets it.
 * One word per device, shared by every call on that device. */
PA_API pa_status pa_device_status(int *status, int clear, void *stream);

/* Check of that failure detection on the current device. Launches, on
 * `stream`, one CTA laid out as the decode kernels' pipeline (a producer warp
 * arming a shared-memory stage, a consumer warp waiting for it) whose stage
 * is armed for a copy that is never issued, so the consumer's bounded wait
 * runs out after timeout_us microseconds instead of the kernels' 2 s. The
 * CTA then records PA_ERR_TIMEOUT in the device status word, stops and
 * returns, as a decode kernel would; no copy is ever in flight. Afterwards
 * pa_device_status reports PA_ERR_TIMEOUT (and clears it if asked), and the
 * device stays usable. The status word is shared: do not run this beside
 * decode calls whose status you mean to read. (Not a step of the pages'
 * method: it tests the library's own failure handling, the counterpart of
 * which on the pages is preemption, "PagedAttention, explained.", procedure
 * steps 7-8.)
 *   timeout_us  1 .. 2,000,000 (else PA_ERR_INVALID_ARG). */
PA_API pa_status pa_check_wait_timeout(unsigned timeout_us, void *stream);

/* ------------------------------------------------------------------------
 * Host slot map: slot_mapping[i] = block_tables[seq[i]][pos[i] / block_size]
 *                 * block_size + pos[i] % block_size   (pos[i] < 0 gives -1)
 * [P5] "Finding a token: position, block, slot"; [P4] section 17 (write_kv).
 * All pointers are HOST memory here. Returns PA_ERR_INVALID_ARG if a position
 * falls past max_blocks_per_seq blocks or a sequence index is out of range.
 * ---------------------------------------------------------------------- */
PA_API pa_status pa_compute_slot_mapping(int64_t *slot_mapping, const int32_t *block_tables,
                                         int num_seqs, int max_blocks_per_seq,
                                         const int32_t *seq_index, const int32_t *positions,
                                         int num_tokens, int block_size);

/* ------------------------------------------------------------------------
 * Host block manager (plain C++, host memory only).
 * [P5] "Paging: blocks handed out as tokens arrive" and "Inside vLLM: the
 * block pool": a pool of fixed-size blocks, a free queue (allocation pops the
 * front), cdiv(num_tokens, block_size) blocks for a prompt, one more block
 * each time the last fills, block 0 reserved as the null block, freed blocks
 * returned to the queue front. [P3] procedure steps 1-4 and 6 and [P1]
 * "Copy-on-write": reference counts; a write into a block whose count is
 * above one first clones it (the caller copies the data with
 * pa_copy_blocks), drops the original's count and repoints only the
 * writer's table.
 * Not thread-safe: one handle per thread, or external locking.
 * Sequence ids are arbitrary int64 values chosen by the caller.
 * ---------------------------------------------------------------------- */
typedef struct pa_bm pa_bm;

typedef struct pa_bm_stats_t {
    int64_t num_blocks;     /* usable blocks (the null block excluded) */
    int64_t free_blocks;    /* blocks on the free queue */
    int64_t used_blocks;    /* physical blocks with refcount >= 1 */
    int64_t shared_blocks;  /* physical blocks with refcount >= 2 */
    int64_t num_seqs;
    int64_t logical_blocks; /* sum over sequences of their table lengths */
    int64_t num_tokens;     /* sum over sequences of their token counts */
    int64_t waste_slots;    /* logical_blocks * block_size - num_tokens */
    int64_t cow_copies;     /* copy-on-write clones made so far */
} pa_bm_stats_t;

/* reserve_null_block != 0 keeps block 0 out of the free queue. The free
 * queue starts in ascending id order. */
PA_API pa_status pa_bm_create(int num_blocks, int block_size, int reserve_null_block,
                              pa_bm **out);
/* As pa_bm_create, with the free queue given explicitly (front first):
 * `free_order` lists n distinct ids in [0, num_blocks). */
PA_API pa_status pa_bm_create_with_free_list(int num_blocks, int block_size,
                                             const int32_t *free_order, int n, pa_bm **out);
PA_API void pa_bm_destroy(pa_bm *bm);

/* New sequence holding num_tokens tokens: takes cdiv(num_tokens, block_size)
 * blocks (refcount 1). PA_ERR_OUT_OF_BLOCKS leaves the manager unchanged;
 * PA_ERR_INVALID_ARG if `seq` already exists. */
PA_API pa_status pa_bm_allocate(pa_bm *bm, int64_t seq, int num_tokens);

/* Room for one more token of `seq`. Writes its slot id, and -1/-1 to
 * cow_src/cow_dst, or the (src, dst) pair to copy before writing when the
 * token falls in a shared block. A full last block takes a fresh block.
 * PA_ERR_OUT_OF_BLOCKS leaves the manager unchanged. */
PA_API pa_status pa_bm_append_slot(pa_bm *bm, int64_t seq, int64_t *slot, int64_t *cow_src,
                                   int64_t *cow_dst);

/* `child` starts as a copy of `parent`: same table and token count, one more
 * reference on each block. */
PA_API pa_status pa_bm_fork(pa_bm *bm, int64_t parent, int64_t child);

/* Drops one reference on each of the sequence's blocks; blocks reaching zero
 * return to the front of the free queue, in block-table order. */
PA_API pa_status pa_bm_free(pa_bm *bm, int64_t seq);

/* Copies the sequence's table into out[0..cap) and its length into *n
 * (PA_ERR_INVALID_ARG if cap < *n; *n is still set). */
PA_API pa_status pa_bm_block_table(const pa_bm *bm, int64_t seq, int32_t *out, int cap, int *n);
PA_API pa_status pa_bm_num_tokens(const pa_bm *bm, int64_t seq, int *n);
PA_API pa_status pa_bm_refcount(const pa_bm *bm, int block, int *refcount);
PA_API pa_status pa_bm_stats(const pa_bm *bm, pa_bm_stats_t *out);
/* Free queue, front first (same cap / n convention as pa_bm_block_table). */
PA_API pa_status pa_bm_free_list(const pa_bm *bm, int32_t *out, int cap, int *n);

/* ------------------------------------------------------------------------
 * Swapping to a CPU pool. [P3] procedure steps 7-8 (when no free block is
 * left, a request's blocks are evicted all at once, sequences that share
 * blocks -- the beams of one request -- together, and later copied back);
 * [P4] section 12 (KV blocks of lower-priority requests moved to CPU memory).
 *
 * pa_bm_enable_swap gives the manager a CPU pool of num_host_blocks blocks
 * (ids 0 .. num_host_blocks-1, an ascending free queue; once per handle).
 *
 * pa_bm_swap_out moves a group of resident sequences (each id once) to the
 * CPU pool. The group must hold every reference to its blocks
 * (PA_ERR_INVALID_ARG otherwise: a shared block cannot be half-evicted).
 * Each distinct GPU block, in order of first appearance across the group's
 * tables, gets the next CPU block; the pairs (GPU id, CPU id) are written to
 * mapping[2*i], mapping[2*i+1] (cap pairs room; *num_pairs set). The GPU
 * blocks return to the front of the free queue in that order, the tables
 * hold the CPU ids, reference counts move with the blocks. The caller copies
 * the data with pa_swap_blocks (GPU pool -> CPU pool) before the freed GPU
 * blocks are written again.
 *
 * pa_bm_swap_in is the reverse: pairs (CPU id, GPU id), fresh GPU blocks
 * from the free queue front, CPU blocks back to their queue front.
 *
 * Both are all-or-nothing: PA_ERR_OUT_OF_BLOCKS if the destination pool is
 * short, PA_ERR_INVALID_ARG if cap is too small (nothing changes either way).
 * While swapped out, pa_bm_append_slot and pa_bm_fork refuse the sequence
 * (PA_ERR_INVALID_ARG); pa_bm_free releases its CPU blocks; pa_bm_stats
 * still counts its tokens and logical blocks (used/shared/free count GPU
 * blocks only).
 * ---------------------------------------------------------------------- */
PA_API pa_status pa_bm_enable_swap(pa_bm *bm, int num_host_blocks);
PA_API pa_status pa_bm_swap_out(pa_bm *bm, const int64_t *seqs, int num_seqs, int64_t *mapping, int cap,
                                int *num_pairs);
PA_API pa_status pa_bm_swap_in(pa_bm *bm, const int64_t *seqs, int num_seqs, int64_t *mapping, int cap,
                               int *num_pairs);
PA_API pa_status pa_bm_is_swapped(const pa_bm *bm, int64_t seq, int *swapped);
PA_API pa_status pa_bm_swap_stats(const pa_bm *bm, int64_t *host_blocks, int64_t *free_host_blocks,
                                  int64_t *swapped_seqs);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
