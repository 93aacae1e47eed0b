/*
 * pkv: paged KV-cache attention for GB300 (sm_103a), C ABI.
 *
 * The operations follow the description of the paged KV cache on these pages:
 *   - "Serving deep dive: KV cache, batching, and inference engines"
 *     (models.specul.com), sections on PagedAttention and chunked prefill;
 *   - the ainews.alishangtian.com article on vLLM, "PagedAttention" (16-token
 *     blocks chained by a block table, shared prefix blocks, copy-on-write);
 *   - chengxuchu.com "PyTorch #47: KV Cache, batching, sampling", sections 2.1
 *     (attention formula), 2.2 (append new K/V at a given position, then the
 *     new query reads all cached K/V), 2.3 (GQA) and 5.2 (the kernel reaches
 *     K/V through the block table);
 *   - caffein.top "modern LLM inference runtime", "Chunked Prefill" and
 *     "Paging".
 *
 * Conventions shared by every call
 *   - Every pointer argument is DEVICE memory owned by the caller, except the
 *     out-parameters of pkv_*_workspace_bytes and pkv_get_status, which are
 *     host pointers.  The library allocates no device memory and keeps no
 *     pointer after a call returns.
 *   - Tensors are dense row-major.  Each KV cache is
 *       [num_blocks][num_kv_heads][block_size][head_dim]
 *     (K and V are separate tensors with the same shape).  Logical token t of
 *     sequence s is row (t % block_size) of physical block
 *     block_tables[s * max_blocks_per_seq + t / block_size].  A slot is
 *     block * block_size + row.
 *   - block_size must be 16; head_dim must be 64 or 128.  dtype is the element
 *     type of q, k, v and both caches (one type for all of them); out_dtype
 *     the element type of out.  Cache, q, k, v and out pointers must be
 *     16-byte aligned.
 *   - Every call only enqueues work on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and returns without waiting.
 *   - Return value: PKV_OK, or PKV_ERR_INVALID when an argument is rejected on
 *     the host (nothing is launched), or PKV_ERR_CUDA when a launch fails.
 *     pkv_last_error_string() describes the last failure on this host thread.
 *   - Indices that are only known on the device (slots, block ids, context
 *     lengths) are checked by the kernels.  A bad one is skipped and recorded
 *     in a per-device status word; no kernel traps.  pkv_get_status() reads
 *     and clears that word.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* return codes */
#define PKV_OK 0
#define PKV_ERR_INVALID 1
#define PKV_ERR_CUDA 2
#define PKV_ERR_OOB 3

/* element types */
#define PKV_F32 0
#define PKV_BF16 1
#define PKV_FP8_E4M3 2  /* cache element: fp8 E4M3 code of value / scale (per kv head); 1 byte */

/* status-word bits (pkv_get_status) */
#define PKV_STATUS_BAD_SLOT 1u       /* kv_append: slot >= num_blocks * block_size */
#define PKV_STATUS_BAD_BLOCK 2u      /* block id < 0 or >= num_blocks (gather or copy) */
#define PKV_STATUS_BAD_LENGTH 4u     /* context_len < 0, > max_blocks_per_seq * block_size,
                                        or > max_context_len */
#define PKV_STATUS_BAD_QLEN 8u       /* prefill: chunk longer than its context, or than max_q_len */
#define PKV_STATUS_INTERNAL 16u      /* a kernel gave up waiting on its own asynchronous work, or its
                                        shared memory was misaligned; its outputs are undefined */

#define PKV_BLOCK_SIZE 16
#define PKV_DEFAULT_PARTITION 512    /* smallest decode split-K partition, tokens */

/*
 * KV append (scatter).  chengxuchu #47 section 2.2: production code
 * preallocates blocks and writes each new token's K/V at its position.
 *   k, v          [num_tokens][num_kv_heads][head_dim], dtype
 *   slot_mapping  [num_tokens] int64; token i goes to slot slot_mapping[i].
 *                 A negative slot skips the token (padding).  A slot at or
 *                 past num_blocks * block_size is skipped and sets
 *                 PKV_STATUS_BAD_SLOT.  Two tokens with the same slot are a
 *                 caller error (which one lands is unspecified).
 *   k_cache, v_cache  updated in place (bit copy, no conversion).
 */
int pkv_kv_append(const void *k, const void *v, const int64_t *slot_mapping, int num_tokens,
                  void *k_cache, void *v_cache, int num_blocks, int num_kv_heads, int head_dim,
                  int block_size, int dtype, void *stream);

/*
 * KV append into an fp8 E4M3 cache (quantised KV cache; the runtime page on
 * KV-cache memory, section 2.4).  As pkv_kv_append, except that each element
 * x of kv head g is stored as the E4M3 code of the binary32 quotient
 * x / k_scale[g] (K) or x / v_scale[g] (V): round to nearest even, magnitudes
 * beyond 448 saturated to 448, NaN to the NaN code.
 *   k, v          [num_tokens][num_kv_heads][head_dim], in_dtype (PKV_F32 or
 *                 PKV_BF16), 16-byte aligned
 *   k_cache, v_cache  [num_blocks][num_kv_heads][16][head_dim] bytes
 *   k_scale, v_scale  [num_kv_heads] float32 device arrays, positive
 */
int pkv_kv_append_fp8(const void *k, const void *v, int in_dtype, const int64_t *slot_mapping,
                      int num_tokens, void *k_cache, void *v_cache, const float *k_scale,
                      const float *v_scale, int num_blocks, int num_kv_heads, int head_dim,
                      int block_size, void *stream);

/*
 * Copy-on-write block copy.  ainews article, "PagedAttention": when requests
 * sharing prefix blocks diverge, only the forked block is copied.
 *   src_dst_pairs  [num_pairs][2] int64 (src, dst): block dst of both caches
 *                  becomes a copy of block src (all kv heads, all 16 rows).
 *                  Destinations must be distinct and must not be sources of
 *                  the same call (caller contract).  An id outside
 *                  [0, num_blocks) skips the pair and sets PKV_STATUS_BAD_BLOCK.
 *   dtype          PKV_F32, PKV_BF16 or PKV_FP8_E4M3 (bytes are copied).
 */
int pkv_copy_blocks(void *k_cache, void *v_cache, const int64_t *src_dst_pairs, int num_pairs,
                    int num_blocks, int num_kv_heads, int head_dim, int block_size, int dtype,
                    void *stream);

/*
 * Workspace (device bytes) that pkv_paged_attention_decode needs for its
 * split-K partials with these sizes.  partition_size 0 means the adaptive
 * default; the size returned then covers every partition it may choose.
 * *bytes is a host pointer.  Returns PKV_ERR_INVALID for bad sizes.
 */
int pkv_decode_workspace_bytes(int num_seqs, int num_q_heads, int head_dim, int max_context_len,
                               int partition_size, size_t *bytes);

/*
 * The split-K partition (tokens) that a decode call with these sizes uses:
 * partition_size itself when it is non-zero, else the adaptive choice
 * described under pkv_paged_attention_decode, made for the current device.
 * A call whose max_context_len (capped at max_blocks_per_seq * 16) exceeds it
 * makes the second, log-sum-exp launch.  *out is a host pointer.  Launches
 * nothing; returns PKV_ERR_INVALID for bad sizes.
 */
int pkv_decode_partition_size(int num_seqs, int num_kv_heads, int max_context_len,
                              int partition_size, int *out);

/*
 * As pkv_decode_partition_size for pkv_paged_attention_decode_fp8, whose
 * adaptive choice differs: when num_seqs x units (units = num_kv_heads x
 * ceil(num_q_heads / num_kv_heads / 8)) is between 2 and 4 times the SM
 * count and max_context_len is at most 8192, one resident wave of its thread
 * blocks covers the batch and no sequence is split (the partition is
 * max_context_len rounded up to a multiple of 16); otherwise the choice of
 * pkv_decode_partition_size.
 */
int pkv_decode_partition_size_fp8(int num_seqs, int num_q_heads, int num_kv_heads, int max_context_len,
                                  int partition_size, int *out);

/*
 * Paged-attention decode.  One query token per sequence and head attends to
 * every cached token of its sequence:
 *   out[s,h,:] = softmax_t(scale * q[s,h,:] . K_t) V_t,  t = 0 .. L_s - 1,
 * chengxuchu #47 sections 2.1-2.2, with K_t and V_t fetched through the block
 * table (section 5.2) and kv head h / (num_q_heads / num_kv_heads) (GQA,
 * section 2.3).  The caller appends the new token first, so context_lens
 * include it.  A sequence with L_s = 0 gets a zero row.
 *   q             [num_seqs][num_q_heads][head_dim], dtype
 *   block_tables  [num_seqs][max_blocks_per_seq] int32; entries at or past
 *                 ceil(L_s / 16) are never read
 *   context_lens  [num_seqs] int32
 *   max_context_len  host-side upper bound on every L_s, sizes the grid; a
 *                 sequence longer than it sets PKV_STATUS_BAD_LENGTH and its
 *                 output is undefined
 *   partition_size   tokens per split-K partition (multiple of 16), or 0 to
 *                 let the library choose: the largest of 3072, 2048, 1536 and
 *                 1024 that leaves about 4 thread blocks per SM (estimated from
 *                 num_seqs, num_kv_heads and max_context_len), else 512.
 *                 Sequences longer than one partition are processed as
 *                 independent partitions whose results are merged by a
 *                 log-sum-exp reduction (a second launch).
 *   out           [num_seqs][num_q_heads][head_dim], out_dtype
 *   workspace     device scratch of at least pkv_decode_workspace_bytes(...)
 *                 bytes (may be NULL when that is 0); contents need no
 *                 initialisation and are clobbered.
 */
int pkv_paged_attention_decode(const void *q, const void *k_cache, const void *v_cache,
                               const int32_t *block_tables, int max_blocks_per_seq,
                               const int32_t *context_lens, int num_seqs, int num_q_heads,
                               int num_kv_heads, int head_dim, int block_size, int num_blocks,
                               int max_context_len, int partition_size, float scale, void *out,
                               int dtype, int out_dtype, void *workspace, size_t workspace_bytes,
                               void *stream);

/*
 * Decode over fp8 E4M3 caches (written by pkv_kv_append_fp8): as
 * pkv_paged_attention_decode with bf16 queries, where cached element x of kv
 * head g stands for x * k_scale[g] (K) or x * v_scale[g] (V).  head_dim must
 * be 128.  The workspace is sized by pkv_decode_workspace_bytes.
 *   q             [num_seqs][num_q_heads][128] bf16
 *   k_cache, v_cache  [num_blocks][num_kv_heads][16][128] bytes
 *   k_scale, v_scale  [num_kv_heads] float32 device arrays
 *   out           [num_seqs][num_q_heads][128], out_dtype
 * partition_size 0 takes the choice of pkv_decode_partition_size_fp8.
 * Precision: codes widen to fp16 exactly; q is rounded to fp16 once (a
 * query beyond the fp16 range, 65504, overflows); the softmax weights enter
 * the value product as fp16; accumulation is fp32.
 */
int pkv_paged_attention_decode_fp8(const void *q, const void *k_cache, const void *v_cache,
                                   const float *k_scale, const float *v_scale,
                                   const int32_t *block_tables, int max_blocks_per_seq,
                                   const int32_t *context_lens, int num_seqs, int num_q_heads,
                                   int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                   int max_context_len, int partition_size, float scale, void *out,
                                   int out_dtype, void *workspace, size_t workspace_bytes,
                                   void *stream);

/*
 * One decode step: append, then attend, in one launch.  Equivalent to
 * pkv_kv_append of each sequence's new token at logical position L_s - 1
 * (slot block_tables[s][(L_s-1)/16] * 16 + (L_s-1) % 16) followed by
 * pkv_paged_attention_decode with the same arguments: the new K/V are
 * scattered into the cache first and the query then reads every cached
 * token (chengxuchu #47 section 2.2).  The thread block that owns a
 * sequence's last partition writes that sequence's new row of its kv head
 * before reading the partition, so no separate append launch is needed.
 *   k_new, v_new  [num_seqs][num_kv_heads][head_dim], dtype, 16-byte aligned
 *   k_cache, v_cache  updated in place (bit copy) and then read
 * Sequences with L_s = 0 append nothing.  A bad block id for position
 * L_s - 1 skips the write and sets PKV_STATUS_BAD_BLOCK.  All other
 * arguments, results and errors are those of pkv_paged_attention_decode.
 */
int pkv_decode_step(const void *q, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                    const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
                    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                    int num_blocks, int max_context_len, int partition_size, float scale, void *out,
                    int dtype, int out_dtype, void *workspace, size_t workspace_bytes, void *stream);

/*
 * pkv_decode_step over fp8 E4M3 caches: pkv_kv_append_fp8 of each sequence's
 * new token at logical position L_s - 1 (code = E4M3(value / scale) of its kv
 * head, the same bytes) followed by pkv_paged_attention_decode_fp8, in one
 * launch.
 *   k_new, v_new  [num_seqs][num_kv_heads][128] bf16, 16-byte aligned
 *   k_cache, v_cache  [num_blocks][num_kv_heads][16][128] E4M3 codes, updated
 *                 in place and then read
 * All other arguments, results and errors are those of
 * pkv_paged_attention_decode_fp8 (partition_size 0: the choice of
 * pkv_decode_partition_size_fp8).
 */
int pkv_decode_step_fp8(const void *q, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                        const float *k_scale, const float *v_scale, const int32_t *block_tables,
                        int max_blocks_per_seq, const int32_t *context_lens, int num_seqs, int num_q_heads,
                        int num_kv_heads, int head_dim, int block_size, int num_blocks, int max_context_len,
                        int partition_size, float scale, void *out, int out_dtype, void *workspace,
                        size_t workspace_bytes, void *stream);

/*
 * Paged-attention decode that allocates nothing, for callers that cannot
 * allocate device memory where they run decode (code inside an allocator or
 * memory-pool hook that must not re-enter the allocator, or embedders whose
 * device memory is budgeted up front).  The pages have no counterpart to this
 * entry point; it exists only for such callers.
 *
 * Same arguments and results as pkv_paged_attention_decode, minus the
 * workspace: the split-K partials go to one scratch array of
 * PKV_NO_ALLOC_SCRATCH_BYTES that is part of this library's device image.
 * Every GPU that loads the library holds that array until the process exits.
 *   - The scratch need is pkv_decode_workspace_bytes at the partition the
 *     call uses (pkv_decode_partition_size: partition_size itself, or the
 *     adaptive choice when it is 0).  Sizes whose need exceeds
 *     PKV_NO_ALLOC_SCRATCH_BYTES are rejected with PKV_ERR_INVALID before
 *     anything is launched.
 *   - The call allocates no memory: no cudaMalloc, cudaFree or allocating
 *     library routine.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress with that device current), which may make the
 *     CUDA driver load this library's device code; make that first call
 *     before any stream capture.
 *   - Every call on a device shares the one array and it keeps the last
 *     call's contents (no call needs it zeroed).  Calls whose work overlaps
 *     on the GPU (other streams, or other host threads) race on it: order
 *     them on one stream or synchronise between them.
 *   - The stream must belong to the current device.
 */
#define PKV_NO_ALLOC_SCRATCH_BYTES (16u << 20)
int pkv_paged_attention_decode_no_alloc(const void *q, const void *k_cache, const void *v_cache,
                                        const int32_t *block_tables, int max_blocks_per_seq,
                                        const int32_t *context_lens, int num_seqs,
                                        int num_q_heads, int num_kv_heads, int head_dim,
                                        int block_size, int num_blocks, int max_context_len,
                                        int partition_size, float scale, void *out, int dtype,
                                        int out_dtype, void *stream);

/*
 * Workspace (device bytes) that pkv_paged_attention_decode_shared_prefix
 * needs with these sizes (head_dim 128; partition_size 0 covers every
 * partition the call may choose).  *bytes is a host pointer.
 */
int pkv_decode_shared_prefix_workspace_bytes(int num_seqs, int num_q_heads, int head_dim,
                                             int max_context_len, int prefix_len, int partition_size,
                                             size_t *bytes);

/*
 * Decode of a batch whose sequences all begin with the same prefix_len tokens
 * stored in the same physical blocks (a shared system prompt; ainews
 * "PagedAttention": blocks of a common prefix are shared, copy-on-write on
 * divergence).  Same result as pkv_decode_step (k_new, v_new given) or
 * pkv_paged_attention_decode (both NULL) on these inputs, computed as a
 * cascade:
 *   1. the prefix once for every query of the batch: the S * Hq query rows
 *      against the prefix keys of block_tables row 0 form a dense tile for
 *      the tcgen05 tensor cores (the chunked-prefill kernel in a non-causal
 *      mode), giving each row's (m, l, O) over the prefix;
 *   2. each sequence's tokens [prefix_len, L_s) with the partitioned decode
 *      kernel (and the fused append of the new token when k_new is given);
 *   3. the log-sum-exp merge of 1 and 2 (chengxuchu #47 section 2.1: the
 *      softmax over the union of the key sets).
 * Contract, not checked: rows 0 .. prefix_len/16 - 1 of every block table
 * are the same block ids.  Requirements: bf16 caches, head_dim 128, 1..16 q
 * heads per kv head, prefix_len a positive multiple of 16 below the context
 * bound, and every L_s > prefix_len (else PKV_STATUS_BAD_LENGTH and that
 * sequence's output is undefined).  Other arguments as
 * pkv_paged_attention_decode / pkv_decode_step; workspace of
 * pkv_decode_shared_prefix_workspace_bytes(...) bytes, 256-byte aligned,
 * needing no initialisation (replays of a captured call are fine, as for
 * pkv_paged_attention_prefill_chunk).
 */
int pkv_paged_attention_decode_shared_prefix(const void *q, const void *k_new, const void *v_new,
                                             void *k_cache, void *v_cache, const int32_t *block_tables,
                                             int max_blocks_per_seq, const int32_t *context_lens,
                                             int num_seqs, int num_q_heads, int num_kv_heads,
                                             int head_dim, int block_size, int num_blocks,
                                             int max_context_len, int prefix_len, int partition_size,
                                             float scale, void *out, int dtype, int out_dtype,
                                             void *workspace, size_t workspace_bytes, void *stream);

/*
 * Workspace (device bytes) that pkv_paged_attention_prefill_chunk needs:
 * 256 for head_dim 128 (the bf16 kernel's work-item counter), else 0.
 */
int pkv_prefill_workspace_bytes(int num_seqs, int total_q, int num_q_heads, int num_kv_heads,
                                int head_dim, int max_q_len, int max_context_len, size_t *bytes);

/*
 * Chunked-prefill attention.  caffein.top "Chunked Prefill" and the
 * "Serving deep dive" page: a long prompt is cut into chunks that run in the
 * same steps as decode.  Sequence s contributes the n_s = cu_q_lens[s+1] -
 * cu_q_lens[s] query rows cu_q_lens[s] .. cu_q_lens[s+1]-1; its cache already
 * holds the chunk (appended by the caller), so its L_s = context_lens[s]
 * tokens end with the chunk and query j sits at position L_s - n_s + j.  It
 * attends causally to tokens 0 .. L_s - n_s + j.
 *   q          [total_q][num_q_heads][head_dim], dtype
 *   cu_q_lens  [num_seqs + 1] int32, non-decreasing, cu_q_lens[0] = 0,
 *              cu_q_lens[num_seqs] = total_q
 *   max_q_len  host-side bound on every n_s (sizes the grid)
 *   max_context_len  host-side bound on every L_s
 *   out        [total_q][num_q_heads][head_dim], out_dtype
 *   workspace  device scratch of pkv_prefill_workspace_bytes(...) bytes,
 *              16-byte aligned; it needs no initialisation (each launch
 *              claims its work counter with a fresh 64-bit tag, and the
 *              launch's last thread block clears it, so a call captured in
 *              a CUDA graph may be replayed any number of times), and calls
 *              that overlap on the GPU must not share it.
 * n_s > L_s or n_s > max_q_len sets PKV_STATUS_BAD_QLEN and skips the sequence.
 */
int pkv_paged_attention_prefill_chunk(const void *q, const int32_t *cu_q_lens,
                                      const void *k_cache, const void *v_cache,
                                      const int32_t *block_tables, int max_blocks_per_seq,
                                      const int32_t *context_lens, int num_seqs, int total_q,
                                      int max_q_len, int max_context_len, int num_q_heads,
                                      int num_kv_heads, int head_dim, int block_size,
                                      int num_blocks, float scale, void *out, int dtype,
                                      int out_dtype, void *workspace, size_t workspace_bytes,
                                      void *stream);

/* ---------------------------------------------------------------------------
 * Host block manager (host memory only; no CUDA call).
 *
 * Keeps the mapping the kernels above consume: which physical cache blocks
 * hold each sequence's tokens (its block table), which blocks are shared and
 * how often (reference counts), and which full blocks hold a known token
 * prefix so that a later prompt starting with the same tokens reuses them.
 * Source: ainews "PagedAttention" (logical blocks mapped to physical blocks,
 * allocated on demand, shared between sequences, copy-on-write when a shared
 * block must change); #47 §5.2 (block table); runtime "Paging" and "Prefix
 * caching" (reuse of cached prefix blocks, least-recently-used eviction).
 *
 * Blocks hold PKV_BLOCK_SIZE tokens.  A block is
 *   - free (in no table, content unknown),
 *   - in use (reference count >= 1: the number of sequences whose table
 *     holds it), or
 *   - cached (reference count 0 but full, with its token content and prefix
 *     registered; reusable by a matching prompt, evicted least recently
 *     used first when no free block is left).
 * Only full blocks are registered.  A block's identity in the prefix index
 * is a 64-bit chain hash of its 16 token ids and the hash of the block
 * before it; a hit also compares the stored token ids.
 *
 * The manager is not thread-safe.  Sequence ids are the caller's (any
 * int64).  Errors: PKV_ERR_INVALID for bad arguments or unknown / duplicate
 * sequence ids, PKV_ERR_OOB when the blocks needed are not available (the
 * call then changes nothing).
 * ------------------------------------------------------------------------- */

/* *bm: a new manager over blocks [0, num_blocks); tables are at most
 * max_blocks_per_seq blocks wide.  prefix_cache 0 disables the prefix index
 * (every block is freed when its last sequence ends). */
int pkv_bm_create(int num_blocks, int max_blocks_per_seq, int prefix_cache, void **bm);

/* Releases the manager. */
int pkv_bm_destroy(void *bm);

/* *free_blocks: blocks a new allocation could take (free + cached);
 * *cached_blocks: those of them that are cached (may be NULL). */
int pkv_bm_num_free_blocks(void *bm, int *free_blocks, int *cached_blocks);

/* A new sequence holding the prompt tokens[0 .. num_tokens).  Its leading
 * full blocks are taken from the prefix index while their token content and
 * prefix match; *num_cached_tokens (may be NULL) receives how many leading
 * tokens were found there (their K/V are already in the cache).  The other
 * tokens get new blocks (the caller writes their K/V, e.g. by a prefill of
 * tokens [*num_cached_tokens, num_tokens)); new full blocks are registered
 * in the prefix index at once, so the caller must write them before any
 * reader of a later prompt uses them. */
int pkv_bm_add_sequence(void *bm, int64_t seq_id, const int32_t *tokens, int num_tokens,
                        int *num_cached_tokens);

/* Sequence `child` starts as a copy of `parent`: the same table, every block
 * shared (reference count + 1).  The first append to either side of a
 * shared, partly filled last block copies it (see pkv_bm_append_tokens). */
int pkv_bm_fork(void *bm, int64_t parent, int64_t child);

/* Reserve the slot of one new token for each of seq_ids[0 .. n) (n host
 * int64 ids; tokens: their token ids, for the prefix index).  The last
 * block is used when it has room and this sequence alone holds it; a full
 * last block gets a new block after it; a shared, partly filled last block
 * is replaced by a new block, and the pair (old, new) is appended to
 * copy_pairs (host int64 [2 * n] at most) for pkv_copy_blocks, which must
 * run before the tokens' K/V are written.  slot_mapping (host int64 [n])
 * receives block * 16 + offset for each token, *num_pairs the number of
 * pairs.  A block that becomes full is registered in the prefix index. */
int pkv_bm_append_tokens(void *bm, const int64_t *seq_ids, int n, const int32_t *tokens,
                         int64_t *slot_mapping, int64_t *copy_pairs, int *num_pairs);

/* Slots of tokens [first, first + n) of a sequence (host int64 [n]), e.g.
 * the prompt tokens a prefill writes. */
int pkv_bm_slots(void *bm, int64_t seq_id, int first, int n, int64_t *slots);

/* The sequence ends: every block's reference count drops by one; a block
 * left unreferenced becomes cached if it is registered, else free. */
int pkv_bm_free_sequence(void *bm, int64_t seq_id);

/* Block tables and lengths for seq_ids[0 .. n): tables is host int32
 * [n][max_blocks] (unused entries -1), context_lens host int32 [n] (may be
 * NULL).  Fails if a table is wider than max_blocks. */
int pkv_bm_block_tables(void *bm, const int64_t *seq_ids, int n, int32_t *tables, int max_blocks,
                        int32_t *context_lens);

/*
 * Synchronises `stream`, then reads and clears the status word of the current
 * device.  *flags (host pointer, may be NULL) receives the PKV_STATUS_* bits.
 * Returns PKV_OK when no bit was set, PKV_ERR_OOB when one was, PKV_ERR_CUDA
 * on a CUDA error.  The word is shared by every stream of the device.
 */
int pkv_get_status(void *stream, unsigned int *flags);

/*
 * Bound on each wait inside the tensor-core kernels (the chunked-prefill tile
 * and the shared-prefix tile of pkv_paged_attention_decode_shared_prefix): a
 * wait on the kernel's own asynchronous copies or MMAs, or on another of its
 * warps, that lasts longer than `ns` nanoseconds (GPU global timer) makes the
 * kernel stop issuing work, let what it already issued finish, record
 * PKV_STATUS_INTERNAL and return; its outputs are then undefined.  0 restores
 * the default, 200 ms (far above any wait of a working launch, which lasts
 * microseconds).  Process-wide; it applies to launches made after the call.
 * Always returns PKV_OK.
 */
int pkv_set_wait_limit_ns(unsigned long long ns);

/* Description of the last failure on the calling host thread ("" if none). */
const char *pkv_last_error_string(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
