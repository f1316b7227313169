/*
 * pagedkv.h -- C ABI of the GB300 paged GQA decode-attention library
 * (libpagedkv.so, CUDA kernels for sm_103a).
 *
 * The library keeps one layer's key/value cache in a fixed pool of
 * fixed-size blocks in HBM, appends each step's new keys and values into
 * their slots, and runs single-token decode attention for a batch of
 * sequences that reach their blocks through per-sequence block tables, with
 * grouped-query attention (n_q query heads share n_kv KV heads).
 *
 * Conventions for every call:
 *   - Pointers named "device" must point to GPU memory of the device the pool
 *     was created on; "host" pointers to ordinary CPU memory.  The caller owns
 *     every buffer it passes and keeps it alive until the work enqueued on
 *     `stream` has finished.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Calls that take a stream only enqueue work and never
 *     synchronise the host.
 *   - A call returns PKV_OK or an error status.  Argument errors are found on
 *     the host before anything is enqueued.  Range errors met on the device
 *     (a slot or block id outside the pool, a context length beyond the block
 *     table) skip the offending item and set a sticky bit read with
 *     pkv_get_error(); kernels never trap.
 *   - pkv_last_error_message() gives a one-line description of the last
 *     failure on the calling thread.
 *   - A pool is not safe to use from two host threads or two streams at once
 *     (it owns one split-KV workspace).
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PKV_OK = 0,
    PKV_EINVAL = 1,        /* bad argument (null pointer, shape, alignment) */
    PKV_ERANGE = 2,        /* a size outside what the call accepts */
    PKV_ENOMEM = 3,        /* device allocation failed */
    PKV_ECUDA = 4,         /* a CUDA runtime call failed (see message) */
    PKV_EUNSUPPORTED = 5,  /* valid but unsupported configuration or device */
    PKV_EDEVICE = 6        /* pkv_get_error: the device recorded range errors */
} pkv_status;

typedef enum {
    PKV_BF16 = 0,      /* keys and values stored as bf16 */
    PKV_FP8_E4M3 = 1,  /* stored as FP8 E4M3 with a per-KV-head fp32 scale */
    PKV_INT4 = 2       /* 4-bit codes: keys with a per-(KV head, channel) scale and zero point, values with a
                          per-(token, KV head) scale and zero point (see kv_pool_set_int4_key_params) */
} pkv_dtype;

/* Bits of the sticky device error word (pkv_get_error). */
#define PKV_DEVERR_SLOT_RANGE  0x1u  /* append: slot >= num_blocks * block_size */
#define PKV_DEVERR_BLOCK_RANGE 0x2u  /* decode: block id outside [0, num_blocks) */
#define PKV_DEVERR_CTX_RANGE   0x4u  /* decode: context_len < 0 or > W * block_size */
#define PKV_DEVERR_TIMEOUT     0x8u  /* a bounded wait on the kernel's own copies ran out */

typedef struct pkv_pool pkv_pool; /* opaque; owns its device memory */

/* Where a pool's blocks live.  Everything one (block, KV head) needs is one
 * contiguous entry: its 16 key rows, then its 16 value rows (and for
 * PKV_INT4 pools then its 16 value rows' fp32 (scale, zero point) pairs).
 * Entries are [num_blocks][n_kv] in one allocation of alloc_bytes starting
 * at k; v points at the first entry's value rows.  Element (blk, g, off, d)
 * of the keys sits at k + blk*stride_block + g*stride_head +
 * off*stride_token + d, and of the values at the same offset from v (strides
 * in elements: bf16 values, E4M3 bytes, or bytes of packed codes).  A row is
 * d_head values, or for PKV_INT4 d_head / 2 bytes each holding channels 2i
 * (low nibble) and 2i+1 (high nibble).  stride_head is 32 * d_head elements
 * (PKV_INT4: 16 * d_head + 128 bytes).  Value row (blk, g, off)'s 4-bit
 * parameters sit at v_params + blk*stride_block + g*stride_head + 8*off
 * bytes. */
typedef struct {
    void *k;                 /* device */
    void *v;                 /* device */
    int64_t stride_block;    /* n_kv * stride_head */
    int64_t stride_head;     /* 2 * block_size * d_head (PKV_INT4: 16 * d_head + 128 bytes) */
    int64_t stride_token;    /* d_head (PKV_INT4: d_head / 2) */
    int64_t num_blocks;
    int32_t block_size;
    int32_t n_kv;
    int32_t d_head;
    int32_t dtype;           /* pkv_dtype */
    int64_t bytes_per_array; /* bytes of key (and, equally, of value) rows in the pool */
    void *v_params;          /* device; PKV_INT4 only (NULL otherwise) */
    int64_t v_params_bytes;  /* bytes of value parameters in the pool (8 per token row) */
    int64_t alloc_bytes;     /* bytes of the allocation k points into: the whole pool */
} pkv_layout;

/* Per-kernel timing gathered with CUDA events while timing is enabled. */
typedef struct {
    int64_t launches;        /* every kernel launch the library enqueued */
    int64_t append_launches;
    int64_t decode_launches;
    int64_t merge_launches;  /* split-KV merge launches (one behind every decode launch) */
    double append_ms;        /* summed event time of timed launches */
    double decode_ms;
    double merge_ms;
    int64_t timed_append, timed_decode, timed_merge;
    int64_t prefix_launches; /* cascade decode: shared-prefix stage launches */
    double prefix_ms;
    int64_t timed_prefix;
    int64_t block_launches;  /* block copy / swap launches */
    double block_ms;
    int64_t timed_block;
    int64_t workspace_bytes; /* bytes of the pool's split-KV workspace allocated so far */
} pkv_timing;

/* Create a pool of `num_blocks` blocks of `block_size` token slots, for
 * `n_kv` KV heads of `d_head` values, stored as `dtype`.  The pool splits the
 * cache into fixed-size blocks that any sequence may own in any order
 * ("KV cache, PagedAttention and FlashAttention", Problem 4, "The idea";
 * "Memory Management in LLM Serving Systems", "Method 3: PagedAttention").
 * One pool holds one layer.  Memory is allocated on the current CUDA device
 * and zero-filled; the pool owns it.
 * Supported: block_size == 16, d_head in {64, 128}, 1 <= n_kv <= 256.
 * Errors: EINVAL (null out, non-positive sizes), EUNSUPPORTED (other block
 * or head sizes, a device that is not sm_103), ENOMEM, ECUDA. */
pkv_status kv_pool_create(int64_t num_blocks, int32_t block_size, int32_t n_kv, int32_t d_head,
                          int32_t dtype, pkv_pool **out);

/* Free the pool and everything it owns (synchronises the device first).
 * NULL is accepted. */
pkv_status kv_pool_destroy(pkv_pool *pool);

/* PKV_INT4 pools: set the keys' per-(KV head, channel) parameters from two
 * host arrays of n_kv x d_head fp32 values, [g][channel]: a key value x is
 * stored as the code c = clamp(rint((x - k_zero) / k_scale), 0, 15)
 * (fp32, round half to even) and read back as c * k_scale + k_zero.  Values
 * need no call: each appended value row gets its own scale (max - min) / 15
 * (1 if max == min) and zero point min.  The pages ask for 4-bit KV with
 * per-channel key scales ("KV cache, PagedAttention and FlashAttention",
 * Problem 3, "Trade-offs"; KIVI, KVQuant); the rest is this library's
 * reading.  Must be called before the first append or decode of a 4-bit
 * pool; scales finite and > 0, zero points finite.  Errors: EINVAL. */
pkv_status kv_pool_set_int4_key_params(pkv_pool *pool, const float *k_scale_host, const float *k_zero_host);

/* FP8 pools: set the per-KV-head dequantisation scales from two host arrays
 * of n_kv fp32 values (stored value = E4M3(x / scale), read back as
 * E4M3 * scale).  Must be called before the first append or decode of an FP8
 * pool; scales must be finite and > 0.  Changing them later does not
 * rewrite stored bytes.  The pages name FP8 KV ("KV cache, PagedAttention
 * and FlashAttention", Problem 3 trade-offs: FP8 halves the bytes of BF16);
 * the per-head scale is this library's reading.  Errors: EINVAL. */
pkv_status kv_pool_set_fp8_scales(pkv_pool *pool, const float *k_scale_host,
                                  const float *v_scale_host);

/* Report the pool's device pointers and layout (see pkv_layout). */
pkv_status kv_pool_layout(const pkv_pool *pool, pkv_layout *out);

/* How paged_decode_attention splits work.  0 (the default): the batch's
 * (sequence, KV head, block) work is cut into one equal slice per resident
 * warp, so every SM gets the same number of blocks whatever the length mix.
 * Otherwise: slices of `tokens` tokens (a multiple of 16 in [16, 2^20]),
 * taken round-robin by the warps.  Results agree up to rounding either way.
 * Errors: ERANGE. */
pkv_status kv_pool_set_partition_tokens(pkv_pool *pool, int32_t tokens);

/* How paged_decode_attention_prefix runs on this pool.
 *   PKV_CASCADE_AUTO (0, the default): the cascade (prefix read once for the
 *     batch) where it measured faster on GB300, plain paged decode over the
 *     whole tables otherwise (where re-reading the prefix from L2 costs less
 *     than the cascade's prefix stage and merge).  bf16 pools: a prefix of at
 *     least 2048 tokens and batch x prefix tokens >= 2^17.  FP8 pools (whose
 *     plain decode converts the prefix again for every sequence): batch x
 *     prefix tokens >= 2^17, or >= 2^16 with a batch of at least 64.  Never
 *     below a batch of 8.
 *   PKV_CASCADE_ALWAYS (1), PKV_CASCADE_NEVER (2): force one of them.
 * Results agree up to rounding either way.  Errors: EINVAL. */
#define PKV_CASCADE_AUTO 0
#define PKV_CASCADE_ALWAYS 1
#define PKV_CASCADE_NEVER 2
pkv_status kv_pool_set_cascade_mode(pkv_pool *pool, int32_t mode);

/* Grow the pool's split-KV workspace now (it otherwise grows inside the
 * first decode call that needs more), so that later decode calls with at
 * most `batch` sequences, `n_q` query heads and `max_blocks_per_seq` table
 * entries allocate nothing.  Errors: EINVAL, ENOMEM. */
pkv_status kv_pool_reserve_workspace(pkv_pool *pool, int32_t batch, int32_t n_q,
                                     int32_t max_blocks_per_seq);

/* Append: write token t's key and value rows into slot slot_mapping[t] of
 * the pool ("The KV Cache from First Principles", "Deriving the cache": each
 * step computes one new key and value per KV head and appends them; "Prefill
 * populates the cache" uses the same call with many tokens).
 *   k_new, v_new  device bf16 [n_tokens][n_kv][d_head], 16-byte aligned.
 *   slot_mapping  device int64 [n_tokens]; slot = physical block *
 *                 block_size + offset ("KV cache, PagedAttention and
 *                 FlashAttention", Problem 4, address arithmetic).  A negative
 *                 slot skips the token; a slot >= num_blocks * block_size is
 *                 skipped and sets PKV_DEVERR_SLOT_RANGE.  Two tokens with the
 *                 same slot in one call leave either one (unspecified).
 * FP8 pools store E4M3(fp32(x) / scale[g]) rounded to nearest even and
 * saturated to +-448.  n_tokens == 0 is a no-op.
 * Errors: EINVAL (null/misaligned pointers, n_tokens < 0, FP8 scales unset). */
pkv_status paged_kv_append(pkv_pool *pool, const void *k_new, const void *v_new,
                           const int64_t *slot_mapping, int64_t n_tokens, void *stream);

/* Decode attention for one new query token per sequence:
 *   out[b][h] = sum_p softmax_p(scale * q[b][h] . K_b[p][g]) V_b[p][g]
 * over positions p < context_lens[b] of sequence b, with g = h / (n_q/n_kv)
 * ("The KV Cache from First Principles", "Implementation" and
 * "Grouped-query attention: the compromise").  K_b[p] lives in block
 * block_tables[b][p / block_size] at offset p % block_size ("KV cache,
 * PagedAttention and FlashAttention", Problem 4, "The idea": the kernel
 * reads keys and values through the block table).  The result equals the
 * plain softmax; internally the kernel keeps a running max and sum
 * (same page, Problem 5, online softmax) and splits long sequences across
 * thread blocks whose partial results are merged by their log-sum-exp
 * (Problem 5, "Serving note").
 *   q             device bf16 [batch][n_q][d_head], 16-byte aligned.
 *   n_q           query heads; a multiple of the pool's n_kv with
 *                 n_q / n_kv in {1, 2, 4, 8}.
 *   block_tables  device int32 [batch][max_blocks_per_seq]; entries past
 *                 ceil(context_len / block_size) are never read.  An entry
 *                 that is read and lies outside [0, num_blocks) is skipped
 *                 (its tokens count as masked) and sets
 *                 PKV_DEVERR_BLOCK_RANGE.
 *   context_lens  device int32 [batch]: tokens cached for each sequence,
 *                 including the one appended this step.  0 gives a zero
 *                 output row; values < 0 or > max_blocks_per_seq *
 *                 block_size are clamped to that range and set
 *                 PKV_DEVERR_CTX_RANGE.
 *   scale         fp32 factor on q.k (normally 1/sqrt(d_head)).
 *   out           device bf16 [batch][n_q][d_head], 16-byte aligned; rounded
 *                 to nearest even from fp32.
 * batch == 0 is a no-op; batch <= 8192 and batch * n_kv * max_blocks_per_seq
 * < 2^30.  Two kernel launches: the decode kernel, which writes every
 * sequence it finishes whole and leaves partials for the ones split across
 * thread blocks, and a merge kernel (a programmatic dependent launch) that
 * combines those partials.  Uses the pool's split-KV workspace, growing it
 * (cudaMalloc, outside any stream capture) when the call needs more.
 * Errors: EINVAL, EUNSUPPORTED (group size), ENOMEM, ECUDA. */
pkv_status paged_decode_attention(pkv_pool *pool, const void *q, int32_t n_q,
                                  const int32_t *block_tables, int32_t max_blocks_per_seq,
                                  const int32_t *context_lens, int32_t batch, float scale,
                                  void *out, void *stream);

/* paged_decode_attention with the page table in the CSR form ("Memory
 * Management in LLM Serving Systems", "Method 3: PagedAttention" and
 * "Walking the table"): sequence b owns the blocks
 * kv_indices[kv_indptr[b] .. kv_indptr[b+1]), logical block j of b being
 * kv_indices[kv_indptr[b] + j].
 *   kv_indptr     device int32 [batch + 1].  A row with kv_indptr[b] < 0,
 *                 kv_indptr[b] > kv_indptr[b+1] or kv_indptr[b+1] >
 *                 n_indices counts as empty and sets PKV_DEVERR_BLOCK_RANGE.
 *   kv_indices    device int32 [n_indices] (may be NULL when n_indices is 0).
 *   context_lens  device int32 [batch]; clamped to 16 x the row's length
 *                 (PKV_DEVERR_CTX_RANGE).
 * n_kv x n_indices < 2^30.  Other arguments, results and errors as
 * paged_decode_attention (the same kernels read the table through the
 * row offsets). */
pkv_status paged_decode_attention_csr(pkv_pool *pool, const void *q, int32_t n_q, const int32_t *kv_indptr,
                                      const int32_t *kv_indices, int64_t n_indices, const int32_t *context_lens,
                                      int32_t batch, float scale, void *out, void *stream);

/* One decode step in one launch: append each sequence's newest token and
 * attend over its whole cache ("The KV Cache from First Principles",
 * "Deriving the cache": compute k_t, v_t, append them, attend with the full
 * cached matrices; "append one row, attend over everything").
 * Equivalent to paged_kv_append of the token at position context_lens[b]-1
 * of every sequence b, into slot block_tables[b][(C-1)/16]*16 + (C-1)%16
 * ("KV cache, PagedAttention and FlashAttention", Problem 4 address
 * arithmetic), followed by paged_decode_attention -- the pool bytes and the
 * output are the same -- but the row is written by the thread block that
 * reads that block anyway, so the step costs the decode's two launches and
 * no append launch.  PKV_INT4 pools (whose value rows need their own min and
 * max before they can be stored) run the append kernel first, finding each
 * slot from the table, then the decode: three launches, same results.
 *   k_new, v_new  device bf16 [batch][n_kv][d_head], 16-byte aligned: the
 *                 new token of each sequence (ignored where context_len == 0).
 *   other arguments as paged_decode_attention.  A sequence's last block must
 *   not be shared with another sequence (as for any append).
 * Errors: as paged_decode_attention. */
pkv_status paged_decode_step(pkv_pool *pool, const void *q, const void *k_new, const void *v_new, int32_t n_q,
                             const int32_t *block_tables, int32_t max_blocks_per_seq,
                             const int32_t *context_lens, int32_t batch, float scale, void *out, void *stream);

/* paged_decode_step for a caller holding its inputs in host memory: brings
 * q, k_new, v_new, block_tables and context_lens (host pointers, same
 * shapes) into a pool-owned device staging area (grown with cudaMalloc when
 * a call needs more), runs the step on `stream`, delivers the output to
 * out_host and synchronises `stream`, so out_host is ready on return.
 * Pinned host memory (cudaHostAlloc / cudaHostRegister, mapped into the
 * device's address space) with q, k_new, v_new and out_host 16-byte aligned
 * (tables and lengths 4-byte): the step's kernels read the inputs in place
 * over the CPU-GPU link and write out_host directly; other pinned inputs:
 * one gather kernel reads them into the staging area first; pageable
 * memory: one copy per array in and one out.  With pinned buffers the
 * call's launches are replayed from a CUDA graph while the arguments stay
 * the same.
 * Errors: as paged_decode_step, plus ENOMEM / ECUDA from staging and copies. */
pkv_status paged_decode_step_host(pkv_pool *pool, const void *q_host, const void *k_new_host,
                                  const void *v_new_host, int32_t n_q, const int32_t *block_tables_host,
                                  int32_t max_blocks_per_seq, const int32_t *context_lens_host, int32_t batch,
                                  float scale, void *out_host, void *stream);

/* Cascade decode for a batch whose sequences all start with the same
 * prefix: the prefix's K and V are read once for the whole batch instead of
 * once per sequence ("Memory Management in LLM Serving Systems", "Prefix
 * sharing": decode-time reads for the shared part drop from n x p to p).
 * Same result as paged_decode_attention (up to rounding order).  The pool's
 * cascade mode (kv_pool_set_cascade_mode) decides whether the call runs the
 * cascade or plain paged decode; the cascade:
 *   stage 1 decodes each sequence's blocks after the prefix; stage 2
 *   attends every query row of each KV head to the prefix on the tcgen05
 *   tensor cores (the prefill kernel of paged_prefill_attention, without
 *   the causal mask) and keeps a (max, sum, output) partial per prefix
 *   chunk; the merge kernel combines each sequence's prefix and tail
 *   partials by log-sum-exp.  Three launches.
 *   prefix_blocks    device int32 [n_prefix_blocks]: physical ids of the
 *                    shared prefix, which is the first n_prefix_blocks * 16
 *                    tokens of every sequence: block_tables[b][0..n) must
 *                    equal prefix_blocks (not checked).
 *   context_lens[b]  at least n_prefix_blocks * 16 (shorter ones are
 *                    treated as prefix-only and set PKV_DEVERR_CTX_RANGE).
 * bf16 and FP8 pools (EUNSUPPORTED for 4-bit ones); on FP8 pools both
 * stages read E4M3 bytes and apply the pool's per-head scales.  Other
 * arguments and errors as paged_decode_attention. */
pkv_status paged_decode_attention_prefix(pkv_pool *pool, const void *q, int32_t n_q,
                                         const int32_t *prefix_blocks, int32_t n_prefix_blocks,
                                         const int32_t *block_tables, int32_t max_blocks_per_seq,
                                         const int32_t *context_lens, int32_t batch, float scale, void *out,
                                         void *stream);

/* Prefill (chunked prefill) attention over the paged cache: for each
 * sequence b, a chunk of T_b new tokens that paged_kv_append has already
 * written at positions C_b - T_b .. C_b - 1 of its cache (C_b =
 * context_lens[b]); token i of the chunk, query head h, attends to cached
 * positions 0 .. C_b - T_b + i with KV head h // (n_q / n_kv) (causal;
 * "Memory Management in LLM Serving Systems", "FlashAttention": exact
 * attention in tiles with an online softmax; "The KV Cache from First
 * Principles", "Deriving the cache": the prefill fills the cache and
 * computes the prompt's attention).  T_b = 1 for every sequence is decode.
 *   q          device bf16 [n_rows][n_q][d_head], 16-byte aligned: the
 *              chunks' tokens, sequence by sequence.
 *   qo_indptr  device int32 [batch + 1]: sequence b's tokens are rows
 *              qo_indptr[b] .. qo_indptr[b+1] (qo_indptr[batch] == n_rows).
 *   context_lens  device int32 [batch]: cache length including the chunk.
 *              A chunk longer than its cache, or a length past the table,
 *              sets PKV_DEVERR_CTX_RANGE.
 *   out        device bf16 [n_rows][n_q][d_head].
 * bf16 and FP8 pools.  One launch (one persistent CTA per SM): tiles of 128
 * query rows per (sequence, KV head) on the tcgen05 tensor cores; each CTA
 * copies the K/V tiles it uses into its own shared memory (TMA, this GPU's
 * pool).  On an FP8 pool the E4M3 tiles are widened to f16 in shared memory
 * (exact) and the products run in f16 (q rounded to f16: |q| must stay in
 * f16's range), with the K scale folded into the score scale and the V
 * scale into the final normalisation.
 * An out-of-range block id is skipped (its keys masked) and sets
 * PKV_DEVERR_BLOCK_RANGE; a qo_indptr that points past n_rows skips those
 * rows' stores and sets PKV_DEVERR_CTX_RANGE.
 * Errors: EINVAL, EUNSUPPORTED (4-bit pools, group size, more than
 * 2^31 query rows x group size), ECUDA. */
pkv_status paged_prefill_attention(pkv_pool *pool, const void *q, int64_t n_rows, int32_t n_q,
                                   const int32_t *qo_indptr, const int32_t *block_tables, int32_t max_blocks_per_seq,
                                   const int32_t *context_lens, int32_t batch, float scale, void *out, void *stream);

/* paged_decode_attention without any allocation.  The pages have no
 * counterpart to this call; it exists for callers that cannot allocate
 * device memory when they decode: an engine that reserved nearly all free
 * HBM for its KV pool at start-up has no room for a workspace, and
 * cudaMalloc/cudaFree may synchronise the whole device, which a caller
 * running other streams' work cannot accept in its decode loop.
 * Same arguments, results and errors as paged_decode_attention, but the
 * split-KV scratch is a fixed 16 MiB array inside the library instead of the
 * pool's workspace; the call allocates nothing and calls no allocating
 * routine, and the pool's workspace stays as it was (empty if this is the
 * only decode call used).
 *   - When the array's memory is taken: kv_pool_create looks up the array's
 *     device address (cudaGetSymbolAddress, with the pool's device current)
 *     and keeps it in the pool.  Under CUDA's lazy module loading that lookup
 *     is what loads the decode code onto the GPU, so the 16 MiB is taken when
 *     the first pool is created on a device, before the caller sizes the
 *     rest of HBM, and stays taken until the process exits.  The call itself
 *     makes no such lookup.
 *   - A call whose scratch would exceed 16 MiB (roughly: more pieces x query
 *     heads x d_head x 4 bytes than fit) fails with PKV_ERANGE before
 *     launching; use paged_decode_attention then.
 *   - The pool's device must be current.  A pool belongs to the CUDA context
 *     it was created in: after cudaDeviceReset, create new pools (the old
 *     ones, and their scratch address, are no longer valid).
 *   - All calls, from every pool and stream, share the one array and it
 *     keeps the last call's contents; nothing in it needs clearing (every
 *     partial a call reads, the same call wrote first).  Calls that overlap
 *     on the GPU race on the array and give wrong results: order them on one
 *     stream, or serialise them.
 * Errors: as paged_decode_attention, plus ERANGE (scratch too small) and
 * EINVAL (pool's device not current). */
pkv_status paged_decode_attention_noalloc(pkv_pool *pool, const void *q, int32_t n_q,
                                          const int32_t *block_tables, int32_t max_blocks_per_seq,
                                          const int32_t *context_lens, int32_t batch, float scale,
                                          void *out, void *stream);

/* ---------------------------------------------------------------------
 * Block management: copy-on-write and swapping ("KV cache, PagedAttention
 * and FlashAttention", Problem 4, "The idea": blocks are shared by
 * reference count, a shared block is copied before it is written, and a
 * preempted sequence's blocks may be swapped to CPU memory; "Memory
 * Management in LLM Serving Systems", "Eviction: recompute or offload?").
 * A block is block_bytes of K plus block_bytes of V: all n_kv heads' 16
 * token rows, held as its n_kv contiguous entries (see pkv_layout).
 * --------------------------------------------------------------------- */

/* Bytes of one block's keys (or, equally, values): n_kv x 16 x d_head x
 * (2 bf16, 1 FP8, 1/2 4-bit).  -1 for a NULL pool. */
int64_t kv_block_bytes(const pkv_pool *pool);

/* Bytes of one swapped block in a host buffer: its K bytes, its V bytes and,
 * for a 4-bit pool, its value rows' (scale, zero point) fp32 pairs
 * (n_kv x 16 x 8 bytes), in that order.  2 x kv_block_bytes for bf16 and FP8
 * pools.  -1 for a NULL pool. */
int64_t kv_swap_entry_bytes(const pkv_pool *pool);

/* Copy blocks inside the pool: block dst_blocks[i] gets the K and V bytes of
 * src_blocks[i], every head and token row, and for a 4-bit pool the value
 * rows' (scale, zero point) pairs too (the copy of copy-on-write).
 *   src_blocks, dst_blocks  device int32 [n]; no dst may appear twice or
 *                           also as a src (unchecked; the copies run in
 *                           parallel).  A pair with an id outside
 *                           [0, num_blocks) is skipped and sets
 *                           PKV_DEVERR_BLOCK_RANGE.
 * One launch, HBM-bound.  Errors: EINVAL, ECUDA. */
pkv_status kv_block_copy(pkv_pool *pool, const int32_t *src_blocks, const int32_t *dst_blocks, int64_t n,
                         void *stream);

/* Swap blocks out to host memory: entry i of host_dst receives block
 * blocks[i] as [K bytes][V bytes][value parameters, 4-bit pools only],
 * kv_swap_entry_bytes per entry.
 *   blocks    device int32 [n]; out-of-range ids are skipped (their entry
 *             left untouched) and set PKV_DEVERR_BLOCK_RANGE.
 *   host_dst  pinned host memory (cudaHostAlloc, or cudaHostRegister),
 *             16-byte aligned, n x kv_swap_entry_bytes bytes; the kernel
 *             writes it directly over the CPU-GPU link.  It holds the data
 *             once the work on `stream` has finished.
 * One launch.  Errors: EINVAL (also for pageable host memory), ECUDA. */
pkv_status kv_swap_out(pkv_pool *pool, const int32_t *blocks, int64_t n, void *host_dst, void *stream);

/* Swap blocks in: block blocks[i] gets entry i of host_src (the layout
 * kv_swap_out writes).  host_src: pinned, 16-byte aligned, caller-owned
 * until the work on `stream` has finished.  Same errors as kv_swap_out. */
pkv_status kv_swap_in(pkv_pool *pool, const void *host_src, const int32_t *blocks, int64_t n, void *stream);

/* Refcounted block allocator (host side; the pages' block manager).  It
 * tracks which of num_blocks physical blocks are in use and how many block
 * table entries refer to each; the caller keeps the tables.  Free blocks
 * are handed out lowest id first, so results are reproducible.  Thread-safe
 * (one internal mutex).  All calls validate everything before changing
 * anything. */
typedef struct pkv_alloc pkv_alloc;

/* num_blocks in [1, 2^31 - 1].  Errors: EINVAL, ENOMEM. */
pkv_status kv_alloc_create(int64_t num_blocks, pkv_alloc **out);
pkv_status kv_alloc_destroy(pkv_alloc *alloc);
/* Free blocks; -1 for a NULL allocator. */
int64_t kv_alloc_free_blocks(pkv_alloc *alloc);
/* References to block id (0 = free).  Errors: EINVAL, ERANGE. */
pkv_status kv_alloc_refcount(pkv_alloc *alloc, int32_t id, int32_t *out);
/* Take n free blocks (reference count 1 each) into ids_out (host int32
 * [n]), lowest ids first; all or nothing.  Errors: EINVAL, ENOMEM (fewer
 * than n free). */
pkv_status kv_alloc_take(pkv_alloc *alloc, int64_t n, int32_t *ids_out);
/* Add one reference to each listed block (a table entry now shares it: a
 * forked sequence, a common prefix).  Every id must be allocated.  Errors:
 * EINVAL (free block), ERANGE. */
pkv_status kv_alloc_share(pkv_alloc *alloc, const int32_t *ids, int64_t n);
/* Drop one reference per listed entry; a block reaching 0 is free again.
 * A block listed k times must hold at least k references.  Errors: EINVAL
 * (a free block or too many releases), ERANGE. */
pkv_status kv_alloc_release(pkv_alloc *alloc, const int32_t *ids, int64_t n);
/* Copy-on-write, before writing into the blocks ids[0..n) (host int32, the
 * caller's table entries): every entry whose block has other references is
 * given a fresh block; the old block loses that reference; the pair
 * (old, fresh) is appended to copy_src / copy_dst (host int32 [n]) and
 * ids[i] is replaced.  *n_copies receives the pair count.  Run
 * kv_block_copy on the pairs before writing.  All or nothing.  Errors:
 * EINVAL, ERANGE, ENOMEM (not enough free blocks for the copies). */
pkv_status kv_alloc_prepare_write(pkv_alloc *alloc, int32_t *ids, int64_t n, int32_t *copy_src, int32_t *copy_dst,
                                  int64_t *n_copies);

/* KV-cache bytes per token: 2 x layers x n_kv x d_head x bytes_per_value
 * ("KV cache, PagedAttention and FlashAttention", Problem 3, "The concepts";
 * "Memory Management in LLM Serving Systems", "KV cache sizing").
 * bytes_per_value may be fractional (0.5 for 4-bit; scales not counted).
 * Host arithmetic only.  Returns a negative value for negative inputs. */
double kv_bytes_per_token(int32_t layers, int32_t n_kv, int32_t d_head, double bytes_per_value);

/* Read the pool's sticky device error word into *bits (NULL allowed),
 * synchronising the device; clear != 0 resets it.  Returns PKV_OK when no
 * bit is set, PKV_EDEVICE when some are, or ECUDA. */
pkv_status pkv_get_error(pkv_pool *pool, int32_t clear, uint32_t *bits);

/* Failure-detection check of the bounded waits every kernel uses: launches
 * one warp on `stream` that waits on an mbarrier nothing ever arrives at,
 * gives up after limit_ns (1 us .. 2 s), records PKV_DEVERR_TIMEOUT in the
 * pool's error word and returns.  Nothing faults and the context stays
 * usable; read the bit with pkv_get_error.  Errors: EINVAL, ERANGE, ECUDA. */
pkv_status pkv_selftest_wait_timeout(pkv_pool *pool, uint64_t limit_ns, void *stream);

/* Timing: while enabled, the library records a CUDA event pair around every
 * kernel it launches, on the launching stream.  pkv_timing_read synchronises
 * those events, fills *out and, if reset != 0, clears the counters.  The
 * launch counters count every launch whether or not timing is enabled. */
pkv_status pkv_timing_enable(pkv_pool *pool, int32_t on);
pkv_status pkv_timing_read(pkv_pool *pool, int32_t reset, pkv_timing *out);

/* Static name of a status; never NULL. */
const char *pkv_status_string(pkv_status s);

/* Description of the last failure on this thread ("" if none). */
const char *pkv_last_error_message(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
