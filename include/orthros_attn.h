/*
 * orthros_attn.h -- C ABI of the Orthros attention hot path on one GPU.
 *
 * Orthros ("Orthros: Phase-Aware Heterogeneous Attention for Efficient
 * Transformers", paperz.arrangedbits.com full text) runs, in every layer:
 *   - a base stream: sliding-window attention of EVERY position t over the keys
 *     max(0, t-w+1) .. t  (Sec. 3.1, Eq. 4; 0-indexed here), which also
 *     produces the layer's K/V cache;
 *   - an output stream: full causal cross-attention of the output positions
 *     over keys 0 .. t of the same K/V (Sec. 3.1, Eq. 5).
 * Both query streams come from one Q projection through their own
 * per-channel scale-offset affine, q = alpha (.) q_raw + beta (Sec. 3.1,
 * Alg. 1 line 5). The four regimes of Sec. 3.2 (pre-training, SFT,
 * prefilling, decoding) differ only in which positions are output rows.
 *
 * Conventions shared by every entry point
 *   - All tensor arguments are DEVICE pointers unless marked HOST. The caller
 *     owns every buffer, including the workspace and the cache pages; the
 *     library never allocates, frees or synchronises on the compute path.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = default stream).
 *   - Layouts are row-major and contiguous. Query heads h map to K/V heads
 *     kv = h / (Hq / Hkv) (contiguous groups; Hq == Hkv is plain multi-head).
 *   - Element type of q, k, v, q_out, k_new, v_new, caches and o_* is given by
 *     `dtype`: ORTHROS_BF16 (bfloat16) or ORTHROS_F32 (float). alpha/beta and
 *     lse are always float. lse is the natural log of sum_j exp(scale q.k_j).
 *   - The logit is scale * (q_affined . k); scale is usually 1/sqrt(d)
 *     (Sec. 2.1, Eq. 1).
 *   - Tensors of element type bf16/f32 must be 16-byte aligned.
 *   - Errors found on the host return before any launch (ORTHROS_EINVAL,
 *     ORTHROS_EUNSUPPORTED, ORTHROS_EWORKSPACE); orthros_last_error() then
 *     describes the problem. Launch failures return ORTHROS_ECUDA. Bad data
 *     that only the GPU can see (a position out of range, a block-table entry
 *     outside the page pool, a cache length past the block table) sets a
 *     status word in the
 *     workspace; the affected rows are skipped or their outputs are NaN, and
 *     orthros_check() reports ORTHROS_EDEVICE. Nothing aborts or traps.
 *   - Supported head sizes: d = 64 or 128.
 *   - The *_workspace_size functions size the scratch for the CUDA device that
 *     is current when they are called (the split-KV partials depend on its SM
 *     count); call them with the device that will run the call current. A
 *     workspace smaller than the call then needs returns ORTHROS_EWORKSPACE.
 */
#ifndef ORTHROS_ATTN_H
#define ORTHROS_ATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ORTHROS_API __attribute__((visibility("default")))
#else
#define ORTHROS_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *orthros_stream_t; /* same type as cudaStream_t */

typedef enum {
    ORTHROS_OK = 0,
    ORTHROS_EINVAL = 1,       /* bad argument, detected on the host */
    ORTHROS_EUNSUPPORTED = 2, /* well-formed but not supported (e.g. d = 96) */
    ORTHROS_ECUDA = 3,        /* a CUDA call or kernel launch failed */
    ORTHROS_EWORKSPACE = 4,   /* workspace NULL or smaller than required */
    ORTHROS_EDEVICE = 5,      /* a kernel flagged bad device-side data */
    ORTHROS_ETIMEOUT = 6      /* a kernel's bounded wait ran out */
} orthros_status;

typedef enum { ORTHROS_BF16 = 0, ORTHROS_F32 = 1 } orthros_dtype;

/* Bits of the device status word (see orthros_check). */
#define ORTHROS_DEV_BAD_POSITION 0x1u  /* out_positions entry outside [0, T) */
#define ORTHROS_DEV_BAD_PAGE 0x2u      /* block-table entry outside [0, num_pages) */
#define ORTHROS_DEV_BAD_LENGTH 0x4u    /* cache_lens[b] < 0 or past the block table */
/* 0x8u is never raised: keys and affined queries beyond the fp16 range of the
 * tensor-core prefill are scaled by exact powers of two (the logit scale
 * takes the inverse), so any finite bf16 input is served. */
#define ORTHROS_DEV_FP16_RANGE 0x8u
#define ORTHROS_DEV_TIMEOUT 0x10u      /* a bounded wait inside a kernel ran out */

/*
 * Workspace bytes orthros_prefill needs for these sizes. n_out is the total
 * number of output rows. Returns 0 for sizes orthros_prefill would reject.
 */
ORTHROS_API size_t orthros_prefill_workspace_size(int B, int T, int Hq, int Hkv, int d,
                                      int n_out, int window, orthros_dtype dtype);

/*
 * Prefill (Sec. 3.2 regimes pre-training / SFT / prefilling): Eq. 4 at every
 * position of B sequences of T tokens, Eq. 5 at the output rows, and
 * optionally the paged K/V cache fill that the decoding phase reads.
 *
 * q            [B, T, Hq, d]   raw queries (the affines are applied inside)
 * k, v         [B, T, Hkv, d]
 * alpha_base, beta_base [Hq, d] float: base-stream affine (alpha, beta)
 * alpha_out,  beta_out  [Hq, d] float: output-stream affine (alpha', beta');
 *              may be NULL when n_out == 0
 * out_indptr   HOST [B+1] int32, out_indptr[0] = 0, non-decreasing,
 *              out_indptr[B] = n_out: output rows of sequence b are
 *              r in [out_indptr[b], out_indptr[b+1])
 * out_positions [n_out] int32: position t_r in [0, T) of output row r (any
 *              order, repeats allowed; each row is independent)
 * q_out        [n_out, Hq, d] raw output-stream queries, or NULL: then the raw
 *              query of row r is q[b, t_r] (one shared Q projection; exact for
 *              a first layer, whose output tokens duplicate the base tokens)
 * window       w >= 1; w >= T gives full causal attention in the base stream
 * scale        logit scale (finite)
 * o_base [B, T, Hq, d], lse_base [B, Hq, T] float
 * o_out  [n_out, Hq, d], lse_out [n_out, Hq] float  (may be NULL if n_out == 0)
 * k_cache, v_cache [num_pages, page_size, Hkv, d], block_table [B, max_pages]
 *              int32: optional (all NULL to skip). When given, token t of
 *              sequence b is also written to page block_table[b*max_pages +
 *              t/page_size], slot t % page_size, for t < T (needs
 *              max_pages * page_size >= T). num_pages bounds the entries.
 * workspace    device scratch of at least orthros_prefill_workspace_size()
 *              bytes, 256-byte aligned; its contents on entry do not matter.
 */
ORTHROS_API orthros_status orthros_prefill(
    const void *q, const void *k, const void *v,
    const float *alpha_base, const float *beta_base,
    const float *alpha_out, const float *beta_out,
    const int32_t *out_indptr, const int32_t *out_positions, int n_out,
    const void *q_out,
    int B, int T, int Hq, int Hkv, int d, int window, float scale,
    orthros_dtype dtype,
    void *o_base, float *lse_base, void *o_out, float *lse_out,
    void *k_cache, void *v_cache, const int32_t *block_table,
    int max_pages, int page_size, int num_pages,
    void *workspace, size_t workspace_bytes, orthros_stream_t stream);

/* Workspace bytes orthros_prefill_from_host needs for these sizes (0 if rejected). */
ORTHROS_API size_t orthros_prefill_from_host_workspace_size(int B, int T, int Hq, int Hkv, int d, int n_out,
                                                            int window, orthros_dtype dtype);

/*
 * orthros_prefill with the step's inputs and outputs in HOST memory: the
 * same computation (Eq. 4 for every position, Eq. 5 for the output rows, the
 * optional cache fill), the host-to-device and device-to-host copies included.
 *
 * HOST:   q, k, v, o_base, lse_base, out_indptr, out_positions, q_out, o_out,
 *         lse_out, with the shapes of orthros_prefill. Page-locked memory
 *         (cudaHostAlloc / cudaHostRegister) lets the copies overlap the
 *         compute; pageable memory gives the same results with copies that do
 *         not overlap. Device memory passed here is rejected (ORTHROS_EINVAL).
 * DEVICE: alpha_base, beta_base, alpha_out, beta_out (model parameters), the
 *         optional k_cache, v_cache, block_table, and the workspace (at least
 *         orthros_prefill_from_host_workspace_size() bytes, 256-byte aligned;
 *         it holds device copies of q, k, v and o_base besides the scratch).
 * out_positions are checked on the host: a position outside [0, T) returns
 * ORTHROS_EINVAL before anything is enqueued.
 *
 * A sequence longer than one chunk (at least 16384 tokens and four halos of
 * w - 1 keys; bf16 only) is computed chunk by chunk as orthros_prefill_shard
 * calls (each chunk's keys with the halo before it, so its base rows are
 * exact, and each output row's partial over the chunk's keys), and the
 * partials are merged as orthros_merge_partials does, so the results equal
 * orthros_prefill's up to the rounding of that merge. Chunk c + 1 is copied
 * in while chunk c computes and chunk c - 1 is copied out, on two copy streams
 * of the library's own (created once per device) ordered after the work
 * already on `stream`; `stream` itself runs the compute and waits for the
 * last copy out, so every output is in host memory once `stream` reaches the
 * point after this call (also after an error return: what the call had
 * already enqueued on its copy streams is joined to `stream`). Calls are
 * enqueued one at a time (an internal lock).
 * Shorter sequences, and f32, copy everything in, compute, and copy out on
 * `stream`. Device-side status as for orthros_prefill (orthros_check on this
 * call's workspace).
 */
ORTHROS_API orthros_status orthros_prefill_from_host(
    const void *q, const void *k, const void *v,
    const float *alpha_base, const float *beta_base,
    const float *alpha_out, const float *beta_out,
    const int32_t *out_indptr, const int32_t *out_positions, int n_out,
    const void *q_out,
    int B, int T, int Hq, int Hkv, int d, int window, float scale,
    orthros_dtype dtype,
    void *o_base, float *lse_base, void *o_out, float *lse_out,
    void *k_cache, void *v_cache, const int32_t *block_table,
    int max_pages, int page_size, int num_pages,
    void *workspace, size_t workspace_bytes, orthros_stream_t stream);

/* Workspace bytes orthros_prefill_shard needs for these sizes (0 if rejected). */
ORTHROS_API size_t orthros_prefill_shard_workspace_size(int B, int Tq, int Tkv, int Hq, int Hkv, int d,
                                                       int n_rows, int window, orthros_dtype dtype);

/*
 * One rank's share of a prefill whose token axis is cut into contiguous chunks
 * across devices (sequence parallelism: the paper runs its 64K-1M-token
 * prefills on 8 GPUs, Sec. 4.5 and the appendix's training/inference setup,
 * without describing the split). Eq. 4 needs only a halo of the w - 1 keys
 * before a chunk; Eq. 5 of an output row spans every chunk up to its position,
 * so each chunk contributes a normalised partial that orthros_merge_partials
 * combines exactly.
 *
 * The chunk holds Tq tokens at global positions P0 .. P0 + Tq - 1. Its keys
 * and values come with the H = Tkv - Tq tokens before it (the halo, received
 * from the ranks that own them; H >= min(w - 1, P0) makes the band rows exact):
 * k, v [B, Tkv, Hkv, d] hold positions P0 - H .. P0 + Tq - 1. Positions below
 * are in this buffer's coordinates (global position - P0 + H).
 *   - base rows (Eq. 4): q [B, Tq, Hq, d] are the chunk's raw queries; query
 *     i sits at position H + i and attends keys max(0, H + i - w + 1) .. H + i.
 *     o_base [B, Tq, Hq, d] (dtype), lse_base [B, Hq, Tq] float.
 *   - partial output rows (Eq. 5 over the chunk's own keys): row r of sequence b
 *     (row_indptr as out_indptr of orthros_prefill, HOST) at position t_r >= 0
 *     attends keys H .. min(t_r, Tkv - 1): rows owned by later ranks have
 *     t_r >= Tkv and read the whole chunk; a row with t_r < H reads nothing and
 *     gets o = 0, lse = -inf. q_rows [n_rows, Hq, d] are their raw
 *     output-stream queries (required when n_rows > 0).
 *     o_part [n_rows, Hq, d] float, lse_part [n_rows, Hq] float.
 * bf16 only (ORTHROS_EUNSUPPORTED otherwise); 1 <= Tq <= Tkv. A negative
 * row position sets ORTHROS_DEV_BAD_POSITION and that row is NaN. Workspace
 * and errors as for orthros_prefill.
 */
ORTHROS_API orthros_status orthros_prefill_shard(
    const void *q, const void *k, const void *v,
    const float *alpha_base, const float *beta_base,
    const float *alpha_out, const float *beta_out,
    const int32_t *row_indptr, const int32_t *row_positions, int n_rows,
    const void *q_rows,
    int B, int Tq, int Tkv, int Hq, int Hkv, int d, int window, float scale,
    orthros_dtype dtype,
    void *o_base, float *lse_base, float *o_part, float *lse_part,
    void *workspace, size_t workspace_bytes, orthros_stream_t stream);

/*
 * Exact merge of normalised attention partials of the same rows over disjoint
 * key sets: lse = log sum_p exp(lse_p), o = sum_p exp(lse_p - lse) o_p (each
 * set's share of the softmax denominator is exp(lse_p)). Merges the chunk
 * partials of orthros_prefill_shard into the rows of Eq. 5.
 * o_parts [n_parts, n_rows, Hq, d] float, lse_parts [n_parts, n_rows, Hq] float
 * o_out [n_rows, Hq, d] of element type dtype, lse_out [n_rows, Hq] float.
 * A partial with lse = -inf holds no keys and weighs nothing; a row whose
 * partials are all empty comes back empty (o = 0, lse = -inf), so partials
 * may be merged in any grouping. Needs no workspace.
 */
ORTHROS_API orthros_status orthros_merge_partials(const float *o_parts, const float *lse_parts, int n_parts,
                                                  int n_rows, int Hq, int d, orthros_dtype dtype,
                                                  void *o_out, float *lse_out, orthros_stream_t stream);

/* Workspace bytes orthros_prefill_backward needs for these sizes (0 if rejected). */
ORTHROS_API size_t orthros_prefill_backward_workspace_size(int B, int T, int Hq, int Hkv, int d,
                                               int n_out, int window, orthros_dtype dtype);

/*
 * Backward of orthros_prefill for training in the pre-training and
 * fine-tuning regimes (Sec. 3.2): the gradients of a loss L with respect to
 * q, k, v, q_out and the four affine vectors, given dL/do of both streams.
 * The paper prints no backward; it is the chain rule through Eq. 4 and Eq. 5
 * (softmax attention) and through the affines q = alpha (.) q_raw + beta.
 * lse is an output the loss is taken not to depend on.
 *
 * Forward arguments (q .. scale, dtype) exactly as given to orthros_prefill,
 * except that out_positions must hold positions in [0, T) (repeats allowed).
 * o_base, lse_base, o_out, lse_out  the outputs orthros_prefill returned for
 *              them (o is used for D = dO . o, lse to recompute softmax weights)
 * do_base [B, T, Hq, d], do_out [n_out, Hq, d]: dL/do_base, dL/do_out
 * dq      [B, T, Hq, d]  dL/dq. When q_out is NULL the output rows read q at
 *              their positions, and their share is included here.
 * dk, dv  [B, T, Hkv, d] (both streams' shares)
 * dq_out  [n_out, Hq, d] dL/dq_out; required when q_out is given, else ignored
 * d_alpha_base, d_beta_base, d_alpha_out, d_beta_out [Hq, d] float
 * All gradients are overwritten (not accumulated into). Element tensors have
 * the dtype of q; lse and the affine gradients are float.
 * workspace    at least orthros_prefill_backward_workspace_size() bytes,
 *              256-byte aligned; contents on entry do not matter.
 * Errors as for orthros_prefill; an output position outside [0, T) sets
 * ORTHROS_DEV_BAD_POSITION and that row's dq_out (or share of dq) is NaN/absent.
 */
ORTHROS_API orthros_status orthros_prefill_backward(
    const void *q, const void *k, const void *v,
    const float *alpha_base, const float *beta_base,
    const float *alpha_out, const float *beta_out,
    const int32_t *out_indptr, const int32_t *out_positions, int n_out,
    const void *q_out,
    int B, int T, int Hq, int Hkv, int d, int window, float scale,
    orthros_dtype dtype,
    const void *o_base, const float *lse_base, const void *o_out, const float *lse_out,
    const void *do_base, const void *do_out,
    void *dq, void *dk, void *dv, void *dq_out,
    float *d_alpha_base, float *d_beta_base, float *d_alpha_out, float *d_beta_out,
    void *workspace, size_t workspace_bytes, orthros_stream_t stream);

/* Workspace bytes orthros_decode needs for these sizes (0 if rejected). */
ORTHROS_API size_t orthros_decode_workspace_size(int B, int Hq, int Hkv, int d,
                                     int max_pages, int page_size,
                                     orthros_dtype dtype);

/*
 * One decoding step for B sequences (Sec. 3.2 "Decoding"; the decoupled
 * token pair of Sec. 3.1). For each sequence b with L = cache_lens[b]:
 *   1. the base token's K/V (k_new[b], v_new[b]) is written at position L of
 *      the paged cache (page block_table[b*max_pages + L/page_size], slot
 *      L % page_size);
 *   2. the base query (alpha/beta affine) attends keys max(0, L-w+1) .. L;
 *   3. the output query (alpha'/beta' affine) attends keys 0 .. L.
 * Both queries read the cache after the append.
 *
 * q            [B, Hq, d] raw query of the base token
 * q_out        [B, Hq, d] raw query of the output token, or NULL (= q)
 * k_new, v_new [B, Hkv, d]
 * k_cache, v_cache [num_pages, page_size, Hkv, d]  (modified: one slot per b)
 * block_table  [B, max_pages] int32 physical page ids
 * cache_lens   [B] int32 lengths BEFORE this step (read only; the caller
 *              increments them afterwards and provides a page for slot L)
 * o_base, o_out [B, Hq, d]; lse_base, lse_out [B, Hq] float
 * workspace    at least orthros_decode_workspace_size() bytes, 256-byte aligned
 */
ORTHROS_API orthros_status orthros_decode(
    const void *q, const void *q_out, const void *k_new, const void *v_new,
    void *k_cache, void *v_cache, const int32_t *block_table, int max_pages,
    int page_size, int num_pages, const int32_t *cache_lens,
    const float *alpha_base, const float *beta_base,
    const float *alpha_out, const float *beta_out,
    int B, int Hq, int Hkv, int d, int window, float scale, orthros_dtype dtype,
    void *o_base, float *lse_base, void *o_out, float *lse_out,
    void *workspace, size_t workspace_bytes, orthros_stream_t stream);

/* Workspace bytes orthros_extend needs for these sizes (0 if rejected). */
ORTHROS_API size_t orthros_extend_workspace_size(int B, int n_new, int n_out, int Hq, int Hkv, int d,
                                     int max_pages, int page_size, orthros_dtype dtype);

/*
 * One continuous-batching step over the paged cache: a batch in which some
 * sequences append a prefill chunk, others decode one token, others nothing.
 * Sec. 3.2 runs every regime as the same computation (a prefill followed by
 * decoding steps agrees exactly with one longer prefill), so one call serves
 * them all; orthros_decode is the case of one new token per sequence.
 *
 * Sequence b (L = cache_lens[b]) appends its n_b = new_indptr[b+1] -
 * new_indptr[b] new tokens (rows new_indptr[b] .. of q, k_new, v_new) at
 * positions L .. L + n_b - 1 of its pages, then
 *   - every new token's base row attends keys max(0, t-w+1) .. t (Eq. 4);
 *   - every output row r (out_indptr[b] <= r < out_indptr[b+1]) at position
 *     out_positions[r] = t in [0, L + n_b) attends keys 0 .. t (Eq. 5), with
 *     raw query q_out[r], or, when q_out is NULL, the q of the new token at
 *     position t (t must then be a new position).
 *
 * q            [n_new, Hq, d] raw base queries of the new tokens
 * q_out        [n_out, Hq, d] raw output queries, or NULL (see above)
 * k_new, v_new [n_new, Hkv, d]
 * k_cache, v_cache [num_pages, page_size, Hkv, d] (modified: the appends)
 * block_table  [B, max_pages] int32; pages for positions < L + n_b must exist
 * cache_lens   [B] int32 device, lengths BEFORE the step (read only)
 * new_indptr, out_indptr  HOST [B+1] int32, start at 0, non-decreasing
 * out_positions [n_out] int32 device, absolute positions
 * o_base [n_new, Hq, d], lse_base [n_new, Hq], o_out [n_out, Hq, d],
 * lse_out [n_out, Hq] float
 * workspace    at least orthros_extend_workspace_size() bytes, 256-byte aligned
 * Rows whose data are impossible (a position outside its sequence, a length
 * past the block table) set ORTHROS_DEV_BAD_POSITION / _BAD_LENGTH and come
 * back as NaN; a page id outside [0, num_pages) sets ORTHROS_DEV_BAD_PAGE.
 */
ORTHROS_API orthros_status orthros_extend(
    const void *q, const void *q_out, const void *k_new, const void *v_new,
    void *k_cache, void *v_cache, const int32_t *block_table, int max_pages,
    int page_size, int num_pages, const int32_t *cache_lens,
    const int32_t *new_indptr, const int32_t *out_indptr, const int32_t *out_positions,
    const float *alpha_base, const float *beta_base,
    const float *alpha_out, const float *beta_out,
    int B, int Hq, int Hkv, int d, int window, float scale, orthros_dtype dtype,
    void *o_base, float *lse_base, void *o_out, float *lse_out,
    void *workspace, size_t workspace_bytes, orthros_stream_t stream);

/*
 * The shared Q/K/V projection that feeds the hot path (Alg. 1 lines 4-5,
 * Sec. 3.1): base-token rows x[0 .. n_base) and output-token rows
 * x[n_base .. n_base+n_out) are multiplied by ONE weight (in decoding, a
 * step's base and output tokens share its read), y = x W, and
 *   q_base = alpha_base (.) y_Q + beta_base   for base rows,
 *   q_out  = alpha_out  (.) y_Q + beta_out    for output rows,
 *   k, v   = y_K, y_V                         for base rows only (only the
 *            base stream writes the cache), to k_out / v_out and/or to the
 *            page slot of (token_seq[i], token_pos[i]).
 * The queries leave with their affine applied: pass identity affines
 * (alpha = 1, beta = 0) to the attention calls that read them.
 *
 * x        [n_base + n_out, d_model] bf16, d_model a multiple of 64
 * w_qkv    [(Hq + 2 Hkv) d, d_model] bf16: row j holds the weights of output
 *          column j (W transposed); columns are Q heads, then K, then V heads
 * alpha_*, beta_* [Hq, d] float
 * q_base [n_base, Hq, d], q_out [n_out, Hq, d] bf16 (q_out NULL if n_out = 0)
 * k_out, v_out [n_base, Hkv, d] bf16, or both NULL
 * k_cache, v_cache [num_pages, page_size, Hkv, d], block_table [B, max_pages],
 * token_seq, token_pos [n_base] device int32: all NULL for no cache writes
 * workspace at least 256 bytes (status word), 256-byte aligned
 * Errors: bf16 only (EUNSUPPORTED otherwise); a row whose page does not exist
 * sets ORTHROS_DEV_BAD_PAGE / _BAD_POSITION and its cache write is skipped.
 * The paper has no kernel for this step; it is the step upstream of the
 * attention that the decoding pair's shared weight read makes worth fusing.
 */
ORTHROS_API orthros_status orthros_qkv_project(
    const void *x, int n_base, int n_out, int d_model, const void *w_qkv,
    int Hq, int Hkv, int d,
    const float *alpha_base, const float *beta_base,
    const float *alpha_out, const float *beta_out,
    void *q_base, void *q_out, void *k_out, void *v_out,
    void *k_cache, void *v_cache, const int32_t *block_table, int B,
    int max_pages, int page_size, int num_pages,
    const int32_t *token_seq, const int32_t *token_pos, orthros_dtype dtype,
    void *workspace, size_t workspace_bytes, orthros_stream_t stream);

/*
 * orthros_decode without a workspace argument, for callers that cannot
 * allocate device memory where they run a decoding step (for example a host
 * framework whose operator interface passes only inputs and outputs, or a
 * serving loop whose allocator must not grow). The paper has no counterpart:
 * this is a deployment convenience, not part of the method.
 *
 * Same arguments, semantics and results as orthros_decode, minus workspace.
 * Scratch comes from one 32 MiB device array inside the library (held by
 * every GPU that loads it until the process exits); sizes whose
 * orthros_decode_workspace_size() exceeds that return ORTHROS_EWORKSPACE
 * before any launch. The first call on a device looks up the array's address
 * (cudaGetSymbolAddress) with that device current: make it before any stream
 * capture. All calls share the array: calls ordered on one stream are fine,
 * calls that overlap on the GPU race. Device-side status bits of this entry
 * point are not exposed; rows with bad data (or whose kernel gave up on a
 * bounded wait) come back as NaN. The array's address is kept per device for
 * the life of the process: resetting a device (cudaDeviceReset) after its
 * first call is not supported.
 */
ORTHROS_API orthros_status orthros_decode_static(
    const void *q, const void *q_out, const void *k_new, const void *v_new,
    void *k_cache, void *v_cache, const int32_t *block_table, int max_pages,
    int page_size, int num_pages, const int32_t *cache_lens,
    const float *alpha_base, const float *beta_base,
    const float *alpha_out, const float *beta_out,
    int B, int Hq, int Hkv, int d, int window, float scale, orthros_dtype dtype,
    void *o_base, float *lse_base, void *o_out, float *lse_out,
    orthros_stream_t stream);

/*
 * Synchronises `stream`, reads the status word that the last call using
 * `workspace` left there and returns ORTHROS_OK, ORTHROS_EDEVICE (data bits) or
 * ORTHROS_ETIMEOUT (timeout bit). *bits (if not NULL) receives the raw
 * ORTHROS_DEV_* bits. This is the one call that blocks the host.
 */
ORTHROS_API orthros_status orthros_check(const void *workspace, orthros_stream_t stream,
                             uint32_t *bits);

/*
 * Per-kernel timing of the library's own launches (tracing aid).
 * orthros_profile_begin() starts recording: every kernel the library launches
 * afterwards is bracketed by two CUDA events recorded on its launch stream.
 * orthros_profile_end() stops recording, waits for the recorded events and
 * fills up to max_entries records, one per kernel name, in first-launch order.
 * It returns the number of distinct kernels (may exceed max_entries), or -1 on
 * a CUDA error. Recording is process-wide and not thread-safe; it adds two
 * event records per launch and nothing else.
 */
typedef struct {
    char name[48];   /* kernel family, e.g. "prefill_tc" */
    int launches;    /* launches recorded */
    double total_ms; /* summed event-to-event time of those launches */
} orthros_kernel_time;

ORTHROS_API orthros_status orthros_profile_begin(void);
ORTHROS_API int orthros_profile_end(orthros_kernel_time *out, int max_entries);

/*
 * Self-test of the failure path (no counterpart in the paper): launches one
 * small kernel whose only wait is on an mbarrier that nothing arrives on,
 * bounded by limit_cycles SM clock cycles (1 .. about 4e9). The wait runs out,
 * the kernel raises ORTHROS_DEV_TIMEOUT in the workspace's status word and
 * returns; orthros_check(workspace, ...) then reports ORTHROS_ETIMEOUT. Every
 * kernel of the library that waits on a barrier uses the same bounded wait
 * (with a limit of about 2 s), so a stalled pipeline ends with this status
 * instead of a hang. workspace: at least 256 bytes, 256-byte aligned.
 */
ORTHROS_API orthros_status orthros_selftest_wait_timeout(long long limit_cycles, void *workspace,
                                                         size_t workspace_bytes, orthros_stream_t stream);

/* Static English name of a status code. */
ORTHROS_API const char *orthros_status_string(orthros_status s);

/* Description of the last host-side error on this thread ("" if none). */
ORTHROS_API const char *orthros_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* ORTHROS_ATTN_H */
