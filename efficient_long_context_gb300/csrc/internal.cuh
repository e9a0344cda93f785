// internal.cuh -- declarations shared by the translation units of liborthros_attn.
//
// Nothing here is part of the public ABI (include/orthros_attn.h is).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "orthros_attn.h"

namespace orthros {

// ---------------------------------------------------------------------------
// Workspace layout (every region 256-byte aligned)
//   [0, 256)        status word (uint32 at offset 0) + spare
//   then per-entry-point regions, sized by the *_workspace_size functions
// ---------------------------------------------------------------------------
constexpr size_t kStatusBytes = 256;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// A kernel's dynamic shared-memory limit is a per-device attribute: raise it
// once on every device that launches the kernel (the first 64 devices are
// remembered; later ones set it on every launch). Concurrent first launches
// may both set it, which is harmless.
class SmemLimit {
  public:
    cudaError_t ensure(const void *func, int bytes) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
        if (bit && (done_.load(std::memory_order_acquire) & bit)) return cudaSuccess;
        e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e == cudaSuccess && bit) done_.fetch_or(bit, std::memory_order_acq_rel);
        return e;
    }

  private:
    std::atomic<uint64_t> done_{0};
};

__device__ __forceinline__ void set_status(uint32_t *status, uint32_t bit) {
    if (status) atomicOr(status, bit);
}

// Element loads / stores for the two supported element types.
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Arguments of the generic row kernels. Every pointer is a device pointer.
struct RowsArgs {
    const void *q;      // prefill [B,T,Hq,d] / decode [B,Hq,d]
    const void *q_out;  // prefill [n_out,Hq,d] / decode [B,Hq,d] or nullptr
    const void *k;      // prefill [B,T,Hkv,d] / decode cache [num_pages,P,Hkv,d]
    const void *v;
    const float *alpha_base, *beta_base, *alpha_out, *beta_out;
    const int32_t *out_indptr;     // device copy [B+1] (prefill output rows)
    const int32_t *out_positions;  // [n_out]
    const int32_t *block_table;    // decode / extend
    const int32_t *cache_lens;     // decode / extend
    const int32_t *new_indptr;     // extend: device [B+1], new tokens of each sequence
    int n_out, max_pages, page_size, num_pages;
    int n_new;                     // extend
    int B, T, Hq, Hkv, window;
    float scale;
    void *o_base;
    float *lse_base;
    void *o_out;
    float *lse_out;
    uint32_t *status;
};

enum RowKind { kPrefillBase = 0, kPrefillOut = 1, kDecodePair = 2, kExtendBase = 3, kExtendOut = 4 };

// orthros_api.cu: records the message returned by orthros_last_error() and
// passes the status through.
orthros_status report_error(orthros_status s, const char *fmt, ...);

// profile.cu: brackets one kernel launch with CUDA events while profiling is on.
class ProfScope {
  public:
    ProfScope(const char *name, cudaStream_t s);
    ~ProfScope();
    ProfScope(const ProfScope &) = delete;
    ProfScope &operator=(const ProfScope &) = delete;

  private:
    const char *name_;
    cudaStream_t stream_;
    void *a_;
};

// prefill_tc.cu: tensor-core banded prefill (bf16 inputs, d = 64 or 128).
struct TcParams {
    const __nv_bfloat16 *q;      // [B,T,Hq,d]
    const __nv_bfloat16 *q_out;  // [n_out,Hq,d] or nullptr
    const float *alpha_base, *beta_base, *alpha_out, *beta_out;
    const int32_t *out_indptr;         // device [B+1]
    const int32_t *out_positions;      // [n_out]
    const int32_t *cross_unit_indptr;  // device [B+1]: output-row units per sequence (prefix sums)
    int B, T, Hq, Hkv, window;  // T: key positions per sequence
    int Tq;     // query rows per sequence; query i sits at key position q_off + i
    int q_off;  // T - Tq (0 for a whole-sequence prefill)
    int shard;  // output rows are partials over keys key_lo .. min(t, T - 1)
    int key_lo; // first key of every output row (0 unless shard)
    float scale, scale_log2;
    int n_cross_units, n_base_units, base_nblk;
    int n_out;  // rows of q_out (its tensor map)
    __nv_bfloat16 *o_base;
    float *lse_base;
    __nv_bfloat16 *o_out;
    float *o_out_f32;  // when set, output rows are written here as float instead of o_out
    float *lse_out;
    uint32_t *status;
    int *unit_counter;  // zero before the launch: the next work unit to take (persistent CTAs)
    // Second launch (rows whose staged query left the fp16 range): row blocks
    // are numbered base blocks first (B * Hq * base_nblk), then the output-row
    // blocks of the sequences whose output rows take this kernel
    // (out_blk_indptr[b] of them before sequence b, device [B+1]); n_blocks in
    // all. redo_bits: bitmap of n_blocks bits, zero before the first launch;
    // redo_list: B * Hq * Tq + n_out * Hq ints of scratch.
    const int32_t *out_blk_indptr;
    int n_blocks;
    uint32_t *redo_bits;
    int *redo_list;
};
// Work units of one (sequence, kv head) for nblk row blocks and group size g.
int tc_units_per_kv(int nblk, int g);
cudaError_t launch_prefill_tc(const TcParams &p, const void *k16, const void *v, int d, cudaStream_t stream);

// splitkv.cu: split-KV attention for few rows over long key ranges + combine.
// kSplitDecodeSplit: a decoding step whose GQA group is too large for one
// 16-row group (8 < g <= 16): group 2 * (b * Hkv + kv) + 0 holds the base rows
// of (sequence b, kv head kv), + 1 its output rows (TMA kernel only).
enum SplitMode { kSplitPrefill = 0, kSplitDecode = 1, kSplitExtend = 2, kSplitDecodeSplit = 3 };
struct SplitParams {
    int mode;
    const __nv_bfloat16 *q, *q_out;  // prefill [B,T,Hq,d] / [n_out,Hq,d]; decode [B,Hq,d] each
    const __nv_bfloat16 *k, *v;      // prefill [B,T,Hkv,d]; decode caches [num_pages,P,Hkv,d]
    const float *alpha_base, *beta_base, *alpha_out, *beta_out;
    const int32_t *out_positions;    // prefill
    const int32_t *group_info;       // prefill: 3 ints per group (b<<16 | kv, first row, positions)
    const int32_t *ext_info;         // extend: 4 ints per group (b<<16 | kv, first new-token row,
                                     // first output row, n_base | n_out << 16): positions of the group are
                                     // its n_base new tokens' base rows, then its n_out output rows
    const int32_t *block_table, *cache_lens;  // decode / extend
    const int32_t *new_indptr;                // extend: device [B+1]
    int n_new;                                // extend: rows of q / k_new / v_new
    int group_offset;                         // first group of this launch (the partial buffer is shared)
    int max_pages, page_size, num_pages;
    int B, T, Hq, Hkv, window;
    int Tq, q_off;       // prefill: query rows per sequence; query i sits at key position q_off + i
    int shard, key_lo;   // prefill: output rows are partials over keys key_lo .. min(t, T - 1)
    float scale, scale_log2;
    int n_groups, chunk, max_chunks;
    long long kv_tokens;  // token rows behind k / v: prefill B*T, decode num_pages*page_size
    float *partial;  // [n_groups, max_chunks, 16, d + 2]
    __nv_bfloat16 *o_base;
    float *lse_base;
    __nv_bfloat16 *o_out;
    float *o_out_f32;  // prefill: when set, output rows are written here as float instead of o_out
    float *lse_out;
    uint32_t *status;
};
// Position index pidx of an extend-mode group (b, L = cache_lens[b]): sets
// kind (0 base row of a new token, 1 output row) and idx (new-token row or
// output row) and returns the position, or -1 when the data make the row
// impossible (length past the block table, output position outside the
// sequence, or a history position without q_out).
__device__ __forceinline__ int extend_position(const SplitParams &p, int group, int b, int L, int pidx, int &kind,
                                               int &idx) {
    const int *e = p.ext_info + 4 * group;
    const int n_base = e[3] & 0xffff;
    const int len = L + (p.new_indptr[b + 1] - p.new_indptr[b]);
    kind = pidx < n_base ? 0 : 1;
    idx = kind == 0 ? e[1] + pidx : e[2] + (pidx - n_base);
    if (L < 0 || (long long)len > (long long)p.max_pages * p.page_size) return -1;
    if (kind == 0) return L + (idx - p.new_indptr[b]);
    const int t = p.out_positions[idx];
    if (t < 0 || t >= len || (!p.q_out && t < L)) return -1;
    return t;
}
// Prefill mode: the last key of an output row at position t (a shard's rows
// past its keys read them all), or -1 when the position is impossible (before
// 0; past the keys outside a shard; without q_out, outside the query rows).
__device__ __forceinline__ int prefill_row_end(const SplitParams &p, int t) {
    if (t < 0 || (!p.shard && t >= p.T)) return -1;
    const int te = min(t, p.T - 1);
    if (!p.q_out && (te < p.q_off || te - p.q_off >= p.Tq)) return -1;
    return te;
}
size_t split_partial_bytes(int n_groups, int max_chunks, int d);
// Runs the split kernel (the TMA-fed persistent one when eligible) and the combine.
cudaError_t launch_splitkv(const SplitParams &p, int d, int rows_per_group, cudaStream_t stream);
// Extend mode: groups [0, n_small) have at most 8 rows, the rest at most 16;
// one TMA launch for each class, then the combine over all p.n_groups groups.
cudaError_t launch_splitkv_extend(const SplitParams &p, int d, int n_small, cudaStream_t stream);
// splitkv_tma.cu
bool splitkv_tma_eligible(const SplitParams &p);
cudaError_t launch_splitkv_tma(const SplitParams &p, int d, int rows_per_group, cudaStream_t stream);
// prefill_tc.cu: 3-D tensor map (d, Hkv, tokens) over bf16 [tokens, Hkv, d] rows,
// box (64 channels, 1 head, box_tokens), 128-byte swizzle, zero fill.
bool encode_kv_map_3d(CUtensorMap *m, const void *base, long long tokens, int Hkv, int d, int box_tokens);

// simt_rows.cu: one warp per (row, head); any element type; the fp32 path.
cudaError_t launch_rows_simt(const RowsArgs &a, RowKind kind, int d, orthros_dtype dtype,
                             cudaStream_t stream);

// backward_simt.cu: gradients of the base and output rows (any element type).
struct BwdArgs {
    const void *q, *q_out, *k, *v;  // forward inputs, layouts as in orthros_prefill
    const float *alpha_base, *beta_base, *alpha_out, *beta_out;
    const int32_t *out_indptr;     // device [B+1]
    const int32_t *out_positions;  // [n_out]
    int32_t *pos_head;             // [B*T]: first output row at (b, t), or -1 (set to -1 by the caller)
    int32_t *row_next;             // [n_out]: next output row at the same position, or -1
    int n_out, B, T, Hq, Hkv, window;
    float scale;
    const void *o_base, *o_out, *do_base, *do_out;  // forward outputs and their gradients
    const float *lse_base, *lse_out;
    float *delta_base;  // [B,Hq,T]  dO . o of every base row
    float *delta_out;   // [n_out,Hq]
    float *dq_rows;     // [n_out,Hq,d] fp32 dq of output rows that read q (q_out == nullptr);
                        // the tensor-core path first accumulates the rows' dqa here
    void *dq, *dk, *dv, *dq_out;
    float *d_alpha_base, *d_beta_base, *d_alpha_out, *d_beta_out;  // zeroed by the caller
    uint32_t *status;
    // tensor-core path only (bf16); nullptr otherwise
    __nv_bfloat16 *qa_base;  // [B,T,Hq,d] affined base queries
    __nv_bfloat16 *qa_out;   // [n_out,Hq,d] affined output-row queries
    float *dq_acc;           // [B,T,Hq,d] fp32 dqa of base rows
    int32_t *omax;           // [n_out]: largest position among rows r .. r+63 of r's sequence
};
// Runs the whole backward; use_tc selects the tensor-core kernel (bf16, d = 64 or 128,
// with the workspace regions above) for the dk/dv/dqa products.
cudaError_t launch_backward(const BwdArgs &a, int d, orthros_dtype dtype, bool use_tc, cudaStream_t stream);

// backward_tc.cu
struct BwdTcParams {
    const int32_t *out_indptr, *out_positions, *omax;
    const float *lse_base, *lse_out, *delta_base, *delta_out;
    float *dq_acc, *dq_out_acc;
    __nv_bfloat16 *dk, *dv;
    int B, T, Hq, Hkv, window, n_out, nkb;
    float scale, scale_log2;
    uint32_t *status;
};
cudaError_t launch_backward_tc(const BwdTcParams &p, int d, const void *k, const void *v, const void *qa_base,
                               const void *do_base, const void *qa_out, const void *do_out, cudaStream_t stream);

// project_tc.cu: shared Q/K/V projection (bf16) with the query affines and
// the cache writes in the epilogue.
struct ProjParams {
    const __nv_bfloat16 *x;    // [n_base + n_out, d_model]
    const __nv_bfloat16 *w_t;  // [(Hq + 2 Hkv) d, d_model]
    int n_base, n_out, d_model, Hq, Hkv, d;
    const float *alpha_base, *beta_base, *alpha_out, *beta_out;
    __nv_bfloat16 *q_base, *q_out, *k_out, *v_out;  // k_out / v_out may be null
    __nv_bfloat16 *k_cache, *v_cache;               // null: no cache writes
    const int32_t *block_table, *token_seq, *token_pos;
    int B, max_pages, page_size, num_pages;
    uint32_t *status;
};
cudaError_t launch_project_tc(const ProjParams &p, cudaStream_t stream);

// merge.cu: exact merge of normalised partials over disjoint key sets.
cudaError_t launch_merge_partials(const float *o_parts, const float *lse_parts, int n_parts, int n_rows, int Hq, int d,
                                  bool f32_out, void *o_out, float *lse_out, cudaStream_t stream);

// cache.cu
// Writes new token i of sequence b (rows new_indptr[b] ..) at position
// cache_lens[b] + (i - new_indptr[b]) of its pages.
cudaError_t launch_extend_append(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                                 const int32_t *block_table, const int32_t *cache_lens, const int32_t *new_indptr,
                                 int B, int n_new, int Hkv, int d, int max_pages, int page_size, int num_pages,
                                 int elem_bytes, uint32_t *status, cudaStream_t stream);
cudaError_t launch_decode_append(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                                 const int32_t *block_table, const int32_t *cache_lens, int B, int Hkv,
                                 int d, int max_pages, int page_size, int num_pages, int elem_bytes,
                                 uint32_t *status, cudaStream_t stream);
// fp16 copy of the keys for the tensor-core prefill, optionally fused with the
// paged cache fill (k_cache == nullptr skips it); records the largest |k| in
// *kmax_bits (atomic max of the float bits; zeroed by the caller).
cudaError_t launch_prefill_prep(const void *k, const void *v, void *k16, void *k_cache, void *v_cache,
                                const int32_t *block_table, int B, int T, int Hkv, int d, int max_pages,
                                int page_size, int num_pages, uint32_t *status, unsigned *kmax_bits,
                                uint32_t *zero_words, int n_zero, cudaStream_t stream);
// The four query affines (alpha_base, beta_base, alpha_out, beta_out; a null
// pointer gives zeros), each of n_aff floats, as consecutive scaled copies in
// aff.
struct AffineSet {
    const float *p[4];
};
// s = 0 unless the largest |k| (*kmax_bits) exceeds the fp16 range; then the
// fp16 keys are rewritten as k * 2^-s. The affines are copied to aff scaled by
// 2^s, so that queries staged with them meet the keys at unchanged logits.
cudaError_t launch_prefill_key_rescale(const void *k, void *k16, int B, int T, int Hkv, int d,
                                       const unsigned *kmax_bits, AffineSet src, float *aff, int n_aff,
                                       cudaStream_t stream);
cudaError_t launch_prefill_cache_fill(const void *k, const void *v, void *k_cache, void *v_cache,
                                      const int32_t *block_table, int B, int T, int Hkv, int d,
                                      int max_pages, int page_size, int num_pages, int elem_bytes,
                                      uint32_t *status, cudaStream_t stream);
// cache.cu: chunked prefill helpers (output-row positions per chunk, status fold).
cudaError_t launch_shift_positions(const int32_t *src, int32_t *dst, int n, int off, cudaStream_t stream);
cudaError_t launch_fold_status(uint32_t *dst, const uint32_t *src, int n, int stride_words, cudaStream_t stream);

}  // namespace orthros
