// orthros_api.cu -- the C ABI: argument checks, workspace carving, dispatch.
//
// Every entry point validates everything the host can see before the first
// launch, then enqueues its kernels on the caller's stream and returns. See
// include/orthros_attn.h for the contract of each call.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>
#include <vector>

#include "internal.cuh"

namespace orthros {
namespace {

thread_local std::string g_last_error;

orthros_status fail(orthros_status s, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

orthros_status cuda_fail(cudaError_t e, const char *what) {
    return fail(ORTHROS_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elem_bytes(orthros_dtype t) { return t == ORTHROS_F32 ? 4 : 2; }

// Split-KV work items cover `chunk` keys of one row group: the longest of
// 8192 .. 512 keys (multiples of the kernels' 128-key stages) that still gives
// every SM three items. Long items amortise each item's query load and state
// merge; short ones keep small batches spread over the GPU.
constexpr int kChunkMax = 8192;
constexpr int kChunkMin = 512;

int device_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
        n > 0)
        return n;
    return 152;
}

int split_chunk(long long n_groups, long long keys) {
    const long long want = 3LL * device_sms();
    for (int c = kChunkMax; c > kChunkMin; c /= 2)
        if (n_groups * ((keys + c - 1) / c) >= want) return c;
    return kChunkMin;
}

// Partial slots (group x chunk) that a launch with at most max_groups groups
// can use: with the largest chunk, n * ceil(keys / 8192); otherwise the chosen
// chunk c was taken because 2c gave fewer than 3 items per SM, so
// n * ceil(keys / c) <= 2 n * ceil(keys / 2c) < 6 items per SM.
long long split_slots_bound(long long max_groups, long long keys) {
    const long long lo = max_groups * ((keys + kChunkMax - 1) / kChunkMax);
    const long long hi = max_groups * ((keys + kChunkMin - 1) / kChunkMin);
    return std::min(hi, std::max(lo, 6LL * device_sms()));
}
// A sequence's output rows take the split-KV kernel when all of its rows fit
// in at most this many 16-row groups per kv head; otherwise the tile kernel.
constexpr int kSplitRowsMax = 256;

int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

// Workspace regions of orthros_prefill.
struct PrefillLayout {
    size_t blob_off, k16_off, part_off, redo_bits_off, redo_list_off, aff_off, total;
    int max_groups;
    long long part_slots;
    int redo_cap;  // row blocks of the tile kernel a call can have (bound)
};

PrefillLayout prefill_layout(int B, int T, int Hq, int Hkv, int d, int n_out, orthros_dtype dtype) {
    PrefillLayout L{};
    size_t at = kStatusBytes;
    L.max_groups = dtype == ORTHROS_BF16 ? (int)std::min<long long>((long long)n_out, 16LL * B) * Hkv : 0;
    L.part_slots = split_slots_bound(L.max_groups, T);
    L.blob_off = at;
    at += align_up(sizeof(int32_t) * (size_t)(3 * (B + 1) + 3 * (size_t)L.max_groups), 256);
    L.k16_off = at;
    if (dtype == ORTHROS_BF16) at += align_up((size_t)B * T * Hkv * d * 2, 256);
    L.part_off = at;
    at += align_up((size_t)L.part_slots * split_partial_bytes(1, 1, d), 256);
    // the tile kernel's second launch: a bitmap over its row blocks (at most
    // B * Hq * ceil(T / 128) base blocks and Hq * (ceil(n_out / 128) + B)
    // output-row blocks, bounded generously below) and a list with one entry
    // per log-sum-exp it scans
    L.redo_bits_off = at;
    L.redo_list_off = at;
    if (dtype == ORTHROS_BF16) {
        const long long cap =
            (long long)Hq * ((long long)B * (ceil_div(T, 128) + 1) + ceil_div(n_out, 128) + 2LL * B);
        L.redo_cap = (int)std::min<long long>(cap, 1LL << 30);
        at += align_up(sizeof(uint32_t) * (size_t)((L.redo_cap + 31) / 32), 256);
        L.redo_list_off = at;
        at += align_up(sizeof(int32_t) * ((size_t)B * Hq * T + (size_t)n_out * Hq), 256);
    }
    // the tile kernel's copies of the four query affines (scaled with the keys)
    L.aff_off = at;
    if (dtype == ORTHROS_BF16) at += align_up(sizeof(float) * 4 * (size_t)Hq * d, 256);
    L.total = at;
    return L;
}

struct DecodeLayout {
    size_t part_off, total;
    int chunk, max_chunks;
};

// Row groups of a decoding step on the split-KV path: one per (sequence, kv
// head) when its g base and g output rows fit 16 rows, else two (base rows,
// output rows) for groups of up to 16 query heads on 64-token-multiple pages.
int decode_groups(int B, int Hq, int Hkv, int page_size) {
    const int g = Hq / Hkv;
    if (2 * g <= 16) return B * Hkv;
    if (g <= 16 && page_size % 64 == 0) return 2 * B * Hkv;
    return 0;  // CUDA-core rows
}

DecodeLayout decode_layout(int B, int Hq, int Hkv, int d, int max_pages, int page_size, orthros_dtype dtype) {
    DecodeLayout L{};
    size_t at = kStatusBytes;
    L.part_off = at;
    const int groups = decode_groups(B, Hq, Hkv, page_size);
    L.chunk = split_chunk(groups > 0 ? groups : 1, (long long)max_pages * page_size);
    L.max_chunks = ceil_div((long long)max_pages * page_size, L.chunk);
    if (dtype == ORTHROS_BF16 && groups > 0) at += align_up(split_partial_bytes(groups, L.max_chunks, d), 256);
    L.total = at;
    return L;
}

// Workspace regions of orthros_prefill_backward.
struct BackwardLayout {
    size_t indptr_off, head_off, next_off, delta_base_off, delta_out_off, dq_rows_off;
    size_t qa_base_off, qa_out_off, dq_acc_off, omax_off, total;
};

// The tensor-core backward (bf16, d = 128) also needs bf16 affined queries,
// an fp32 dqa accumulator for the base rows and the output tiles' largest positions.
BackwardLayout backward_layout(int B, int T, int Hq, int d, int n_out, orthros_dtype dtype) {
    BackwardLayout L{};
    size_t at = kStatusBytes;
    L.indptr_off = at;
    at += align_up(sizeof(int32_t) * (size_t)(B + 1), 256);
    L.head_off = at;
    at += align_up(sizeof(int32_t) * (size_t)B * T, 256);
    L.next_off = at;
    at += align_up(sizeof(int32_t) * (size_t)n_out, 256);
    L.delta_base_off = at;
    at += align_up(sizeof(float) * (size_t)B * Hq * T, 256);
    L.delta_out_off = at;
    at += align_up(sizeof(float) * (size_t)n_out * Hq, 256);
    L.dq_rows_off = at;
    at += align_up(sizeof(float) * (size_t)n_out * Hq * d, 256);
    const bool tc = dtype == ORTHROS_BF16;
    L.qa_base_off = at;
    if (tc) at += align_up((size_t)2 * B * T * Hq * d, 256);
    L.qa_out_off = at;
    if (tc) at += align_up((size_t)2 * n_out * Hq * d, 256);
    L.dq_acc_off = at;
    if (tc) at += align_up(sizeof(float) * (size_t)B * T * Hq * d, 256);
    L.omax_off = at;
    if (tc) at += align_up(sizeof(int32_t) * (size_t)n_out, 256);
    L.total = at;
    return L;
}

// Workspace regions of orthros_extend.
struct ExtendLayout {
    size_t blob_off, part_off, total;
    int max_groups;
    long long part_slots;
};

ExtendLayout extend_layout(int B, int n_new, int n_out, int Hq, int Hkv, int d, int max_pages, int page_size,
                           orthros_dtype dtype) {
    ExtendLayout L{};
    (void)Hq;
    size_t at = kStatusBytes;
    // at most one group per position of each (sequence, kv head), plus one partial group per class
    const long long groups = ((long long)n_new + n_out + 2LL * B) * Hkv;
    L.max_groups = dtype == ORTHROS_BF16 ? (int)std::min<long long>(groups, 1LL << 30) : 0;
    L.part_slots = split_slots_bound(L.max_groups, (long long)max_pages * page_size);
    L.blob_off = at;
    at += align_up(sizeof(int32_t) * (size_t)(2 * (B + 1) + 4 * (size_t)L.max_groups), 256);
    L.part_off = at;
    at += align_up((size_t)L.part_slots * split_partial_bytes(1, 1, d), 256);
    L.total = at;
    return L;
}

orthros_status check_shapes(int B, int Hq, int Hkv, int d, int window, float scale, orthros_dtype dtype) {
    if (B < 0) return fail(ORTHROS_EINVAL, "B = %d must be >= 0", B);
    if (Hq < 1 || Hkv < 1) return fail(ORTHROS_EINVAL, "head counts Hq = %d, Hkv = %d must be >= 1", Hq, Hkv);
    if (Hq % Hkv != 0) return fail(ORTHROS_EINVAL, "Hq = %d is not a multiple of Hkv = %d", Hq, Hkv);
    if (window < 1) return fail(ORTHROS_EINVAL, "window = %d must be >= 1", window);
    if (!std::isfinite(scale)) return fail(ORTHROS_EINVAL, "scale must be finite");
    if (dtype != ORTHROS_BF16 && dtype != ORTHROS_F32) return fail(ORTHROS_EINVAL, "unknown dtype %d", (int)dtype);
    if (d != 64 && d != 128) return fail(ORTHROS_EUNSUPPORTED, "head size d = %d (supported: 64, 128)", d);
    return ORTHROS_OK;
}

// orthros_prefill (Tq == T, whole sequences) and orthros_prefill_shard (Tq <=
// T: the queries are the last Tq key positions; with `shard` the output rows
// are float partials over the last Tq keys) share this body. T counts keys.
orthros_status prefill_core(const void *q, const void *k, const void *v, const float *alpha_base,
                            const float *beta_base, const float *alpha_out, const float *beta_out,
                            const int32_t *out_indptr, const int32_t *out_positions, int n_out,
                            const void *q_out, int B, int T, int Tq, bool shard, int Hq, int Hkv, int d,
                            int window, float scale, orthros_dtype dtype, void *o_base, float *lse_base,
                            void *o_out, float *o_out_f32, float *lse_out, void *k_cache, void *v_cache,
                            const int32_t *block_table, int max_pages, int page_size, int num_pages,
                            void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    orthros_status st = check_shapes(B, Hq, Hkv, d, window, scale, dtype);
    if (st != ORTHROS_OK) return st;
    if (T < 0) return fail(ORTHROS_EINVAL, "T = %d must be >= 0", T);
    if (Tq < 0 || Tq > T) return fail(ORTHROS_EINVAL, "Tq = %d must lie in [0, T = %d]", Tq, T);
    if (n_out < 0) return fail(ORTHROS_EINVAL, "n_out = %d must be >= 0", n_out);
    const long long rows = (long long)B * T;
    if (rows > (1LL << 31)) return fail(ORTHROS_EUNSUPPORTED, "B*T = %lld tokens exceeds 2^31", rows);
    if (shard && dtype != ORTHROS_BF16) return fail(ORTHROS_EUNSUPPORTED, "shards take bf16 only");
    if (shard && n_out > 0 && !q_out) return fail(ORTHROS_EINVAL, "a shard's output rows need q_out");
    if ((long long)B * Tq > 0) {
        if (!q || !k || !v) return fail(ORTHROS_EINVAL, "q, k and v must not be NULL");
        if (!alpha_base || !beta_base) return fail(ORTHROS_EINVAL, "alpha_base and beta_base must not be NULL");
        if (!o_base || !lse_base) return fail(ORTHROS_EINVAL, "o_base and lse_base must not be NULL");
        if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o_base))
            return fail(ORTHROS_EINVAL, "q, k, v and o_base must be 16-byte aligned");
        if (!aligned16(alpha_base) || !aligned16(beta_base))
            return fail(ORTHROS_EINVAL, "alpha_base and beta_base must be 16-byte aligned");
    }
    if (B > 0 && !out_indptr) return fail(ORTHROS_EINVAL, "out_indptr (host) must not be NULL");
    if (B > 0) {
        if (out_indptr[0] != 0) return fail(ORTHROS_EINVAL, "out_indptr[0] = %d must be 0", out_indptr[0]);
        for (int b = 0; b < B; ++b)
            if (out_indptr[b + 1] < out_indptr[b])
                return fail(ORTHROS_EINVAL, "out_indptr decreases at %d", b);
        if (out_indptr[B] != n_out)
            return fail(ORTHROS_EINVAL, "out_indptr[B] = %d differs from n_out = %d", out_indptr[B], n_out);
    } else if (n_out != 0) {
        return fail(ORTHROS_EINVAL, "n_out = %d with B = 0", n_out);
    }
    if (n_out > 0) {
        if (T == 0) return fail(ORTHROS_EINVAL, "output rows with T = 0");
        if (!out_positions) return fail(ORTHROS_EINVAL, "out_positions must not be NULL when n_out > 0");
        if (!alpha_out || !beta_out) return fail(ORTHROS_EINVAL, "alpha_out and beta_out must not be NULL when n_out > 0");
        if (!(shard ? (void *)o_out_f32 : o_out) || !lse_out)
            return fail(ORTHROS_EINVAL, "o_out and lse_out must not be NULL when n_out > 0");
        if (!aligned16(shard ? (void *)o_out_f32 : o_out) || (q_out && !aligned16(q_out)) || !aligned16(alpha_out) ||
            !aligned16(beta_out))
            return fail(ORTHROS_EINVAL, "o_out, q_out, alpha_out and beta_out must be 16-byte aligned");
    }
    const bool fill = k_cache || v_cache || block_table;
    if (fill) {
        if (!k_cache || !v_cache || !block_table)
            return fail(ORTHROS_EINVAL, "k_cache, v_cache and block_table must be all NULL or all set");
        if (page_size < 1 || max_pages < 1 || num_pages < 1)
            return fail(ORTHROS_EINVAL, "page_size, max_pages, num_pages must be >= 1 for the cache fill");
        if ((long long)max_pages * page_size < T)
            return fail(ORTHROS_EINVAL, "max_pages * page_size = %lld < T = %d",
                        (long long)max_pages * page_size, T);
        if (!aligned16(k_cache) || !aligned16(v_cache))
            return fail(ORTHROS_EINVAL, "k_cache and v_cache must be 16-byte aligned");
    }
    const PrefillLayout lay = prefill_layout(B, T, Hq, Hkv, d, n_out, dtype);
    if (!workspace || workspace_bytes < lay.total)
        return fail(ORTHROS_EWORKSPACE, "workspace needs %zu bytes, got %zu", lay.total,
                    workspace ? workspace_bytes : (size_t)0);
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(ORTHROS_EINVAL, "workspace must be 256-byte aligned");

    char *ws = static_cast<char *>(workspace);
    uint32_t *status = reinterpret_cast<uint32_t *>(ws);
    // the status word and, next to it, the tile kernel's work-unit counter, a
    // spare word and the keys' largest magnitude
    cudaError_t e = cudaMemsetAsync(status, 0, 4 * sizeof(uint32_t), stream);
    if (e != cudaSuccess) return cuda_fail(e, "status reset");
    if (rows == 0) return ORTHROS_OK;

    const int g = Hq / Hkv;
    const bool tc = dtype == ORTHROS_BF16;

    // Plan (host): which sequences' output rows take the split-KV kernel, the
    // tile kernel's output-row units, and the split groups. One upload.
    // blob: out_indptr, cross_unit_indptr, out_blk_indptr (B + 1 each), split groups
    std::vector<int32_t> blob((size_t)3 * (B + 1), 0);
    int n_cross_units = 0, n_groups = 0, rows_per_group = 0, n_out_blocks = 0;
    bool any_simt_out = false;
    std::copy(out_indptr, out_indptr + B + 1, blob.begin());
    for (int b = 0; b < B; ++b) {
        const int nb = out_indptr[b + 1] - out_indptr[b];
        blob[(size_t)B + 1 + b] = n_cross_units;
        blob[(size_t)2 * (B + 1) + b] = n_out_blocks;
        if (nb == 0) continue;
        if (!tc) {
            any_simt_out = true;
        } else if (g <= 16 && (long long)nb * g <= kSplitRowsMax) {
            const int per = 16 / g;  // positions per 16-row group
            for (int kvh = 0; kvh < Hkv; ++kvh)
                for (int r0 = 0; r0 < nb; r0 += per) {
                    const int cnt = std::min(per, nb - r0);
                    blob.push_back((b << 16) | kvh);
                    blob.push_back(out_indptr[b] + r0);
                    blob.push_back(cnt);
                    rows_per_group = std::max(rows_per_group, cnt * g);
                    ++n_groups;
                }
        } else {
            n_cross_units += Hkv * tc_units_per_kv(ceil_div(nb, 128), g);
            n_out_blocks += Hq * ceil_div(nb, 128);
        }
    }
    blob[(size_t)2 * B + 1] = n_cross_units;
    blob[(size_t)3 * B + 2] = n_out_blocks;
    if (n_groups > lay.max_groups) return fail(ORTHROS_EWORKSPACE, "internal: split groups exceed the workspace plan");
    int32_t *blob_dev = reinterpret_cast<int32_t *>(ws + lay.blob_off);
    const int32_t *indptr_dev = blob_dev;
    const int32_t *cross_indptr_dev = blob_dev + B + 1;
    const int32_t *out_blk_dev = blob_dev + 2 * (B + 1);
    const int32_t *groups_dev = blob_dev + 3 * (B + 1);
    if (n_out > 0) {
        e = cudaMemcpyAsync(blob_dev, blob.data(), sizeof(int32_t) * blob.size(), cudaMemcpyHostToDevice, stream);
        if (e != cudaSuccess) return cuda_fail(e, "plan upload");
    }

    if (!tc) {
        if (fill) {
            ProfScope ps("cache_fill", stream);
            e = launch_prefill_cache_fill(k, v, k_cache, v_cache, block_table, B, T, Hkv, d, max_pages, page_size,
                                          num_pages, elem_bytes(dtype), status, stream);
            if (e != cudaSuccess) return cuda_fail(e, "cache fill launch");
        }
        RowsArgs a{};
        a.q = q;
        a.q_out = q_out;
        a.k = k;
        a.v = v;
        a.alpha_base = alpha_base;
        a.beta_base = beta_base;
        a.alpha_out = alpha_out;
        a.beta_out = beta_out;
        a.out_indptr = indptr_dev;
        a.out_positions = out_positions;
        a.n_out = n_out;
        a.B = B;
        a.T = T;
        a.Hq = Hq;
        a.Hkv = Hkv;
        a.window = window;
        a.scale = scale;
        a.o_base = o_base;
        a.lse_base = lse_base;
        a.o_out = o_out;
        a.lse_out = lse_out;
        a.status = status;
        {
            ProfScope ps("rows_simt_base", stream);
            e = launch_rows_simt(a, kPrefillBase, d, dtype, stream);
        }
        if (e != cudaSuccess) return cuda_fail(e, "base-stream launch");
        if (any_simt_out) {
            ProfScope ps("rows_simt_out", stream);
            e = launch_rows_simt(a, kPrefillOut, d, dtype, stream);
            if (e != cudaSuccess) return cuda_fail(e, "output-stream launch");
        }
        return ORTHROS_OK;
    }

    // bf16: fp16 keys (+ cache fill) -> split-KV output rows -> tensor-core tiles
    void *k16 = ws + lay.k16_off;
    {
        ProfScope ps("prefill_prep", stream);
        e = launch_prefill_prep(k, v, k16, fill ? k_cache : nullptr, fill ? v_cache : nullptr, block_table, B, T, Hkv,
                                d, max_pages, page_size, num_pages, status, reinterpret_cast<unsigned *>(ws) + 3,
                                reinterpret_cast<uint32_t *>(ws + lay.redo_bits_off), (lay.redo_cap + 31) / 32,
                                stream);
    }
    if (e != cudaSuccess) return cuda_fail(e, "prep launch");
    {
        ProfScope ps("prefill_key_rescale", stream);
        const AffineSet src{{alpha_base, beta_base, alpha_out, beta_out}};
        e = launch_prefill_key_rescale(k, k16, B, T, Hkv, d, reinterpret_cast<const unsigned *>(ws) + 3, src,
                                       reinterpret_cast<float *>(ws + lay.aff_off), Hq * d, stream);
    }
    if (e != cudaSuccess) return cuda_fail(e, "key rescale launch");
    const float log2e = 1.4426950408889634f;
    if (n_groups > 0) {
        SplitParams sp{};
        sp.mode = kSplitPrefill;
        sp.q = static_cast<const __nv_bfloat16 *>(q);
        sp.q_out = static_cast<const __nv_bfloat16 *>(q_out);
        sp.k = static_cast<const __nv_bfloat16 *>(k);
        sp.v = static_cast<const __nv_bfloat16 *>(v);
        sp.alpha_base = alpha_base;
        sp.beta_base = beta_base;
        sp.alpha_out = alpha_out;
        sp.beta_out = beta_out;
        sp.out_positions = out_positions;
        sp.group_info = groups_dev;
        sp.B = B;
        sp.T = T;
        sp.Tq = Tq;
        sp.q_off = T - Tq;
        sp.shard = shard;
        sp.key_lo = shard ? T - Tq : 0;
        sp.Hq = Hq;
        sp.Hkv = Hkv;
        sp.window = window;
        sp.scale = scale;
        sp.scale_log2 = scale * log2e;
        sp.n_groups = n_groups;
        sp.chunk = split_chunk(n_groups, T);
        sp.max_chunks = ceil_div(T, sp.chunk);
        if ((long long)n_groups * sp.max_chunks > lay.part_slots)
            return fail(ORTHROS_EWORKSPACE, "internal: split partials exceed the workspace plan");
        sp.kv_tokens = (long long)B * T;
        sp.partial = reinterpret_cast<float *>(ws + lay.part_off);
        sp.o_out = static_cast<__nv_bfloat16 *>(o_out);
        sp.o_out_f32 = shard ? o_out_f32 : nullptr;
        sp.lse_out = lse_out;
        sp.status = status;
        ProfScope ps("splitkv_prefill", stream);
        e = launch_splitkv(sp, d, rows_per_group, stream);
        if (e != cudaSuccess) return cuda_fail(e, "split-KV launch");
    }
    TcParams tp{};
    tp.q = static_cast<const __nv_bfloat16 *>(q);
    tp.q_out = static_cast<const __nv_bfloat16 *>(q_out);
    {
        // the affines scaled with the keys (copies written by the rescale pass)
        const float *aff = reinterpret_cast<const float *>(ws + lay.aff_off);
        const size_t n_aff = (size_t)Hq * d;
        tp.alpha_base = aff;
        tp.beta_base = aff + n_aff;
        tp.alpha_out = aff + 2 * n_aff;
        tp.beta_out = aff + 3 * n_aff;
    }
    tp.out_indptr = indptr_dev;
    tp.out_positions = out_positions;
    tp.cross_unit_indptr = cross_indptr_dev;
    tp.B = B;
    tp.T = T;
    tp.Tq = Tq;
    tp.q_off = T - Tq;
    tp.shard = shard;
    tp.key_lo = shard ? T - Tq : 0;
    tp.Hq = Hq;
    tp.Hkv = Hkv;
    tp.window = window;
    tp.scale = scale;
    tp.scale_log2 = scale * log2e;
    tp.base_nblk = ceil_div(Tq, 128);
    tp.n_cross_units = n_cross_units;
    tp.n_out = n_out;
    tp.n_base_units = B * Hkv * tc_units_per_kv(tp.base_nblk, g);
    tp.o_base = static_cast<__nv_bfloat16 *>(o_base);
    tp.lse_base = lse_base;
    tp.o_out = static_cast<__nv_bfloat16 *>(o_out);
    tp.o_out_f32 = shard ? o_out_f32 : nullptr;
    tp.lse_out = lse_out;
    tp.status = status;
    tp.unit_counter = reinterpret_cast<int *>(ws + sizeof(uint32_t));
    tp.out_blk_indptr = out_blk_dev;
    tp.n_blocks = B * Hq * tp.base_nblk + n_out_blocks;
    tp.redo_bits = reinterpret_cast<uint32_t *>(ws + lay.redo_bits_off);
    tp.redo_list = reinterpret_cast<int *>(ws + lay.redo_list_off);
    if (tp.n_blocks > lay.redo_cap) return fail(ORTHROS_EWORKSPACE, "internal: row blocks exceed the workspace plan");
    {
        ProfScope ps("prefill_tc", stream);
        e = launch_prefill_tc(tp, k16, v, d, stream);
    }
    if (e != cudaSuccess) return cuda_fail(e, "tensor-core prefill launch");
    return ORTHROS_OK;
}


// ---------------------------------------------------------------------------
// orthros_prefill_from_host: the prefill with its inputs and outputs in host
// memory. Sequences longer than one chunk are cut into chunks of the token
// axis that run as shards (base rows exact with a halo of keys; output rows as
// partials merged at the end), so that the host-to-device copy of chunk c + 1,
// the compute of chunk c and the device-to-host copy of chunk c - 1 overlap on
// three streams.
// ---------------------------------------------------------------------------
constexpr int kHostChunkMin = 16384;
constexpr size_t kSlotBytes = 256;  // one shard call's status words

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Rows per chunk: at least 16384 and at least four halos, so that the halo
// keys each chunk converts again stay a small share of its work.
int host_chunk_rows(int T, int window) {
    const long long halo = std::max(window - 1, 1);
    const long long c = std::max<long long>(kHostChunkMin, 4 * ((halo + 127) / 128) * 128);
    return (int)std::min<long long>(c, std::max(T, 1));
}

// Chunk boundaries of a sequence of T tokens: a quarter chunk first (the
// compute starts after a short copy in), full chunks, and the remainder ending
// in a quarter chunk (a short copy out after the last compute).
std::vector<int> chunk_starts(int T, int chunk) {
    std::vector<int> st;
    if (T <= chunk) {
        st.push_back(0);
    } else {
        const int quarter = std::max(128, (chunk / 4) & ~127);
        int t = 0;
        st.push_back(t);
        t += quarter;
        while (T - t > chunk + quarter) {
            st.push_back(t);
            t += chunk;
        }
        if (T - t > quarter) {
            st.push_back(t);
            t = T - quarter;
        }
        st.push_back(t);
    }
    st.push_back(T);
    return st;  // chunk c covers [st[c], st[c + 1])
}

struct FromHostLayout {
    bool pipelined;
    std::vector<int> starts;
    int chunk, n_chunks, halo_max, max_rows;
    size_t q_off, k_off, v_off, o_off, lse_off, qrows_off, pos_off, pos_chunk_off, parts_off, lparts_off, oout_off,
        lout_off, core_off, core_bytes, total;
};

FromHostLayout from_host_layout(int B, int T, int Hq, int Hkv, int d, int n_out, int window, orthros_dtype dtype) {
    FromHostLayout L{};
    const size_t eb = elem_bytes(dtype);
    L.chunk = host_chunk_rows(T, window);
    L.starts = chunk_starts(T, L.chunk);
    L.n_chunks = T > 0 ? (int)L.starts.size() - 1 : 0;
    L.pipelined = dtype == ORTHROS_BF16 && L.n_chunks >= 2;
    L.halo_max = std::min(std::max(window - 1, 1), std::max(T, 1));
    L.max_rows = n_out;  // a sequence's output rows, at most
    const size_t bt = (size_t)B * T;
    size_t off;
    if (L.pipelined) {
        L.core_bytes = prefill_layout(1, L.chunk + L.halo_max, Hq, Hkv, d, L.max_rows, dtype).total;
        off = kSlotBytes;  // this call's own status words
        L.core_off = off;  // one status slot per shard call, then the shard workspace
        off = align256(off + (size_t)B * L.n_chunks * kSlotBytes + L.core_bytes);
        L.lse_off = off;  // two chunk-sized lse_base buffers (double-buffered against the copy out)
        off = align256(off + 2 * (size_t)Hq * L.chunk * 4);
        L.qrows_off = off;
        off = align256(off + (size_t)n_out * Hq * d * eb);
        L.pos_chunk_off = off;
        off = align256(off + (size_t)n_out * 4);
        L.parts_off = off;
        off = align256(off + (size_t)L.n_chunks * n_out * Hq * d * 4);
        L.lparts_off = off;
        off = align256(off + (size_t)L.n_chunks * n_out * Hq * 4);
    } else {
        L.core_bytes = prefill_layout(B, T, Hq, Hkv, d, n_out, dtype).total;
        L.core_off = 0;  // its status words are this call's
        off = align256(L.core_bytes);
        L.lse_off = off;
        off = align256(off + (size_t)B * Hq * T * 4);
        L.qrows_off = off;  // q_out, when given
        off = align256(off + (size_t)n_out * Hq * d * eb);
    }
    L.pos_off = off;
    off = align256(off + (size_t)n_out * 4);
    L.oout_off = off;
    off = align256(off + (size_t)n_out * Hq * d * eb);
    L.lout_off = off;
    off = align256(off + (size_t)n_out * Hq * 4);
    L.q_off = off;
    off = align256(off + bt * Hq * d * eb);
    L.k_off = off;
    off = align256(off + bt * Hkv * d * eb);
    L.v_off = off;
    off = align256(off + bt * Hkv * d * eb);
    L.o_off = off;
    off = align256(off + bt * Hq * d * eb);
    L.total = off;
    return L;
}

// Copy streams and events of the pipelined path, created once per device.
struct HostPipe {
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, in_done = nullptr, comp_done = nullptr, out_done[2] = {nullptr, nullptr},
                end = nullptr;
};
constexpr int kPipeDevices = 64;
std::mutex g_pipe_mu;  // held for a whole call's enqueueing: the events are shared
HostPipe g_pipe[kPipeDevices];

cudaError_t host_pipe(HostPipe **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kPipeDevices) return cudaErrorInvalidDevice;
    HostPipe &hp = g_pipe[dev];
    if (!hp.end) {
        if ((e = cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking)) != cudaSuccess) return e;
        if ((e = cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking)) != cudaSuccess) return e;
        for (cudaEvent_t *ev : {&hp.start, &hp.in_done, &hp.comp_done, &hp.out_done[0], &hp.out_done[1], &hp.end})
            if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess) return e;
    }
    *out = &hp;
    return cudaSuccess;
}

// A host argument must not be device memory (page-locked host memory lets the
// copies overlap; pageable memory works, with copies that do not).
bool is_host_memory(const void *p) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return true;  // unknown to CUDA: plain pageable memory
    }
    return at.type == cudaMemoryTypeHost || at.type == cudaMemoryTypeUnregistered;
}

orthros_status from_host_core(const void *q, const void *k, const void *v, const float *alpha_base,
                              const float *beta_base, const float *alpha_out, const float *beta_out,
                              const int32_t *out_indptr, const int32_t *out_positions, int n_out, const void *q_out,
                              int B, int T, int Hq, int Hkv, int d, int window, float scale, orthros_dtype dtype,
                              void *o_base, float *lse_base, void *o_out, float *lse_out, void *k_cache,
                              void *v_cache, const int32_t *block_table, int max_pages, int page_size, int num_pages,
                              void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    orthros_status st = check_shapes(B, Hq, Hkv, d, window, scale, dtype);
    if (st != ORTHROS_OK) return st;
    if (T < 0 || n_out < 0) return fail(ORTHROS_EINVAL, "T = %d and n_out = %d must be >= 0", T, n_out);
    if (B > 0 && !out_indptr) return fail(ORTHROS_EINVAL, "out_indptr (host) must not be NULL");
    if (B > 0 && (out_indptr[0] != 0 || out_indptr[B] != n_out))
        return fail(ORTHROS_EINVAL, "out_indptr must run from 0 to n_out = %d", n_out);
    for (int b = 0; b < B; ++b)
        if (out_indptr[b + 1] < out_indptr[b]) return fail(ORTHROS_EINVAL, "out_indptr decreases at %d", b);
    if (n_out > 0) {
        if (!out_positions || !o_out || !lse_out)
            return fail(ORTHROS_EINVAL, "out_positions, o_out and lse_out must not be NULL when n_out > 0");
        for (int r = 0; r < n_out; ++r)
            if (out_positions[r] < 0 || out_positions[r] >= T)
                return fail(ORTHROS_EINVAL, "out_positions[%d] = %d lies outside [0, T = %d)", r, out_positions[r], T);
    }
    const long long bt = (long long)B * T;
    if (bt > 0 && (!q || !k || !v || !o_base || !lse_base))
        return fail(ORTHROS_EINVAL, "q, k, v, o_base and lse_base must not be NULL");
    for (const void *h : {q, k, v, (const void *)o_base, (const void *)lse_base, q_out, (const void *)o_out,
                          (const void *)lse_out, (const void *)out_positions})
        if (h && !is_host_memory(h)) return fail(ORTHROS_EINVAL, "inputs and outputs must be host memory");
    const FromHostLayout L = from_host_layout(B, T, Hq, Hkv, d, n_out, window, dtype);
    if (!workspace || workspace_bytes < L.total)
        return fail(ORTHROS_EWORKSPACE, "workspace needs %zu bytes, got %zu", L.total, workspace ? workspace_bytes : (size_t)0);
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(ORTHROS_EINVAL, "workspace must be 256-byte aligned");
    char *ws = static_cast<char *>(workspace);
    const size_t eb = elem_bytes(dtype);
    const size_t qrow = (size_t)Hq * d * eb, kvrow = (size_t)Hkv * d * eb;
    char *qd = ws + L.q_off, *kd = ws + L.k_off, *vd = ws + L.v_off, *od = ws + L.o_off;
    int32_t *pos_d = reinterpret_cast<int32_t *>(ws + L.pos_off);
    char *oout_d = ws + L.oout_off;
    float *lout_d = reinterpret_cast<float *>(ws + L.lout_off);
    cudaError_t e;
#define ORTHROS_CU(call, what)                          \
    do {                                                \
        if ((e = (call)) != cudaSuccess) return cuda_fail(e, what); \
    } while (0)

    if (!L.pipelined) {
        // one chunk per sequence: copy in, compute, copy out, all on the caller's stream
        ORTHROS_CU(cudaMemcpyAsync(qd, q, bt * qrow, cudaMemcpyHostToDevice, stream), "q copy in");
        ORTHROS_CU(cudaMemcpyAsync(kd, k, bt * kvrow, cudaMemcpyHostToDevice, stream), "k copy in");
        ORTHROS_CU(cudaMemcpyAsync(vd, v, bt * kvrow, cudaMemcpyHostToDevice, stream), "v copy in");
        const void *qo_d = nullptr;
        if (n_out > 0) {
            ORTHROS_CU(cudaMemcpyAsync(pos_d, out_positions, (size_t)n_out * 4, cudaMemcpyHostToDevice, stream),
                       "positions copy in");
            if (q_out) {
                ORTHROS_CU(cudaMemcpyAsync(ws + L.qrows_off, q_out, (size_t)n_out * qrow, cudaMemcpyHostToDevice, stream),
                           "q_out copy in");
                qo_d = ws + L.qrows_off;
            }
        }
        float *lse_d = reinterpret_cast<float *>(ws + L.lse_off);
        st = prefill_core(qd, kd, vd, alpha_base, beta_base, alpha_out, beta_out, out_indptr, pos_d, n_out, qo_d, B, T,
                          T, false, Hq, Hkv, d, window, scale, dtype, od, lse_d, oout_d, nullptr, lout_d, k_cache,
                          v_cache, block_table, max_pages, page_size, num_pages, ws + L.core_off, L.core_bytes, stream);
        if (st != ORTHROS_OK) return st;
        ORTHROS_CU(cudaMemcpyAsync(o_base, od, bt * qrow, cudaMemcpyDeviceToHost, stream), "o_base copy out");
        ORTHROS_CU(cudaMemcpyAsync(lse_base, lse_d, bt * Hq * 4, cudaMemcpyDeviceToHost, stream), "lse_base copy out");
        if (n_out > 0) {
            ORTHROS_CU(cudaMemcpyAsync(o_out, oout_d, (size_t)n_out * qrow, cudaMemcpyDeviceToHost, stream),
                       "o_out copy out");
            ORTHROS_CU(cudaMemcpyAsync(lse_out, lout_d, (size_t)n_out * Hq * 4, cudaMemcpyDeviceToHost, stream),
                       "lse_out copy out");
        }
        return ORTHROS_OK;
    }

    // ---- pipelined: chunks of the token axis as shards ----
    if (n_out > 0 && (!alpha_out || !beta_out)) return fail(ORTHROS_EINVAL, "alpha_out and beta_out must not be NULL");
    const bool fill = k_cache || v_cache || block_table;
    if (fill) {
        if (!k_cache || !v_cache || !block_table)
            return fail(ORTHROS_EINVAL, "k_cache, v_cache and block_table must be all NULL or all set");
        if (page_size < 1 || max_pages < 1 || num_pages < 1 || (long long)max_pages * page_size < T)
            return fail(ORTHROS_EINVAL, "the cache fill needs page_size, max_pages, num_pages >= 1, max_pages * page_size >= T");
    }
    HostPipe *hp = nullptr;
    std::lock_guard<std::mutex> lock(g_pipe_mu);
    ORTHROS_CU(host_pipe(&hp), "copy streams");
    uint32_t *status = reinterpret_cast<uint32_t *>(ws);
    ORTHROS_CU(cudaMemsetAsync(status, 0, 4 * sizeof(uint32_t), stream), "status reset");
    if (n_out > 0)
        ORTHROS_CU(cudaMemcpyAsync(pos_d, out_positions, (size_t)n_out * 4, cudaMemcpyHostToDevice, stream),
                   "positions copy in");
    ORTHROS_CU(cudaEventRecord(hp->start, stream), "event");
    ORTHROS_CU(cudaStreamWaitEvent(hp->in, hp->start, 0), "event wait");
    ORTHROS_CU(cudaStreamWaitEvent(hp->out, hp->start, 0), "event wait");
    // On an error return, the caller's stream still waits for whatever this
    // call has put on the copy streams, so that its buffers may be freed once
    // `stream` has passed this call.
    struct JoinOnError {
        HostPipe *hp;
        cudaStream_t s;
        bool armed = true;
        ~JoinOnError() {
            if (!armed) return;
            cudaEventRecord(hp->in_done, hp->in);
            cudaStreamWaitEvent(s, hp->in_done, 0);
            cudaEventRecord(hp->end, hp->out);
            cudaStreamWaitEvent(s, hp->end, 0);
        }
    } join{hp, stream};
    // the output rows' raw queries, needed by every chunk: q_out, or runs of
    // consecutive positions of q
    char *qrows_d = ws + L.qrows_off;
    if (n_out > 0) {
        if (q_out) {
            ORTHROS_CU(cudaMemcpyAsync(qrows_d, q_out, (size_t)n_out * qrow, cudaMemcpyHostToDevice, hp->in),
                       "q_out copy in");
        } else {
            for (int b = 0; b < B; ++b)
                for (int r = out_indptr[b]; r < out_indptr[b + 1];) {
                    int n = 1;
                    while (r + n < out_indptr[b + 1] && out_positions[r + n] == out_positions[r] + n) ++n;
                    ORTHROS_CU(cudaMemcpyAsync(qrows_d + (size_t)r * qrow,
                                               static_cast<const char *>(q) + ((size_t)b * T + out_positions[r]) * qrow,
                                               (size_t)n * qrow, cudaMemcpyHostToDevice, hp->in),
                               "output-row queries copy in");
                    r += n;
                }
        }
    }
    int32_t *pos_chunk = reinterpret_cast<int32_t *>(ws + L.pos_chunk_off);
    float *parts = reinterpret_cast<float *>(ws + L.parts_off);
    float *lparts = reinterpret_cast<float *>(ws + L.lparts_off);
    const size_t part_stride = (size_t)n_out * Hq * d, lpart_stride = (size_t)n_out * Hq;
    int slot = 0;
    for (int b = 0; b < B; ++b) {
        const int r0 = out_indptr[b], nb = out_indptr[b + 1] - out_indptr[b];
        for (int c = 0; c < L.n_chunks; ++c, ++slot) {
            const int t0 = L.starts[c], tq = L.starts[c + 1] - t0;
            const int halo = c == 0 ? 0 : std::min(L.halo_max, t0);
            const size_t row0 = (size_t)b * T + t0;
            // in: this chunk's rows (its halo came with the chunks before it)
            ORTHROS_CU(cudaMemcpyAsync(qd + row0 * qrow, static_cast<const char *>(q) + row0 * qrow, (size_t)tq * qrow,
                                       cudaMemcpyHostToDevice, hp->in), "q copy in");
            ORTHROS_CU(cudaMemcpyAsync(kd + row0 * kvrow, static_cast<const char *>(k) + row0 * kvrow,
                                       (size_t)tq * kvrow, cudaMemcpyHostToDevice, hp->in), "k copy in");
            ORTHROS_CU(cudaMemcpyAsync(vd + row0 * kvrow, static_cast<const char *>(v) + row0 * kvrow,
                                       (size_t)tq * kvrow, cudaMemcpyHostToDevice, hp->in), "v copy in");
            ORTHROS_CU(cudaEventRecord(hp->in_done, hp->in), "event");
            ORTHROS_CU(cudaStreamWaitEvent(stream, hp->in_done, 0), "event wait");
            // compute: the chunk as a shard (its lse_base buffer waits for the copy
            // out of the chunk that used it two chunks ago)
            if (slot >= 2) ORTHROS_CU(cudaStreamWaitEvent(stream, hp->out_done[slot & 1], 0), "event wait");
            float *lse_c = reinterpret_cast<float *>(ws + L.lse_off) + (size_t)(slot & 1) * Hq * L.chunk;
            if (nb > 0) ORTHROS_CU(launch_shift_positions(pos_d + r0, pos_chunk + r0, nb, t0 - halo, stream), "positions");
            const int32_t rows_indptr[2] = {0, nb};
            st = prefill_core(qd + row0 * qrow, kd + (row0 - halo) * kvrow, vd + (row0 - halo) * kvrow, alpha_base,
                              beta_base, alpha_out, beta_out, rows_indptr, pos_chunk + r0, nb,
                              nb > 0 ? qrows_d + (size_t)r0 * qrow : nullptr, 1, halo + tq, tq, true, Hq, Hkv, d,
                              window, scale, dtype, od + row0 * qrow, lse_c, nullptr,
                              nb > 0 ? parts + c * part_stride + (size_t)r0 * Hq * d : nullptr,
                              nb > 0 ? lparts + c * lpart_stride + (size_t)r0 * Hq : nullptr, nullptr, nullptr,
                              nullptr, 0, 0, 0, ws + L.core_off + (size_t)slot * kSlotBytes, L.core_bytes, stream);
            if (st != ORTHROS_OK) return st;
            ORTHROS_CU(cudaEventRecord(hp->comp_done, stream), "event");
            // out: the chunk's o_base rows and its lse_base columns
            ORTHROS_CU(cudaStreamWaitEvent(hp->out, hp->comp_done, 0), "event wait");
            ORTHROS_CU(cudaMemcpyAsync(static_cast<char *>(o_base) + row0 * qrow, od + row0 * qrow, (size_t)tq * qrow,
                                       cudaMemcpyDeviceToHost, hp->out), "o_base copy out");
            ORTHROS_CU(cudaMemcpy2DAsync(lse_base + (size_t)b * Hq * T + t0, (size_t)T * 4, lse_c, (size_t)tq * 4,
                                         (size_t)tq * 4, Hq, cudaMemcpyDeviceToHost, hp->out), "lse_base copy out");
            ORTHROS_CU(cudaEventRecord(hp->out_done[slot & 1], hp->out), "event");
        }
    }
    // the output rows' partials merged; the cache filled from the keys and values
    // now on the device; every shard's status folded into this call's
    if (n_out > 0) {
        ProfScope ps("merge_partials", stream);
        ORTHROS_CU(launch_merge_partials(parts, lparts, L.n_chunks, n_out, Hq, d, false, oout_d, lout_d, stream),
                   "merge launch");
    }
    if (fill) {
        ProfScope ps("cache_fill", stream);
        ORTHROS_CU(launch_prefill_cache_fill(kd, vd, k_cache, v_cache, block_table, B, T, Hkv, d, max_pages, page_size,
                                             num_pages, (int)eb, status, stream), "cache fill launch");
    }
    ORTHROS_CU(launch_fold_status(status, reinterpret_cast<const uint32_t *>(ws + L.core_off), slot,
                                  (int)(kSlotBytes / 4), stream), "status fold");
    if (n_out > 0) {
        ORTHROS_CU(cudaEventRecord(hp->comp_done, stream), "event");
        ORTHROS_CU(cudaStreamWaitEvent(hp->out, hp->comp_done, 0), "event wait");
        ORTHROS_CU(cudaMemcpyAsync(o_out, oout_d, (size_t)n_out * qrow, cudaMemcpyDeviceToHost, hp->out), "o_out copy out");
        ORTHROS_CU(cudaMemcpyAsync(lse_out, lout_d, (size_t)n_out * Hq * 4, cudaMemcpyDeviceToHost, hp->out),
                   "lse_out copy out");
    }
    // the caller's stream resumes once everything above, copies out included, is done
    ORTHROS_CU(cudaEventRecord(hp->end, hp->out), "event");
    ORTHROS_CU(cudaStreamWaitEvent(stream, hp->end, 0), "event wait");
    join.armed = false;
#undef ORTHROS_CU
    return ORTHROS_OK;
}

}  // namespace

orthros_status report_error(orthros_status s, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

}  // namespace orthros

using namespace orthros;

extern "C" {

const char *orthros_status_string(orthros_status s) {
    switch (s) {
        case ORTHROS_OK: return "ok";
        case ORTHROS_EINVAL: return "invalid argument";
        case ORTHROS_EUNSUPPORTED: return "unsupported configuration";
        case ORTHROS_ECUDA: return "CUDA error";
        case ORTHROS_EWORKSPACE: return "workspace missing or too small";
        case ORTHROS_EDEVICE: return "bad device-side data flagged by a kernel";
        case ORTHROS_ETIMEOUT: return "bounded wait inside a kernel ran out";
    }
    return "unknown status";
}

const char *orthros_last_error(void) { return g_last_error.c_str(); }

size_t orthros_prefill_workspace_size(int B, int T, int Hq, int Hkv, int d, int n_out, int window,
                                      orthros_dtype dtype) {
    if (T < 0 || n_out < 0) return 0;
    if (check_shapes(B, Hq, Hkv, d, window, 1.0f, dtype) != ORTHROS_OK) return 0;
    return prefill_layout(B, T, Hq, Hkv, d, n_out, dtype).total;
}

orthros_status orthros_prefill(const void *q, const void *k, const void *v, const float *alpha_base,
                               const float *beta_base, const float *alpha_out, const float *beta_out,
                               const int32_t *out_indptr, const int32_t *out_positions, int n_out,
                               const void *q_out, int B, int T, int Hq, int Hkv, int d, int window,
                               float scale, orthros_dtype dtype, void *o_base, float *lse_base,
                               void *o_out, float *lse_out, void *k_cache, void *v_cache,
                               const int32_t *block_table, int max_pages, int page_size, int num_pages,
                               void *workspace, size_t workspace_bytes, orthros_stream_t stream) {
    g_last_error.clear();
    return prefill_core(q, k, v, alpha_base, beta_base, alpha_out, beta_out, out_indptr, out_positions, n_out, q_out,
                        B, T, T, false, Hq, Hkv, d, window, scale, dtype, o_base, lse_base, o_out, nullptr, lse_out,
                        k_cache, v_cache, block_table, max_pages, page_size, num_pages, workspace, workspace_bytes,
                        reinterpret_cast<cudaStream_t>(stream));
}

size_t orthros_prefill_shard_workspace_size(int B, int Tq, int Tkv, int Hq, int Hkv, int d, int n_rows, int window,
                                            orthros_dtype dtype) {
    if (Tkv < 0 || Tq < 0 || Tq > Tkv || n_rows < 0 || dtype != ORTHROS_BF16) return 0;
    if (check_shapes(B, Hq, Hkv, d, window, 1.0f, dtype) != ORTHROS_OK) return 0;
    return prefill_layout(B, Tkv, Hq, Hkv, d, n_rows, dtype).total;
}

orthros_status orthros_prefill_shard(const void *q, const void *k, const void *v, const float *alpha_base,
                                     const float *beta_base, const float *alpha_out, const float *beta_out,
                                     const int32_t *row_indptr, const int32_t *row_positions, int n_rows,
                                     const void *q_rows, int B, int Tq, int Tkv, int Hq, int Hkv, int d, int window,
                                     float scale, orthros_dtype dtype, void *o_base, float *lse_base,
                                     float *o_part, float *lse_part, void *workspace, size_t workspace_bytes,
                                     orthros_stream_t stream) {
    g_last_error.clear();
    if (Tq < 1) return fail(ORTHROS_EINVAL, "Tq = %d: a shard holds at least one query row", Tq);
    return prefill_core(q, k, v, alpha_base, beta_base, alpha_out, beta_out, row_indptr, row_positions, n_rows,
                        q_rows, B, Tkv, Tq, true, Hq, Hkv, d, window, scale, dtype, o_base, lse_base, nullptr,
                        o_part, lse_part, nullptr, nullptr, nullptr, 0, 0, 0, workspace, workspace_bytes,
                        reinterpret_cast<cudaStream_t>(stream));
}

size_t orthros_prefill_from_host_workspace_size(int B, int T, int Hq, int Hkv, int d, int n_out, int window,
                                                orthros_dtype dtype) {
    if (T < 0 || n_out < 0) return 0;
    if (check_shapes(B, Hq, Hkv, d, window, 1.0f, dtype) != ORTHROS_OK) return 0;
    return from_host_layout(B, T, Hq, Hkv, d, n_out, window, dtype).total;
}

orthros_status orthros_prefill_from_host(const void *q, const void *k, const void *v, const float *alpha_base,
                                         const float *beta_base, const float *alpha_out, const float *beta_out,
                                         const int32_t *out_indptr, const int32_t *out_positions, int n_out,
                                         const void *q_out, int B, int T, int Hq, int Hkv, int d, int window,
                                         float scale, orthros_dtype dtype, void *o_base, float *lse_base, void *o_out,
                                         float *lse_out, void *k_cache, void *v_cache, const int32_t *block_table,
                                         int max_pages, int page_size, int num_pages, void *workspace,
                                         size_t workspace_bytes, orthros_stream_t stream) {
    g_last_error.clear();
    return from_host_core(q, k, v, alpha_base, beta_base, alpha_out, beta_out, out_indptr, out_positions, n_out, q_out,
                          B, T, Hq, Hkv, d, window, scale, dtype, o_base, lse_base, o_out, lse_out, k_cache, v_cache,
                          block_table, max_pages, page_size, num_pages, workspace, workspace_bytes,
                          reinterpret_cast<cudaStream_t>(stream));
}

orthros_status orthros_merge_partials(const float *o_parts, const float *lse_parts, int n_parts, int n_rows, int Hq,
                                      int d, orthros_dtype dtype, void *o_out, float *lse_out,
                                      orthros_stream_t stream_) {
    g_last_error.clear();
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (n_parts < 1 || n_rows < 0 || Hq < 1) return fail(ORTHROS_EINVAL, "n_parts >= 1, n_rows >= 0, Hq >= 1");
    if (d != 64 && d != 128) return fail(ORTHROS_EUNSUPPORTED, "head size d = %d (supported: 64, 128)", d);
    if (dtype != ORTHROS_BF16 && dtype != ORTHROS_F32) return fail(ORTHROS_EINVAL, "unknown dtype %d", (int)dtype);
    if ((long long)n_rows * Hq > (1LL << 31) / 32)
        return fail(ORTHROS_EUNSUPPORTED, "n_rows * Hq = %lld exceeds the launch grid", (long long)n_rows * Hq);
    if (n_rows == 0) return ORTHROS_OK;
    if (!o_parts || !lse_parts || !o_out || !lse_out) return fail(ORTHROS_EINVAL, "pointers must not be NULL");
    if (!aligned16(o_parts) || !aligned16(o_out)) return fail(ORTHROS_EINVAL, "o_parts and o_out must be 16-byte aligned");
    cudaError_t e;
    {
        ProfScope ps("merge_partials", stream);
        e = launch_merge_partials(o_parts, lse_parts, n_parts, n_rows, Hq, d, dtype == ORTHROS_F32, o_out, lse_out,
                                  stream);
    }
    if (e != cudaSuccess) return cuda_fail(e, "merge launch");
    return ORTHROS_OK;
}

size_t orthros_prefill_backward_workspace_size(int B, int T, int Hq, int Hkv, int d, int n_out, int window,
                                               orthros_dtype dtype) {
    if (T < 0 || n_out < 0) return 0;
    if (check_shapes(B, Hq, Hkv, d, window, 1.0f, dtype) != ORTHROS_OK) return 0;
    return backward_layout(B, T, Hq, d, n_out, dtype).total;
}

orthros_status orthros_prefill_backward(const void *q, const void *k, const void *v, const float *alpha_base,
                                        const float *beta_base, const float *alpha_out, const float *beta_out,
                                        const int32_t *out_indptr, const int32_t *out_positions, int n_out,
                                        const void *q_out, int B, int T, int Hq, int Hkv, int d, int window,
                                        float scale, orthros_dtype dtype, const void *o_base,
                                        const float *lse_base, const void *o_out, const float *lse_out,
                                        const void *do_base, const void *do_out, void *dq, void *dk, void *dv,
                                        void *dq_out, float *d_alpha_base, float *d_beta_base,
                                        float *d_alpha_out, float *d_beta_out, void *workspace,
                                        size_t workspace_bytes, orthros_stream_t stream_) {
    g_last_error.clear();
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    orthros_status st = check_shapes(B, Hq, Hkv, d, window, scale, dtype);
    if (st != ORTHROS_OK) return st;
    if (T < 0) return fail(ORTHROS_EINVAL, "T = %d must be >= 0", T);
    if (n_out < 0) return fail(ORTHROS_EINVAL, "n_out = %d must be >= 0", n_out);
    const long long rows = (long long)B * T;
    if (rows > (1LL << 31)) return fail(ORTHROS_EUNSUPPORTED, "B*T = %lld tokens exceeds 2^31", rows);
    if (B > 65535) return fail(ORTHROS_EUNSUPPORTED, "B = %d exceeds 65535 sequences per call", B);
    if (!d_alpha_base || !d_beta_base || !d_alpha_out || !d_beta_out)
        return fail(ORTHROS_EINVAL, "the four affine gradients must not be NULL");
    if (rows > 0) {
        if (!q || !k || !v || !o_base || !lse_base || !do_base || !dq || !dk || !dv)
            return fail(ORTHROS_EINVAL, "q, k, v, o_base, lse_base, do_base, dq, dk and dv must not be NULL");
        if (!alpha_base || !beta_base) return fail(ORTHROS_EINVAL, "alpha_base and beta_base must not be NULL");
        if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o_base) || !aligned16(do_base) ||
            !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
            return fail(ORTHROS_EINVAL, "element tensors must be 16-byte aligned");
        if (!aligned16(alpha_base) || !aligned16(beta_base))
            return fail(ORTHROS_EINVAL, "alpha_base and beta_base must be 16-byte aligned");
    }
    if (B > 0 && !out_indptr) return fail(ORTHROS_EINVAL, "out_indptr (host) must not be NULL");
    if (B > 0) {
        if (out_indptr[0] != 0) return fail(ORTHROS_EINVAL, "out_indptr[0] = %d must be 0", out_indptr[0]);
        for (int b = 0; b < B; ++b)
            if (out_indptr[b + 1] < out_indptr[b])
                return fail(ORTHROS_EINVAL, "out_indptr decreases at %d", b);
        if (out_indptr[B] != n_out)
            return fail(ORTHROS_EINVAL, "out_indptr[B] = %d differs from n_out = %d", out_indptr[B], n_out);
    } else if (n_out != 0) {
        return fail(ORTHROS_EINVAL, "n_out = %d with B = 0", n_out);
    }
    if (n_out > 0) {
        if (T == 0) return fail(ORTHROS_EINVAL, "output rows with T = 0");
        if (!out_positions || !alpha_out || !beta_out || !o_out || !lse_out || !do_out)
            return fail(ORTHROS_EINVAL, "out_positions, alpha_out, beta_out, o_out, lse_out and do_out "
                                        "must not be NULL when n_out > 0");
        if (q_out && !dq_out) return fail(ORTHROS_EINVAL, "dq_out must not be NULL when q_out is given");
        if (!aligned16(o_out) || !aligned16(do_out) || (q_out && (!aligned16(q_out) || !aligned16(dq_out))) ||
            !aligned16(alpha_out) || !aligned16(beta_out))
            return fail(ORTHROS_EINVAL, "output-row tensors and affines must be 16-byte aligned");
    }
    const BackwardLayout lay = backward_layout(B, T, Hq, d, n_out, dtype);
    if (!workspace || workspace_bytes < lay.total)
        return fail(ORTHROS_EWORKSPACE, "workspace needs %zu bytes, got %zu", lay.total,
                    workspace ? workspace_bytes : (size_t)0);
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(ORTHROS_EINVAL, "workspace must be 256-byte aligned");

    char *ws = static_cast<char *>(workspace);
    uint32_t *status = reinterpret_cast<uint32_t *>(ws);
    cudaError_t e = cudaMemsetAsync(status, 0, sizeof(uint32_t), stream);
    if (e != cudaSuccess) return cuda_fail(e, "status reset");
    const size_t affine_bytes = sizeof(float) * (size_t)Hq * d;
    for (float *g : {d_alpha_base, d_beta_base, d_alpha_out, d_beta_out})
        if ((e = cudaMemsetAsync(g, 0, affine_bytes, stream)) != cudaSuccess) return cuda_fail(e, "gradient reset");
    if (rows == 0) return ORTHROS_OK;
    int32_t *indptr_dev = reinterpret_cast<int32_t *>(ws + lay.indptr_off);
    int32_t *head = reinterpret_cast<int32_t *>(ws + lay.head_off);
    if (n_out > 0) {
        e = cudaMemcpyAsync(indptr_dev, out_indptr, sizeof(int32_t) * (size_t)(B + 1), cudaMemcpyHostToDevice,
                            stream);
        if (e != cudaSuccess) return cuda_fail(e, "indptr upload");
        if ((e = cudaMemsetAsync(head, 0xff, sizeof(int32_t) * (size_t)rows, stream)) != cudaSuccess)
            return cuda_fail(e, "row-list reset");
    }
    BwdArgs a{};
    a.q = q;
    a.q_out = q_out;
    a.k = k;
    a.v = v;
    a.alpha_base = alpha_base;
    a.beta_base = beta_base;
    a.alpha_out = alpha_out;
    a.beta_out = beta_out;
    a.out_indptr = indptr_dev;
    a.out_positions = out_positions;
    a.pos_head = head;
    a.row_next = reinterpret_cast<int32_t *>(ws + lay.next_off);
    a.n_out = n_out;
    a.B = B;
    a.T = T;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.window = window;
    a.scale = scale;
    a.o_base = o_base;
    a.o_out = o_out;
    a.do_base = do_base;
    a.do_out = do_out;
    a.lse_base = lse_base;
    a.lse_out = lse_out;
    a.delta_base = reinterpret_cast<float *>(ws + lay.delta_base_off);
    a.delta_out = reinterpret_cast<float *>(ws + lay.delta_out_off);
    a.dq_rows = reinterpret_cast<float *>(ws + lay.dq_rows_off);
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.dq_out = q_out ? dq_out : nullptr;
    a.d_alpha_base = d_alpha_base;
    a.d_beta_base = d_beta_base;
    a.d_alpha_out = d_alpha_out;
    a.d_beta_out = d_beta_out;
    a.status = status;
    const bool use_tc = dtype == ORTHROS_BF16;
    if (use_tc) {
        a.qa_base = reinterpret_cast<__nv_bfloat16 *>(ws + lay.qa_base_off);
        a.qa_out = reinterpret_cast<__nv_bfloat16 *>(ws + lay.qa_out_off);
        a.dq_acc = reinterpret_cast<float *>(ws + lay.dq_acc_off);
        a.omax = reinterpret_cast<int32_t *>(ws + lay.omax_off);
    }
    e = launch_backward(a, d, dtype, use_tc, stream);
    if (e != cudaSuccess) return cuda_fail(e, "backward launch");
    return ORTHROS_OK;
}

size_t orthros_extend_workspace_size(int B, int n_new, int n_out, int Hq, int Hkv, int d, int max_pages,
                                     int page_size, orthros_dtype dtype) {
    if (n_new < 0 || n_out < 0 || max_pages < 1 || page_size < 1) return 0;
    if (check_shapes(B, Hq, Hkv, d, 1, 1.0f, dtype) != ORTHROS_OK) return 0;
    return extend_layout(B, n_new, n_out, Hq, Hkv, d, max_pages, page_size, dtype).total;
}

orthros_status orthros_extend(const void *q, const void *q_out, const void *k_new, const void *v_new, void *k_cache,
                              void *v_cache, const int32_t *block_table, int max_pages, int page_size, int num_pages,
                              const int32_t *cache_lens, const int32_t *new_indptr, const int32_t *out_indptr,
                              const int32_t *out_positions, const float *alpha_base, const float *beta_base,
                              const float *alpha_out, const float *beta_out, int B, int Hq, int Hkv, int d,
                              int window, float scale, orthros_dtype dtype, void *o_base, float *lse_base,
                              void *o_out, float *lse_out, void *workspace, size_t workspace_bytes,
                              orthros_stream_t stream_) {
    g_last_error.clear();
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    orthros_status st = check_shapes(B, Hq, Hkv, d, window, scale, dtype);
    if (st != ORTHROS_OK) return st;
    if (B > 32767) return fail(ORTHROS_EUNSUPPORTED, "B = %d exceeds 32767 sequences per step", B);
    if (page_size < 1 || max_pages < 1 || num_pages < 1)
        return fail(ORTHROS_EINVAL, "page_size, max_pages and num_pages must be >= 1");
    if (B > 0 && (!new_indptr || !out_indptr)) return fail(ORTHROS_EINVAL, "new_indptr and out_indptr (host) must not be NULL");
    for (const int32_t *ip : {new_indptr, out_indptr}) {
        if (B == 0) break;
        if (ip[0] != 0) return fail(ORTHROS_EINVAL, "indptr[0] = %d must be 0", ip[0]);
        for (int b = 0; b < B; ++b)
            if (ip[b + 1] < ip[b]) return fail(ORTHROS_EINVAL, "indptr decreases at %d", b);
    }
    const int n_new = B > 0 ? new_indptr[B] : 0;
    const int n_out = B > 0 ? out_indptr[B] : 0;
    if (B > 0) {
        if (!k_cache || !v_cache || !block_table || !cache_lens)
            return fail(ORTHROS_EINVAL, "k_cache, v_cache, block_table and cache_lens must not be NULL");
        if (!aligned16(k_cache) || !aligned16(v_cache)) return fail(ORTHROS_EINVAL, "caches must be 16-byte aligned");
    }
    if (n_new > 0) {
        if (!q || !k_new || !v_new || !alpha_base || !beta_base || !o_base || !lse_base)
            return fail(ORTHROS_EINVAL, "q, k_new, v_new, alpha_base, beta_base, o_base, lse_base must not be NULL");
        if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(o_base) ||
            !aligned16(alpha_base) || !aligned16(beta_base))
            return fail(ORTHROS_EINVAL, "new-token tensors and base affines must be 16-byte aligned");
    }
    if (n_out > 0) {
        if (!out_positions || !alpha_out || !beta_out || !o_out || !lse_out)
            return fail(ORTHROS_EINVAL, "out_positions, alpha_out, beta_out, o_out, lse_out must not be NULL");
        if (!q_out && !q) return fail(ORTHROS_EINVAL, "output rows need q_out or the new tokens' q");
        if (!aligned16(o_out) || (q_out && !aligned16(q_out)) || !aligned16(alpha_out) || !aligned16(beta_out))
            return fail(ORTHROS_EINVAL, "output-row tensors and affines must be 16-byte aligned");
    }
    const ExtendLayout lay = extend_layout(B, n_new, n_out, Hq, Hkv, d, max_pages, page_size, dtype);
    if (!workspace || workspace_bytes < lay.total)
        return fail(ORTHROS_EWORKSPACE, "workspace needs %zu bytes, got %zu", lay.total,
                    workspace ? workspace_bytes : (size_t)0);
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(ORTHROS_EINVAL, "workspace must be 256-byte aligned");
    char *ws = static_cast<char *>(workspace);
    uint32_t *status = reinterpret_cast<uint32_t *>(ws);
    cudaError_t e = cudaMemsetAsync(status, 0, sizeof(uint32_t), stream);
    if (e != cudaSuccess) return cuda_fail(e, "status reset");
    if (n_new + n_out == 0) return ORTHROS_OK;

    // plan: both indptrs, then the split groups (bf16 fast path)
    const int g = Hq / Hkv;
    const long long kv_tokens = (long long)num_pages * page_size;
    const bool fast = dtype == ORTHROS_BF16 && g <= 16 && page_size % 64 == 0 && kv_tokens < 0x7fffffffLL;
    std::vector<int32_t> blob((size_t)2 * (B + 1));
    std::copy(new_indptr, new_indptr + B + 1, blob.begin());
    std::copy(out_indptr, out_indptr + B + 1, blob.begin() + B + 1);
    // Groups of one (sequence, kv head): all its positions in one group when
    // they fit 8 rows (a decoding token's base and output rows then share one
    // pass over the cache); otherwise new-token base rows in groups of up to
    // 16 rows (neighbouring windows overlap) and output rows in groups of up
    // to 8. Groups of <= 8 rows come first (their own launch).
    int n_groups = 0, n_small = 0;
    if (fast) {
        std::vector<int32_t> small, big;
        auto add = [&](std::vector<int32_t> &v, int b, int kvh, int base0, int nb, int out0, int no) {
            v.push_back((b << 16) | kvh);
            v.push_back(base0);
            v.push_back(out0);
            v.push_back(nb | (no << 16));
        };
        const int p8 = std::max(1, 8 / g), p16 = 16 / g;
        for (int b = 0; b < B; ++b) {
            const int nb = new_indptr[b + 1] - new_indptr[b], no = out_indptr[b + 1] - out_indptr[b];
            for (int kvh = 0; kvh < Hkv; ++kvh) {
                if (nb + no == 0) continue;
                if (g <= 8 && (nb + no) * g <= 8) {
                    add(small, b, kvh, new_indptr[b], nb, out_indptr[b], no);
                    continue;
                }
                for (int i = 0; i < nb; i += p16)
                    add(big, b, kvh, new_indptr[b] + i, std::min(p16, nb - i), out_indptr[b], 0);
                for (int i = 0; i < no; i += p8)
                    add(g <= 8 ? small : big, b, kvh, new_indptr[b], 0, out_indptr[b] + i, std::min(p8, no - i));
            }
        }
        n_small = (int)small.size() / 4;
        n_groups = n_small + (int)big.size() / 4;
        blob.insert(blob.end(), small.begin(), small.end());
        blob.insert(blob.end(), big.begin(), big.end());
        if (n_groups > lay.max_groups) return fail(ORTHROS_EWORKSPACE, "internal: extend groups exceed the plan");
    }
    int32_t *blob_dev = reinterpret_cast<int32_t *>(ws + lay.blob_off);
    e = cudaMemcpyAsync(blob_dev, blob.data(), sizeof(int32_t) * blob.size(), cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return cuda_fail(e, "plan upload");
    const int32_t *new_dev = blob_dev, *out_dev = blob_dev + B + 1, *groups_dev = blob_dev + 2 * (B + 1);
    {
        ProfScope ps("extend_append", stream);
        e = launch_extend_append(k_new, v_new, k_cache, v_cache, block_table, cache_lens, new_dev, B, n_new, Hkv, d,
                                 max_pages, page_size, num_pages, elem_bytes(dtype), status, stream);
    }
    if (e != cudaSuccess) return cuda_fail(e, "append launch");
    if (fast) {
        SplitParams sp{};
        sp.mode = kSplitExtend;
        sp.q = static_cast<const __nv_bfloat16 *>(q);
        sp.q_out = static_cast<const __nv_bfloat16 *>(q_out);
        sp.k = static_cast<const __nv_bfloat16 *>(k_cache);
        sp.v = static_cast<const __nv_bfloat16 *>(v_cache);
        sp.alpha_base = alpha_base;
        sp.beta_base = beta_base;
        sp.alpha_out = alpha_out;
        sp.beta_out = beta_out;
        sp.out_positions = out_positions;
        sp.ext_info = groups_dev;
        sp.block_table = block_table;
        sp.cache_lens = cache_lens;
        sp.new_indptr = new_dev;
        sp.n_new = n_new;
        sp.max_pages = max_pages;
        sp.page_size = page_size;
        sp.num_pages = num_pages;
        sp.B = B;
        sp.Hq = Hq;
        sp.Hkv = Hkv;
        sp.window = window;
        sp.scale = scale;
        sp.scale_log2 = scale * 1.4426950408889634f;
        sp.n_groups = n_groups;
        sp.chunk = split_chunk(n_groups, (long long)max_pages * page_size);
        sp.max_chunks = ceil_div((long long)max_pages * page_size, sp.chunk);
        if ((long long)n_groups * sp.max_chunks > lay.part_slots)
            return fail(ORTHROS_EWORKSPACE, "internal: split partials exceed the workspace plan");
        sp.kv_tokens = kv_tokens;
        sp.partial = reinterpret_cast<float *>(ws + lay.part_off);
        sp.o_base = static_cast<__nv_bfloat16 *>(o_base);
        sp.lse_base = lse_base;
        sp.o_out = static_cast<__nv_bfloat16 *>(o_out);
        sp.lse_out = lse_out;
        sp.status = status;
        ProfScope ps("splitkv_extend", stream);
        e = launch_splitkv_extend(sp, d, n_small, stream);
        if (e != cudaSuccess) return cuda_fail(e, "split-KV extend launch");
        return ORTHROS_OK;
    }
    RowsArgs a{};
    a.q = q;
    a.q_out = q_out;
    a.k = k_cache;
    a.v = v_cache;
    a.alpha_base = alpha_base;
    a.beta_base = beta_base;
    a.alpha_out = alpha_out;
    a.beta_out = beta_out;
    a.out_indptr = out_dev;
    a.out_positions = out_positions;
    a.block_table = block_table;
    a.cache_lens = cache_lens;
    a.new_indptr = new_dev;
    a.n_new = n_new;
    a.n_out = n_out;
    a.max_pages = max_pages;
    a.page_size = page_size;
    a.num_pages = num_pages;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.window = window;
    a.scale = scale;
    a.o_base = o_base;
    a.lse_base = lse_base;
    a.o_out = o_out;
    a.lse_out = lse_out;
    a.status = status;
    if (n_new > 0) {
        ProfScope ps("rows_simt_extend", stream);
        if ((e = launch_rows_simt(a, kExtendBase, d, dtype, stream)) != cudaSuccess) return cuda_fail(e, "extend rows");
    }
    if (n_out > 0) {
        ProfScope ps("rows_simt_extend_out", stream);
        if ((e = launch_rows_simt(a, kExtendOut, d, dtype, stream)) != cudaSuccess) return cuda_fail(e, "extend rows");
    }
    return ORTHROS_OK;
}

orthros_status orthros_qkv_project(const void *x, int n_base, int n_out, int d_model, const void *w_qkv, int Hq,
                                   int Hkv, int d, const float *alpha_base, const float *beta_base,
                                   const float *alpha_out, const float *beta_out, void *q_base, void *q_out,
                                   void *k_out, void *v_out, void *k_cache, void *v_cache,
                                   const int32_t *block_table, int B, int max_pages, int page_size, int num_pages,
                                   const int32_t *token_seq, const int32_t *token_pos, orthros_dtype dtype,
                                   void *workspace, size_t workspace_bytes, orthros_stream_t stream_) {
    g_last_error.clear();
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (dtype != ORTHROS_BF16) return fail(ORTHROS_EUNSUPPORTED, "the projection takes bf16 only");
    if (n_base < 0 || n_out < 0) return fail(ORTHROS_EINVAL, "n_base = %d, n_out = %d must be >= 0", n_base, n_out);
    if (Hq < 1 || Hkv < 1) return fail(ORTHROS_EINVAL, "head counts must be >= 1");
    if (d != 64 && d != 128) return fail(ORTHROS_EUNSUPPORTED, "head size d = %d (supported: 64, 128)", d);
    if (d_model < 64 || d_model % 64 != 0)
        return fail(ORTHROS_EUNSUPPORTED, "d_model = %d must be a positive multiple of 64", d_model);
    if ((long long)n_base + n_out > 65535LL * 128)
        return fail(ORTHROS_EUNSUPPORTED, "%lld rows exceed 65535 tiles of 128", (long long)n_base + n_out);
    if (!workspace || workspace_bytes < kStatusBytes)
        return fail(ORTHROS_EWORKSPACE, "workspace needs %zu bytes", kStatusBytes);
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(ORTHROS_EINVAL, "workspace must be 256-byte aligned");
    if (n_base + n_out > 0) {
        if (!x || !w_qkv) return fail(ORTHROS_EINVAL, "x and w_qkv must not be NULL");
        if (!aligned16(x) || !aligned16(w_qkv)) return fail(ORTHROS_EINVAL, "x and w_qkv must be 16-byte aligned");
    }
    if (n_base > 0) {
        if (!q_base || !alpha_base || !beta_base) return fail(ORTHROS_EINVAL, "q_base and the base affine must not be NULL");
        if ((k_out == nullptr) != (v_out == nullptr)) return fail(ORTHROS_EINVAL, "k_out and v_out: both or neither");
        const bool cache = k_cache || v_cache || block_table;
        if (cache && (!k_cache || !v_cache || !block_table || !token_seq || !token_pos))
            return fail(ORTHROS_EINVAL, "cache writes need k_cache, v_cache, block_table, token_seq and token_pos");
        if (cache && (page_size < 1 || max_pages < 1 || num_pages < 1 || B < 1))
            return fail(ORTHROS_EINVAL, "B, page_size, max_pages and num_pages must be >= 1 for cache writes");
        if (!aligned16(q_base) || (k_out && (!aligned16(k_out) || !aligned16(v_out))) ||
            (k_cache && (!aligned16(k_cache) || !aligned16(v_cache))))
            return fail(ORTHROS_EINVAL, "outputs must be 16-byte aligned");
    }
    if (n_out > 0) {
        if (!q_out || !alpha_out || !beta_out) return fail(ORTHROS_EINVAL, "q_out and the output affine must not be NULL");
        if (!aligned16(q_out)) return fail(ORTHROS_EINVAL, "q_out must be 16-byte aligned");
    }
    uint32_t *status = static_cast<uint32_t *>(workspace);
    cudaError_t e = cudaMemsetAsync(status, 0, sizeof(uint32_t), stream);
    if (e != cudaSuccess) return cuda_fail(e, "status reset");
    if (n_base + n_out == 0) return ORTHROS_OK;
    ProjParams pp{};
    pp.x = static_cast<const __nv_bfloat16 *>(x);
    pp.w_t = static_cast<const __nv_bfloat16 *>(w_qkv);
    pp.n_base = n_base;
    pp.n_out = n_out;
    pp.d_model = d_model;
    pp.Hq = Hq;
    pp.Hkv = Hkv;
    pp.d = d;
    pp.alpha_base = alpha_base;
    pp.beta_base = beta_base;
    pp.alpha_out = alpha_out;
    pp.beta_out = beta_out;
    pp.q_base = static_cast<__nv_bfloat16 *>(q_base);
    pp.q_out = static_cast<__nv_bfloat16 *>(q_out);
    pp.k_out = static_cast<__nv_bfloat16 *>(k_out);
    pp.v_out = static_cast<__nv_bfloat16 *>(v_out);
    pp.k_cache = static_cast<__nv_bfloat16 *>(k_cache);
    pp.v_cache = static_cast<__nv_bfloat16 *>(v_cache);
    pp.block_table = block_table;
    pp.token_seq = token_seq;
    pp.token_pos = token_pos;
    pp.B = B;
    pp.max_pages = max_pages;
    pp.page_size = page_size;
    pp.num_pages = num_pages;
    pp.status = status;
    {
        ProfScope ps("project_tc", stream);
        e = launch_project_tc(pp, stream);
    }
    if (e != cudaSuccess) return cuda_fail(e, "projection launch");
    return ORTHROS_OK;
}

size_t orthros_decode_workspace_size(int B, int Hq, int Hkv, int d, int max_pages, int page_size,
                                     orthros_dtype dtype) {
    if (max_pages < 1 || page_size < 1) return 0;
    if (check_shapes(B, Hq, Hkv, d, 1, 1.0f, dtype) != ORTHROS_OK) return 0;
    return decode_layout(B, Hq, Hkv, d, max_pages, page_size, dtype).total;
}

orthros_status orthros_decode(const void *q, const void *q_out, const void *k_new, const void *v_new,
                              void *k_cache, void *v_cache, const int32_t *block_table, int max_pages,
                              int page_size, int num_pages, const int32_t *cache_lens,
                              const float *alpha_base, const float *beta_base, const float *alpha_out,
                              const float *beta_out, int B, int Hq, int Hkv, int d, int window, float scale,
                              orthros_dtype dtype, void *o_base, float *lse_base, void *o_out, float *lse_out,
                              void *workspace, size_t workspace_bytes, orthros_stream_t stream_) {
    g_last_error.clear();
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    orthros_status st = check_shapes(B, Hq, Hkv, d, window, scale, dtype);
    if (st != ORTHROS_OK) return st;
    if (page_size < 1 || max_pages < 1 || num_pages < 1)
        return fail(ORTHROS_EINVAL, "page_size, max_pages and num_pages must be >= 1");
    if (B > 0) {
        if (!q || !k_new || !v_new || !k_cache || !v_cache || !block_table || !cache_lens)
            return fail(ORTHROS_EINVAL, "q, k_new, v_new, caches, block_table, cache_lens must not be NULL");
        if (!alpha_base || !beta_base || !alpha_out || !beta_out)
            return fail(ORTHROS_EINVAL, "the four affine vectors must not be NULL");
        if (!aligned16(alpha_base) || !aligned16(beta_base) || !aligned16(alpha_out) || !aligned16(beta_out))
            return fail(ORTHROS_EINVAL, "the four affine vectors must be 16-byte aligned");
        if (!o_base || !lse_base || !o_out || !lse_out)
            return fail(ORTHROS_EINVAL, "outputs must not be NULL");
        if (!aligned16(q) || (q_out && !aligned16(q_out)) || !aligned16(k_new) || !aligned16(v_new) ||
            !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o_base) || !aligned16(o_out))
            return fail(ORTHROS_EINVAL, "element tensors must be 16-byte aligned");
    }
    const DecodeLayout lay = decode_layout(B, Hq, Hkv, d, max_pages, page_size, dtype);
    if (!workspace || workspace_bytes < lay.total)
        return fail(ORTHROS_EWORKSPACE, "workspace needs %zu bytes, got %zu", lay.total,
                    workspace ? workspace_bytes : (size_t)0);
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(ORTHROS_EINVAL, "workspace must be 256-byte aligned");
    uint32_t *status = static_cast<uint32_t *>(workspace);
    cudaError_t e = cudaMemsetAsync(status, 0, sizeof(uint32_t), stream);
    if (e != cudaSuccess) return cuda_fail(e, "status reset");
    if (B == 0) return ORTHROS_OK;

    {
        ProfScope ps("decode_append", stream);
        e = launch_decode_append(k_new, v_new, k_cache, v_cache, block_table, cache_lens, B, Hkv, d, max_pages,
                                 page_size, num_pages, elem_bytes(dtype), status, stream);
    }
    if (e != cudaSuccess) return cuda_fail(e, "append launch");

    const int g = Hq / Hkv;
    const int groups = decode_groups(B, Hq, Hkv, page_size);
    if (dtype == ORTHROS_BF16 && groups > 0) {
        // both rows of every query head of a kv group share one pass over the
        // cache; groups of more than 8 query heads read it once per row kind
        // (the base rows only their window)
        SplitParams sp{};
        sp.mode = groups == B * Hkv ? kSplitDecode : kSplitDecodeSplit;
        sp.q = static_cast<const __nv_bfloat16 *>(q);
        sp.q_out = static_cast<const __nv_bfloat16 *>(q_out);
        sp.k = static_cast<const __nv_bfloat16 *>(k_cache);
        sp.v = static_cast<const __nv_bfloat16 *>(v_cache);
        sp.alpha_base = alpha_base;
        sp.beta_base = beta_base;
        sp.alpha_out = alpha_out;
        sp.beta_out = beta_out;
        sp.block_table = block_table;
        sp.cache_lens = cache_lens;
        sp.max_pages = max_pages;
        sp.page_size = page_size;
        sp.num_pages = num_pages;
        sp.B = B;
        sp.Hq = Hq;
        sp.Hkv = Hkv;
        sp.window = window;
        sp.scale = scale;
        sp.scale_log2 = scale * 1.4426950408889634f;
        sp.n_groups = groups;
        sp.chunk = lay.chunk;
        sp.max_chunks = lay.max_chunks;
        sp.kv_tokens = (long long)num_pages * page_size;
        sp.partial = reinterpret_cast<float *>(static_cast<char *>(workspace) + lay.part_off);
        sp.o_base = static_cast<__nv_bfloat16 *>(o_base);
        sp.lse_base = lse_base;
        sp.o_out = static_cast<__nv_bfloat16 *>(o_out);
        sp.lse_out = lse_out;
        sp.status = status;
        ProfScope ps("splitkv_decode", stream);
        e = launch_splitkv(sp, d, sp.mode == kSplitDecode ? 2 * g : g, stream);
        if (e != cudaSuccess) return cuda_fail(e, "split-KV decode launch");
        return ORTHROS_OK;
    }

    RowsArgs a{};
    a.q = q;
    a.q_out = q_out;
    a.k = k_cache;
    a.v = v_cache;
    a.alpha_base = alpha_base;
    a.beta_base = beta_base;
    a.alpha_out = alpha_out;
    a.beta_out = beta_out;
    a.block_table = block_table;
    a.cache_lens = cache_lens;
    a.max_pages = max_pages;
    a.page_size = page_size;
    a.num_pages = num_pages;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.window = window;
    a.scale = scale;
    a.o_base = o_base;
    a.lse_base = lse_base;
    a.o_out = o_out;
    a.lse_out = lse_out;
    a.status = status;
    {
        ProfScope ps("rows_simt_decode", stream);
        e = launch_rows_simt(a, kDecodePair, d, dtype, stream);
    }
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    return ORTHROS_OK;
}

orthros_status orthros_check(const void *workspace, orthros_stream_t stream_, uint32_t *bits) {
    if (!workspace) return fail(ORTHROS_EINVAL, "workspace must not be NULL");
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    uint32_t word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, workspace, sizeof word, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "status read");
    if (bits) *bits = word;
    if (word & ORTHROS_DEV_TIMEOUT) return fail(ORTHROS_ETIMEOUT, "a kernel's bounded wait ran out (bits 0x%x)", word);
    if (word) return fail(ORTHROS_EDEVICE, "device status bits 0x%x", word);
    return ORTHROS_OK;
}

}  // extern "C"
