// orthros_api.cu -- the C ABI: argument checks, workspace carving, dispatch.
//
// Every entry point validates everything the host can see before the first
// launch, then enqueues its kernels on the caller's stream and returns. See
// include/orthros_attn.h for the contract of each call.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <string>

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

// Workspace regions of orthros_prefill.
struct PrefillLayout {
    size_t indptr_off, total;
};

PrefillLayout prefill_layout(int B) {
    PrefillLayout L{};
    size_t at = kStatusBytes;
    L.indptr_off = at;
    at += align_up(sizeof(int32_t) * (size_t)(B + 1), 256);
    L.total = at;
    return L;
}

struct DecodeLayout {
    size_t total;
};

DecodeLayout decode_layout() {
    DecodeLayout L{};
    L.total = kStatusBytes;
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

}  // namespace
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
    return prefill_layout(B).total;
}

orthros_status orthros_prefill(const void *q, const void *k, const void *v, const float *alpha_base,
                               const float *beta_base, const float *alpha_out, const float *beta_out,
                               const int32_t *out_indptr, const int32_t *out_positions, int n_out,
                               const void *q_out, int B, int T, int Hq, int Hkv, int d, int window,
                               float scale, orthros_dtype dtype, void *o_base, float *lse_base,
                               void *o_out, float *lse_out, void *k_cache, void *v_cache,
                               const int32_t *block_table, int max_pages, int page_size, int num_pages,
                               void *workspace, size_t workspace_bytes, orthros_stream_t stream_) {
    g_last_error.clear();
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    orthros_status st = check_shapes(B, Hq, Hkv, d, window, scale, dtype);
    if (st != ORTHROS_OK) return st;
    if (T < 0) return fail(ORTHROS_EINVAL, "T = %d must be >= 0", T);
    if (n_out < 0) return fail(ORTHROS_EINVAL, "n_out = %d must be >= 0", n_out);
    const long long rows = (long long)B * T;
    if (rows > (1LL << 31)) return fail(ORTHROS_EUNSUPPORTED, "B*T = %lld tokens exceeds 2^31", rows);
    if (rows > 0) {
        if (!q || !k || !v) return fail(ORTHROS_EINVAL, "q, k and v must not be NULL");
        if (!alpha_base || !beta_base) return fail(ORTHROS_EINVAL, "alpha_base and beta_base must not be NULL");
        if (!o_base || !lse_base) return fail(ORTHROS_EINVAL, "o_base and lse_base must not be NULL");
        if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o_base))
            return fail(ORTHROS_EINVAL, "q, k, v and o_base must be 16-byte aligned");
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
        if (!o_out || !lse_out) return fail(ORTHROS_EINVAL, "o_out and lse_out must not be NULL when n_out > 0");
        if (!aligned16(o_out) || (q_out && !aligned16(q_out)))
            return fail(ORTHROS_EINVAL, "o_out and q_out must be 16-byte aligned");
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
    const PrefillLayout lay = prefill_layout(B);
    if (!workspace || workspace_bytes < lay.total)
        return fail(ORTHROS_EWORKSPACE, "workspace needs %zu bytes, got %zu", lay.total,
                    workspace ? workspace_bytes : (size_t)0);
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(ORTHROS_EINVAL, "workspace must be 256-byte aligned");

    char *ws = static_cast<char *>(workspace);
    uint32_t *status = reinterpret_cast<uint32_t *>(ws);
    cudaError_t e = cudaMemsetAsync(status, 0, sizeof(uint32_t), stream);
    if (e != cudaSuccess) return cuda_fail(e, "status reset");
    if (rows == 0) return ORTHROS_OK;

    int32_t *indptr_dev = reinterpret_cast<int32_t *>(ws + lay.indptr_off);
    if (n_out > 0) {
        e = cudaMemcpyAsync(indptr_dev, out_indptr, sizeof(int32_t) * (size_t)(B + 1), cudaMemcpyHostToDevice,
                            stream);
        if (e != cudaSuccess) return cuda_fail(e, "out_indptr upload");
    }

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
    if (n_out > 0) {
        ProfScope ps("rows_simt_out", stream);
        e = launch_rows_simt(a, kPrefillOut, d, dtype, stream);
        if (e != cudaSuccess) return cuda_fail(e, "output-stream launch");
    }
    return ORTHROS_OK;
}

size_t orthros_decode_workspace_size(int B, int Hq, int Hkv, int d, int max_pages, int page_size,
                                     orthros_dtype dtype) {
    if (max_pages < 1 || page_size < 1) return 0;
    if (check_shapes(B, Hq, Hkv, d, 1, 1.0f, dtype) != ORTHROS_OK) return 0;
    return decode_layout().total;
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
        if (!o_base || !lse_base || !o_out || !lse_out)
            return fail(ORTHROS_EINVAL, "outputs must not be NULL");
        if (!aligned16(q) || (q_out && !aligned16(q_out)) || !aligned16(k_new) || !aligned16(v_new) ||
            !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o_base) || !aligned16(o_out))
            return fail(ORTHROS_EINVAL, "element tensors must be 16-byte aligned");
    }
    const DecodeLayout lay = decode_layout();
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
