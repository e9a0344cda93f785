// simt_rows.cu -- generic one-warp-per-row attention (CUDA cores, fp32 math).
//
// Serves every row kind of the Orthros hot path for any element type:
//   prefill base rows   (Sec. 3.1 Eq. 4: keys max(0, t-w+1) .. t)
//   prefill output rows (Sec. 3.1 Eq. 5: keys 0 .. t)
//   decoding pairs      (Sec. 3.2 "Decoding": base row over the window, output
//                        row over the whole paged history, after the append)
// It is the fp32 path (no tensor cores: the fp32 contract is tighter than
// tf32 allows) and the bf16 path for shapes the tensor-core kernels do not
// take. The affine q = alpha (.) q_raw + beta is applied in registers as the
// query row is loaded (Alg. 1 line 5) and never written back.
//
// A warp owns one (row, head): lane l holds channels [l*E, l*E+E) of the query
// and of the output accumulator (E = d/32). Keys are visited in order with an
// online softmax; each logit is a warp-shuffle reduction of the lanes' partial
// dot products.
#include "internal.cuh"

namespace orthros {
namespace {

template <typename T, int E> struct Vec;
template <> struct Vec<float, 2> { using type = float2; };
template <> struct Vec<float, 4> { using type = float4; };
template <> struct Vec<__nv_bfloat16, 2> { using type = __nv_bfloat162; };
template <> struct Vec<__nv_bfloat16, 4> { using type = uint2; };

template <typename T, int E>
__device__ __forceinline__ void load_vec(const T *p, float (&x)[E]) {
    if constexpr (sizeof(T) == 4) {
        const typename Vec<T, E>::type r = *reinterpret_cast<const typename Vec<T, E>::type *>(p);
        const float *f = reinterpret_cast<const float *>(&r);
#pragma unroll
        for (int e = 0; e < E; ++e) x[e] = f[e];
    } else {
        const typename Vec<T, E>::type r = *reinterpret_cast<const typename Vec<T, E>::type *>(p);
        const __nv_bfloat16 *h = reinterpret_cast<const __nv_bfloat16 *>(&r);
#pragma unroll
        for (int e = 0; e < E; ++e) x[e] = __bfloat162float(h[e]);
    }
}

template <typename T, int E>
__device__ __forceinline__ void store_vec(T *p, const float (&x)[E]) {
#pragma unroll
    for (int e = 0; e < E; ++e) p[e] = from_f32<T>(x[e]);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Token j of one K/V head: contiguous [B,T,Hkv,d] (prefill) or paged (decode).
struct KeyAddr {
    const int32_t *bt;  // block-table row of this sequence, nullptr when contiguous
    long long base;     // element offset of token 0 (contiguous) / head offset (paged)
    long long tok_stride;
    int page_size;
    int num_pages;
    __device__ __forceinline__ long long at(int j, bool &ok) const {
        if (!bt) return base + (long long)j * tok_stride;
        const int pg = bt[j / page_size];
        ok = ok && pg >= 0 && pg < num_pages;
        const int pgc = pg < 0 ? 0 : (pg >= num_pages ? num_pages - 1 : pg);
        return base + ((long long)pgc * page_size + j % page_size) * tok_stride;
    }
};

template <typename T, int D>
__global__ void __launch_bounds__(256) rows_simt_kernel(RowsArgs a, int kind, long long n_units) {
    constexpr int E = D / 32;
    const int lane = threadIdx.x & 31;
    const long long unit = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (unit >= n_units) return;
    const int g = a.Hq / a.Hkv;

    int b, h, t, lo, hi;
    const T *qrow;
    const float *alpha, *beta;
    T *orow;
    float *lse_ptr;
    KeyAddr ka{};
    ka.tok_stride = (long long)a.Hkv * D;

    if (kind == kPrefillBase) {
        h = (int)(unit % a.Hq);
        t = (int)((unit / a.Hq) % a.T);
        b = (int)(unit / ((long long)a.Hq * a.T));
        const long long row = ((long long)b * a.T + t) * a.Hq + h;
        qrow = reinterpret_cast<const T *>(a.q) + row * D;
        orow = reinterpret_cast<T *>(a.o_base) + row * D;
        lse_ptr = a.lse_base + ((long long)b * a.Hq + h) * a.T + t;
        alpha = a.alpha_base + (long long)h * D;
        beta = a.beta_base + (long long)h * D;
        lo = max(0, t - a.window + 1);
        hi = t;
        ka.base = (long long)b * a.T * a.Hkv * D + (long long)(h / g) * D;
    } else if (kind == kPrefillOut) {
        h = (int)(unit % a.Hq);
        const int r = (int)(unit / a.Hq);
        int lo_b = 0, hi_b = a.B - 1;  // sequence of row r: last b with indptr[b] <= r
        while (lo_b < hi_b) {
            const int mid = (lo_b + hi_b + 1) >> 1;
            if (a.out_indptr[mid] <= r) lo_b = mid; else hi_b = mid - 1;
        }
        b = lo_b;
        t = a.out_positions[r];
        orow = reinterpret_cast<T *>(a.o_out) + ((long long)r * a.Hq + h) * D;
        lse_ptr = a.lse_out + (long long)r * a.Hq + h;
        if (t < 0 || t >= a.T) {
            set_status(a.status, ORTHROS_DEV_BAD_POSITION);
            float nanv[E];
#pragma unroll
            for (int e = 0; e < E; ++e) nanv[e] = __int_as_float(0x7fc00000);
            store_vec<T, E>(orow + lane * E, nanv);
            if (lane == 0) *lse_ptr = __int_as_float(0x7fc00000);
            return;
        }
        qrow = a.q_out ? reinterpret_cast<const T *>(a.q_out) + ((long long)r * a.Hq + h) * D
                       : reinterpret_cast<const T *>(a.q) + (((long long)b * a.T + t) * a.Hq + h) * D;
        alpha = a.alpha_out + (long long)h * D;
        beta = a.beta_out + (long long)h * D;
        lo = 0;
        hi = t;
        ka.base = (long long)b * a.T * a.Hkv * D + (long long)(h / g) * D;
    } else if (kind == kExtendBase || kind == kExtendOut) {
        // unit = (row, h): rows are new tokens (base) or output rows
        h = (int)(unit % a.Hq);
        const int r = (int)(unit / a.Hq);
        const int32_t *ip = kind == kExtendBase ? a.new_indptr : a.out_indptr;
        int lo_b = 0, hi_b = a.B - 1;  // sequence of row r
        while (lo_b < hi_b) {
            const int mid = (lo_b + hi_b + 1) >> 1;
            if (ip[mid] <= r) lo_b = mid; else hi_b = mid - 1;
        }
        b = lo_b;
        const int L = a.cache_lens[b];
        const int len = L + (a.new_indptr[b + 1] - a.new_indptr[b]);
        const long long row = (long long)r * a.Hq + h;
        const bool base = kind == kExtendBase;
        orow = reinterpret_cast<T *>(base ? a.o_base : a.o_out) + row * D;
        lse_ptr = (base ? a.lse_base : a.lse_out) + row;
        t = base ? L + (r - a.new_indptr[b]) : a.out_positions[r];
        const bool bad_len = L < 0 || (long long)len > (long long)a.max_pages * a.page_size;
        const bool bad_pos = !base && (t < 0 || t >= len || (!a.q_out && t < L));
        if (bad_len || bad_pos) {
            set_status(a.status, bad_len ? ORTHROS_DEV_BAD_LENGTH : ORTHROS_DEV_BAD_POSITION);
            float nanv[E];
#pragma unroll
            for (int e = 0; e < E; ++e) nanv[e] = __int_as_float(0x7fc00000);
            store_vec<T, E>(orow + lane * E, nanv);
            if (lane == 0) *lse_ptr = __int_as_float(0x7fc00000);
            return;
        }
        if (base) qrow = reinterpret_cast<const T *>(a.q) + row * D;
        else if (a.q_out) qrow = reinterpret_cast<const T *>(a.q_out) + row * D;
        else qrow = reinterpret_cast<const T *>(a.q) + ((long long)(a.new_indptr[b] + t - L) * a.Hq + h) * D;
        alpha = (base ? a.alpha_base : a.alpha_out) + (long long)h * D;
        beta = (base ? a.beta_base : a.beta_out) + (long long)h * D;
        lo = base ? max(0, t - a.window + 1) : 0;
        hi = t;
        ka.bt = a.block_table + (long long)b * a.max_pages;
        ka.page_size = a.page_size;
        ka.num_pages = a.num_pages;
        ka.base = (long long)(h / g) * D;
    } else {  // decoding pair: unit = (b, h, stream)
        const int stream = (int)(unit & 1);
        h = (int)((unit >> 1) % a.Hq);
        b = (int)((unit >> 1) / a.Hq);
        const long long row = (long long)b * a.Hq + h;
        const int L = a.cache_lens[b];
        const bool base = stream == 0;
        orow = reinterpret_cast<T *>(base ? a.o_base : a.o_out) + row * D;
        lse_ptr = (base ? a.lse_base : a.lse_out) + row;
        if (L < 0 || L / a.page_size >= a.max_pages) {
            set_status(a.status, ORTHROS_DEV_BAD_LENGTH);
            float nanv[E];
#pragma unroll
            for (int e = 0; e < E; ++e) nanv[e] = __int_as_float(0x7fc00000);
            store_vec<T, E>(orow + lane * E, nanv);
            if (lane == 0) *lse_ptr = __int_as_float(0x7fc00000);
            return;
        }
        const void *qsrc = (!base && a.q_out) ? a.q_out : a.q;
        qrow = reinterpret_cast<const T *>(qsrc) + row * D;
        alpha = (base ? a.alpha_base : a.alpha_out) + (long long)h * D;
        beta = (base ? a.beta_base : a.beta_out) + (long long)h * D;
        lo = base ? max(0, L - a.window + 1) : 0;
        hi = L;
        t = L;
        ka.bt = a.block_table + (long long)b * a.max_pages;
        ka.page_size = a.page_size;
        ka.num_pages = a.num_pages;
        ka.base = (long long)(h / g) * D;
    }

    // Alg. 1 line 5: affine in fp32 as the row is loaded.
    float qa[E];
    load_vec<T, E>(qrow + lane * E, qa);
#pragma unroll
    for (int e = 0; e < E; ++e) qa[e] = fmaf(alpha[lane * E + e], qa[e], beta[lane * E + e]);

    const T *kbase = reinterpret_cast<const T *>(a.k);
    const T *vbase = reinterpret_cast<const T *>(a.v);
    float m = -INFINITY, l = 0.f, acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    bool ok = true;
    for (int j = lo; j <= hi; ++j) {
        const long long off = ka.at(j, ok);
        float kx[E], vx[E];
        load_vec<T, E>(kbase + off + lane * E, kx);
        load_vec<T, E>(vbase + off + lane * E, vx);
        float s = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) s = fmaf(qa[e], kx[e], s);
        s = warp_sum(s) * a.scale;
        const float m_new = fmaxf(m, s);
        const float corr = expf(m - m_new);
        const float p = expf(s - m_new);
        l = l * corr + p;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = fmaf(acc[e], corr, p * vx[e]);
        m = m_new;
    }
    if (!ok) {
        set_status(a.status, ORTHROS_DEV_BAD_PAGE);
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = __int_as_float(0x7fc00000);
        if (lane == 0) *lse_ptr = __int_as_float(0x7fc00000);
        store_vec<T, E>(orow + lane * E, acc);
        return;
    }
    const float inv = 1.f / l;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] *= inv;
    store_vec<T, E>(orow + lane * E, acc);
    if (lane == 0) *lse_ptr = m + logf(l);
}

template <typename T>
cudaError_t launch_t(const RowsArgs &a, RowKind kind, int d, cudaStream_t stream) {
    long long n_units;
    if (kind == kPrefillBase) n_units = (long long)a.B * a.T * a.Hq;
    else if (kind == kPrefillOut || kind == kExtendOut) n_units = (long long)a.n_out * a.Hq;
    else if (kind == kExtendBase) n_units = (long long)a.n_new * a.Hq;
    else n_units = (long long)a.B * a.Hq * 2;
    if (n_units == 0) return cudaSuccess;
    constexpr int kWarps = 8;
    const long long blocks = (n_units + kWarps - 1) / kWarps;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (d == 128)
        rows_simt_kernel<T, 128><<<(unsigned)blocks, kWarps * 32, 0, stream>>>(a, (int)kind, n_units);
    else
        rows_simt_kernel<T, 64><<<(unsigned)blocks, kWarps * 32, 0, stream>>>(a, (int)kind, n_units);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rows_simt(const RowsArgs &a, RowKind kind, int d, orthros_dtype dtype,
                             cudaStream_t stream) {
    return dtype == ORTHROS_F32 ? launch_t<float>(a, kind, d, stream)
                                : launch_t<__nv_bfloat16>(a, kind, d, stream);
}

}  // namespace orthros
