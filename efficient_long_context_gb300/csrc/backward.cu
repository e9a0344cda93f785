// backward.cu -- gradients of the banded and cross rows: the CUDA-core path
// and the pre/post passes of the tensor-core path (backward_tc.cu).
//
// The backward of Sec. 3.1 Eq. 4 (every position t over keys max(0,t-w+1)..t)
// and Eq. 5 (every output row at position t_r over keys 0..t_r), both behind
// the query affine q = alpha (.) q_raw + beta (Alg. 1 line 5). With the
// forward's log-sum-exp L and D = dO . o of each row, each (row, key) pair
// contributes
//   p  = exp(scale * qa . k - L)
//   ds = p * (dO . v - D)
//   dv_key += p * dO,   dk_key += scale * ds * qa,   dqa_row += scale * ds * k
// and, through the affine, dq_raw = alpha (.) dqa, dalpha += dqa (.) q_raw,
// dbeta += dqa. Output rows that read q at their own position (no separate
// q_out) add their dq_raw into that position's dq.
//
// CUDA-core path (any element type, fp32 arithmetic):
//   delta kernel  one warp per row: D = dO . o
//   dk/dv kernel  one warp per (sequence, kv head, key): walks every query
//                 row of the group's heads that sees the key, in both streams;
//                 each key's dk and dv are written once, no atomics
//   dq kernel     one warp per (row, head): walks the row's keys; a block of 8
//                 warps shares one head and reduces its affine gradients in
//                 shared memory before one atomic add per channel
// Lane l holds channels [l*E, l*E+E), E = d/32, of every row it touches.
//
// Tensor-core path (bf16, d = 64 or 128): the delta kernel also writes qa in bf16,
// backward_tc.cu computes dk, dv and accumulates dqa in fp32, and the dq
// kernel (FromAcc) applies the affine and reduces the affine gradients.
#include "internal.cuh"

namespace orthros {
namespace {

constexpr int kWarps = 8;

// E consecutive elements of this lane as one vector load (E = 2 or 4).
template <typename T, int E>
__device__ __forceinline__ void ld(const T *p, float (&x)[E]) {
    if constexpr (sizeof(T) == 4) {
        if constexpr (E == 4) {
            const float4 r = *reinterpret_cast<const float4 *>(p);
            x[0] = r.x; x[1] = r.y; x[2] = r.z; x[3] = r.w;
        } else {
            const float2 r = *reinterpret_cast<const float2 *>(p);
            x[0] = r.x; x[1] = r.y;
        }
    } else {
        if constexpr (E == 4) {
            const uint2 r = *reinterpret_cast<const uint2 *>(p);
            const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162 *>(&r.x);
            const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&r.y);
            x[0] = __low2float(a); x[1] = __high2float(a); x[2] = __low2float(b); x[3] = __high2float(b);
        } else {
            const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162 *>(p);
            x[0] = __low2float(a); x[1] = __high2float(a);
        }
    }
}

template <typename T, int E>
__device__ __forceinline__ void st(T *p, const float (&x)[E]) {
    if constexpr (sizeof(T) == 4) {
        if constexpr (E == 4) *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
        else *reinterpret_cast<float2 *>(p) = make_float2(x[0], x[1]);
    } else {
        const __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]);
        if constexpr (E == 4) {
            const __nv_bfloat162 b = __floats2bfloat162_rn(x[2], x[3]);
            uint2 r;
            r.x = *reinterpret_cast<const uint32_t *>(&a);
            r.y = *reinterpret_cast<const uint32_t *>(&b);
            *reinterpret_cast<uint2 *>(p) = r;
        } else {
            *reinterpret_cast<__nv_bfloat162 *>(p) = a;
        }
    }
}

__device__ __forceinline__ float wsum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

template <int E>
__device__ __forceinline__ float dot(const float (&a)[E], const float (&b)[E]) {
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) s = fmaf(a[e], b[e], s);
    return s;
}

// Sequence of output row r: the last b with indptr[b] <= r.
__device__ __forceinline__ int seq_of_row(const int32_t *indptr, int B, int r) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (indptr[mid] <= r) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// D = dO . o of every row; with WriteQa (bf16 tensor-core path) also the
// affined query of the row, qa = alpha (.) q_raw + beta, rounded to bf16.
template <typename T, int D, bool WriteQa>
__global__ void __launch_bounds__(256) bwd_delta_kernel(BwdArgs a, long long n_base) {
    constexpr int E = D / 32;
    const int lane = threadIdx.x & 31;
    const long long unit = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
    const long long n_units = n_base + (long long)a.n_out * a.Hq;
    if (unit >= n_units) return;
    float o[E], dO[E];
    if (unit < n_base) {  // unit = (b, t, h) in [B,T,Hq] order
        const int h = (int)(unit % a.Hq);
        const long long bt = unit / a.Hq;
        const int t = (int)(bt % a.T), b = (int)(bt / a.T);
        ld<T, E>(static_cast<const T *>(a.o_base) + unit * D + lane * E, o);
        ld<T, E>(static_cast<const T *>(a.do_base) + unit * D + lane * E, dO);
        const float s = wsum(dot<E>(o, dO));
        if (lane == 0) a.delta_base[((long long)b * a.Hq + h) * a.T + t] = s;
        if constexpr (WriteQa) {
            float q[E], al[E], be[E];
            ld<T, E>(static_cast<const T *>(a.q) + unit * D + lane * E, q);
            ld<float, E>(a.alpha_base + h * D + lane * E, al);
            ld<float, E>(a.beta_base + h * D + lane * E, be);
#pragma unroll
            for (int e = 0; e < E; ++e) q[e] = fmaf(al[e], q[e], be[e]);
            st<__nv_bfloat16, E>(a.qa_base + unit * D + lane * E, q);
        }
    } else {
        const long long u = unit - n_base;  // (r, h)
        ld<T, E>(static_cast<const T *>(a.o_out) + u * D + lane * E, o);
        ld<T, E>(static_cast<const T *>(a.do_out) + u * D + lane * E, dO);
        const float s = wsum(dot<E>(o, dO));
        if (lane == 0) a.delta_out[u] = s;
        if constexpr (WriteQa) {
            const int h = (int)(u % a.Hq), r = (int)(u / a.Hq);
            float q[E], al[E], be[E];
#pragma unroll
            for (int e = 0; e < E; ++e) q[e] = 0.f;
            bool ok = true;
            if (a.q_out) {
                ld<T, E>(static_cast<const T *>(a.q_out) + u * D + lane * E, q);
            } else {
                const int b = seq_of_row(a.out_indptr, a.B, r);
                const int t = a.out_positions[r];
                ok = t >= 0 && t < a.T;  // bad positions are flagged (and masked) elsewhere
                if (ok) ld<T, E>(static_cast<const T *>(a.q) + (((long long)b * a.T + t) * a.Hq + h) * D + lane * E, q);
            }
            ld<float, E>(a.alpha_out + h * D + lane * E, al);
            ld<float, E>(a.beta_out + h * D + lane * E, be);
#pragma unroll
            for (int e = 0; e < E; ++e) q[e] = ok ? fmaf(al[e], q[e], be[e]) : 0.f;
            st<__nv_bfloat16, E>(a.qa_out + u * D + lane * E, q);
        }
    }
}

// omax[r] = largest position among output rows r .. r+63 of r's sequence: the
// tensor-core kernel skips a 64-row tile whose largest position precedes its keys.
__global__ void bwd_omax_kernel(BwdArgs a) {
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= a.n_out) return;
    const int b = seq_of_row(a.out_indptr, a.B, r);
    const int end = min(r + 64, a.out_indptr[b + 1]);
    int m = -1;
    for (int i = r; i < end; ++i) m = max(m, a.out_positions[i]);
    a.omax[r] = m;
}

// Threads the output rows of each position into a list (positions may repeat):
// pos_head[b*T + t] is the first row at (b, t), row_next[r] the next one, -1 ends.
__global__ void bwd_row_lists_kernel(BwdArgs a) {
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= a.n_out) return;
    const int b = seq_of_row(a.out_indptr, a.B, r);
    const int t = a.out_positions[r];
    if (t < 0 || t >= a.T) {
        set_status(a.status, ORTHROS_DEV_BAD_POSITION);
        a.row_next[r] = -1;
        return;
    }
    a.row_next[r] = atomicExch(a.pos_head + (long long)b * a.T + t, r);
}

// One (row, key) pair seen from the key's side: accumulates dv and dk (unscaled).
template <int E>
__device__ __forceinline__ void key_pair(const float (&k)[E], const float (&v)[E], const float (&qa)[E],
                                         const float (&dO)[E], float lse, float delta, float scale,
                                         float (&dk)[E], float (&dv)[E]) {
    const float s = wsum(dot<E>(qa, k)) * scale;
    const float p = __expf(s - lse);
    const float dp = wsum(dot<E>(dO, v));
    const float ds = p * (dp - delta);
#pragma unroll
    for (int e = 0; e < E; ++e) {
        dv[e] = fmaf(p, dO[e], dv[e]);
        dk[e] = fmaf(ds, qa[e], dk[e]);
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(256) bwd_dkdv_kernel(BwdArgs a) {
    constexpr int E = D / 32;
    const int lane = threadIdx.x & 31;
    const long long unit = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);  // (b, j, kv)
    if (unit >= (long long)a.B * a.T * a.Hkv) return;
    const int kv = (int)(unit % a.Hkv);
    const long long bj = unit / a.Hkv;
    const int j = (int)(bj % a.T), b = (int)(bj / a.T);
    const int g = a.Hq / a.Hkv;
    float k[E], v[E], dk[E], dv[E];
    ld<T, E>(static_cast<const T *>(a.k) + unit * D + lane * E, k);
    ld<T, E>(static_cast<const T *>(a.v) + unit * D + lane * E, v);
#pragma unroll
    for (int e = 0; e < E; ++e) dk[e] = dv[e] = 0.f;
    const int t_hi = (int)min((long long)a.T - 1, (long long)j + a.window - 1);
    const int r0 = a.n_out ? a.out_indptr[b] : 0, r1 = a.n_out ? a.out_indptr[b + 1] : 0;
    for (int h = kv * g; h < (kv + 1) * g; ++h) {
        float al[E], be[E], qa[E], dO[E];
        ld<float, E>(a.alpha_base + h * D + lane * E, al);
        ld<float, E>(a.beta_base + h * D + lane * E, be);
        for (int t = j; t <= t_hi; ++t) {  // base rows that see key j
            const long long row = ((long long)b * a.T + t) * a.Hq + h;
            ld<T, E>(static_cast<const T *>(a.q) + row * D + lane * E, qa);
#pragma unroll
            for (int e = 0; e < E; ++e) qa[e] = fmaf(al[e], qa[e], be[e]);
            ld<T, E>(static_cast<const T *>(a.do_base) + row * D + lane * E, dO);
            const long long li = ((long long)b * a.Hq + h) * a.T + t;
            key_pair<E>(k, v, qa, dO, a.lse_base[li], a.delta_base[li], a.scale, dk, dv);
        }
        if (r1 > r0) {
            ld<float, E>(a.alpha_out + h * D + lane * E, al);
            ld<float, E>(a.beta_out + h * D + lane * E, be);
        }
        for (int r = r0; r < r1; ++r) {  // output rows at positions >= j
            const int t = a.out_positions[r];
            if (t < j || t >= a.T) continue;
            const long long ro = (long long)r * a.Hq + h;
            const T *qraw = a.q_out ? static_cast<const T *>(a.q_out) + ro * D
                                    : static_cast<const T *>(a.q) + (((long long)b * a.T + t) * a.Hq + h) * D;
            ld<T, E>(qraw + lane * E, qa);
#pragma unroll
            for (int e = 0; e < E; ++e) qa[e] = fmaf(al[e], qa[e], be[e]);
            ld<T, E>(static_cast<const T *>(a.do_out) + ro * D + lane * E, dO);
            key_pair<E>(k, v, qa, dO, a.lse_out[ro], a.delta_out[ro], a.scale, dk, dv);
        }
    }
#pragma unroll
    for (int e = 0; e < E; ++e) dk[e] *= a.scale;
    st<T, E>(static_cast<T *>(a.dk) + unit * D + lane * E, dk);
    st<T, E>(static_cast<T *>(a.dv) + unit * D + lane * E, dv);
}

// kind 0: base rows, grid (ceil(T/(8 RPW)), Hq, B); kind 1: output rows,
// grid (ceil(n_out/(8 RPW)), Hq). Each warp handles RPW rows of one head and
// keeps its share of the affine gradients in registers; the block reduces
// them once. FromAcc: dqa (scale included) was accumulated by the tensor-core
// kernel (dq_acc for base rows, dq_rows for output rows); only the affine
// step and the affine gradients remain.
template <typename T, int D, bool FromAcc, int RPW>
__global__ void __launch_bounds__(256) bwd_dq_kernel(BwdArgs a, int kind) {
    constexpr int E = D / 32;
    __shared__ float red[2][kWarps][D];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int h = blockIdx.y;
    const int kv = h / (a.Hq / a.Hkv);
    float acc_a[E], acc_b[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc_a[e] = acc_b[e] = 0.f;
    const float *alpha = kind == 0 ? a.alpha_base : a.alpha_out;
    const float *beta = kind == 0 ? a.beta_base : a.beta_out;
    for (int it = 0; it < RPW; ++it) {
    const int row_id = (blockIdx.x * RPW + it) * kWarps + warp;
    float dqa[E], qraw[E];
#pragma unroll
    for (int e = 0; e < E; ++e) dqa[e] = qraw[e] = 0.f;
    int b = 0, t = -1, r = -1;
    bool active;
    if (kind == 0) {
        b = blockIdx.z;
        t = row_id;
        active = t < a.T;
    } else {
        r = row_id;
        active = r < a.n_out;
        if (active) {
            b = seq_of_row(a.out_indptr, a.B, r);
            t = a.out_positions[r];
            if (t < 0 || t >= a.T) {
                set_status(a.status, ORTHROS_DEV_BAD_POSITION);
                float nanv[E];
#pragma unroll
                for (int e = 0; e < E; ++e) nanv[e] = __int_as_float(0x7fc00000);
                const long long ro = (long long)r * a.Hq + h;
                if (a.q_out) st<T, E>(static_cast<T *>(a.dq_out) + ro * D + lane * E, nanv);
                else st<float, E>(a.dq_rows + ro * D + lane * E, nanv);
                active = false;
            }
        }
    }
    if (active) {
        float al[E], be[E];
        [[maybe_unused]] float qa[E], dO[E], k[E], v[E];
        ld<float, E>(alpha + h * D + lane * E, al);
        ld<float, E>(beta + h * D + lane * E, be);
        const long long row = ((long long)b * a.T + t) * a.Hq + h;
        const long long ro = (long long)r * a.Hq + h;
        const T *qp = (kind == 1 && a.q_out) ? static_cast<const T *>(a.q_out) + ro * D
                                             : static_cast<const T *>(a.q) + row * D;
        ld<T, E>(qp + lane * E, qraw);
        if constexpr (FromAcc) {
            ld<float, E>((kind == 0 ? a.dq_acc + row * D : a.dq_rows + ro * D) + lane * E, dqa);
        } else {
#pragma unroll
        for (int e = 0; e < E; ++e) qa[e] = fmaf(al[e], qraw[e], be[e]);
        float lse, delta;
        if (kind == 0) {
            ld<T, E>(static_cast<const T *>(a.do_base) + row * D + lane * E, dO);
            const long long li = ((long long)b * a.Hq + h) * a.T + t;
            lse = a.lse_base[li];
            delta = a.delta_base[li];
        } else {
            ld<T, E>(static_cast<const T *>(a.do_out) + ro * D + lane * E, dO);
            lse = a.lse_out[ro];
            delta = a.delta_out[ro];
        }
        const int lo = kind == 0 ? max(0, t - a.window + 1) : 0;
        const T *kb = static_cast<const T *>(a.k) + ((long long)b * a.T * a.Hkv + kv) * D + lane * E;
        const T *vb = static_cast<const T *>(a.v) + ((long long)b * a.T * a.Hkv + kv) * D + lane * E;
        for (int j = lo; j <= t; ++j) {
            ld<T, E>(kb + (long long)j * a.Hkv * D, k);
            ld<T, E>(vb + (long long)j * a.Hkv * D, v);
            const float s = wsum(dot<E>(qa, k)) * a.scale;
            const float p = __expf(s - lse);
            const float dp = wsum(dot<E>(dO, v));
            const float ds = p * (dp - delta);
#pragma unroll
            for (int e = 0; e < E; ++e) dqa[e] = fmaf(ds, k[e], dqa[e]);
        }
#pragma unroll
        for (int e = 0; e < E; ++e) dqa[e] *= a.scale;
        }
        float dq[E];
#pragma unroll
        for (int e = 0; e < E; ++e) dq[e] = al[e] * dqa[e];
        if (kind == 0) {
            // output rows at this position that read this q add their share
            int rr = (a.q_out || a.n_out == 0) ? -1 : a.pos_head[(long long)b * a.T + t];
            for (int guard = 0; rr >= 0 && rr < a.n_out && guard < a.n_out; ++guard) {
                float add[E];
                ld<float, E>(a.dq_rows + ((long long)rr * a.Hq + h) * D + lane * E, add);
#pragma unroll
                for (int e = 0; e < E; ++e) dq[e] += add[e];
                rr = a.row_next[rr];
            }
            st<T, E>(static_cast<T *>(a.dq) + row * D + lane * E, dq);
        } else if (a.q_out) {
            st<T, E>(static_cast<T *>(a.dq_out) + ro * D + lane * E, dq);
        } else {
            st<float, E>(a.dq_rows + ro * D + lane * E, dq);
        }
    }
#pragma unroll
    for (int e = 0; e < E; ++e) {
        acc_a[e] = fmaf(dqa[e], qraw[e], acc_a[e]);  // zero for inactive rows
        acc_b[e] += dqa[e];
    }
    }
#pragma unroll
    for (int e = 0; e < E; ++e) {
        red[0][warp][lane * E + e] = acc_a[e];
        red[1][warp][lane * E + e] = acc_b[e];
    }
    __syncthreads();
    float *ga = kind == 0 ? a.d_alpha_base : a.d_alpha_out;
    float *gb = kind == 0 ? a.d_beta_base : a.d_beta_out;
    for (int i = threadIdx.x; i < 2 * D; i += blockDim.x) {
        const int which = i / D, c = i % D;
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) s += red[which][w][c];
        atomicAdd((which ? gb : ga) + h * D + c, s);
    }
}

template <typename T, int D, bool Tc>
cudaError_t launch_t(const BwdArgs &a, cudaStream_t stream) {
    const long long n_base = (long long)a.B * a.T * a.Hq;
    const long long n_rows = n_base + (long long)a.n_out * a.Hq;
    cudaError_t e;
    if (a.n_out > 0) {
        {
            ProfScope ps("bwd_row_lists", stream);
            bwd_row_lists_kernel<<<(a.n_out + 255) / 256, 256, 0, stream>>>(a);
        }
        if constexpr (Tc) {
            ProfScope ps("bwd_omax", stream);
            bwd_omax_kernel<<<(a.n_out + 255) / 256, 256, 0, stream>>>(a);
        }
    }
    {
        ProfScope ps("bwd_prep", stream);
        bwd_delta_kernel<T, D, Tc><<<(unsigned)((n_rows + kWarps - 1) / kWarps), kWarps * 32, 0, stream>>>(a, n_base);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if constexpr (Tc) {
        if ((e = cudaMemsetAsync(a.dq_acc, 0, sizeof(float) * (size_t)n_base * D, stream)) != cudaSuccess) return e;
        if (a.n_out > 0 &&
            (e = cudaMemsetAsync(a.dq_rows, 0, sizeof(float) * (size_t)a.n_out * a.Hq * D, stream)) != cudaSuccess)
            return e;
        BwdTcParams tp{};
        tp.out_indptr = a.out_indptr;
        tp.out_positions = a.out_positions;
        tp.omax = a.omax;
        tp.lse_base = a.lse_base;
        tp.lse_out = a.lse_out;
        tp.delta_base = a.delta_base;
        tp.delta_out = a.delta_out;
        tp.dq_acc = a.dq_acc;
        tp.dq_out_acc = a.dq_rows;
        tp.dk = static_cast<__nv_bfloat16 *>(a.dk);
        tp.dv = static_cast<__nv_bfloat16 *>(a.dv);
        tp.B = a.B;
        tp.T = a.T;
        tp.Hq = a.Hq;
        tp.Hkv = a.Hkv;
        tp.window = a.window;
        tp.n_out = a.n_out;
        tp.nkb = (a.T + 127) / 128;
        tp.scale = a.scale;
        tp.scale_log2 = a.scale * 1.4426950408889634f;
        tp.status = a.status;
        ProfScope ps("bwd_tc", stream);
        e = launch_backward_tc(tp, D, a.k, a.v, a.qa_base, a.do_base, a.qa_out, a.do_out, stream);
    } else {
        ProfScope ps("bwd_dkdv_simt", stream);
        const long long n = (long long)a.B * a.T * a.Hkv;
        bwd_dkdv_kernel<T, D><<<(unsigned)((n + kWarps - 1) / kWarps), kWarps * 32, 0, stream>>>(a);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
    // the tensor-core path's finishing pass is light per row: 8 rows per warp
    constexpr int kRpw = Tc ? 8 : 1;
    constexpr int kRowsPerBlock = kWarps * kRpw;
    if (a.n_out > 0) {
        ProfScope ps(Tc ? "bwd_finish_out" : "bwd_dq_out_simt", stream);
        bwd_dq_kernel<T, D, Tc, kRpw><<<dim3((a.n_out + kRowsPerBlock - 1) / kRowsPerBlock, a.Hq), kWarps * 32, 0,
                                         stream>>>(a, 1);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    {
        ProfScope ps(Tc ? "bwd_finish" : "bwd_dq_simt", stream);
        bwd_dq_kernel<T, D, Tc, kRpw><<<dim3((a.T + kRowsPerBlock - 1) / kRowsPerBlock, a.Hq, a.B), kWarps * 32, 0,
                                         stream>>>(a, 0);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_backward(const BwdArgs &a, int d, orthros_dtype dtype, bool use_tc, cudaStream_t stream) {
    if (dtype == ORTHROS_F32)
        return d == 64 ? launch_t<float, 64, false>(a, stream) : launch_t<float, 128, false>(a, stream);
    if (use_tc) return d == 64 ? launch_t<__nv_bfloat16, 64, true>(a, stream) : launch_t<__nv_bfloat16, 128, true>(a, stream);
    return d == 64 ? launch_t<__nv_bfloat16, 64, false>(a, stream) : launch_t<__nv_bfloat16, 128, false>(a, stream);
}

}  // namespace orthros
