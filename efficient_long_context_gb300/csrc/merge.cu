// merge.cu -- exact merge of attention partials over disjoint key sets.
//
// Softmax attention of one query over a union of disjoint key sets S_1..S_P
// follows from each set's normalised result (o_p, lse_p) alone:
//   lse = log sum_p exp(lse_p),   o = sum_p exp(lse_p - lse) o_p,
// because exp(lse_p) is set p's share of the softmax denominator. A
// sequence-parallel prefill (Orthros paper, Sec. 4.5 and the appendix's
// training/inference setup: the 64K-1M-token prefills run on 8 GPUs) computes
// every output row's Eq. 5 as one partial per chunk of the token axis and
// merges them here. An empty partial (lse = -inf, o = 0) weighs nothing, and
// the merge of empty partials is again empty, so partials can be merged in
// any grouping.
#include "internal.cuh"

namespace orthros {
namespace {

// One warp per (row, head); lane c holds channels c, c + 32, ...
template <int D, bool F32>
__global__ void __launch_bounds__(256) merge_partials_kernel(const float *__restrict__ o_parts,
                                                             const float *__restrict__ lse_parts, int n_parts,
                                                             long long n_rh, void *o_out, float *lse_out) {
    const long long rh = blockIdx.x * 8LL + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (rh >= n_rh) return;
    float M = -INFINITY;
    for (int p = lane; p < n_parts; p += 32) M = fmaxf(M, lse_parts[p * n_rh + rh]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    constexpr int E = D / 32;
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    float lse = -INFINITY;
    if (M != -INFINITY) {
        float S = 0.f;
        for (int p = lane; p < n_parts; p += 32) S += expf(lse_parts[p * n_rh + rh] - M);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
        lse = M + logf(S);
        for (int p = 0; p < n_parts; ++p) {
            const float lp = lse_parts[p * n_rh + rh];
            if (lp == -INFINITY) continue;
            const float w = expf(lp - lse);
            const float *src = o_parts + (p * n_rh + rh) * D;
#pragma unroll
            for (int e = 0; e < E; ++e) acc[e] += w * src[lane + 32 * e];
        }
    }
#pragma unroll
    for (int e = 0; e < E; ++e) {
        if (F32) static_cast<float *>(o_out)[rh * D + lane + 32 * e] = acc[e];
        else static_cast<__nv_bfloat16 *>(o_out)[rh * D + lane + 32 * e] = __float2bfloat16_rn(acc[e]);
    }
    if (lane == 0) lse_out[rh] = lse;
}

template <int D>
cudaError_t launch_d(const float *o_parts, const float *lse_parts, int n_parts, long long n_rh, bool f32_out,
                     void *o_out, float *lse_out, cudaStream_t stream) {
    const long long blocks = (n_rh + 7) / 8;
    if (f32_out)
        merge_partials_kernel<D, true><<<(unsigned)blocks, 256, 0, stream>>>(o_parts, lse_parts, n_parts, n_rh, o_out,
                                                                             lse_out);
    else
        merge_partials_kernel<D, false><<<(unsigned)blocks, 256, 0, stream>>>(o_parts, lse_parts, n_parts, n_rh,
                                                                              o_out, lse_out);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_merge_partials(const float *o_parts, const float *lse_parts, int n_parts, int n_rows, int Hq, int d,
                                  bool f32_out, void *o_out, float *lse_out, cudaStream_t stream) {
    const long long n_rh = (long long)n_rows * Hq;
    if (n_rh == 0) return cudaSuccess;
    return d == 128 ? launch_d<128>(o_parts, lse_parts, n_parts, n_rh, f32_out, o_out, lse_out, stream)
                    : launch_d<64>(o_parts, lse_parts, n_parts, n_rh, f32_out, o_out, lse_out, stream);
}

}  // namespace orthros
