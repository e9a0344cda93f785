// project_tc.cu -- the shared Q/K/V projection that feeds the hot path, on
// the 5th-generation tensor cores, with the query affine and the paged-cache
// writes in the epilogue.
//
// What it computes (Orthros paper, Alg. 1 lines 4-5 and Sec. 3.1): the base
// tokens' hidden rows and the output tokens' hidden rows go through ONE
// Q/K/V weight, y = x W; the query part of each row gets its stream's affine
// (q = alpha (.) y_Q + beta), and the base tokens' K/V parts are the cache
// entries (the output stream never writes the cache). In decoding the base
// and output token of every sequence share one read of the weight.
//
// Design: a CTA computes a BM-row x BN-column tile of y (BN = 256, or 64 when
// there are few rows, so that enough CTAs stream the weight; BM = 128, or 64
// when the call has at most 64 rows). Warp 4 streams K slices of x and of the
// weight (stored K-major, one output column per row) with TMA, 128-byte
// swizzle, one, two or four 64-channel atoms per stage; warp 5 issues tcgen05.mma
// (M=BM, N=BN, K=16) into a TMEM accumulator; warps 0-3 read the accumulator
// 32 columns at a time (one thread per tile row), apply the affine to query
// columns, round to bf16 and store: queries to q_base / q_out, keys and values
// to k_out / v_out and/or straight into the row's page slot.
#include <cuda.h>

#include "ptx.cuh"

namespace orthros {

using namespace ptx;

namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;  // one 128-byte swizzle atom of bf16 along K
constexpr int kThreadsP = 192;
constexpr int kProducerWarpP = 4;
constexpr int kMmaWarpP = 5;

// KS = 128-byte swizzle atoms of K per stage (one stage = KS * 64 channels).
// BM = rows per tile: 128, or 64 when the whole call has at most 64 rows (a
// decoding step); an M=64 accumulator puts rows 16q .. 16q+15 in TMEM lanes
// 32q .. 32q+15, so epilogue warp q owns 16 rows in its lanes 0-15.
template <int BN, int KS, int BM> struct PCfg {
    static constexpr int kStages = (BN == 256 ? 4 : (BM == 64 ? 12 : 8)) / KS;
    static constexpr int kASub = BM * kBK * 2;   // 16 KB (8 KB) per atom
    static constexpr int kBSub = BN * kBK * 2;   // 32 KB or 8 KB per atom
    static constexpr int kABytes = KS * kASub;
    static constexpr int kBBytes = KS * kBSub;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kBar = kStages * kStageBytes;
    static constexpr int kSmem = kBar + 256 + 1024;
};

template <int BN, int KS, int BM>
__global__ void __launch_bounds__(kThreadsP, 1)
    project_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                      const ProjParams p) {
    using C = PCfg<BN, KS, BM>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::kBar);
    uint64_t *empty = full + C::kStages;
    uint64_t *acc_full = empty + C::kStages;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_full + 1);
    int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);
    volatile int *abort = abort_flag;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n0 = blockIdx.x * BN, m0 = blockIdx.y * BM;
    const int k_tiles = p.d_model / (kBK * KS);

    if (tid == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kProducerWarpP && lane == 0) {
        prefetch_tmap(&tm_x);
        prefetch_tmap(&tm_w);
    }
    __syncthreads();
    if (warp == kMmaWarpP) {
        tmem_alloc(tmem_slot, BN);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kProducerWarpP) {
        if (lane == 0) {
            int issued = 0;
            for (int kt = 0; kt < k_tiles; ++kt) {
                const int s = kt % C::kStages;
                if (kt >= C::kStages && !mbar_wait(&empty[s], ((kt / C::kStages) - 1) & 1, abort, p.status)) break;
                uint8_t *a = smem + s * C::kStageBytes;
                mbar_arrive_expect_tx(&full[s], C::kStageBytes);
#pragma unroll
                for (int j = 0; j < KS; ++j) {
                    tma_load_3d(a + j * C::kASub, &tm_x, &full[s], (kt * KS + j) * kBK, 0, m0);
                    tma_load_3d(a + C::kABytes + j * C::kBSub, &tm_w, &full[s], (kt * KS + j) * kBK, 0, n0);
                }
                issued = kt + 1;
            }
            // nothing may land in shared memory after the CTA exits
            for (int kt = issued > C::kStages ? issued - C::kStages : 0; kt < issued; ++kt)
                mbar_wait_drain(&full[kt % C::kStages], (kt / C::kStages) & 1, p.status);
        }
    } else if (warp == kMmaWarpP) {
        if (lane == 0) {
            constexpr uint32_t kId = idesc_f16(1, 1, 0, 0, BM, BN);
            const uint64_t da = desc_sw128(smem_u32(smem), 16, 1024);
            const uint64_t db = desc_sw128(smem_u32(smem + C::kABytes), 16, 1024);
            constexpr uint32_t kStageU = C::kStageBytes >> 4;
            for (int kt = 0; kt < k_tiles; ++kt) {
                const int s = kt % C::kStages;
                if (!mbar_wait(&full[s], (kt / C::kStages) & 1, abort, p.status)) break;
                tc_fence_after();
#pragma unroll
                for (int j = 0; j < KS; ++j)
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        mma_ss(tmem, da + s * kStageU + ((j * C::kASub + kk * 32) >> 4),
                               db + s * kStageU + ((j * C::kBSub + kk * 32) >> 4), kId,
                               (kt > 0 || j > 0 || kk > 0) ? 1u : 0u);
                tc_commit(&empty[s]);
            }
            tc_commit(acc_full);
            mbar_wait_drain(acc_full, 0, p.status);
        }
    } else {
        // ---------------- epilogue: thread = tile row ----------------
        const int r = m0 + warp * (BM / 4) + lane;
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        const bool got = mbar_wait_warp(acc_full, 0, abort, p.status);
        if (got) {
            tc_fence_after();
            const int Nq = p.Hq * p.d, Nkv = p.Hkv * p.d;
            const bool base = r < p.n_base;
            const bool live = lane < BM / 4 && r < p.n_base + p.n_out;
            // the page slot of a base row's K/V
            long long slot = -1;
            if (live && base && p.k_cache) {
                const int t = p.token_pos[r], b = p.token_seq[r];
                if (t >= 0 && t / p.page_size < p.max_pages && b >= 0 && b < p.B) {
                    const int pg = p.block_table[(long long)b * p.max_pages + t / p.page_size];
                    if (pg >= 0 && pg < p.num_pages) slot = (long long)pg * p.page_size + t % p.page_size;
                    else set_status(p.status, ORTHROS_DEV_BAD_PAGE);
                } else {
                    set_status(p.status, ORTHROS_DEV_BAD_POSITION);
                }
            }
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(tmem + lane_off + 32 * c, v);
                tmem_ld_wait();
                const int n = n0 + 32 * c;
                if (!live) continue;
                uint4 w[4];
                uint32_t *wp = reinterpret_cast<uint32_t *>(w);
                __nv_bfloat16 *dst = nullptr, *dst2 = nullptr;
                if (n < Nq) {
                    const float *al = (base ? p.alpha_base : p.alpha_out) + n;
                    const float *be = (base ? p.beta_base : p.beta_out) + n;
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        wp[e] = pack_bf16(fmaf(al[2 * e], __uint_as_float(v[2 * e]), be[2 * e]),
                                          fmaf(al[2 * e + 1], __uint_as_float(v[2 * e + 1]), be[2 * e + 1]));
                    dst = base ? p.q_base + (long long)r * Nq + n : p.q_out + (long long)(r - p.n_base) * Nq + n;
                } else if (base) {
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        wp[e] = pack_bf16(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
                    const bool is_k = n - Nq < Nkv;
                    const int off = is_k ? n - Nq : n - Nq - Nkv;
                    __nv_bfloat16 *plain = is_k ? p.k_out : p.v_out;
                    if (plain) dst = plain + (long long)r * Nkv + off;
                    __nv_bfloat16 *cache = is_k ? p.k_cache : p.v_cache;
                    if (cache && slot >= 0) dst2 = cache + slot * Nkv + off;
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (dst) reinterpret_cast<uint4 *>(dst)[e] = w[e];
                    if (dst2) reinterpret_cast<uint4 *>(dst2)[e] = w[e];
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarpP) {
        tc_fence_after();
        tmem_dealloc(tmem, BN);
    }
}

template <int BN, int KS, int BM>
cudaError_t launch_bn(const ProjParams &p, cudaStream_t stream) {
    using C = PCfg<BN, KS, BM>;
    CUtensorMap tx, tw;
    const int N = (p.Hq + 2 * p.Hkv) * p.d;
    if (!encode_kv_map_3d(&tx, p.x, (long long)p.n_base + p.n_out, 1, p.d_model, BM) ||
        !encode_kv_map_3d(&tw, p.w_t, N, 1, p.d_model, BN))
        return cudaErrorInvalidValue;
    static SmemLimit limit;
    if (cudaError_t e = limit.ensure((const void *)project_tc_kernel<BN, KS, BM>, C::kSmem); e != cudaSuccess)
        return e;
    const dim3 grid(N / BN, (p.n_base + p.n_out + BM - 1) / BM);
    project_tc_kernel<BN, KS, BM><<<grid, kThreadsP, C::kSmem, stream>>>(tx, tw, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_project_tc(const ProjParams &p, cudaStream_t stream) {
    const int N = (p.Hq + 2 * p.Hkv) * p.d;
    const long long m_tiles = ((long long)p.n_base + p.n_out + kBM - 1) / kBM;
    if (m_tiles == 0) return cudaSuccess;
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // wide tiles when they already fill the GPU, narrow ones for few rows
    if (N % 256 == 0 && m_tiles * (N / 256) >= sms) return launch_bn<256, 1, kBM>(p, stream);
    const bool k2 = p.d_model % (2 * kBK) == 0, k4 = p.d_model % (4 * kBK) == 0;
    // few rows: the weight streams as 512-byte runs of each of its rows per stage
    // (longer runs per DRAM row: 21.2 vs 22.6 us for the 32-sequence decoding pair)
    if ((long long)p.n_base + p.n_out <= 64)
        return k4 ? launch_bn<64, 4, 64>(p, stream) : (k2 ? launch_bn<64, 2, 64>(p, stream) : launch_bn<64, 1, 64>(p, stream));
    return k2 ? launch_bn<64, 2, kBM>(p, stream) : launch_bn<64, 1, kBM>(p, stream);
}

}  // namespace orthros
