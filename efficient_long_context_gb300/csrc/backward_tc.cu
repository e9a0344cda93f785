// backward_tc.cu -- gradients of the banded and cross rows on the 5th-generation
// tensor cores (tcgen05, TMEM, TMA); bf16, head size d = 128 or 64.
//
// What it computes: the chain rule through Sec. 3.1 Eq. 4 (base rows, keys
// max(0, t-w+1) .. t) and Eq. 5 (output rows, keys 0 .. t_r). With the
// forward's log-sum-exp L and D = dO . o of each row (prepared by a pre-pass
// together with the affined queries qa = alpha (.) q + beta in bf16):
//   P  = exp(scale * qa k^T - L)          dP = dO v^T
//   dS = scale * P (.) (dP - D)
//   dV = P^T dO     dK = dS^T qa     dQa = dS K
// dV and dK are complete per key; dQa is reduced over key blocks in fp32.
//
// Design: one CTA per (sequence, kv head, block of 128 keys), 320 threads.
//   It visits every 64-row query tile that sees its keys: for each query head
//   of the GQA group, the base-stream tiles of the band [j0, j0 + 127 + w - 1]
//   and the output-row tiles whose largest position reaches j0.
//   Keys are the M dimension of every product, so dK and dV accumulate in
//   TMEM over all tiles and are written once:
//     S^T  = K qa^T   (M 128 keys, N 64 rows, K = d)        TMEM [0, 64)
//     dP^T = V dO^T                                          TMEM [64, 128)
//     dV  += P^T dO   (P^T from TMEM; dO read MN-major)      TMEM [128, 256)
//     dK  += dS^T qa  (dS^T from shared memory)              TMEM [256, 384)
//     dQ^T = K^T dS^T (M = d channels, N = 64 rows, both operands MN-major)
//                                                            TMEM [384, 448)
//     (d = 64: dV, dK take 64 columns each; dQ^T is an M = 64 accumulator,
//     channel 16 q + i in TMEM lane 32 q + i, i < 16)
//     P^T as packed bf16, two buffers                        TMEM [448, 512)
//   warp 8: TMA producer (K, V once; qa and dO tiles, 3 stages) and the
//           per-tile row metadata (positions, L, D), loaded while the tiles fly.
//   warp 9: one thread issues the MMAs in the order S_i, dP_i, dV_{i-1},
//           dK_{i-1}, dQ_{i-1}, so the tensor core works on tile i while the
//           softmax warps turn tile i-1's scores into P and dS.
//   warps 0-7: thread (lane quarter q, half h) owns key 32 q + lane and 32 of
//           the 64 rows: P and dS in fp32; P^T back to TMEM as bf16, dS^T to
//           shared memory as bf16 in a swizzled layout that is K-major for
//           dK and MN-major for dQ^T at once; then they drain dQ^T of the
//           previous tile into the fp32 accumulator with coalesced
//           reductions, and at the end store dK and dV.
#include <cuda.h>

#include <algorithm>

#include "ptx.cuh"

namespace orthros {

using namespace ptx;

namespace {

constexpr int kKeys = 128;
constexpr int kRows = 64;
constexpr int kStages = 3;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 320;
constexpr int kSoftThreads = 256;

constexpr int kBoxK = kKeys * 128;     // one 64-channel box of 128 keys: 16 KB
constexpr int kBoxQ = kRows * 128;     // one 64-channel box of 64 rows: 8 KB
constexpr int kDSBytes = kKeys * kRows * 2;  // 16 KB
// TMEM columns
constexpr uint32_t kTS = 0, kTdP = 64, kTdV = 128, kTdK = 256, kTdQ = 384, kTP = 448;

// 16-byte aligned: the softmax warps read pos / lse2 / ndelta four at a time
struct __align__(16) StageMeta {
    int pos[kRows];      // row position, -1 for rows past the tile's end
    float lse2[kRows];   // L * log2(e), +inf for rows past the end
    float ndelta[kRows]; // -D * scale, D = dO . o
    int2 tile;           // x = 2 * head + kind (0 base, 1 output rows), y = first row
};
static_assert(sizeof(StageMeta) % 16 == 0, "stage metadata must keep every stage 16-byte aligned");

// The query tiles one key block visits, in order: for each query head of the
// GQA group, the base-stream tiles of the band [j0, j0 + 127 + w - 1], then
// the output-row tiles whose largest position reaches j0. Produced one at a
// time by the (warp-uniform) producer warp, so a key block may visit any
// number of tiles.
struct TileGen {
    int hh = 0, bi = 0, mbase = 0, phase = 0;
    unsigned mask = 0;
    // next tile (x = -1 when none is left); every lane of the warp calls it
    __device__ int2 next(const BwdTcParams &p, int kv, int g, int j0, int n_base, int r0b, int r1b, int lane) {
        const int n_cand = (r1b - r0b + kRows - 1) / kRows;
        while (hh < g) {
            const int h = kv * g + hh;
            if (phase == 0) {
                if (bi < n_base) return make_int2(2 * h, j0 + kRows * bi++);
                phase = 1;
                mbase = 0;
                mask = 0;
            }
            if (mask) {
                const int k = __ffs(mask) - 1;
                mask &= mask - 1;
                return make_int2(2 * h + 1, r0b + (mbase - 32 + k) * kRows);
            }
            if (mbase >= n_cand) {
                ++hh;
                phase = 0;
                bi = 0;
                continue;
            }
            const int m = mbase + lane;
            const int r = r0b + m * kRows;
            mask = __ballot_sync(0xffffffffu, m < n_cand && p.omax[r] >= j0);
            mbase += 32;
        }
        return make_int2(-1, 0);
    }
};

struct Meta {
    uint64_t kv_full, q_full[kStages], q_empty[kStages];
    uint64_t s_full, s_free, p_full[2], pds_free[2], dq_full, dq_free, mma_done;
    uint32_t tmem_base;
    int abort;
    int n_tiles;
    int pad;
    StageMeta st[kStages];
};

// Shared-memory layout for head size D (D / 64 boxes of 64 channels per tile).
template <int D> struct BCfg {
    static constexpr int kAtoms = D / 64;
    static constexpr int kKBytes = kAtoms * kBoxK;  // 32 KB (16 KB at d = 64)
    static constexpr int kQBytes = kAtoms * kBoxQ;  // 16 KB (8 KB)
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kOffK + kKBytes;
    static constexpr int kOffQ = kOffV + kKBytes;  // stage s: qa at +s*2*kQBytes, dO after it
    static constexpr int kOffDS = kOffQ + kStages * 2 * kQBytes;
    static constexpr int kOffMeta = kOffDS + 2 * kDSBytes;
    static constexpr int kSmem = kOffMeta + (int)sizeof(Meta) + 1024;
};

__device__ __forceinline__ void reg_fence(uint32_t (&r)[32]) {
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                   "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]),
                   "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]),
                   "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]));
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    backward_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_qb, const __grid_constant__ CUtensorMap tm_db,
                       const __grid_constant__ CUtensorMap tm_qo, const __grid_constant__ CUtensorMap tm_do,
                       const BwdTcParams p) {
    using C = BCfg<D>;
    constexpr int kOffK = C::kOffK, kOffV = C::kOffV, kOffQ = C::kOffQ, kOffDS = C::kOffDS, kOffMeta = C::kOffMeta;
    constexpr int kKBytes = C::kKBytes, kQBytes = C::kQBytes;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Meta &mt = *reinterpret_cast<Meta *>(smem + kOffMeta);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    volatile int *abort = &mt.abort;

    // unit: (sequence, kv head) slowest, key block fastest: the CTAs running at
    // one time reduce into the dQ rows of a few (sequence, kv head) pairs,
    // which then stay in L2; inside a pair the early key blocks (those that
    // the most output rows reach) start first
    const int jb = blockIdx.x % p.nkb;
    const int b = blockIdx.x / p.nkb / p.Hkv;
    const int kv = (blockIdx.x / p.nkb) % p.Hkv;
    const int j0 = jb * kKeys;
    const int g = p.Hq / p.Hkv;
    const int r0b = p.n_out ? p.out_indptr[b] : 0;
    const int r1b = p.n_out ? p.out_indptr[b + 1] : 0;

    if (tid == 0) {
        mbar_init(&mt.kv_full, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&mt.q_full[s], 1);
            mbar_init(&mt.q_empty[s], 1);
        }
        mbar_init(&mt.s_full, 1);
        mbar_init(&mt.s_free, kSoftThreads);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&mt.p_full[s], kSoftThreads);
            mbar_init(&mt.pds_free[s], 1);
        }
        mbar_init(&mt.dq_full, 1);
        mbar_init(&mt.dq_free, kSoftThreads);
        mbar_init(&mt.mma_done, 1);
        mt.abort = 0;
        fence_mbar_init();
    }
    // base tiles of the band of one head: rows j0 .. min(T - 1, j0 + 127 + w - 1)
    const long long t_hi_ll = min((long long)p.T - 1, (long long)j0 + kKeys - 1 + (long long)p.window - 1);
    const int n_base = (int)((t_hi_ll - j0) / kRows) + 1;
    if (warp == 0) {
        // tiles to visit: the same output-row tiles reach this key block for every head
        int n_out_tiles = 0;
        for (int r0 = r0b; r0 < r1b; r0 += 32 * kRows) {
            const int r = r0 + lane * kRows;
            n_out_tiles += __popc(__ballot_sync(0xffffffffu, r < r1b && p.omax[r] >= j0));
        }
        if (lane == 0) mt.n_tiles = g * (n_base + n_out_tiles);
    }
    if (warp == kProducerWarp && lane == 0) {
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_qb);
        prefetch_tmap(&tm_db);
    }
    __syncthreads();
    if (warp == kMmaWarp) {
        tmem_alloc(&mt.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = mt.tmem_base;
    const int n_tiles = mt.n_tiles;
    const long long seq_tok = (long long)b * p.T;

    if (warp == kProducerWarp) {
        // ---------------- TMA producer + row metadata ----------------
        int issued = 0;
        if (lane == 0 && n_tiles > 0) {
            mbar_arrive_expect_tx(&mt.kv_full, 2 * kKBytes);
            for (int j = 0; j < C::kAtoms; ++j) {
                tma_load_3d(smem + kOffK + j * kBoxK, &tm_k, &mt.kv_full, 64 * j, kv, (int)(seq_tok + j0));
                tma_load_3d(smem + kOffV + j * kBoxK, &tm_v, &mt.kv_full, 64 * j, kv, (int)(seq_tok + j0));
            }
        }
        const float log2e = 1.4426950408889634f;
        // Row metadata of tile i (2 rows per lane) is loaded into registers one
        // tile ahead, so its global-memory latency overlaps the wait for a stage.
        int m_pos[2];
        float m_l2[2], m_dl[2];
        TileGen gen;
        auto fetch = [&](int2 tl) {
            const int h = tl.x >> 1, kind = tl.x & 1, row0 = tl.y;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int c = lane + 32 * u;
                m_pos[u] = -1;
                m_l2[u] = INFINITY;
                m_dl[u] = 0.f;
                if (kind == 0) {
                    const int t = row0 + c;
                    if (t < p.T) {
                        const long long idx = ((long long)b * p.Hq + h) * p.T + t;
                        m_pos[u] = t;
                        m_l2[u] = p.lse_base[idx];
                        m_dl[u] = p.delta_base[idx];
                    }
                } else {
                    const int r = row0 + c;
                    if (r < r1b) {
                        const long long idx = (long long)r * p.Hq + h;
                        m_pos[u] = p.out_positions[r];
                        m_l2[u] = p.lse_out[idx];
                        m_dl[u] = p.delta_out[idx];
                    }
                }
            }
        };
        int2 tl_next = make_int2(-1, 0);
        if (n_tiles > 0) {
            tl_next = gen.next(p, kv, g, j0, n_base, r0b, r1b, lane);
            fetch(tl_next);
        }
        for (int i = 0; i < n_tiles; ++i) {
            const int s = i % kStages;
            if (i >= kStages) {
                if (!mbar_wait_warp(&mt.q_empty[s], ((i / kStages) - 1) & 1, abort, p.status)) break;
            }
            const int2 tl = tl_next;
            const int h = tl.x >> 1, kind = tl.x & 1, row0 = tl.y;
            if (lane == 0) {
                uint8_t *qa = smem + kOffQ + s * 2 * kQBytes;
                uint8_t *dO = qa + kQBytes;
                mbar_expect_tx(&mt.q_full[s], 2 * kQBytes);
                const int row_tok = kind == 0 ? (int)(seq_tok + row0) : row0;
                const CUtensorMap *mq = kind == 0 ? &tm_qb : &tm_qo;
                const CUtensorMap *md = kind == 0 ? &tm_db : &tm_do;
                for (int j = 0; j < C::kAtoms; ++j) {
                    tma_load_3d(qa + j * kBoxQ, mq, &mt.q_full[s], 64 * j, h, row_tok);
                    tma_load_3d(dO + j * kBoxQ, md, &mt.q_full[s], 64 * j, h, row_tok);
                }
            }
            StageMeta &sm = mt.st[s];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int c = lane + 32 * u;
                const int t = m_pos[u];
                const bool valid = t >= 0 && t < p.T;  // rows past the end carry -1
                sm.pos[c] = valid ? t : -1;
                sm.lse2[c] = valid ? m_l2[u] * log2e : INFINITY;
                sm.ndelta[c] = valid ? -m_dl[u] * p.scale : 0.f;
            }
            if (lane == 0) sm.tile = tl;
            __syncwarp();
            if (lane == 0) mbar_arrive(&mt.q_full[s]);
            if (i + 1 < n_tiles) {
                tl_next = gen.next(p, kv, g, j0, n_base, r0b, r1b, lane);
                fetch(tl_next);
            }
            issued = i + 1;
        }
        // nothing may land in shared memory after the CTA exits
        if (lane == 0) {
            if (n_tiles > 0) mbar_wait_drain(&mt.kv_full, 0, p.status);
            for (int i = max(0, issued - kStages); i < issued; ++i)
                mbar_wait_drain(&mt.q_full[i % kStages], (i / kStages) & 1, p.status);
        }
    } else if (warp == kMmaWarp) {
        // ---------------- tcgen05.mma issuer ----------------
        if (lane == 0 && n_tiles > 0) {
            constexpr uint32_t kIdS = idesc_f16(1, 1, 0, 0, kKeys, kRows);   // S^T, dP^T
            constexpr uint32_t kIdKV = idesc_f16(1, 1, 0, 1, kKeys, D);      // dV, dK: B MN-major
            constexpr uint32_t kIdQ = idesc_f16(1, 1, 1, 1, D, kRows);       // dQ^T: A and B MN-major
            // start-address field is (byte address >> 4); all operands lie below
            // 256 KB, so adding (offset >> 4) never carries out of the field
            const uint64_t d_k = desc_sw128(smem_u32(smem + kOffK), 16, 1024);          // K-major
            const uint64_t d_v = desc_sw128(smem_u32(smem + kOffV), 16, 1024);
            const uint64_t d_kmn = desc_sw128(smem_u32(smem + kOffK), kBoxK, 1024);     // K as MN-major A
            const uint64_t d_q0 = desc_sw128(smem_u32(smem + kOffQ), 16, 1024);         // qa stage 0, K-major
            const uint64_t d_qmn0 = desc_sw128(smem_u32(smem + kOffQ), kBoxQ, 1024);    // qa stage 0, MN-major
            const uint64_t d_ds0 = desc_sw128(smem_u32(smem + kOffDS), 16, 1024);
            const uint64_t d_dsmn0 = desc_sw128(smem_u32(smem + kOffDS), kBoxQ, 1024);
            constexpr uint32_t kStageU = (2 * kQBytes) >> 4, kQU = kQBytes >> 4, kDSU = kDSBytes >> 4;
            bool ok = mbar_wait(&mt.kv_full, 0, abort, p.status);
            for (int i = 0; ok && i <= n_tiles; ++i) {
                if (i < n_tiles) {
                    const int s = i % kStages;
                    if (!(ok = mbar_wait(&mt.q_full[s], (i / kStages) & 1, abort, p.status))) break;
                    if (i >= 1 && !(ok = mbar_wait(&mt.s_free, (i - 1) & 1, abort, p.status))) break;
                    tc_fence_after();
                    const uint64_t dq = d_q0 + s * kStageU, ddo = dq + kQU;
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint32_t ok_ = ((ks >> 2) * kBoxK + (ks & 3) * 32) >> 4;
                        const uint32_t oq = ((ks >> 2) * kBoxQ + (ks & 3) * 32) >> 4;
                        mma_ss(tmem + kTS, d_k + ok_, dq + oq, kIdS, ks > 0);
                    }
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint32_t ok_ = ((ks >> 2) * kBoxK + (ks & 3) * 32) >> 4;
                        const uint32_t oq = ((ks >> 2) * kBoxQ + (ks & 3) * 32) >> 4;
                        mma_ss(tmem + kTdP, d_v + ok_, ddo + oq, kIdS, ks > 0);
                    }
                    tc_commit(&mt.s_full);
                }
                if (i >= 1) {
                    const int pi = i - 1, ps = pi % 2, qs = pi % kStages;
                    if (!(ok = mbar_wait(&mt.p_full[ps], (pi / 2) & 1, abort, p.status))) break;
                    tc_fence_after();
                    const uint64_t dqmn = d_qmn0 + qs * kStageU, ddomn = dqmn + kQU;
                    const uint64_t dds = d_ds0 + ps * kDSU, ddsmn = d_dsmn0 + ps * kDSU;
                    // dV += P^T dO: P^T packed bf16 in TMEM, 16 rows (8 columns) per step
#pragma unroll
                    for (int kk = 0; kk < kRows / 16; ++kk)
                        mma_ts(tmem + kTdV, tmem + kTP + 32 * ps + 8 * kk, ddomn + ((kk * 16 * 128) >> 4), kIdKV,
                               (pi > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
                    for (int kk = 0; kk < kRows / 16; ++kk)
                        mma_ss(tmem + kTdK, dds + ((kk * 32) >> 4), dqmn + ((kk * 16 * 128) >> 4), kIdKV,
                               (pi > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(&mt.q_empty[qs]);
                    if (pi >= 1 && !(ok = mbar_wait(&mt.dq_free, (pi - 1) & 1, abort, p.status))) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kKeys / 16; ++kk)
                        mma_ss(tmem + kTdQ, d_kmn + ((kk * 16 * 128) >> 4), ddsmn + ((kk * 16 * 128) >> 4), kIdQ,
                               kk > 0);
                    tc_commit(&mt.dq_full);
                    tc_commit(&mt.pds_free[ps]);
                }
            }
            tc_commit(&mt.mma_done);
            mbar_wait_drain(&mt.mma_done, 0, p.status);
        }
    } else {
        // ---------------- P, dS; dQ drain; dK, dV store ----------------
        const int qd = warp & 3, hh = warp >> 2;
        const int key = qd * 32 + lane;  // TMEM lane of this thread
        const int j = j0 + key;
        const uint32_t lane_off = static_cast<uint32_t>(qd * 32) << 16;
        const float c2 = p.scale_log2;
        int2 prev_tile = make_int2(0, 0);  // the tile whose dQ is drained next
        auto drain = [&](int pi) -> bool {
            if (!mbar_wait_warp(&mt.dq_full, pi & 1, abort, p.status)) return false;
            tc_fence_after();
            uint32_t v[32];
            tmem_ld32(tmem + lane_off + kTdQ + 32 * hh, v);
            tmem_ld_wait();
            reg_fence(v);
            tc_fence_before();
            mbar_arrive(&mt.dq_free);
            const int2 tl = prev_tile;
            const int h = tl.x >> 1, kind = tl.x & 1, row0 = tl.y;
            // dQ^T lanes are channels (d = 64: lanes 32 q .. 32 q + 15 hold channels 16 q ..)
            const int ch = D == 128 ? key : qd * 16 + lane;
            const bool own = D == 128 || lane < 16;
            if (kind == 0) {
                float *dst = p.dq_acc + ((seq_tok + row0 + 32 * hh) * p.Hq + h) * D + ch;
                const long long stride = (long long)p.Hq * D;
                const int n = own ? min(32, p.T - (row0 + 32 * hh)) : 0;
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    if (e < n) red_add_f32(dst + e * stride, __uint_as_float(v[e]));
            } else {
                float *dst = p.dq_out_acc + ((long long)(row0 + 32 * hh) * p.Hq + h) * D + ch;
                const long long stride = (long long)p.Hq * D;
                const int n = own ? min(32, r1b - (row0 + 32 * hh)) : 0;
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    if (e < n) red_add_f32(dst + e * stride, __uint_as_float(v[e]));
            }
            return true;
        };
        bool ok = true;
        for (int i = 0; i < n_tiles; ++i) {
            const int s = i % kStages, ps = i % 2;
            if (!(ok = mbar_wait_warp(&mt.s_full, i & 1, abort, p.status))) break;
            tc_fence_after();
            uint32_t sv[32], dv[32];
            tmem_ld32(tmem + lane_off + kTS + 32 * hh, sv);
            tmem_ld32(tmem + lane_off + kTdP + 32 * hh, dv);
            tmem_ld_wait();
            reg_fence(sv);
            reg_fence(dv);
            tc_fence_before();
            mbar_arrive(&mt.s_free);
            // the row metadata was published with q_full (already complete for this tile)
            if (!(ok = mbar_wait_warp(&mt.q_full[s], (i / kStages) & 1, abort, p.status))) break;
            const int2 cur_tile = mt.st[s].tile;
            const int kind = cur_tile.x & 1;
            const unsigned wlim = kind ? 0x7fffffffu : (unsigned)p.window;  // valid: 0 <= t - j < wlim
            const StageMeta &sm = mt.st[s];
            uint32_t pk[16], dk[16];
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
                const int col = 32 * hh + 4 * q4;
                const int4 t4 = *reinterpret_cast<const int4 *>(&sm.pos[col]);
                const float4 l4 = *reinterpret_cast<const float4 *>(&sm.lse2[col]);
                const float4 d4 = *reinterpret_cast<const float4 *>(&sm.ndelta[col]);
                const int tt[4] = {t4.x, t4.y, t4.z, t4.w};
                const float ll[4] = {l4.x, l4.y, l4.z, l4.w};
                const float dd[4] = {d4.x, d4.y, d4.z, d4.w};
                float pv[4], dsv[4];
                // pairs of rows: one packed instruction each for the exponent's argument,
                // dP * scale + (-D * scale), and P times that
#pragma unroll
                for (int u = 0; u < 4; u += 2) {
                    const int e = 4 * q4 + u;
                    float a0, a1, g0, g1;
                    fma2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1]), c2, c2, -ll[u], -ll[u + 1], a0, a1);
                    pv[u] = (unsigned)(tt[u] - j) < wlim ? ex2(a0) : 0.f;
                    pv[u + 1] = (unsigned)(tt[u + 1] - j) < wlim ? ex2(a1) : 0.f;
                    fma2(__uint_as_float(dv[e]), __uint_as_float(dv[e + 1]), p.scale, p.scale, dd[u], dd[u + 1], g0, g1);
                    mul2(pv[u], pv[u + 1], g0, g1, dsv[u], dsv[u + 1]);
                }
                pk[2 * q4] = pack_bf16(pv[0], pv[1]);
                pk[2 * q4 + 1] = pack_bf16(pv[2], pv[3]);
                dk[2 * q4] = pack_bf16(dsv[0], dsv[1]);
                dk[2 * q4 + 1] = pack_bf16(dsv[2], dsv[3]);
            }
            if (i >= 2 && !(ok = mbar_wait_warp(&mt.pds_free[ps], ((i / 2) - 1) & 1, abort, p.status))) break;
            // P^T rows 32 hh .. +31 of this key -> 16 packed columns of this P buffer
            tmem_st16(tmem + lane_off + kTP + 32 * ps + 16 * hh, pk);
            uint8_t *db = smem + kOffDS + ps * kDSBytes + key * 128;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int phys = ((4 * hh + q) ^ (key & 7)) << 4;
                *reinterpret_cast<uint4 *>(db + phys) = make_uint4(dk[4 * q], dk[4 * q + 1], dk[4 * q + 2], dk[4 * q + 3]);
            }
            tmem_st_wait();
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&mt.p_full[ps]);
            if (i >= 1 && !(ok = drain(i - 1))) break;
            prev_tile = cur_tile;
        }
        if (ok && n_tiles > 0) ok = drain(n_tiles - 1);
        // dK, dV of this thread's key: columns [D/2 hh, D/2 hh + D/2) of each
        const bool done = n_tiles > 0 && ok && mbar_wait_warp(&mt.mma_done, 0, abort, p.status);
        if (done) {
            tc_fence_after();
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                __nv_bfloat16 *dst = (which ? p.dk : p.dv) + ((seq_tok + j) * p.Hkv + kv) * D + (D / 2) * hh;
#pragma unroll
                for (int half = 0; half < D / 64; ++half) {
                    uint32_t v[32];
                    tmem_ld32(tmem + lane_off + kTdV + 128 * which + (D / 2) * hh + 32 * half, v);
                    tmem_ld_wait();
                    reg_fence(v);
                    if (j < p.T) {
                        uint4 w[4];
                        uint32_t *wp = reinterpret_cast<uint32_t *>(w);
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            wp[e] = pack_bf16(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
#pragma unroll
                        for (int e = 0; e < 4; ++e) reinterpret_cast<uint4 *>(dst + 32 * half)[e] = w[e];
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

namespace {

template <int D>
cudaError_t launch_d(const BwdTcParams &p, const void *k, const void *v, const void *qa_base, const void *do_base,
                     const void *qa_out, const void *do_out, cudaStream_t stream) {
    const long long tokens = (long long)p.B * p.T;
    CUtensorMap tk, tv, tqb, tdb, tqo, tdo;
    const long long n_out_rows = p.n_out > 0 ? p.n_out : 1;
    if (!encode_kv_map_3d(&tk, k, tokens, p.Hkv, D, kKeys) || !encode_kv_map_3d(&tv, v, tokens, p.Hkv, D, kKeys) ||
        !encode_kv_map_3d(&tqb, qa_base, tokens, p.Hq, D, kRows) ||
        !encode_kv_map_3d(&tdb, do_base, tokens, p.Hq, D, kRows) ||
        !encode_kv_map_3d(&tqo, p.n_out > 0 ? qa_out : qa_base, n_out_rows, p.Hq, D, kRows) ||
        !encode_kv_map_3d(&tdo, p.n_out > 0 ? do_out : do_base, n_out_rows, p.Hq, D, kRows))
        return cudaErrorInvalidValue;
    static SmemLimit limit;
    if (cudaError_t e = limit.ensure((const void *)backward_tc_kernel<D>, BCfg<D>::kSmem); e != cudaSuccess) return e;
    const long long units = (long long)p.nkb * p.B * p.Hkv;
    if (units == 0) return cudaSuccess;
    backward_tc_kernel<D><<<(unsigned)units, kThreads, BCfg<D>::kSmem, stream>>>(tk, tv, tqb, tdb, tqo, tdo, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_backward_tc(const BwdTcParams &p, int d, const void *k, const void *v, const void *qa_base,
                               const void *do_base, const void *qa_out, const void *do_out, cudaStream_t stream) {
    return d == 128 ? launch_d<128>(p, k, v, qa_base, do_base, qa_out, do_out, stream)
                    : launch_d<64>(p, k, v, qa_base, do_base, qa_out, do_out, stream);
}

}  // namespace orthros
