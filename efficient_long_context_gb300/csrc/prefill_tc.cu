// prefill_tc.cu -- banded sliding-window attention (base stream) and dense
// output-stream rows on the 5th-generation tensor cores (tcgen05, TMEM, TMA).
//
// What it computes (Orthros paper, Sec. 3.1):
//   Eq. 4: o_t  = softmax_j(scale * q_t . k_j)  v_j over j in [max(0, t-w+1), t]
//   Eq. 5: o'_t = softmax_j(scale * q'_t . k_j) v_j over j in [0, t]
// with q = alpha (.) q_raw + beta applied while the query tile is staged
// (Alg. 1 line 5), for every base position and for output rows handed to this
// kernel (those of sequences with many output rows; sequences with few output
// rows take the split-KV kernel instead).
//
// Design (one CTA per SM, 576 threads):
//   * A work unit is two 128-row query tiles that read the SAME key/value
//     tiles: two query heads of one GQA group at the same positions, or (when
//     the group size is odd, e.g. plain multi-head) two consecutive row blocks
//     of one head. Key/value tiles of 128 tokens are visited only inside the
//     union of the tiles' bands; tiles outside the band are never loaded.
//   * warp 16 (one thread): TMA producer. Keys come from an fp16 copy made by
//     the pre-pass kernel (3 stages), values in bf16 (2 stages), 128B swizzle.
//   * warp 17 (one thread): tcgen05.mma issuer. S_s = Q_s K^T (M=128, N=128,
//     fp16 operands from shared memory) into TMEM; O_s += P_s V (M=128, N=d,
//     P read from TMEM as bf16, V from shared memory, MN-major).
//   * warps 0-15: softmax, two threads per row. Warp w serves slot
//     (w >> 2) & 1, key half w >> 3 of each 128-key tile, rows 32 (w & 3) ..
//     +31 (TMEM lane quarter w & 3). A thread reads its 64 logits with
//     tcgen05.ld, masks the two band edge tiles, agrees with its partner on
//     the row's shift, keeps a running max with lazy rescaling (O in TMEM is
//     only rescaled when the max grows by more than 2^8), writes P as packed
//     bf16 back over its logits, and finally normalises its half of O and
//     stores o and lse.
//   TMEM (512 columns): S0 [0,128) S1 [128,256) O0 [256,256+d) O1 [384,384+d).
//
// Precision: the query affine runs in fp32 and is rounded to fp16 (11-bit
// significand) rather than bf16 for the QK^T product; the pre-pass converts
// keys bf16 -> fp16, which is exact in the fp16 range (the pre-pass flags any
// key beyond it). P is rounded to bf16 for the PV product, accumulation fp32.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "ptx.cuh"

namespace orthros {

using namespace ptx;

namespace {

constexpr int kRowsPerTile = 128;  // M of every MMA, rows of a query tile
constexpr int kKeysPerTile = 128;  // N of QK^T, K of PV
constexpr int kSoftmaxWarps = 16;  // 2 slots x 2 column halves x 4 lane quarters
constexpr int kThreads = (kSoftmaxWarps + 2) * 32;
constexpr int kProducerWarp = 16;
constexpr int kMmaWarp = 17;
constexpr int kNumK = 3;  // key stages
constexpr int kNumV = 2;  // value stages

template <int D> struct Cfg {
    static constexpr int kSub = D / 64;                                 // 128-byte swizzle atoms per row
    static constexpr int kTileBytes = kRowsPerTile * D * 2;             // one 128 x D fp16/bf16 tile
    static constexpr int kQ0 = 0;                                       // two query tiles
    static constexpr int kK0 = kQ0 + 2 * kTileBytes;                    // key stages
    static constexpr int kV0 = kK0 + kNumK * kTileBytes;                // value stages
    static constexpr int kBar = kV0 + kNumV * kTileBytes;               // barriers + metadata
    static constexpr int kSmem = kBar + 1536 + 1024;                    // + alignment slack
    static constexpr int kTmemO = 256;                                  // first O column
};

struct Meta {
    uint64_t k_full[kNumK], k_empty[kNumK], v_full[kNumV], v_empty[kNumV];
    uint64_t s_full[2], p_full[2], o_full[2], mma_done;
    uint64_t q_full[2];  // per slot: raw query tile landed (TMA; rows contiguous in q or q_out)
    uint64_t os_bar[2];  // per slot: normalised output tile staged for the TMA store
    uint64_t xm_bar[2], lx_bar[2];  // per slot: row maxima / row sums exchanged between column halves
    uint32_t tmem_base;
    int abort;
    int t_min[2], t_max[2];
    __nv_bfloat16 xmax[2][2][kRowsPerTile];  // [slot][half][row] tile maxima (a shared shift; rounding is harmless)
};

struct Slot {
    int kind;  // 0 base positions, 1 output rows, -1 empty
    int b, h, row0, n;
};

// Work-unit decoding. Units [0, n_cross) are output-row units (heavier, so
// they start first), then base units. Inside one (sequence, kv head) the order
// is reversed so that late, fully populated row blocks start first.
__device__ __forceinline__ int units_per_kv(int nblk, int g) {
    return (g % 2 == 0) ? nblk * (g / 2) : g * ((nblk + 1) / 2);
}

__device__ void decode_unit(const TcParams &p, int u, Slot &s0, Slot &s1) {
    const int g = p.Hq / p.Hkv;
    int b, lu, rows, rowbase, kind;
    if (u < p.n_cross_units) {
        kind = 1;
        int lo = 0, hi = p.B - 1;  // last b with cross_unit_indptr[b] <= u
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.cross_unit_indptr[mid] <= u) lo = mid; else hi = mid - 1;
        }
        b = lo;
        lu = u - p.cross_unit_indptr[b];
        rowbase = p.out_indptr[b];
        rows = p.out_indptr[b + 1] - rowbase;
    } else {
        kind = 0;
        lu = u - p.n_cross_units;
        const int upb = p.Hkv * units_per_kv(p.base_nblk, g);
        b = lu / upb;
        lu -= b * upb;
        rowbase = 0;
        rows = p.Tq;
    }
    const int nblk = (rows + kRowsPerTile - 1) / kRowsPerTile;
    const int upk = units_per_kv(nblk, g);
    const int kv = lu / upk;
    const int q = upk - 1 - (lu - kv * upk);
    int blk0, blk1, h0, h1;
    if (g % 2 == 0) {
        blk0 = blk1 = q / (g / 2);
        h0 = kv * g + 2 * (q % (g / 2));
        h1 = h0 + 1;
    } else {
        const int per = (nblk + 1) / 2;
        h0 = h1 = kv * g + q / per;
        blk0 = 2 * (q % per);
        blk1 = blk0 + 1;
    }
    s0.kind = kind;
    s0.b = b;
    s0.h = h0;
    s0.row0 = rowbase + blk0 * kRowsPerTile;
    s0.n = min(kRowsPerTile, rows - blk0 * kRowsPerTile);
    s1.kind = blk1 < nblk ? kind : -1;
    s1.b = b;
    s1.h = h1;
    s1.row0 = rowbase + blk1 * kRowsPerTile;
    s1.n = blk1 < nblk ? min(kRowsPerTile, rows - blk1 * kRowsPerTile) : 0;
}

__device__ __forceinline__ void reg_fence(uint32_t (&r)[32]) {
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                   "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]),
                   "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]),
                   "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]));
}

// Byte offset of (row, 16-byte chunk c) inside a 128B-swizzled tile of D columns.
template <int D>
__device__ __forceinline__ uint32_t sw128_offset(int row, int c) {
    const int sub = c >> 3;  // 64-column atom
    const int cc = c & 7;
    return sub * (kRowsPerTile * 128) + row * 128 + ((cc ^ (row & 7)) << 4);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_qo,
                      const __grid_constant__ CUtensorMap tm_ob, const TcParams p) {
    using C = Cfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Meta &mt = *reinterpret_cast<Meta *>(smem + C::kBar);
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    volatile int *abort = &mt.abort;

    Slot sl0, sl1;
    decode_unit(p, blockIdx.x, sl0, sl1);

    if (tid == 0) {
        for (int i = 0; i < kNumK; ++i) {
            mbar_init(&mt.k_full[i], 1);
            mbar_init(&mt.k_empty[i], 1);
        }
        for (int i = 0; i < kNumV; ++i) {
            mbar_init(&mt.v_full[i], 1);
            mbar_init(&mt.v_empty[i], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&mt.s_full[s], 1);
            mbar_init(&mt.p_full[s], 2 * kRowsPerTile);
            mbar_init(&mt.o_full[s], 1);
            mbar_init(&mt.xm_bar[s], 2 * kRowsPerTile);
            mbar_init(&mt.lx_bar[s], 2 * kRowsPerTile);
            mbar_init(&mt.q_full[s], 1);
            mbar_init(&mt.os_bar[s], 2 * kRowsPerTile);
            mt.t_min[s] = 0x7fffffff;
            mt.t_max[s] = -1;
        }
        mbar_init(&mt.mma_done, 1);
        mt.abort = 0;
        fence_mbar_init();
    }
    if (warp == kProducerWarp && lane == 0) {
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
    }
    __syncthreads();
    if (warp == kMmaWarp) {
        tmem_alloc(&mt.tmem_base, 512);
        tmem_relinquish();
    }

    // Query tiles whose rows are contiguous (base positions; output rows with
    // their own q_out) arrive by TMA as raw bf16 and are turned into affined
    // fp16 in place below; output rows that read q at their positions are
    // gathered by the softmax threads.
    auto q_by_tma = [&](const Slot &S) { return S.kind == 0 || (S.kind == 1 && p.q_out != nullptr); };
    if (warp == kProducerWarp && lane == 0) {
        for (int s = 0; s < 2; ++s) {
            const Slot S = s ? sl1 : sl0;
            if (S.kind < 0 || !q_by_tma(S)) continue;
            mbar_arrive_expect_tx(&mt.q_full[s], C::kTileBytes);
            const int row = S.kind == 0 ? S.b * p.Tq + S.row0 : S.row0;
            for (int j = 0; j < C::kSub; ++j)
                tma_load_3d(smem + C::kQ0 + s * C::kTileBytes + j * (kRowsPerTile * 128), S.kind == 0 ? &tm_q : &tm_qo,
                            &mt.q_full[s], 64 * j, S.h, row);
        }
    }

    // Base-position tiles know their band without reading any data, so the
    // producer starts the first key/value loads now and they overlap the query
    // staging below (tiles with output rows wait for their positions).
    int pre_k = 0, pre_v = 0;
    const bool closed_form = sl0.kind == 0 && sl1.kind != 1;
    if (warp == kProducerWarp && lane == 0 && closed_form) {
        const int t0 = sl0.row0 + p.q_off;
        const int lo0 = max(0, t0 - p.window + 1) / kKeysPerTile;
        const int hi0 = (t0 + sl0.n - 1) / kKeysPerTile;
        int lo = lo0, hi = hi0;
        if (sl1.kind == 0) {
            const int t1 = sl1.row0 + p.q_off;
            lo = min(lo, max(0, t1 - p.window + 1) / kKeysPerTile);
            hi = max(hi, (t1 + sl1.n - 1) / kKeysPerTile);
        }
        const int n_cf = hi - lo + 1;
        const int kvh = sl0.h / (p.Hq / p.Hkv);
        pre_k = min(n_cf, kNumK);
        pre_v = min(n_cf, kNumV);
        for (int i = 0; i < pre_k; ++i) {
            mbar_arrive_expect_tx(&mt.k_full[i], C::kTileBytes);
            for (int j = 0; j < C::kSub; ++j)
                tma_load_4d(smem + C::kK0 + i * C::kTileBytes + j * (kKeysPerTile * 128), &tm_k, &mt.k_full[i], 64 * j,
                            kvh, (lo + i) * kKeysPerTile, sl0.b);
        }
        for (int i = 0; i < pre_v; ++i) {
            mbar_arrive_expect_tx(&mt.v_full[i], C::kTileBytes);
            for (int j = 0; j < C::kSub; ++j)
                tma_load_4d(smem + C::kV0 + i * C::kTileBytes + j * (kKeysPerTile * 128), &tm_v, &mt.v_full[i], 64 * j,
                            kvh, (lo + i) * kKeysPerTile, sl0.b);
        }
    }

    // ---------------- prologue: stage both query tiles (affine fused) ----------------
    // Softmax warp w: slot (w >> 2) & 1, column half w >> 3, rows 32 (w & 3) .. +31;
    // each half stages its own D/2 channels of the row.
    const bool softmax_thread = warp < kSoftmaxWarps;
    const int s_me = (warp >> 2) & 1;
    const int h_me = warp >> 3;
    const int row = ((warp & 3) << 5) | lane;
    int my_t = 0;  // the row's position in key coordinates
    bool my_valid = false, my_bad = false;
    if (softmax_thread) {
        const Slot S = s_me ? sl1 : sl0;
        if (S.kind >= 0 && row < S.n) {
            if (S.kind == 0) {
                my_t = S.row0 + row + p.q_off;
                my_valid = true;
            } else {
                const int t = p.out_positions[S.row0 + row];
                // a shard's output rows may sit past its keys (they read them all)
                my_t = p.shard ? min(t, p.T - 1) : t;
                my_valid = t >= 0 && (p.shard || t < p.T);
                // without q_out the row's query is the base query at its position
                if (!p.q_out && (my_t < p.q_off || my_t - p.q_off >= p.Tq)) my_valid = false;
            }
            my_bad = !my_valid;
            if (my_bad && h_me == 0) set_status(p.status, ORTHROS_DEV_BAD_POSITION);
        }
        uint8_t *qs = smem + C::kQ0 + s_me * C::kTileBytes;
        constexpr int kHalfChunks = D / 16;  // 16-byte chunks per half row
        const bool tma = S.kind >= 0 && q_by_tma(S);
        if (tma && !mbar_wait_warp(&mt.q_full[s_me], 0, abort, p.status)) my_valid = false;
        if (my_valid) {
            const float *al = (S.kind == 0 ? p.alpha_base : p.alpha_out) + S.h * D;
            const float *be = (S.kind == 0 ? p.beta_base : p.beta_out) + S.h * D;
            bool over = false;
            uint4 raws[kHalfChunks];  // every load of the half row in flight at once
            if (tma) {
#pragma unroll
                for (int cc = 0; cc < kHalfChunks; ++cc)
                    raws[cc] = *reinterpret_cast<const uint4 *>(qs + sw128_offset<D>(row, h_me * kHalfChunks + cc));
            } else {
                const __nv_bfloat16 *src = p.q + (((long long)S.b * p.Tq + (my_t - p.q_off)) * p.Hq + S.h) * D;
#pragma unroll
                for (int cc = 0; cc < kHalfChunks; ++cc)
                    raws[cc] = reinterpret_cast<const uint4 *>(src)[h_me * kHalfChunks + cc];
            }
#pragma unroll
            for (int cc = 0; cc < kHalfChunks; ++cc) {
                const int c = h_me * kHalfChunks + cc;
                const uint4 raw = raws[cc];
                const float4 a0 = reinterpret_cast<const float4 *>(al)[2 * c];
                const float4 a1 = reinterpret_cast<const float4 *>(al)[2 * c + 1];
                const float4 b0 = reinterpret_cast<const float4 *>(be)[2 * c];
                const float4 b1 = reinterpret_cast<const float4 *>(be)[2 * c + 1];
                const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&raw);
                float2 x0 = __bfloat1622float2(h2[0]), x1 = __bfloat1622float2(h2[1]);
                float2 x2 = __bfloat1622float2(h2[2]), x3 = __bfloat1622float2(h2[3]);
                float v[8] = {fmaf(a0.x, x0.x, b0.x), fmaf(a0.y, x0.y, b0.y), fmaf(a0.z, x1.x, b0.z),
                              fmaf(a0.w, x1.y, b0.w), fmaf(a1.x, x2.x, b1.x), fmaf(a1.y, x2.y, b1.y),
                              fmaf(a1.z, x3.x, b1.z), fmaf(a1.w, x3.y, b1.w)};
#pragma unroll
                for (int e = 0; e < 8; ++e) over |= fabsf(v[e]) > 65504.f;
                uint4 o;
                o.x = pack_f16(v[0], v[1]);
                o.y = pack_f16(v[2], v[3]);
                o.z = pack_f16(v[4], v[5]);
                o.w = pack_f16(v[6], v[7]);
                *reinterpret_cast<uint4 *>(qs + sw128_offset<D>(row, c)) = o;
            }
            if (over) set_status(p.status, ORTHROS_DEV_FP16_RANGE);
            if (h_me == 0) {
                atomicMin(&mt.t_min[s_me], my_t);
                atomicMax(&mt.t_max[s_me], my_t);
            }
        } else {
#pragma unroll 4
            for (int cc = 0; cc < kHalfChunks; ++cc)
                *reinterpret_cast<uint4 *>(qs + sw128_offset<D>(row, h_me * kHalfChunks + cc)) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---------------- band of each tile, in key-tile units ----------------
    // Band of each tile in key-tile units: [kt_lo, kt_hi]; lo_max = latest
    // window start of its rows (key tiles before it need the window mask).
    struct Band {
        int kt_lo, kt_hi, lo_max, t_min, t_max;
    };
    auto band_of = [&](const Slot &S, int tmin, int tmax) {
        Band bd;
        bd.t_min = tmin;
        bd.t_max = tmax;
        if (S.kind < 0 || tmax < 0) {
            bd.kt_lo = 1;
            bd.kt_hi = 0;
            bd.lo_max = 0;
            return bd;
        }
        const int lo_min = S.kind == 0 ? max(0, tmin - p.window + 1) : p.key_lo;
        bd.lo_max = S.kind == 0 ? max(0, tmax - p.window + 1) : p.key_lo;
        bd.kt_lo = lo_min / kKeysPerTile;
        bd.kt_hi = tmax / kKeysPerTile;
        return bd;
    };
    const Band bd0 = band_of(sl0, mt.t_min[0], mt.t_max[0]);
    const Band bd1 = band_of(sl1, mt.t_min[1], mt.t_max[1]);
    const bool any0 = bd0.kt_lo <= bd0.kt_hi, any1 = bd1.kt_lo <= bd1.kt_hi;
    const int kt_min = any0 && any1 ? min(bd0.kt_lo, bd1.kt_lo) : (any0 ? bd0.kt_lo : bd1.kt_lo);
    const int kt_max = any0 && any1 ? max(bd0.kt_hi, bd1.kt_hi) : (any0 ? bd0.kt_hi : bd1.kt_hi);
    const int n_it = (any0 || any1) ? kt_max - kt_min + 1 : 0;
    const uint32_t tmem = mt.tmem_base;
    const int kv = sl0.h / (p.Hq / p.Hkv);
    const int bseq = sl0.b;

    if (warp == kProducerWarp) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            for (int i = 0; i < n_it && !*abort; ++i) {
                const int kt = kt_min + i;
                const int sk = i % kNumK;
                if (i >= pre_k) {
                    if (i >= kNumK && !mbar_wait(&mt.k_empty[sk], ((i / kNumK) - 1) & 1, abort, p.status)) break;
                    mbar_arrive_expect_tx(&mt.k_full[sk], C::kTileBytes);
                    for (int j = 0; j < C::kSub; ++j)
                        tma_load_4d(smem + C::kK0 + sk * C::kTileBytes + j * (kKeysPerTile * 128), &tm_k,
                                    &mt.k_full[sk], 64 * j, kv, kt * kKeysPerTile, bseq);
                }
                const int sv = i % kNumV;
                if (i >= pre_v) {
                    if (i >= kNumV && !mbar_wait(&mt.v_empty[sv], ((i / kNumV) - 1) & 1, abort, p.status)) break;
                    mbar_arrive_expect_tx(&mt.v_full[sv], C::kTileBytes);
                    for (int j = 0; j < C::kSub; ++j)
                        tma_load_4d(smem + C::kV0 + sv * C::kTileBytes + j * (kKeysPerTile * 128), &tm_v,
                                    &mt.v_full[sv], 64 * j, kv, kt * kKeysPerTile, bseq);
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // ---------------- tcgen05.mma issuer ----------------
        if (lane == 0 && n_it > 0) {
            constexpr uint32_t kIdescS = idesc_f16(0, 0, 0, 0, kRowsPerTile, kKeysPerTile);  // fp16, K-major
            constexpr uint32_t kIdescO = idesc_f16(1, 1, 0, 1, kRowsPerTile, D);             // bf16, V MN-major
            // Descriptors are built once; the start-address field is the low 14 bits
            // (byte address >> 4) and every operand lies below 256 KB of shared
            // memory, so adding (byte offset >> 4) never carries out of the field.
            constexpr uint32_t kTileU = C::kTileBytes >> 4;
            const uint64_t dq = desc_sw128(smem_u32(smem + C::kQ0), 16, 1024);
            const uint64_t dk = desc_sw128(smem_u32(smem + C::kK0), 16, 1024);
            const uint64_t dv = desc_sw128(smem_u32(smem + C::kV0), kKeysPerTile * 128, 1024);
            const uint32_t d_s0 = tmem, d_s1 = tmem + 128;
            const uint32_t d_o0 = tmem + C::kTmemO, d_o1 = tmem + C::kTmemO + 128;
            const int lo0 = bd0.kt_lo, hi0 = bd0.kt_hi, lo1 = bd1.kt_lo, hi1 = bd1.kt_hi;
            // S = Q K^T: 16 channels per instruction; inside a 128B atom the start
            // address advances 32 bytes per step.
#define ORTHROS_ISSUE_S(D_TMEM, QDESC, KDESC)                                           \
    _Pragma("unroll") for (int ks = 0; ks < D / 16; ++ks) {                            \
        const uint32_t off = ((ks >> 2) * (kRowsPerTile * 128) + (ks & 3) * 32) >> 4; \
        mma_ss((D_TMEM), (QDESC) + off, (KDESC) + off, kIdescS, ks > 0);             \
    }
            // O += P V: 16 keys per instruction; P packed bf16x2 in the S columns
            // (8 columns per step), V rows 128 bytes apart.
#define ORTHROS_ISSUE_PV(D_TMEM, P_TMEM, VDESC, ACC0)                                            \
    _Pragma("unroll") for (int kk = 0; kk < kKeysPerTile / 16; ++kk)                            \
        mma_ts((D_TMEM), (P_TMEM) + kk * 8, (VDESC) + (uint64_t)((kk * 16 * 128) >> 4), kIdescO, \
               kk > 0 ? 1u : (ACC0));
            uint32_t pc0 = 0, pc1 = 0, o_init0 = 0, o_init1 = 0;
            bool ok = mbar_wait(&mt.k_full[0], 0, abort, p.status);
            if (ok) {
                tc_fence_after();
                if (kt_min >= lo0 && kt_min <= hi0) {
                    ORTHROS_ISSUE_S(d_s0, dq, dk)
                    tc_commit(&mt.s_full[0]);
                }
                if (kt_min >= lo1 && kt_min <= hi1) {
                    ORTHROS_ISSUE_S(d_s1, dq + kTileU, dk)
                    tc_commit(&mt.s_full[1]);
                }
                tc_commit(&mt.k_empty[0]);
            }
            // per tile and slot: PV_s(i), then S_s(i+1) into the TMEM that held P_s(i)
            // (tcgen05.mma from one thread execute in issue order)
            for (int i = 0; ok && i < n_it; ++i) {
                const int kt = kt_min + i;
                const int sv = i % kNumV;
                const uint64_t vdesc = dv + (uint64_t)(sv * kTileU);
                const bool more = i + 1 < n_it;
                const int skn = (i + 1) % kNumK;
                const uint64_t kdesc = dk + (uint64_t)(skn * kTileU);
                if (!(ok = mbar_wait(&mt.v_full[sv], (i / kNumV) & 1, abort, p.status))) break;
                // slot 0
                if (kt >= lo0 && kt <= hi0) {
                    if (!(ok = mbar_wait(&mt.p_full[0], pc0 & 1, abort, p.status))) break;
                    ++pc0;
                    tc_fence_after();
                    ORTHROS_ISSUE_PV(d_o0, d_s0, vdesc, o_init0)
                    o_init0 = 1;
                }
                if (more) {
                    if (!(ok = mbar_wait(&mt.k_full[skn], ((i + 1) / kNumK) & 1, abort, p.status))) break;
                    tc_fence_after();
                    if (kt + 1 >= lo0 && kt + 1 <= hi0) {
                        ORTHROS_ISSUE_S(d_s0, dq, kdesc)
                        tc_commit(&mt.s_full[0]);
                    }
                }
                // slot 1
                if (kt >= lo1 && kt <= hi1) {
                    if (!(ok = mbar_wait(&mt.p_full[1], pc1 & 1, abort, p.status))) break;
                    ++pc1;
                    tc_fence_after();
                    ORTHROS_ISSUE_PV(d_o1, d_s1, vdesc, o_init1)
                    o_init1 = 1;
                }
                if (more) {
                    if (kt + 1 >= lo1 && kt + 1 <= hi1) {
                        ORTHROS_ISSUE_S(d_s1, dq + kTileU, kdesc)
                        tc_commit(&mt.s_full[1]);
                    }
                    tc_commit(&mt.k_empty[skn]);
                }
                tc_commit(&mt.v_empty[sv]);
            }
#undef ORTHROS_ISSUE_S
#undef ORTHROS_ISSUE_PV
            tc_commit(&mt.o_full[0]);
            tc_commit(&mt.o_full[1]);
            tc_commit(&mt.mma_done);
            mbar_wait(&mt.mma_done, 0, abort, p.status);
        }
    } else {
        // ---------------- softmax: two threads per row (one per 64-key half) ----------------
        const int s = s_me, hh = h_me;
        const Slot S = s ? sl1 : sl0;
        const Band bd = s ? bd1 : bd0;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t t_s = tmem + lane_off + s * 128;                // S_s columns of this lane quarter
        const uint32_t t_o = tmem + lane_off + C::kTmemO + s * 128 + hh * (D / 2);  // this half of O_s
        const int t_row = my_valid ? my_t : bd.t_max;
        const int lo_row = S.kind == 0 ? max(0, t_row - p.window + 1) : p.key_lo;
        const float c2 = p.scale_log2;
        const int t_min_s = bd.t_min;
        float m_ref = -INFINITY, l = 0.f;
        uint32_t cnt = 0;
        for (int i = 0; i < n_it; ++i) {
            const int kt = kt_min + i;
            if (kt < bd.kt_lo || kt > bd.kt_hi) continue;
            const bool got = mbar_wait(&mt.s_full[s], cnt & 1, abort, p.status);
            if (!__all_sync(0xffffffffu, got)) break;
            tc_fence_after();
            // this half's 64 logits of the row, in two 32-column loads, one wait
            uint32_t ra[32], rb[32];
            tmem_ld32(t_s + 64 * hh, ra);
            tmem_ld32(t_s + 64 * hh + 32, rb);
            tmem_ld_wait();
            reg_fence(ra);
            reg_fence(rb);
            const int key0 = kt * kKeysPerTile + 64 * hh;
            if (kt * kKeysPerTile + kKeysPerTile - 1 > t_min_s || kt * kKeysPerTile < bd.lo_max) {
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    if (key0 + c > t_row || key0 + c < lo_row) ra[c] = __float_as_uint(-INFINITY);
                    if (key0 + 32 + c > t_row || key0 + 32 + c < lo_row) rb[c] = __float_as_uint(-INFINITY);
                }
            }
            const float *xa = reinterpret_cast<const float *>(ra);
            const float *xb = reinterpret_cast<const float *>(rb);
            float mq[8];
#pragma unroll
            for (int q = 0; q < 8; ++q)
                mq[q] = max3(max3(xa[4 * q], xa[4 * q + 1], xa[4 * q + 2]), max3(xa[4 * q + 3], xb[4 * q], xb[4 * q + 1]),
                             fmaxf(xb[4 * q + 2], xb[4 * q + 3]));
            const float mine = max3(max3(mq[0], mq[1], mq[2]), max3(mq[3], mq[4], mq[5]), fmaxf(mq[6], mq[7]));
            // both halves combine the same two bf16-rounded maxima, so they agree on the shift
            const __nv_bfloat16 mine_b = __float2bfloat16_rn(mine);
            mt.xmax[s][hh][row] = mine_b;
            mbar_arrive(&mt.xm_bar[s]);
            if (!__all_sync(0xffffffffu, mbar_wait(&mt.xm_bar[s], cnt & 1, abort, p.status))) break;
            const float m_tile = fmaxf(__bfloat162float(mine_b), __bfloat162float(mt.xmax[s][hh ^ 1][row]));
            const float m_new = fmaxf(m_ref, m_tile);
            const bool resc = (m_new - m_ref) * c2 > 8.f;  // true on the first finite max
            const bool any_resc = __any_sync(0xffffffffu, resc);
            const float alpha = resc ? ex2((m_ref - m_new) * c2) : 1.f;
            if (resc) {
                l *= alpha;
                m_ref = m_new;
            }
            const float mb = m_ref == -INFINITY ? 0.f : m_ref * c2;
            float ls[4] = {0.f, 0.f, 0.f, 0.f};
            // P for keys 64 hh .. 64 hh + 63 -> packed columns 32 hh .. 32 hh + 31
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const float *x = j ? xb : xa;
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float p0 = ex2(fmaf(x[2 * e], c2, -mb));
                    const float p1 = ex2(fmaf(x[2 * e + 1], c2, -mb));
                    ls[e & 3] += p0 + p1;
                    pk[e] = pack_bf16(p0, p1);
                }
                tmem_st16(t_s + 32 * hh + 16 * j, pk);
            }
            l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
            // O_s is idle here (PV_s of the previous tile completed before S_s of
            // this tile was signalled; the next PV_s waits for p_full): each half
            // rescales its own D/2 columns of the running output.
            if (any_resc && cnt > 0) {
#pragma unroll
                for (int j = 0; j < D / 64; ++j) {
                    uint32_t o[32];
                    tmem_ld32(t_o + 32 * j, o);
                    tmem_ld_wait();
                    reg_fence(o);
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st32(t_o + 32 * j, o);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&mt.p_full[s]);
            ++cnt;
        }
        // ---------------- epilogue: o = O / l, lse = scale*m + ln l ----------------
        // Every MMA has completed once o_full fires, so the key stages and the
        // query tile are idle: row sums are exchanged through the first key
        // stage; a base-position tile's normalised output is staged in its
        // query tile (128-byte swizzle) and leaves by one TMA store (rows past
        // T fall outside the map); output-row tiles store row by row.
        bool have = cnt > 0 && mbar_wait(&mt.o_full[s], 0, abort, p.status);
        have = __all_sync(0xffffffffu, have);
        if (have) {
            tc_fence_after();
            float *lx = reinterpret_cast<float *>(smem + C::kK0 + s * 1024);  // [2][128]
            lx[hh * kRowsPerTile + row] = l;
            mbar_arrive(&mt.lx_bar[s]);
            have = __all_sync(0xffffffffu, mbar_wait(&mt.lx_bar[s], 0, abort, p.status));
            const float l_all = l + lx[(hh ^ 1) * kRowsPerTile + row];
            const bool tile_store = S.kind == 0;  // warp-uniform
            const bool store = have && S.kind >= 0 && row < S.n;
            uint8_t *stage = smem + C::kQ0 + s * C::kTileBytes;
            __nv_bfloat16 *dst = nullptr;
            float *dst32 = nullptr;  // output rows written as float (shard partials)
            float *lse_dst = nullptr;
            if (store && S.kind == 0) {
                lse_dst = p.lse_base + ((long long)S.b * p.Hq + S.h) * p.Tq + (my_t - p.q_off);
            } else if (store) {
                const long long o_off = ((long long)(S.row0 + row) * p.Hq + S.h) * D + hh * (D / 2);
                if (p.o_out_f32) dst32 = p.o_out_f32 + o_off;
                else dst = p.o_out + o_off;
                lse_dst = p.lse_out + (long long)(S.row0 + row) * p.Hq + S.h;
            }
            // a shard's output row before the shard's first key has no keys: o = 0, lse = -inf
            const float inv = my_bad ? __int_as_float(0x7fc00000) : (l_all > 0.f ? 1.f / l_all : 0.f);
#pragma unroll
            for (int j = 0; j < D / 64; ++j) {
                uint32_t o[32];
                tmem_ld32(t_o + 32 * j, o);
                tmem_ld_wait();
                reg_fence(o);
                uint4 w[4];
                uint32_t *wp = reinterpret_cast<uint32_t *>(w);
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    wp[e] = pack_bf16(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
                if (tile_store) {
                    const int c0 = (hh * (D / 2) + 32 * j) / 8;  // first 16-byte chunk of these 32 channels
#pragma unroll
                    for (int e = 0; e < 4; ++e) *reinterpret_cast<uint4 *>(stage + sw128_offset<D>(row, c0 + e)) = w[e];
                } else if (dst32) {
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        reinterpret_cast<float4 *>(dst32 + 32 * j)[e] =
                            make_float4(__uint_as_float(o[4 * e]) * inv, __uint_as_float(o[4 * e + 1]) * inv,
                                        __uint_as_float(o[4 * e + 2]) * inv, __uint_as_float(o[4 * e + 3]) * inv);
                } else if (store) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) reinterpret_cast<uint4 *>(dst + 32 * j)[e] = w[e];
                }
            }
            if (store && hh == 0)
                *lse_dst = my_bad ? __int_as_float(0x7fc00000)
                                  : (l_all > 0.f ? m_ref * p.scale + logf(l_all) : -INFINITY);
            if (tile_store && have) {
                fence_proxy_async_smem();
                mbar_arrive(&mt.os_bar[s]);
                const bool staged = __all_sync(0xffffffffu, mbar_wait(&mt.os_bar[s], 0, abort, p.status));
                if (staged && row == 0 && hh == 0 && lane == 0) {
                    for (int j = 0; j < C::kSub; ++j)
                        tma_store_4d(&tm_ob, stage + j * (kRowsPerTile * 128), 64 * j, S.h, S.row0, S.b);
                    bulk_commit();
                    bulk_wait_read();
                }
            }
        } else if (cnt == 0 && !*abort && S.kind == 1 && row < S.n && my_valid) {
            // no key tile in the slot's band (a shard's rows that all precede its keys)
            const long long o_off = ((long long)(S.row0 + row) * p.Hq + S.h) * D + hh * (D / 2);
            for (int c = 0; c < D / 2; ++c) {
                if (p.o_out_f32) p.o_out_f32[o_off + c] = 0.f;
                else p.o_out[o_off + c] = __float2bfloat16_rn(0.f);
            }
            if (hh == 0) p.lse_out[(long long)(S.row0 + row) * p.Hq + S.h] = -INFINITY;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// [B, T, Hkv, D] 2-byte elements -> 4-D map (D, Hkv, T, B), box (64, 1, 128, 1).
bool make_kv_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int B, int T, int Hkv, int D) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)T, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)Hkv * D * 2, (cuuint64_t)T * Hkv * D * 2};
    cuuint32_t box[4] = {64, 1, kKeysPerTile, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(m, dt, 4, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_d(const TcParams &p, const void *k16, const void *v, int units, cudaStream_t stream) {
    CUtensorMap tk, tv, tq, tqo, tob;
    if (!make_kv_map(&tk, k16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, p.B, p.T, p.Hkv, D) ||
        !make_kv_map(&tv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.B, p.T, p.Hkv, D) ||
        !make_kv_map(&tob, p.o_base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.B, p.Tq, p.Hq, D) ||
        !encode_kv_map_3d(&tq, p.q, (long long)p.B * p.Tq, p.Hq, D, kRowsPerTile) ||
        !encode_kv_map_3d(&tqo, p.q_out ? (const void *)p.q_out : (const void *)p.q,
                          p.q_out ? (long long)p.n_out : (long long)p.B * p.Tq, p.Hq, D, kRowsPerTile))
        return cudaErrorInvalidValue;
    static SmemLimit limit;
    if (cudaError_t e = limit.ensure((const void *)prefill_tc_kernel<D>, Cfg<D>::kSmem); e != cudaSuccess) return e;
    prefill_tc_kernel<D><<<units, kThreads, Cfg<D>::kSmem, stream>>>(tk, tv, tq, tqo, tob, p);
    return cudaGetLastError();
}

}  // namespace

bool encode_kv_map_3d(CUtensorMap *m, const void *base, long long tokens, int Hkv, int d, int box_tokens) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)Hkv, (cuuint64_t)tokens};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)Hkv * d * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)box_tokens};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int tc_units_per_kv(int nblk, int g) { return (g % 2 == 0) ? nblk * (g / 2) : g * ((nblk + 1) / 2); }

cudaError_t launch_prefill_tc(const TcParams &p, const void *k16, const void *v, int d, cudaStream_t stream) {
    const int units = p.n_cross_units + p.n_base_units;
    if (units == 0) return cudaSuccess;
    return d == 128 ? launch_d<128>(p, k16, v, units, stream) : launch_d<64>(p, k16, v, units, stream);
}

}  // namespace orthros
