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
// Design (one CTA per SM; 576 threads, or 320 for windows of 4096 keys and more):
//   * A work unit is two 128-row query tiles that read the SAME key/value
//     tiles: two query heads of one GQA group at the same positions, or (when
//     the group size is odd, e.g. plain multi-head) two consecutive row blocks
//     of one head. Key/value tiles of 128 tokens are visited only inside the
//     union of the tiles' bands; tiles outside the band are never loaded.
//   * the warp after the softmax warps (one thread): TMA producer. Keys come
//     from an fp16 copy made by the pre-pass kernel (3 stages), values in bf16
//     (2 stages), 128B swizzle.
//   * the last warp (one thread): tcgen05.mma issuer. S_s = Q_s K^T (M=128,
//     N=128, fp16 operands from shared memory) into TMEM; O_s += P_s V (M=128,
//     N=d, P read from TMEM as bf16, V from shared memory, MN-major).
//   * softmax warps, two layouts (template kRow):
//     - two threads per row (warps 0-15): warp w serves slot (w >> 2) & 1, key
//       half w >> 3 of each 128-key tile, rows 32 (w & 3) .. +31 (TMEM lane
//       quarter w & 3). A thread reads its 64 logits with tcgen05.ld, masks
//       the two band edge tiles, agrees with its partner on the row's shift,
//       keeps a running max with lazy rescaling (O in TMEM is only rescaled
//       when the max grows by more than 2^8), writes P as packed bf16 back
//       over its logits, and finally normalises its half of O and stores o
//       and lse. 96 registers a thread.
//     - one thread per row (warps 0-7, windows of 4096 keys and more): warp w
//       serves slot w >> 2, rows 32 (w & 3) .. +31, all 128 logits of a tile
//       at once, with no exchange between threads; it stages and stores the
//       whole row, gathering its query from global memory (prefetched into L2
//       one unit ahead) instead of a TMA tile. 168 registers a thread: its
//       tiles are faster, its unit boundaries slower, so it is taken where
//       units are long.
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
// Two layouts of the softmax warps. kRow = false: two threads per row (one per
// 64-key half), 16 softmax warps, 18 in all: five warps on two of the four
// schedulers leave 96 registers a thread. kRow = true: one thread per row, 8
// softmax warps, 10 in all: three warps on two schedulers leave 168 registers
// a thread (3 x 32 x 168 fits a scheduler's 16K), so the register bound is
// taken for 384 threads while the launch has 320.
template <bool kRow> struct Warps {
    static constexpr int kSoftmax = kRow ? 8 : 16;   // 2 slots x (2 halves x) 4 lane quarters
    static constexpr int kThreads = (kSoftmax + 2) * 32;
    static constexpr int kProducer = kSoftmax;
    static constexpr int kMma = kSoftmax + 1;
    static constexpr int kBound = kRow ? 384 : kThreads;
    static constexpr int kPerRow = kRow ? 1 : 2;      // softmax threads per row
};
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

// 2^e for an integer e in [-126, 127] (exact).
__device__ __forceinline__ float exp2_int(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }

struct Slot {
    int kind;  // 0 base positions, 1 output rows, -1 empty
    int b, h, row0, n;
    int qrow;  // first row of the raw query tile in q (or q_out) when its rows are contiguous there, else -1
};

// Band of a slot in key-tile units: [kt_lo, kt_hi]; lo_max = latest window
// start of its rows (key tiles before it need the window mask); t_min / t_max
// = first / last position of its usable rows.
struct Band {
    int kt_lo, kt_hi, lo_max, t_min, t_max;
};

// What every role needs to know about one work unit (written by the
// producer, read by the MMA issuer and the softmax warps).
struct UnitDesc {
    Slot sl[2];
    Band bd[2];
    int kt_min, n_it;  // key tiles kt_min .. kt_min + n_it - 1: the union of the two bands
    int end;           // no more units: every role leaves its loop
};

constexpr int kDescRing = 2;  // unit descriptors in flight

struct Meta {
    uint64_t k_full[kNumK], k_empty[kNumK], v_full[kNumV], v_empty[kNumV];
    uint64_t s_full[2], p_full[2], o_full[2], mma_done;
    uint64_t q_full[2];   // per slot: raw query tile landed (TMA) or nothing to land (gathered / empty)
    uint64_t q_ready[2];  // per slot: affined query tile staged for the products
    uint64_t q_free[2];   // per slot: the unit is done with its query tile (epilogue stored)
    uint64_t os_bar[2];   // per slot: normalised output tile staged for the TMA store
    uint64_t xm_bar[2], lx_bar[2];  // per slot: row maxima / row sums exchanged between column halves
                                    // (xm_bar completes one phase per s_full phase)
    uint64_t u_full[kDescRing], u_empty[kDescRing];  // unit descriptor ring
    uint32_t tmem_base;
    int abort;
    int n_redo;  // second launch: row blocks this CTA lists to compute again
    UnitDesc desc[kDescRing];
    __nv_bfloat16 xmax[2][2][kRowsPerTile];  // [slot][half][row] tile maxima (a shared shift; rounding is harmless)
};
static_assert(sizeof(Meta) <= 1536, "barriers and metadata must fit their shared-memory region");

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
    // base rows are contiguous in q, output rows in q_out; output rows that
    // read q at their positions are checked for contiguity by make_desc
    for (Slot *S : {&s0, &s1})
        S->qrow = S->kind == 0 ? S->b * p.Tq + S->row0 : (S->kind == 1 && p.q_out ? S->row0 : -1);
}

// Second launch: row block idx as slot 0 of a unit. Blocks [0, B Hq nblk) are
// base-position blocks (b, h, blk); the rest are output-row blocks of the
// sequences whose output rows take this kernel, out_blk_indptr[b] of them
// before sequence b, head-major within a sequence.
__device__ void decode_block(const TcParams &p, int idx, Slot &S) {
    const int nb_base = p.B * p.Hq * p.base_nblk;
    if (idx < nb_base) {
        const int b = idx / (p.Hq * p.base_nblk), rem = idx % (p.Hq * p.base_nblk);
        S.kind = 0;
        S.b = b;
        S.h = rem / p.base_nblk;
        S.row0 = (rem % p.base_nblk) * kRowsPerTile;
        S.n = min(kRowsPerTile, p.Tq - S.row0);
        S.qrow = b * p.Tq + S.row0;
        return;
    }
    const int o = idx - nb_base;
    int lo = 0, hi = p.B - 1;  // last b with out_blk_indptr[b] <= o
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.out_blk_indptr[mid] <= o) lo = mid; else hi = mid - 1;
    }
    const int b = lo, local = o - p.out_blk_indptr[b];
    const int rows = p.out_indptr[b + 1] - p.out_indptr[b];
    const int nbb = (rows + kRowsPerTile - 1) / kRowsPerTile;
    S.kind = 1;
    S.b = b;
    S.h = local / nbb;
    S.row0 = p.out_indptr[b] + (local % nbb) * kRowsPerTile;
    S.n = min(kRowsPerTile, p.out_indptr[b + 1] - S.row0);
    S.qrow = p.q_out ? S.row0 : -1;
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

// Position (in key coordinates) of output row r and whether the row is usable:
// its position lies in [0, T) (a shard's rows past its keys read them all), and
// without q_out the base query at that position exists.
__device__ __forceinline__ bool out_row_position(const TcParams &p, int r, int &te) {
    const int t = p.out_positions[r];
    te = p.shard ? min(t, p.T - 1) : t;
    bool ok = t >= 0 && (p.shard || t < p.T);
    if (!p.q_out && (te < p.q_off || te - p.q_off >= p.Tq)) ok = false;
    return ok;
}

__device__ __forceinline__ Band band_of(const TcParams &p, const Slot &S, int tmin, int tmax) {
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
}

// Descriptor of unit u (u < 0: the end marker). Called by all 32 lanes of the
// producer warp, which read an output-row slot's positions together; every
// lane returns the same descriptor.
__device__ void make_desc(const TcParams &p, int u, int lane, UnitDesc &D, bool block_unit) {
    D.end = u < 0;
    D.kt_min = 0;
    D.n_it = 0;
    if (D.end) {
        for (int s = 0; s < 2; ++s) {
            D.sl[s] = Slot{-1, 0, 0, 0, 0, -1};
            D.bd[s] = Band{1, 0, 0, 0, -1};
        }
        return;
    }
    if (block_unit) {
        decode_block(p, u, D.sl[0]);
        D.sl[1] = Slot{-1, 0, 0, 0, 0, -1};
    } else {
        decode_unit(p, u, D.sl[0], D.sl[1]);
    }
    for (int s = 0; s < 2; ++s) {
        const Slot S = D.sl[s];
        int tmin = 0x7fffffff, tmax = -1;
        if (S.kind == 0) {
            tmin = S.row0 + p.q_off;
            tmax = S.row0 + S.n - 1 + p.q_off;
        } else if (S.kind == 1) {
            // output rows at consecutive positions (an answer span, every position)
            // have their raw queries contiguous in q: one TMA tile instead of a gather
            const int t_first = p.out_positions[S.row0];
            bool contig = !p.q_out;
            for (int r = lane; r < S.n; r += 32) {
                int te;
                const bool ok = out_row_position(p, S.row0 + r, te);
                if (ok) {
                    tmin = min(tmin, te);
                    tmax = max(tmax, te);
                }
                contig = contig && ok && p.out_positions[S.row0 + r] == t_first + r;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                tmin = min(tmin, __shfl_xor_sync(0xffffffffu, tmin, o));
                tmax = max(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
            }
            contig = __all_sync(0xffffffffu, contig);
            if (contig) D.sl[s].qrow = S.b * p.Tq + (t_first - p.q_off);
        }
        D.bd[s] = band_of(p, S, tmin, tmax);
    }
    const Band &b0 = D.bd[0], &b1 = D.bd[1];
    const bool any0 = b0.kt_lo <= b0.kt_hi, any1 = b1.kt_lo <= b1.kt_hi;
    if (any0 || any1) {
        D.kt_min = any0 && any1 ? min(b0.kt_lo, b1.kt_lo) : (any0 ? b0.kt_lo : b1.kt_lo);
        const int kt_max = any0 && any1 ? max(b0.kt_hi, b1.kt_hi) : (any0 ? b0.kt_hi : b1.kt_hi);
        D.n_it = kt_max - D.kt_min + 1;
    }
}

// kRedo: the second launch. Each CTA scans a slice of the log-sum-exps for
// rows that came out non-finite although they have keys (a staged query value
// past the fp16 range gives such rows) and computes their row blocks again,
// every row staged with its own power-of-two shift and the inverse shift on
// its logit scale. Without such rows every CTA leaves after the scan.
template <int D, bool kRedo, bool kRow>
__global__ void __launch_bounds__(Warps<kRow>::kBound, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_qo,
                      const __grid_constant__ CUtensorMap tm_ob, const TcParams p) {
    using C = Cfg<D>;
    using Wp = Warps<kRow>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Meta &mt = *reinterpret_cast<Meta *>(smem + C::kBar);
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    volatile int *abort = &mt.abort;
    const int total_units = p.n_cross_units + p.n_base_units;
    // The second launch is a programmatic dependent launch: its CTAs may start
    // as the first launch's leave, and wait here until all of it has finished.
    if constexpr (kRedo) asm volatile("griddepcontrol.wait;" ::: "memory");
    else asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

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
            mbar_init(&mt.p_full[s], Wp::kPerRow * kRowsPerTile);
            mbar_init(&mt.o_full[s], 1);
            mbar_init(&mt.xm_bar[s], 2 * kRowsPerTile);
            mbar_init(&mt.lx_bar[s], 2 * kRowsPerTile);
            mbar_init(&mt.q_full[s], 1);
            mbar_init(&mt.q_ready[s], Wp::kPerRow * kRowsPerTile);
            mbar_init(&mt.q_free[s], Wp::kPerRow * kRowsPerTile);
            mbar_init(&mt.os_bar[s], Wp::kPerRow * kRowsPerTile);
        }
        for (int r = 0; r < kDescRing; ++r) {
            mbar_init(&mt.u_full[r], 1);
            mbar_init(&mt.u_empty[r], Wp::kSoftmax + 1);
        }
        mbar_init(&mt.mma_done, 1);
        mt.abort = 0;
        mt.n_redo = 0;
        fence_mbar_init();
    }
    if (warp == Wp::kProducer && lane == 0) {
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_qo);
        prefetch_tmap(&tm_ob);
    }
    __syncthreads();
    // Second launch: this CTA scans its slice of the log-sum-exps (lse_base,
    // then lse_out, as one flat range; coalesced) for rows that have keys but a
    // non-finite value. The first CTA to find a row block claims it in the
    // bitmap redo_bits (zeroed before the first launch) and lists it in its own
    // part of redo_list (one entry per scanned value at most), so every block is
    // computed again once, by the CTA that found it.
    long long redo_lo = 0;
    if constexpr (kRedo) {
        const long long fb = (long long)p.B * p.Hq * p.Tq, ft = fb + (long long)p.n_out * p.Hq;
        const long long per = (ft + gridDim.x - 1) / gridDim.x;
        redo_lo = min((long long)blockIdx.x * per, ft);
        const long long redo_hi = min(redo_lo + per, ft);
        const int nb_base = p.B * p.Hq * p.base_nblk;
        auto claim = [&](long long f) {
            int idx;
            if (f < fb) {
                idx = (int)(f / p.Tq) * p.base_nblk + (int)(f % p.Tq) / kRowsPerTile;
            } else {
                const int row = (int)((f - fb) / p.Hq), h = (int)((f - fb) % p.Hq);
                int te;
                if (!out_row_position(p, row, te) || te < p.key_lo) return;  // NaN by design / no keys
                int lo = 0, hi = p.B - 1;  // the row's sequence: last b with out_indptr[b] <= row
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (p.out_indptr[mid] <= row) lo = mid; else hi = mid - 1;
                }
                const int b = lo;
                if (p.out_blk_indptr[b + 1] == p.out_blk_indptr[b]) return;  // rows of the split-KV kernel
                const int nbb = (p.out_indptr[b + 1] - p.out_indptr[b] + kRowsPerTile - 1) / kRowsPerTile;
                idx = nb_base + p.out_blk_indptr[b] + h * nbb + (row - p.out_indptr[b]) / kRowsPerTile;
            }
            const uint32_t m = 1u << (idx & 31);
            if (!(atomicOr(&p.redo_bits[idx >> 5], m) & m)) p.redo_list[redo_lo + atomicAdd(&mt.n_redo, 1)] = idx;
        };
        constexpr int kBatch = 8;  // loads in flight per thread
        for (long long f0 = redo_lo + tid; f0 < redo_hi; f0 += (long long)kBatch * Wp::kThreads) {
            float x[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const long long f = f0 + (long long)j * Wp::kThreads;
                x[j] = f >= redo_hi ? 0.f : __ldcg(f < fb ? p.lse_base + f : p.lse_out + (f - fb));
            }
#pragma unroll
            for (int j = 0; j < kBatch; ++j)
                if (!(fabsf(x[j]) <= 3.4e38f)) claim(f0 + (long long)j * Wp::kThreads);
        }
        __syncthreads();
        if (mt.n_redo == 0) return;  // the common case: nothing to compute again
    }
    if (warp == Wp::kMma) {
        tmem_alloc(&mt.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = mt.tmem_base;

    // Query tiles whose rows are contiguous in q or q_out (base positions;
    // output rows with their own q_out or at consecutive positions) arrive by
    // TMA as raw bf16 and are turned into affined fp16 in place; other output
    // rows are gathered by the softmax threads.

    if (warp == Wp::kProducer) {
        // ---------------- producer: unit descriptors, then TMA loads ----------------
        // Takes units from a device-wide counter (heaviest first: the numbering
        // puts output-row units and late row blocks first), publishes each
        // unit's descriptor, and streams its K/V tiles through the rings with
        // phases that run on across units. The first K/V tiles of a unit go
        // out before its query tiles, which wait for the previous unit's
        // epilogue to release the query buffers.
        uint32_t gk = 0;            // K/V iterations issued (all units so far)
        uint32_t nq[2] = {0, 0};    // per slot: units whose query phase was armed
        // Descriptors run one unit ahead of the loads, so the other roles never
        // wait for the next unit's counter fetch and position reads.
        int taken = 0;  // second launch: blocks of this CTA's list taken so far
        auto next_desc = [&](UnitDesc &ud) {
            int u = 0;
            if constexpr (kRedo) {
                u = taken < mt.n_redo ? __ldcg(p.redo_list + redo_lo + taken) : -1;
                ++taken;
            } else {
                if (lane == 0) u = atomicAdd(p.unit_counter, 1);
                u = __shfl_sync(0xffffffffu, u, 0);
                u = u < total_units ? u : -1;
            }
            make_desc(p, u, lane, ud, kRedo);
        };
        auto publish = [&](int i, const UnitDesc &ud) -> bool {
            const int r = i % kDescRing;
            if (i >= kDescRing && !mbar_wait_warp(&mt.u_empty[r], ((i / kDescRing) - 1) & 1, abort, p.status))
                return false;
            if (lane == 0) {
                mt.desc[r] = ud;
                mbar_arrive(&mt.u_full[r]);  // releases the descriptor to the other roles
            }
            __syncwarp();
            return true;
        };
        UnitDesc dsc;
        next_desc(dsc);
        bool alive = publish(0, dsc);
        for (int i = 0; alive && !dsc.end; ++i) {
            UnitDesc nxt;
            next_desc(nxt);
            if (!publish(i + 1, nxt)) break;
            if (lane == 0) {
                const int kvh = dsc.sl[0].h / (p.Hq / p.Hkv);
                const int bseq = dsc.sl[0].b;
                auto issue_kv = [&](int it) -> bool {
                    const uint32_t g = gk + it;
                    const int kt = dsc.kt_min + it;
                    const int sk = g % kNumK, sv = g % kNumV;
                    if (g >= (uint32_t)kNumK && !mbar_wait(&mt.k_empty[sk], ((g / kNumK) - 1) & 1, abort, p.status))
                        return false;
                    mbar_arrive_expect_tx(&mt.k_full[sk], C::kTileBytes);
                    for (int j = 0; j < C::kSub; ++j)
                        tma_load_4d(smem + C::kK0 + sk * C::kTileBytes + j * (kKeysPerTile * 128), &tm_k,
                                    &mt.k_full[sk], 64 * j, kvh, kt * kKeysPerTile, bseq);
                    if (g >= (uint32_t)kNumV && !mbar_wait(&mt.v_empty[sv], ((g / kNumV) - 1) & 1, abort, p.status))
                        return false;
                    mbar_arrive_expect_tx(&mt.v_full[sv], C::kTileBytes);
                    for (int j = 0; j < C::kSub; ++j)
                        tma_load_4d(smem + C::kV0 + sv * C::kTileBytes + j * (kKeysPerTile * 128), &tm_v,
                                    &mt.v_full[sv], 64 * j, kvh, kt * kKeysPerTile, bseq);
                    return true;
                };
                auto issue_q = [&](int s) -> bool {
                    if (i >= 1 && !mbar_wait(&mt.q_free[s], (i - 1) & 1, abort, p.status)) return false;
                    const Slot &S = dsc.sl[s];
                    nq[s] = i + 1;
                    if (!kRow && S.qrow >= 0) {  // (the one-thread-per-row layout gathers its rows)
                        mbar_arrive_expect_tx(&mt.q_full[s], C::kTileBytes);
                        for (int j = 0; j < C::kSub; ++j)
                            tma_load_3d(smem + C::kQ0 + s * C::kTileBytes + j * (kRowsPerTile * 128),
                                        S.kind == 1 && p.q_out ? &tm_qo : &tm_q, &mt.q_full[s], 64 * j, S.h, S.qrow);
                    } else {
                        mbar_arrive(&mt.q_full[s]);  // nothing to copy (gathered rows or an empty slot)
                    }
                    return true;
                };
                // the first tile's key/value loads need only stages the previous
                // unit has released; the query tiles wait for its epilogue
                bool ok = dsc.n_it == 0 || issue_kv(0);
                ok = ok && issue_q(0);
                ok = ok && issue_q(1);
                for (int it = 1; ok && it < dsc.n_it; ++it) ok = issue_kv(it);
                gk += dsc.n_it;
                alive = ok;
            }
            alive = __shfl_sync(0xffffffffu, alive, 0);
            dsc = nxt;
        }
        if (lane == 0) {
            // nothing may be in flight when the CTA leaves: wait (bounded) for the
            // copies of the last stages and query tiles issued
            for (uint32_t g = gk > (uint32_t)kNumK ? gk - kNumK : 0; g < gk; ++g)
                mbar_wait_drain(&mt.k_full[g % kNumK], (g / kNumK) & 1, p.status);
            for (uint32_t g = gk > (uint32_t)kNumV ? gk - kNumV : 0; g < gk; ++g)
                mbar_wait_drain(&mt.v_full[g % kNumV], (g / kNumV) & 1, p.status);
            for (int s = 0; s < 2; ++s)
                if (nq[s] > 0) mbar_wait_drain(&mt.q_full[s], (nq[s] - 1) & 1, p.status);
        }
    } else if (warp == Wp::kMma) {
        // ---------------- tcgen05.mma issuer ----------------
        if (lane == 0) {
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
            uint32_t g = 0;              // K/V iterations consumed (all units so far)
            uint32_t pc0 = 0, pc1 = 0;   // P tiles consumed per slot
            uint32_t qr0 = 0, qr1 = 0;   // second launch: q_ready phases consumed per slot
            bool ok = true;
            for (int i = 0; ok; ++i) {
                const int r = i % kDescRing;
                if (!(ok = mbar_wait(&mt.u_full[r], (i / kDescRing) & 1, abort, p.status))) break;
                const UnitDesc &dr = mt.desc[r];
                const int end = dr.end;
                const int lo0 = dr.bd[0].kt_lo, hi0 = dr.bd[0].kt_hi, lo1 = dr.bd[1].kt_lo, hi1 = dr.bd[1].kt_hi;
                const int kt_min = dr.kt_min, n_it = dr.n_it;
                mbar_arrive(&mt.u_empty[r]);
                if (end) break;
                // Second launch: a slot with key tiles gets, in place of its first
                // product, a go-ahead on s_full to stage its rows again with per-row
                // shifts; the products wait for that second staging (two q_ready
                // phases per unit there, one in the first launch).
                auto restage = [&](int sl, int lo, int hi, uint32_t &qr) -> bool {
                    if (!kRedo || max(lo, kt_min) > min(hi, kt_min + n_it - 1)) return true;
                    mbar_arrive(&mt.s_full[sl]);
                    if (!mbar_wait(&mt.q_ready[sl], qr & 1, abort, p.status)) return false;
                    ++qr;
                    return true;
                };
                // each slot's query tile staged before its first product (this also
                // orders the product after that slot's previous epilogue)
                if (!(ok = mbar_wait(&mt.q_ready[0], (kRedo ? qr0 : (uint32_t)i) & 1, abort, p.status))) break;
                if (kRedo) ++qr0;
                if (n_it == 0) {
                    if (!(ok = mbar_wait(&mt.q_ready[1], (kRedo ? qr1 : (uint32_t)i) & 1, abort, p.status))) break;
                    if (kRedo) ++qr1;
                    continue;
                }
                if (!(ok = restage(0, lo0, hi0, qr0))) break;
                if (!(ok = mbar_wait(&mt.k_full[g % kNumK], (g / kNumK) & 1, abort, p.status))) break;
                tc_fence_after();
                const uint64_t dk0 = dk + (uint64_t)((g % kNumK) * kTileU);
                if (kt_min >= lo0 && kt_min <= hi0) {
                    ORTHROS_ISSUE_S(d_s0, dq, dk0)
                    tc_commit(&mt.s_full[0]);
                }
                if (!(ok = mbar_wait(&mt.q_ready[1], (kRedo ? qr1 : (uint32_t)i) & 1, abort, p.status))) break;
                if (kRedo) ++qr1;
                if (!(ok = restage(1, lo1, hi1, qr1))) break;
                tc_fence_after();
                if (kt_min >= lo1 && kt_min <= hi1) {
                    ORTHROS_ISSUE_S(d_s1, dq + kTileU, dk0)
                    tc_commit(&mt.s_full[1]);
                }
                tc_commit(&mt.k_empty[g % kNumK]);
                // per tile and slot: PV_s(i), then S_s(i+1) into the TMEM that held P_s(i)
                // (tcgen05.mma from one thread execute in issue order)
                uint32_t o_init0 = 0, o_init1 = 0;
                for (int it = 0; ok && it < n_it; ++it) {
                    const uint32_t gi = g + it;
                    const int kt = kt_min + it;
                    const int sv = gi % kNumV;
                    const uint64_t vdesc = dv + (uint64_t)(sv * kTileU);
                    const bool more = it + 1 < n_it;
                    const int skn = (gi + 1) % kNumK;
                    const uint64_t kdesc = dk + (uint64_t)(skn * kTileU);
                    if (!(ok = mbar_wait(&mt.v_full[sv], (gi / kNumV) & 1, abort, p.status))) break;
                    // slot 0
                    if (kt >= lo0 && kt <= hi0) {
                        if (!(ok = mbar_wait(&mt.p_full[0], pc0 & 1, abort, p.status))) break;
                        ++pc0;
                        tc_fence_after();
                        ORTHROS_ISSUE_PV(d_o0, d_s0, vdesc, o_init0)
                        o_init0 = 1;
                        if (kt == hi0) tc_commit(&mt.o_full[0]);  // slot 0's epilogue may start
                    }
                    if (more) {
                        if (!(ok = mbar_wait(&mt.k_full[skn], ((gi + 1) / kNumK) & 1, abort, p.status))) break;
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
                        if (kt == hi1) tc_commit(&mt.o_full[1]);
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
                if (!ok) break;
                g += n_it;
            }
#undef ORTHROS_ISSUE_S
#undef ORTHROS_ISSUE_PV
            // every product issued must be complete before tensor memory is freed
            tc_commit(&mt.mma_done);
            mbar_wait_drain(&mt.mma_done, 0, p.status);
        }
    } else if constexpr (kRow) {
        // ---------------- softmax: one thread per row ----------------
        // Softmax warp w: slot w >> 2, rows 32 (w & 3) .. +31 (TMEM lane quarter
        // w & 3); each thread holds its row's 128 logits of a tile at once.
        const int s = warp >> 2;
        const int row = ((warp & 3) << 5) | lane;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t t_s = tmem + lane_off + s * 128;               // S_s columns of this lane quarter
        const uint32_t t_o = tmem + lane_off + C::kTmemO + s * 128;  // O_s
        const float c2 = p.scale_log2;
        uint8_t *qs = smem + C::kQ0 + s * C::kTileBytes;
        constexpr int kChunks = D / 8;  // 16-byte chunks of a row
        uint32_t cnt = 0;    // S tiles of this slot handled (all units so far)
        uint32_t ucnt = 0;   // units in which this slot had tiles
        uint32_t bcnt = 0;   // base-position tiles stored
        bool stored = false; // this thread issued TMA stores
        for (int i = 0;; ++i) {
            const int r = i % kDescRing;
            if (!mbar_wait_warp(&mt.u_full[r], (i / kDescRing) & 1, abort, p.status)) break;
            const UnitDesc &dr = mt.desc[r];
            const int end = dr.end;
            const Slot S = dr.sl[s];
            const Band bd = dr.bd[s];
            const int kt_min = dr.kt_min, n_it = dr.n_it;
            __syncwarp();
            if (lane == 0) mbar_arrive(&mt.u_empty[r]);
            if (end) break;

            // ---- the row's position and its query, affine fused ----
            int my_t = 0;  // the row's position in key coordinates
            bool my_valid = false, my_bad = false;
            if (S.kind >= 0 && row < S.n) {
                if (S.kind == 0) {
                    my_t = S.row0 + row + p.q_off;
                    my_valid = true;
                } else {
                    my_valid = out_row_position(p, S.row0 + row, my_t);
                }
                my_bad = !my_valid;
                if (my_bad) set_status(p.status, ORTHROS_DEV_BAD_POSITION);
            }
            const bool tma = false;  // gathered in this layout
            if (!mbar_wait_warp(&mt.q_full[s], i & 1, abort, p.status)) break;
            if (S.kind >= 0) {
                if (my_valid) {
                    const float *al = (S.kind == 0 ? p.alpha_base : p.alpha_out) + S.h * D;
                    const float *be = (S.kind == 0 ? p.beta_base : p.beta_out) + S.h * D;
                    const __nv_bfloat16 *src =
                        (S.kind == 1 && p.q_out) ? p.q_out + ((long long)(S.row0 + row) * p.Hq + S.h) * D
                                                 : p.q + (((long long)S.b * p.Tq + (my_t - p.q_off)) * p.Hq + S.h) * D;
                    // two passes of half a row each: every load of a pass in flight at once
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        uint4 raws[kChunks / 2];
#pragma unroll
                        for (int cc = 0; cc < kChunks / 2; ++cc) {
                            const int c = hh * (kChunks / 2) + cc;
                            raws[cc] = tma ? *reinterpret_cast<const uint4 *>(qs + sw128_offset<D>(row, c))
                                           : reinterpret_cast<const uint4 *>(src)[c];
                        }
#pragma unroll
                        for (int cc = 0; cc < kChunks / 2; ++cc) {
                            const int c = hh * (kChunks / 2) + cc;
                            const uint4 raw = raws[cc];
                            const float4 a0 = reinterpret_cast<const float4 *>(al)[2 * c];
                            const float4 a1 = reinterpret_cast<const float4 *>(al)[2 * c + 1];
                            const float4 b0 = reinterpret_cast<const float4 *>(be)[2 * c];
                            const float4 b1 = reinterpret_cast<const float4 *>(be)[2 * c + 1];
                            const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&raw);
                            float2 x0 = __bfloat1622float2(h2[0]), x1 = __bfloat1622float2(h2[1]);
                            float2 x2 = __bfloat1622float2(h2[2]), x3 = __bfloat1622float2(h2[3]);
                            uint4 o;
                            o.x = pack_f16(fmaf(a0.x, x0.x, b0.x), fmaf(a0.y, x0.y, b0.y));
                            o.y = pack_f16(fmaf(a0.z, x1.x, b0.z), fmaf(a0.w, x1.y, b0.w));
                            o.z = pack_f16(fmaf(a1.x, x2.x, b1.x), fmaf(a1.y, x2.y, b1.y));
                            o.w = pack_f16(fmaf(a1.z, x3.x, b1.z), fmaf(a1.w, x3.y, b1.w));
                            *reinterpret_cast<uint4 *>(qs + sw128_offset<D>(row, c)) = o;
                        }
                    }
                } else {
#pragma unroll 4
                    for (int c = 0; c < kChunks; ++c)
                        *reinterpret_cast<uint4 *>(qs + sw128_offset<D>(row, c)) = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
            }
            mbar_arrive(&mt.q_ready[s]);

            // ---- tiles: S -> P (online softmax), band mask on edge tiles only ----
            const int t_row = my_valid ? my_t : bd.t_max;
            const int lo_row = S.kind == 0 ? max(0, t_row - p.window + 1) : p.key_lo;
            const int t_min_s = bd.t_min;
            float m_ref = -INFINITY, l = 0.f;
            bool ok = true;
            uint32_t tiles = 0;
            int row_shift = 0;  // second launch: the products give this row's logits times 2^-row_shift
            if (kRedo && max(bd.kt_lo, kt_min) <= min(bd.kt_hi, kt_min + n_it - 1)) {
                // The issuer's go-ahead comes in place of the first product: each row is
                // staged again as qa * 2^-r, r the smallest shift that brings its largest
                // value below 2^15.
                ok = __all_sync(0xffffffffu, mbar_wait(&mt.s_full[s], cnt & 1, abort, p.status));
                ++cnt;
                if (ok) {
                    const float *al = (S.kind == 0 ? p.alpha_base : p.alpha_out) + S.h * D;
                    const float *be = (S.kind == 0 ? p.beta_base : p.beta_out) + S.h * D;
                    float amax = 0.f;
                    const __nv_bfloat16 *src = nullptr;
                    if (my_valid) {
                        src = S.qrow >= 0
                                  ? (S.kind == 1 && p.q_out ? p.q_out : p.q) + ((long long)(S.qrow + row) * p.Hq + S.h) * D
                                  : p.q + (((long long)S.b * p.Tq + (my_t - p.q_off)) * p.Hq + S.h) * D;
                        for (int ch = 0; ch < D; ++ch)
                            amax = fmaxf(amax, fabsf(fmaf(al[ch], __bfloat162float(src[ch]), be[ch])));
                    }
                    if (amax > 65504.f && __float_as_uint(amax) < 0x7f800000u)
                        row_shift = min((int)((__float_as_uint(amax) >> 23) & 0xff) - 127 - 14, 126);
                    if (my_valid && row_shift > 0) {
                        const float f = exp2_int(-row_shift);
                        for (int c = 0; c < kChunks; ++c) {
                            float qa[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                qa[e] = fmaf(al[8 * c + e], __bfloat162float(src[8 * c + e]), be[8 * c + e]) * f;
                            uint4 o;
                            o.x = pack_f16(qa[0], qa[1]);
                            o.y = pack_f16(qa[2], qa[3]);
                            o.z = pack_f16(qa[4], qa[5]);
                            o.w = pack_f16(qa[6], qa[7]);
                            *reinterpret_cast<uint4 *>(qs + sw128_offset<D>(row, c)) = o;
                        }
                    }
                    fence_proxy_async_smem();
                    mbar_arrive(&mt.q_ready[s]);
                    ok = __all_sync(0xffffffffu, mbar_wait(&mt.s_full[s], cnt & 1, abort, p.status));
                }
                if (!ok) break;
            }
            const float c2u = kRedo ? c2 * exp2_int(row_shift) : c2;  // the row's logit scale
            for (int it = 0; it < n_it; ++it) {
                const int kt = kt_min + it;
                if (kt < bd.kt_lo || kt > bd.kt_hi) continue;
                if (!kRedo || tiles > 0) {  // (second launch: the first tile's wait came above)
                    const bool got = mbar_wait(&mt.s_full[s], cnt & 1, abort, p.status);
                    if (!(ok = __all_sync(0xffffffffu, got))) break;
                }
                tc_fence_after();
                // the row's 128 logits, in four 32-column loads, one wait
                uint32_t xr[kKeysPerTile];
                using Cols = uint32_t[32];
#pragma unroll
                for (int q = 0; q < kKeysPerTile / 32; ++q)
                    tmem_ld32(t_s + 32 * q, *reinterpret_cast<Cols *>(xr + 32 * q));
                tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < kKeysPerTile / 32; ++q) reg_fence(*reinterpret_cast<Cols *>(xr + 32 * q));
                const int key0 = kt * kKeysPerTile;
                if (key0 + kKeysPerTile - 1 > t_min_s || key0 < bd.lo_max) {
#pragma unroll
                    for (int c = 0; c < kKeysPerTile; ++c)
                        if (key0 + c > t_row || key0 + c < lo_row) xr[c] = __float_as_uint(-INFINITY);
                }
                const float *x = reinterpret_cast<const float *>(xr);
                float mq[16];
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    mq[q] = max3(max3(x[8 * q], x[8 * q + 1], x[8 * q + 2]), max3(x[8 * q + 3], x[8 * q + 4], x[8 * q + 5]),
                                 fmaxf(x[8 * q + 6], x[8 * q + 7]));
                const float m_tile = max3(max3(max3(mq[0], mq[1], mq[2]), max3(mq[3], mq[4], mq[5]), max3(mq[6], mq[7], mq[8])),
                                          max3(mq[9], mq[10], mq[11]), max3(mq[12], mq[13], fmaxf(mq[14], mq[15])));
                const float m_new = fmaxf(m_ref, m_tile);
                const bool resc = (m_new - m_ref) * c2u > 8.f;  // true on the first finite max
                const bool any_resc = __any_sync(0xffffffffu, resc);
                const float alpha = resc ? ex2((m_ref - m_new) * c2u) : 1.f;
                if (resc) {
                    l *= alpha;
                    m_ref = m_new;
                }
                const float mb = m_ref == -INFINITY ? 0.f : m_ref * c2u;
                float ls[4] = {0.f, 0.f, 0.f, 0.f};
                // (c2, c2) and (-mb, -mb) as f32x2 operands: the scaled, shifted logits and
                // the row sums take one packed instruction per pair of keys
                const uint64_t cv = f32x2(c2u, c2u), mv = f32x2(-mb, -mb);
                // P for keys 32 j .. 32 j + 31 -> packed columns 16 j .. 16 j + 15 (over
                // logits this thread has already read)
#pragma unroll
                for (int j = 0; j < kKeysPerTile / 32; ++j) {
                    const float *xj = x + 32 * j;
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float a0, a1;
                        fma_f32x2(xj[2 * e], xj[2 * e + 1], cv, mv, a0, a1);
                        // the row's last pair on the FMA pipe, the other 126
                        // exponentials on the special-function unit
                        float p0, p1;
                        if (j == kKeysPerTile / 32 - 1 && e == 15) exp2_fma_x2(a0, a1, p0, p1);
                        else p0 = ex2(a0), p1 = ex2(a1);
                        add_f32x2(ls[2 * (e & 1)], ls[2 * (e & 1) + 1], p0, p1);
                        pk[e] = pack_bf16(p0, p1);
                    }
                    tmem_st16(t_s + 16 * j, pk);
                }
                l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
                // O_s is idle here (PV_s of the previous tile completed before S_s of
                // this tile was signalled; the next PV_s waits for p_full)
                if (any_resc && tiles > 0) {
#pragma unroll
                    for (int j = 0; j < D / 32; ++j) {
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
                ++tiles;
            }
            if (!ok) break;
            if (kRedo) m_ref *= exp2_int(row_shift);  // back to logit units for the epilogue
            // The next unit's query rows into L2 now (this layout gathers its rows
            // from global memory at the staging), so that their loads there hit
            // L2: the descriptor ring runs a unit ahead of the softmax.
            {
                const int r2 = (i + 1) % kDescRing;
                if (mbar_wait_warp(&mt.u_full[r2], ((i + 1) / kDescRing) & 1, abort, p.status)) {
                    const UnitDesc &d2 = mt.desc[r2];
                    const Slot S2 = d2.sl[s];
                    if (!d2.end && S2.kind >= 0 && row < S2.n) {
                        int t2 = 0;
                        bool v2 = true;
                        if (S2.kind == 0) t2 = S2.row0 + row + p.q_off;
                        else if (!p.q_out) v2 = out_row_position(p, S2.row0 + row, t2);
                        if (v2) {
                            const char *a2 = reinterpret_cast<const char *>(
                                (S2.kind == 1 && p.q_out) ? p.q_out + ((long long)(S2.row0 + row) * p.Hq + S2.h) * D
                                                          : p.q + (((long long)S2.b * p.Tq + (t2 - p.q_off)) * p.Hq + S2.h) * D);
#pragma unroll
                            for (int cb = 0; cb < D * 2; cb += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(a2 + cb));
                        }
                    }
                }
            }

            // ---- epilogue: o = O / l, lse = scale*m + ln l ----
            // o_full fires once every product of the slot's unit has completed, so
            // the slot's query tile is idle: a base-position tile's normalised output
            // is staged in it (128-byte swizzle) and leaves by one TMA store (rows
            // past the query rows fall outside the map); output-row tiles store row
            // by row.
            if (tiles > 0) {
                if (!mbar_wait_warp(&mt.o_full[s], ucnt & 1, abort, p.status)) break;
                tc_fence_after();
                ++ucnt;
                const bool tile_store = S.kind == 0;  // warp-uniform
                const bool store = S.kind >= 0 && row < S.n;
                __nv_bfloat16 *dst = nullptr;
                float *dst32 = nullptr;  // output rows written as float (shard partials)
                float *lse_dst = nullptr;
                if (store && S.kind == 0) {
                    lse_dst = p.lse_base + ((long long)S.b * p.Hq + S.h) * p.Tq + (my_t - p.q_off);
                } else if (store) {
                    const long long o_off = ((long long)(S.row0 + row) * p.Hq + S.h) * D;
                    if (p.o_out_f32) dst32 = p.o_out_f32 + o_off;
                    else dst = p.o_out + o_off;
                    lse_dst = p.lse_out + (long long)(S.row0 + row) * p.Hq + S.h;
                }
                // a shard's output row before the shard's first key has no keys: o = 0, lse = -inf
                const float inv = my_bad ? __int_as_float(0x7fc00000) : (l > 0.f ? 1.f / l : 0.f);
#pragma unroll
                for (int j = 0; j < D / 32; ++j) {
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
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            *reinterpret_cast<uint4 *>(qs + sw128_offset<D>(row, 4 * j + e)) = w[e];
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
                if (store)
                    *lse_dst = my_bad ? __int_as_float(0x7fc00000) : (l > 0.f ? m_ref * p.scale + logf(l) : -INFINITY);
                if (tile_store) {
                    fence_proxy_async_smem();
                    mbar_arrive(&mt.os_bar[s]);
                    if (!mbar_wait_warp(&mt.os_bar[s], bcnt & 1, abort, p.status)) break;
                    ++bcnt;
                    if (row == 0) {
                        for (int j = 0; j < C::kSub; ++j)
                            tma_store_4d(&tm_ob, qs + j * (kRowsPerTile * 128), 64 * j, S.h, S.row0, S.b);
                        bulk_commit();
                        bulk_wait_read();  // the query tile is free again once the store has read it
                        stored = true;
                    }
                }
            } else if (S.kind == 1 && row < S.n && my_valid) {
                // no key tile in the slot's band (a shard's rows that all precede its keys)
                const long long o_off = ((long long)(S.row0 + row) * p.Hq + S.h) * D;
                for (int c = 0; c < D; ++c) {
                    if (p.o_out_f32) p.o_out_f32[o_off + c] = 0.f;
                    else p.o_out[o_off + c] = __float2bfloat16_rn(0.f);
                }
                p.lse_out[(long long)(S.row0 + row) * p.Hq + S.h] = -INFINITY;
            }
            tc_fence_before();
            mbar_arrive(&mt.q_free[s]);
        }
        if (stored) bulk_wait_all();
    } else {
        // ---------------- softmax: two threads per row (one per 64-key half) ----------------
        // Softmax warp w: slot (w >> 2) & 1, column half w >> 3, rows 32 (w & 3) .. +31;
        // each half stages its own D/2 channels of the row.
        const int s = (warp >> 2) & 1;
        const int hh = warp >> 3;
        const int row = ((warp & 3) << 5) | lane;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t t_s = tmem + lane_off + s * 128;                     // S_s columns of this lane quarter
        const uint32_t t_o = tmem + lane_off + C::kTmemO + s * 128 + hh * (D / 2);  // this half of O_s
        const float c2 = p.scale_log2;
        uint8_t *qs = smem + C::kQ0 + s * C::kTileBytes;
        uint32_t cnt = 0;    // S tiles of this slot handled (all units so far)
        uint32_t ucnt = 0;   // units in which this slot had tiles
        uint32_t bcnt = 0;   // base-position tiles stored
        bool stored = false; // this thread issued TMA stores
        for (int i = 0;; ++i) {
            const int r = i % kDescRing;
            if (!mbar_wait_warp(&mt.u_full[r], (i / kDescRing) & 1, abort, p.status)) break;
            const UnitDesc &dr = mt.desc[r];
            const int end = dr.end;
            const Slot S = dr.sl[s];
            const Band bd = dr.bd[s];
            const int kt_min = dr.kt_min, n_it = dr.n_it;
            __syncwarp();
            if (lane == 0) mbar_arrive(&mt.u_empty[r]);
            if (end) break;

            // ---- the row's position and its query, affine fused ----
            int my_t = 0;  // the row's position in key coordinates
            bool my_valid = false, my_bad = false;
            if (S.kind >= 0 && row < S.n) {
                if (S.kind == 0) {
                    my_t = S.row0 + row + p.q_off;
                    my_valid = true;
                } else {
                    my_valid = out_row_position(p, S.row0 + row, my_t);
                }
                my_bad = !my_valid;
                if (my_bad && hh == 0) set_status(p.status, ORTHROS_DEV_BAD_POSITION);
            }
            const bool tma = S.qrow >= 0;
            if (!mbar_wait_warp(&mt.q_full[s], i & 1, abort, p.status)) break;
            if (S.kind >= 0) {
                constexpr int kHalfChunks = D / 16;  // 16-byte chunks per half row
                if (my_valid) {
                    const float *al = (S.kind == 0 ? p.alpha_base : p.alpha_out) + S.h * D;
                    const float *be = (S.kind == 0 ? p.beta_base : p.beta_out) + S.h * D;
                    uint4 raws[kHalfChunks];  // every load of the half row in flight at once
                    if (tma) {
#pragma unroll
                        for (int cc = 0; cc < kHalfChunks; ++cc)
                            raws[cc] = *reinterpret_cast<const uint4 *>(qs + sw128_offset<D>(row, hh * kHalfChunks + cc));
                    } else {
                        const __nv_bfloat16 *src =
                            p.q + (((long long)S.b * p.Tq + (my_t - p.q_off)) * p.Hq + S.h) * D;
#pragma unroll
                        for (int cc = 0; cc < kHalfChunks; ++cc)
                            raws[cc] = reinterpret_cast<const uint4 *>(src)[hh * kHalfChunks + cc];
                    }
#pragma unroll
                    for (int cc = 0; cc < kHalfChunks; ++cc) {
                        const int c = hh * kHalfChunks + cc;
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
                        uint4 o;
                        o.x = pack_f16(v[0], v[1]);
                        o.y = pack_f16(v[2], v[3]);
                        o.z = pack_f16(v[4], v[5]);
                        o.w = pack_f16(v[6], v[7]);
                        *reinterpret_cast<uint4 *>(qs + sw128_offset<D>(row, c)) = o;
                    }
                } else {
#pragma unroll 4
                    for (int cc = 0; cc < kHalfChunks; ++cc)
                        *reinterpret_cast<uint4 *>(qs + sw128_offset<D>(row, hh * kHalfChunks + cc)) =
                            make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
            }
            mbar_arrive(&mt.q_ready[s]);

            // ---- tiles: S -> P (online softmax), band mask on edge tiles only ----
            const int t_row = my_valid ? my_t : bd.t_max;
            const int lo_row = S.kind == 0 ? max(0, t_row - p.window + 1) : p.key_lo;
            const int t_min_s = bd.t_min;
            float m_ref = -INFINITY, l = 0.f;
            bool ok = true;
            uint32_t tiles = 0;
            int row_shift = 0;  // second launch: the products give this row's logits times 2^-row_shift
            if (kRedo && max(bd.kt_lo, kt_min) <= min(bd.kt_hi, kt_min + n_it - 1)) {
                // The issuer's go-ahead comes in place of the first product: each row is
                // staged again as qa * 2^-r, r the smallest shift that brings its largest
                // value below 2^15. The two halves of a row combine the same two rounded
                // maxima (exchanged like a tile's maxima, one xm_bar phase for the one
                // s_full phase), so they agree on r.
                ok = __all_sync(0xffffffffu, mbar_wait(&mt.s_full[s], cnt & 1, abort, p.status));
                if (ok) {
                    constexpr int kHalfChunks = D / 16;
                    const float *al = (S.kind == 0 ? p.alpha_base : p.alpha_out) + S.h * D;
                    const float *be = (S.kind == 0 ? p.beta_base : p.beta_out) + S.h * D;
                    float qa[D / 2];  // this half row, affined (re-read: the tile holds the first staging)
                    float amax = 0.f;
                    if (my_valid) {
                        const __nv_bfloat16 *src =
                            S.qrow >= 0
                                ? (S.kind == 1 && p.q_out ? p.q_out : p.q) + ((long long)(S.qrow + row) * p.Hq + S.h) * D
                                : p.q + (((long long)S.b * p.Tq + (my_t - p.q_off)) * p.Hq + S.h) * D;
#pragma unroll
                        for (int c = 0; c < D / 2; ++c) {
                            const int ch = hh * (D / 2) + c;
                            qa[c] = fmaf(al[ch], __bfloat162float(src[ch]), be[ch]);
                            amax = fmaxf(amax, fabsf(qa[c]));
                        }
                    }
                    const __nv_bfloat16 amax_b = __float2bfloat16_ru(amax);
                    mt.xmax[s][hh][row] = amax_b;
                    mbar_arrive(&mt.xm_bar[s]);
                    ok = __all_sync(0xffffffffu, mbar_wait(&mt.xm_bar[s], cnt & 1, abort, p.status));
                    ++cnt;
                    if (ok) {
                        const float rmax = fmaxf(__bfloat162float(amax_b), __bfloat162float(mt.xmax[s][hh ^ 1][row]));
                        if (rmax > 65504.f && __float_as_uint(rmax) < 0x7f800000u)
                            row_shift = min((int)((__float_as_uint(rmax) >> 23) & 0xff) - 127 - 14, 126);
                        if (my_valid && row_shift > 0) {
                            const float f = exp2_int(-row_shift);
#pragma unroll
                            for (int cc = 0; cc < kHalfChunks; ++cc) {
                                uint4 o;
                                o.x = pack_f16(qa[8 * cc] * f, qa[8 * cc + 1] * f);
                                o.y = pack_f16(qa[8 * cc + 2] * f, qa[8 * cc + 3] * f);
                                o.z = pack_f16(qa[8 * cc + 4] * f, qa[8 * cc + 5] * f);
                                o.w = pack_f16(qa[8 * cc + 6] * f, qa[8 * cc + 7] * f);
                                *reinterpret_cast<uint4 *>(qs + sw128_offset<D>(row, hh * kHalfChunks + cc)) = o;
                            }
                        }
                        fence_proxy_async_smem();
                        mbar_arrive(&mt.q_ready[s]);
                        ok = __all_sync(0xffffffffu, mbar_wait(&mt.s_full[s], cnt & 1, abort, p.status));
                    }
                }
                if (!ok) break;
            }
            const float c2u = kRedo ? c2 * exp2_int(row_shift) : c2;  // the row's logit scale
            for (int it = 0; it < n_it; ++it) {
                const int kt = kt_min + it;
                if (kt < bd.kt_lo || kt > bd.kt_hi) continue;
                if (!kRedo || tiles > 0) {  // (second launch: the first tile's wait came above)
                    const bool got = mbar_wait(&mt.s_full[s], cnt & 1, abort, p.status);
                    if (!(ok = __all_sync(0xffffffffu, got))) break;
                }
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
                    mq[q] = max3(max3(xa[4 * q], xa[4 * q + 1], xa[4 * q + 2]),
                                 max3(xa[4 * q + 3], xb[4 * q], xb[4 * q + 1]), fmaxf(xb[4 * q + 2], xb[4 * q + 3]));
                const float mine = max3(max3(mq[0], mq[1], mq[2]), max3(mq[3], mq[4], mq[5]), fmaxf(mq[6], mq[7]));
                // both halves combine the same two bf16-rounded maxima, so they agree on the shift
                const __nv_bfloat16 mine_b = __float2bfloat16_rn(mine);
                mt.xmax[s][hh][row] = mine_b;
                mbar_arrive(&mt.xm_bar[s]);
                if (!(ok = __all_sync(0xffffffffu, mbar_wait(&mt.xm_bar[s], cnt & 1, abort, p.status)))) break;
                const float m_tile = fmaxf(__bfloat162float(mine_b), __bfloat162float(mt.xmax[s][hh ^ 1][row]));
                const float m_new = fmaxf(m_ref, m_tile);
                const bool resc = (m_new - m_ref) * c2u > 8.f;  // true on the first finite max
                const bool any_resc = __any_sync(0xffffffffu, resc);
                const float alpha = resc ? ex2((m_ref - m_new) * c2u) : 1.f;
                if (resc) {
                    l *= alpha;
                    m_ref = m_new;
                }
                const float mb = m_ref == -INFINITY ? 0.f : m_ref * c2u;
                float ls[4] = {0.f, 0.f, 0.f, 0.f};
                // (c2, c2) and (-mb, -mb) as f32x2 operands: the scaled, shifted logits and
                // the row sums take one packed instruction per pair of keys
                const uint64_t cv = f32x2(c2u, c2u), mv = f32x2(-mb, -mb);
                // P for keys 64 hh .. 64 hh + 63 -> packed columns 32 hh .. 32 hh + 31
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const float *x = j ? xb : xa;
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float a0, a1;
                        fma_f32x2(x[2 * e], x[2 * e + 1], cv, mv, a0, a1);
                        // the half row's last pair on the FMA pipe, the other 62
                        // exponentials on the special-function unit (3-5 % per
                        // launch at every workload shape timed; more pairs, or
                        // earlier ones, timed slower)
                        float p0, p1;
                        if (j == 1 && e == 15) exp2_fma_x2(a0, a1, p0, p1);
                        else p0 = ex2(a0), p1 = ex2(a1);
                        add_f32x2(ls[2 * (e & 1)], ls[2 * (e & 1) + 1], p0, p1);
                        pk[e] = pack_bf16(p0, p1);
                    }
                    tmem_st16(t_s + 32 * hh + 16 * j, pk);
                }
                l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
                // O_s is idle here (PV_s of the previous tile completed before S_s of
                // this tile was signalled; the next PV_s waits for p_full): each half
                // rescales its own D/2 columns of the running output.
                if (any_resc && tiles > 0) {
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
                ++tiles;
            }
            if (!ok) break;
            if (kRedo) m_ref *= exp2_int(row_shift);  // back to logit units for the epilogue

            // ---- epilogue: o = O / l, lse = scale*m + ln l ----
            // o_full fires once every product of the slot's unit has completed, so
            // the slot's S columns and its query tile are idle: the two halves of a
            // row exchange their row sums through two S columns of their TMEM lane;
            // a base-position tile's normalised output is staged in its query tile
            // (128-byte swizzle) and leaves by one TMA store (rows past the query
            // rows fall outside the map); output-row tiles store row by row.
            if (tiles > 0) {
                if (!mbar_wait_warp(&mt.o_full[s], ucnt & 1, abort, p.status)) break;
                tc_fence_after();
                tmem_st1(t_s + 96 + hh, __float_as_uint(l));
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&mt.lx_bar[s]);
                if (!mbar_wait_warp(&mt.lx_bar[s], ucnt & 1, abort, p.status)) break;
                tc_fence_after();
                uint32_t l_other = tmem_ld1(t_s + 96 + (hh ^ 1));
                tmem_ld_wait();
                asm volatile("" : "+r"(l_other));  // not read before the wait
                const float l_all = l + __uint_as_float(l_other);
                ++ucnt;
                const bool tile_store = S.kind == 0;  // warp-uniform
                const bool store = S.kind >= 0 && row < S.n;
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
                        for (int e = 0; e < 4; ++e)
                            *reinterpret_cast<uint4 *>(qs + sw128_offset<D>(row, c0 + e)) = w[e];
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
                if (tile_store) {
                    fence_proxy_async_smem();
                    mbar_arrive(&mt.os_bar[s]);
                    if (!mbar_wait_warp(&mt.os_bar[s], bcnt & 1, abort, p.status)) break;
                    ++bcnt;
                    if (row == 0 && hh == 0) {
                        for (int j = 0; j < C::kSub; ++j)
                            tma_store_4d(&tm_ob, qs + j * (kRowsPerTile * 128), 64 * j, S.h, S.row0, S.b);
                        bulk_commit();
                        bulk_wait_read();  // the query tile is free again once the store has read it
                        stored = true;
                    }
                }
            } else if (S.kind == 1 && row < S.n && my_valid) {
                // no key tile in the slot's band (a shard's rows that all precede its keys)
                const long long o_off = ((long long)(S.row0 + row) * p.Hq + S.h) * D + hh * (D / 2);
                for (int c = 0; c < D / 2; ++c) {
                    if (p.o_out_f32) p.o_out_f32[o_off + c] = 0.f;
                    else p.o_out[o_off + c] = __float2bfloat16_rn(0.f);
                }
                if (hh == 0) p.lse_out[(long long)(S.row0 + row) * p.Hq + S.h] = -INFINITY;
            }
            tc_fence_before();
            mbar_arrive(&mt.q_free[s]);
        }
        if (stored) bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == Wp::kMma) {
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

template <int D, bool kRow>
cudaError_t launch_dr(const TcParams &p, const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tq,
                      const CUtensorMap &tqo, const CUtensorMap &tob, int units, cudaStream_t stream) {
    using Wp = Warps<kRow>;
    static SmemLimit limit, limit_redo;
    if (cudaError_t e = limit.ensure((const void *)prefill_tc_kernel<D, false, kRow>, Cfg<D>::kSmem); e != cudaSuccess)
        return e;
    if (cudaError_t e = limit_redo.ensure((const void *)prefill_tc_kernel<D, true, kRow>, Cfg<D>::kSmem); e != cudaSuccess)
        return e;
    // persistent: one CTA per SM takes units from the counter until none is left
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int grid = units < sms ? units : sms;
    prefill_tc_kernel<D, false, kRow><<<grid, Wp::kThreads, Cfg<D>::kSmem, stream>>>(tk, tv, tq, tqo, tob, p);
    if (cudaError_t e = cudaGetLastError(); e != cudaSuccess) return e;
    // second launch: scans the log-sum-exps for rows with a query past the fp16
    // range and computes their blocks again (none: every CTA leaves after the scan)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sms);
    cfg.blockDim = dim3(Wp::kThreads);
    cfg.dynamicSmemBytes = Cfg<D>::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaError_t e = cudaLaunchKernelEx(&cfg, prefill_tc_kernel<D, true, kRow>, tk, tv, tq, tqo, tob, p);
        e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

// Windows of at least this many keys take the one-thread-per-row softmax:
// their base units run 33 key tiles or more, where its shorter per-tile
// softmax wins (128K shape: 7.18 vs 7.35 ms), while the per-unit query
// staging and epilogue, twice as long per thread, cost more than that on
// short units (fine-tuning shape, w = 1024: 1.14 vs 1.08 ms; pre-training
// shape, w = 512: 0.41 vs 0.33 ms).
constexpr int kRowWindowMin = 4096;

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
    return p.window >= kRowWindowMin ? launch_dr<D, true>(p, tk, tv, tq, tqo, tob, units, stream)
                                     : launch_dr<D, false>(p, tk, tv, tq, tqo, tob, units, stream);
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
