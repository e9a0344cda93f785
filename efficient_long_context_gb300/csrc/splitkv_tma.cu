// splitkv_tma.cu -- persistent, TMA-fed split-KV attention (same contract as
// splitkv.cu's kernel: per (row group, key chunk) partials for the combine).
//
// Decoding is bound by HBM bandwidth: every cached key/value byte is read once
// per step (Orthros paper, Sec. 3.3: decoding is I/O-bound; Sec. 3.2
// "Decoding": the base and the output token of a step read the same cache).
// This version keeps the memory system busy without per-thread address work:
//   * one CTA per SM loops over work items (row group, key chunk), chunk-major;
//   * one producer thread streams 128-key stages with TMA (64-token boxes,
//     128-byte swizzle) through a 3-stage ring (6 for d = 64) and keeps
//     streaming across item boundaries, so no pipeline refill between items;
//   * four consumer warps each take 32 keys of a stage (mma.sync m16n8k16,
//     keys as M, up to 16 query rows as N, hi/lo split of the affined query),
//     keep a running (max, sum, output) per row, and at the end of an item
//     merge their states in shared memory and write the chunk partial.
// Paged caches need page_size % 64 == 0 (a 64-token box must not cross a
// page); other page sizes take splitkv.cu. Boxes past the last needed key read
// an out-of-bounds coordinate, which TMA fills with zeros.
#include "ptx.cuh"

namespace orthros {

using namespace ptx;

namespace {

constexpr int kConsumers = 4;
constexpr int kThreadsT = (kConsumers + 1) * 32;
constexpr int kStageKeys = 128;
constexpr int kBoxTokens = 64;
constexpr int kBoxBytes = kBoxTokens * 128;  // 64 tokens x 64 channels x 2 bytes
constexpr int kMaxRowsT = 16;

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &a0, uint32_t &a1, uint32_t &a2, uint32_t &a3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &a0, uint32_t &a1, uint32_t &a2, uint32_t &a3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                 : "r"(addr));
}
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// A 128-key stage of one tensor: boxes (channel half h, token half tb) of
// 64 rows x 128 bytes; 16-byte chunk c of key row r sits at chunk c ^ (r & 7).
__device__ __forceinline__ uint32_t stage_off(int r, int c) {
    return (((c >> 3) * 2 + (r >> 6)) * kBoxBytes) + (r & 63) * 128 + (((c & 7) ^ (r & 7)) << 4);
}

// Rows of one work item (group): key range per row and where its query lives.
struct ItemInfo {
    int b, kv, nrows, pos_base, L;
    int group;     // global group index (extend rows are looked up through it)
    int union_hi;  // last key any row needs (-1: none)
    int union_lo;  // first key any row needs, rounded down to a whole stage (keys before it are skipped)
};

__device__ __forceinline__ ItemInfo item_info(const SplitParams &p, int group) {
    ItemInfo it{};
    const int gsz = p.Hq / p.Hkv;
    it.group = group;
    if (p.mode == kSplitDecode) {
        it.b = group / p.Hkv;
        it.kv = group % p.Hkv;
        it.nrows = 2 * gsz;
        it.L = p.cache_lens[it.b];
        it.union_hi = (it.L >= 0 && it.L / p.page_size < p.max_pages) ? it.L : -1;
    } else if (p.mode == kSplitDecodeSplit) {
        const int pair = group >> 1;
        it.b = pair / p.Hkv;
        it.kv = pair % p.Hkv;
        it.nrows = gsz;
        it.L = p.cache_lens[it.b];
        it.union_hi = (it.L >= 0 && it.L / p.page_size < p.max_pages) ? it.L : -1;
        // the base rows' group reads only the window
        it.union_lo = (group & 1) == 0 && it.union_hi >= 0 ? (max(0, it.L - p.window + 1) / kStageKeys) * kStageKeys : 0;
    } else if (p.mode == kSplitExtend) {
        const int *e = p.ext_info + 4 * group;
        it.b = e[0] >> 16;
        it.kv = e[0] & 0xffff;
        const int npos = (e[3] & 0xffff) + (e[3] >> 16);
        it.nrows = npos * gsz;
        it.L = p.cache_lens[it.b];
        int hi = -1, lo = 0x7fffffff, kind, idx;
        for (int i = 0; i < npos; ++i) {
            const int t = extend_position(p, group, it.b, it.L, i, kind, idx);
            if (t < 0) continue;
            hi = max(hi, t);
            lo = min(lo, kind == 0 ? max(0, t - p.window + 1) : 0);
        }
        it.union_hi = hi;
        // base rows of a prefill chunk need only their windows
        it.union_lo = hi >= 0 ? (lo / kStageKeys) * kStageKeys : 0;
    } else {
        const int gi = p.group_info[3 * group];
        it.b = gi >> 16;
        it.kv = gi & 0xffff;
        it.pos_base = p.group_info[3 * group + 1];
        const int npos = p.group_info[3 * group + 2];
        it.nrows = npos * gsz;
        int hi = -1;
        for (int i = 0; i < npos; ++i) {
            const int t = prefill_row_end(p, p.out_positions[it.pos_base + i]);
            if (t >= p.key_lo) hi = max(hi, t);
        }
        it.union_hi = hi;
        it.union_lo = (p.key_lo / kStageKeys) * kStageKeys;
    }
    return it;
}

// Key range of row r of an item (lo > hi: the row takes no keys).
__device__ __forceinline__ void row_range(const SplitParams &p, const ItemInfo &it, int r, int &lo, int &hi) {
    const int gsz = p.Hq / p.Hkv;
    lo = 1;
    hi = 0;
    if (r >= it.nrows) return;
    if (p.mode == kSplitDecode || p.mode == kSplitDecodeSplit) {
        if (it.union_hi < 0) return;
        hi = it.L;
        const bool base = p.mode == kSplitDecode ? r < gsz : (it.group & 1) == 0;
        lo = base ? max(0, it.L - p.window + 1) : 0;
    } else if (p.mode == kSplitExtend) {
        int kind, idx;
        const int t = extend_position(p, it.group, it.b, it.L, r / gsz, kind, idx);
        if (t >= 0) {
            hi = t;
            lo = kind == 0 ? max(0, t - p.window + 1) : 0;
        }
    } else {
        const int t = prefill_row_end(p, p.out_positions[it.pos_base + r / gsz]);
        if (t >= 0) {
            lo = p.key_lo;
            hi = t;
        }
    }
}

template <int D> struct TCfg {
    static constexpr int kTile = kStageKeys * D * 2;  // one tensor's stage
    static constexpr int kStages = D == 128 ? 3 : 6;
    static constexpr int kStageBytes = 2 * kTile;  // K + V
    static constexpr int kScratch = kConsumers * kMaxRowsT * (D + 2) * 4;
    static constexpr int kBar = kStages * kStageBytes + kScratch;
    // barriers (2 kStages + 2) x 8 B, the abort flag and kStages stage flags
    static constexpr int kMetaBytes = (2 * kStages + 2) * 8 + 4 + 4 * kStages;
    static_assert(kMetaBytes <= 192, "stage metadata must fit its region");
    static constexpr int kSmem = kBar + 192 + 1024;
};

template <int D, int NT>
__global__ void __launch_bounds__(kThreadsT, 1)
    splitkv_tma_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const SplitParams p, int total_items) {
    using C = TCfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *scratch = reinterpret_cast<float *>(smem + C::kStages * C::kStageBytes);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::kBar);
    uint64_t *empty = full + C::kStages;
    uint64_t *merge_bar = empty + C::kStages;  // [2]: states written / partial written (one arrive per consumer warp)
    int *abort_flag = reinterpret_cast<int *>(merge_bar + 2);
    volatile int *abort = abort_flag;
    // per stage: 1 when a block-table entry of its keys was outside the page
    // pool (the producer then loaded page 0 in its place); written before the
    // stage's full barrier is armed, read by the consumers after it completes
    volatile int *stage_bad = abort_flag + 1;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gsz = p.Hq / p.Hkv;
    // Items run chunk-major: CTAs that run at the same time read the same
    // token range of every group (all kv heads of a token row, 2 KB of
    // contiguous cache for GQA 32/8), not distant ranges of one head.
    const int n_groups = total_items / p.max_chunks;

    if (tid == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumers);
        }
        mbar_init(&merge_bar[0], kConsumers);
        mbar_init(&merge_bar[1], kConsumers);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kConsumers && lane == 0) {
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
    }
    __syncthreads();

    if (warp == kConsumers) {
        // ---------------- producer: one thread streams every stage of every item ----------------
        if (lane != 0) return;
        uint32_t sc = 0;  // stages issued so far
        // Before leaving (normally or on abort) wait, bounded, for the copies of
        // the last stages issued, so that none is in flight when the CTA exits.
        auto drain = [&]() {
            for (uint32_t i = sc > (uint32_t)C::kStages ? sc - C::kStages : 0; i < sc; ++i)
                mbar_wait_drain(&full[i % C::kStages], (i / C::kStages) & 1, p.status);
        };
        for (int item = blockIdx.x; item < total_items && !*abort; item += gridDim.x) {
            const int group = p.group_offset + item % n_groups, chunk = item / n_groups;
            const ItemInfo it = item_info(p, group);
            const int key_lo = max(chunk * p.chunk, it.union_lo);
            const int key_hi = min(it.union_hi, chunk * p.chunk + p.chunk - 1);
            if (key_lo > key_hi) continue;
            const int32_t *bt = p.mode != kSplitPrefill ? p.block_table + (long long)it.b * p.max_pages : nullptr;
            for (int j0 = key_lo; j0 <= key_hi; j0 += kStageKeys, ++sc) {
                const int st = sc % C::kStages;
                if (sc >= (uint32_t)C::kStages &&
                    !mbar_wait(&empty[st], ((sc / C::kStages) - 1) & 1, abort, p.status)) {
                    drain();
                    return;
                }
                int tok[2], bad = 0;
#pragma unroll
                for (int tb = 0; tb < 2; ++tb) {
                    const int j = j0 + tb * kBoxTokens;
                    tok[tb] = (int)p.kv_tokens;  // past the end: TMA fills zeros
                    if (j <= key_hi) {
                        if (bt) {
                            int pg = bt[j / p.page_size];
                            if (pg < 0 || pg >= p.num_pages) {
                                set_status(p.status, ORTHROS_DEV_BAD_PAGE);
                                bad = 1;
                                pg = 0;
                            }
                            tok[tb] = pg * p.page_size + j % p.page_size;
                        } else {
                            tok[tb] = it.b * p.T + j;
                        }
                    }
                }
                stage_bad[st] = bad;  // released to the consumers by the arrive below
                mbar_arrive_expect_tx(&full[st], C::kStageBytes);
                uint8_t *ks = smem + st * C::kStageBytes;
                uint8_t *vs = ks + C::kTile;
#pragma unroll
                for (int tb = 0; tb < 2; ++tb)
#pragma unroll
                    for (int h = 0; h < D / 64; ++h) {
                        tma_load_3d(ks + (h * 2 + tb) * kBoxBytes, &tm_k, &full[st], 64 * h, it.kv, tok[tb]);
                        tma_load_3d(vs + (h * 2 + tb) * kBoxBytes, &tm_v, &full[st], 64 * h, it.kv, tok[tb]);
                    }
            }
        }
        drain();
        return;
    }

    // ---------------- consumers ----------------
    const int g4 = lane >> 2, t4 = lane & 3;
    const float c2 = p.scale_log2;
    constexpr int kRowStride = D + 2;
    uint32_t sc = 0, merges = 0;
    // bounded rendezvous of the four consumer warps (never a plain bar.sync, so
    // that a warp leaving on a timed-out wait cannot strand the others)
    auto consumer_sync = [&](int which) -> bool {
        __syncwarp();
        if (lane == 0) mbar_arrive(&merge_bar[which]);
        const bool got = mbar_wait(&merge_bar[which], merges & 1, abort, p.status);
        return __all_sync(0xffffffffu, got);
    };
    for (int item = blockIdx.x; item < total_items; item += gridDim.x) {
        const int group = p.group_offset + item % n_groups, chunk = item / n_groups;
        const ItemInfo it = item_info(p, group);
        const int key_lo = max(chunk * p.chunk, it.union_lo);
        const int key_hi = min(it.union_hi, chunk * p.chunk + p.chunk - 1);
        float *part = p.partial + ((long long)group * p.max_chunks + chunk) * kMaxRowsT * kRowStride;
        if (chunk == 0 && tid < kMaxRowsT && tid < it.nrows) {
            // report rows the data makes impossible (their combined outputs are NaN)
            if (p.mode == kSplitDecode || p.mode == kSplitDecodeSplit) {
                if (it.union_hi < 0 && tid == 0) set_status(p.status, ORTHROS_DEV_BAD_LENGTH);
            } else if (p.mode == kSplitExtend) {
                int kind, idx;
                if (tid % gsz == 0 && extend_position(p, group, it.b, it.L, tid / gsz, kind, idx) < 0)
                    set_status(p.status, (it.L < 0 || kind == 0) ? ORTHROS_DEV_BAD_LENGTH : ORTHROS_DEV_BAD_POSITION);
            } else if (tid % gsz == 0) {
                if (prefill_row_end(p, p.out_positions[it.pos_base + tid / gsz]) < 0)
                    set_status(p.status, ORTHROS_DEV_BAD_POSITION);
            }
        }
        if (key_lo > key_hi) {
            if (tid < kMaxRowsT) {
                part[tid * kRowStride + D] = -INFINITY;
                part[tid * kRowStride + D + 1] = 0.f;
            }
            continue;
        }
        // query fragments of this item's rows (affine in fp32, bf16 hi + lo)
        uint32_t qh[NT][D / 16][2], ql[NT][D / 16][2];
        int rlo[NT][2], rhi[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int r = nt * 8 + g4;
            const bool valid = r < it.nrows;
            const __nv_bfloat16 *qrow = nullptr;
            const float *al = nullptr, *be = nullptr;
            if (valid) {
                if (p.mode == kSplitDecode || p.mode == kSplitDecodeSplit) {
                    const bool base = p.mode == kSplitDecode ? r < gsz : (it.group & 1) == 0;
                    const int h = it.kv * gsz + (r < gsz ? r : r - gsz);
                    const __nv_bfloat16 *src = (!base && p.q_out) ? p.q_out : p.q;
                    qrow = src + ((long long)it.b * p.Hq + h) * D;
                    al = (base ? p.alpha_base : p.alpha_out) + h * D;
                    be = (base ? p.beta_base : p.beta_out) + h * D;
                } else if (p.mode == kSplitExtend) {
                    const int h = it.kv * gsz + r % gsz;
                    int kind, idx;
                    const int t = extend_position(p, it.group, it.b, it.L, r / gsz, kind, idx);
                    if (kind == 0) {
                        qrow = p.q + ((long long)idx * p.Hq + h) * D;
                    } else if (p.q_out) {
                        qrow = p.q_out + ((long long)idx * p.Hq + h) * D;
                    } else {  // the new token at the row's position (its first new token if the row is invalid)
                        const int i = p.new_indptr[it.b] + (t >= 0 ? t - it.L : 0);
                        qrow = p.q + ((long long)min(i, max(p.n_new - 1, 0)) * p.Hq + h) * D;
                    }
                    al = (kind == 0 ? p.alpha_base : p.alpha_out) + h * D;
                    be = (kind == 0 ? p.beta_base : p.beta_out) + h * D;
                } else {
                    const int pi = it.pos_base + r / gsz;
                    const int h = it.kv * gsz + r % gsz;
                    const int i = min(max(p.out_positions[pi] - p.q_off, 0), p.Tq - 1);  // query row of the position
                    qrow = p.q_out ? p.q_out + ((long long)pi * p.Hq + h) * D
                                   : p.q + (((long long)it.b * p.Tq + i) * p.Hq + h) * D;
                    al = p.alpha_out + h * D;
                    be = p.beta_out + h * D;
                }
            }
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int ch = ks * 16 + half * 8 + 2 * t4;
                    float x0 = 0.f, x1 = 0.f;
                    if (valid) {
                        const __nv_bfloat162 raw = *reinterpret_cast<const __nv_bfloat162 *>(qrow + ch);
                        x0 = fmaf(al[ch], __bfloat162float(raw.x), be[ch]);
                        x1 = fmaf(al[ch + 1], __bfloat162float(raw.y), be[ch + 1]);
                    }
                    const uint32_t hi = pack_bf16(x0, x1);
                    qh[nt][ks][half] = hi;
                    ql[nt][ks][half] =
                        pack_bf16(x0 - __uint_as_float(hi << 16), x1 - __uint_as_float(hi & 0xffff0000u));
                }
#pragma unroll
            for (int e = 0; e < 2; ++e) row_range(p, it, nt * 8 + 2 * t4 + e, rlo[nt][e], rhi[nt][e]);
        }
        float m[NT][2], l[NT][2], o[NT][D / 16][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            m[nt][0] = m[nt][1] = -INFINITY;
            l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
            for (int cm = 0; cm < D / 16; ++cm)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[nt][cm][e] = 0.f;
        }
        bool ok = true;
        uint32_t bad_rows = 0;  // bit 2 nt + e: a row of this thread read a stage loaded from a bad page
        for (int j0 = key_lo; j0 <= key_hi; j0 += kStageKeys, ++sc) {
            const int st = sc % C::kStages;
            ok = __all_sync(0xffffffffu, mbar_wait(&full[st], (sc / C::kStages) & 1, abort, p.status));
            if (!ok) break;
            if (stage_bad[st]) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e)
                        if (rlo[nt][e] <= j0 + kStageKeys - 1 && rhi[nt][e] >= j0) bad_rows |= 1u << (2 * nt + e);
            }
            const uint32_t kt = smem_u32(smem + st * C::kStageBytes);
            const uint32_t vt = kt + C::kTile;
            const int r0 = warp * 32;  // this warp's 32 keys of the stage
            // S^T = K (Q_hi + Q_lo)^T, four independent accumulator chains
            float sh[NT][2][4], sl[NT][2][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) sh[nt][mt][e] = sl[nt][mt][e] = 0.f;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(kt + stage_off(r0 + 16 * mt + (lane & 15), 2 * ks + (lane >> 4)), a0, a1, a2, a3);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        mma_bf16(sh[nt][mt], a0, a1, a2, a3, qh[nt][ks][0], qh[nt][ks][1]);
                        mma_bf16(sl[nt][mt], a0, a1, a2, a3, ql[nt][ks][0], ql[nt][ks][1]);
                    }
                }
            }
            // online softmax over the warp's 32 keys; thread holds keys
            // {g4, g4+8} of each 16-key m-tile for rows 2t4, 2t4+1
            uint32_t pb[NT][2][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float pr[2][4];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float sv[4];
#pragma unroll
                    for (int mt = 0; mt < 2; ++mt) {
                        const int ja = j0 + r0 + 16 * mt + g4, jb = ja + 8;
                        sv[2 * mt] = (ja >= rlo[nt][e] && ja <= rhi[nt][e]) ? sh[nt][mt][e] + sl[nt][mt][e] : -INFINITY;
                        sv[2 * mt + 1] =
                            (jb >= rlo[nt][e] && jb <= rhi[nt][e]) ? sh[nt][mt][2 + e] + sl[nt][mt][2 + e] : -INFINITY;
                    }
                    float mx = max3(sv[0], sv[1], fmaxf(sv[2], sv[3]));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                    const float m_new = fmaxf(m[nt][e], mx);
                    const float mb = m_new == -INFINITY ? 0.f : m_new * c2;
                    const float alpha = ex2(m[nt][e] * c2 - mb);
                    float ls = 0.f;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float pv = ex2(fmaf(sv[k], c2, -mb));
                        ls += pv;
                        pr[e][k] = pv;
                    }
                    ls += __shfl_xor_sync(0xffffffffu, ls, 4);
                    ls += __shfl_xor_sync(0xffffffffu, ls, 8);
                    ls += __shfl_xor_sync(0xffffffffu, ls, 16);
                    l[nt][e] = l[nt][e] * alpha + ls;
                    m[nt][e] = m_new;
#pragma unroll
                    for (int cm = 0; cm < D / 16; ++cm) {
                        o[nt][cm][e] *= alpha;
                        o[nt][cm][2 + e] *= alpha;
                    }
                }
                // P^T blocks (keys x rows) -> B fragments of the PV product
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    pb[nt][mt][0] = movmatrix_t(pack_bf16(pr[0][2 * mt], pr[1][2 * mt]));
                    pb[nt][mt][1] = movmatrix_t(pack_bf16(pr[0][2 * mt + 1], pr[1][2 * mt + 1]));
                }
            }
            // O^T += V^T P^T
#pragma unroll
            for (int cm = 0; cm < D / 16; ++cm) {
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    uint32_t a0, a1, a2, a3;
                    const int vr = r0 + 16 * mt + (lane & 7) + ((lane >> 4) << 3);
                    ldsm_x4_t(vt + stage_off(vr, 2 * cm + ((lane >> 3) & 1)), a0, a1, a2, a3);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) mma_bf16(o[nt][cm], a0, a1, a2, a3, pb[nt][mt][0], pb[nt][mt][1]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
        }
        if (!ok) return;
        // merge the four warps' states, write the chunk partial
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float *dst = scratch + (warp * kMaxRowsT + nt * 8 + 2 * t4 + e) * kRowStride;
#pragma unroll
                for (int cm = 0; cm < D / 16; ++cm) {
                    dst[16 * cm + g4] = o[nt][cm][e];
                    dst[16 * cm + g4 + 8] = o[nt][cm][2 + e];
                }
                if (g4 == 0) {
                    // a NaN row sum makes the combined row NaN (the data behind it is not the row's)
                    dst[D] = m[nt][e];
                    dst[D + 1] = (bad_rows >> (2 * nt + e)) & 1u ? __int_as_float(0x7fc00000) : l[nt][e];
                }
            }
        if (!consumer_sync(0)) return;
        for (int idx = tid; idx < NT * 8 * kRowStride; idx += kConsumers * 32) {
            const int r = idx / kRowStride, c = idx % kRowStride;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kConsumers; ++w) M = fmaxf(M, scratch[(w * kMaxRowsT + r) * kRowStride + D]);
            const float Mb = M == -INFINITY ? 0.f : M * c2;
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumers; ++w) {
                const float *src = scratch + (w * kMaxRowsT + r) * kRowStride;
                const float wgt = ex2(src[D] * c2 - Mb);
                if (c < D) acc += wgt * src[c];
                else if (c == D + 1) acc += wgt * src[D + 1];
            }
            part[r * kRowStride + c] = c == D ? M : acc;
        }
        if (!consumer_sync(1)) return;
        ++merges;
    }
}

template <int D, int NT>
cudaError_t launch_t(const SplitParams &p, cudaStream_t stream) {
    CUtensorMap tk, tv;
    if (!encode_kv_map_3d(&tk, p.k, p.kv_tokens, p.Hkv, D, kBoxTokens) ||
        !encode_kv_map_3d(&tv, p.v, p.kv_tokens, p.Hkv, D, kBoxTokens))
        return cudaErrorInvalidValue;
    static SmemLimit limit;
    if (cudaError_t e = limit.ensure((const void *)splitkv_tma_kernel<D, NT>, TCfg<D>::kSmem); e != cudaSuccess)
        return e;
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long items = (long long)p.n_groups * p.max_chunks;
    if (items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const int grid = (int)(items < sms ? items : sms);
    splitkv_tma_kernel<D, NT><<<grid, kThreadsT, TCfg<D>::kSmem, stream>>>(tk, tv, p, (int)items);
    return cudaGetLastError();
}

}  // namespace

bool splitkv_tma_eligible(const SplitParams &p) {
    return p.chunk % kStageKeys == 0 && (p.mode == kSplitPrefill || p.page_size % kBoxTokens == 0) &&
           p.kv_tokens > 0 && p.kv_tokens < 0x7fffffffLL;
}

cudaError_t launch_splitkv_tma(const SplitParams &p, int d, int rows_per_group, cudaStream_t stream) {
    const int nt = rows_per_group > 8 ? 2 : 1;
    if (d == 128) return nt == 2 ? launch_t<128, 2>(p, stream) : launch_t<128, 1>(p, stream);
    return nt == 2 ? launch_t<64, 2>(p, stream) : launch_t<64, 1>(p, stream);
}

}  // namespace orthros
