// splitkv.cu -- split-KV flash attention for few query rows over long key
// ranges, plus the combine pass. Serves
//   * the decoding pair (Orthros paper, Sec. 3.2 "Decoding"): per (sequence,
//     kv head) the g base rows (window max(0, L-w+1)..L, Eq. 4) and the g
//     output rows (whole history 0..L, Eq. 5) read ONE pass over the paged
//     cache;
//   * output rows of a prefill whose sequence has only a few of them (the
//     prefilling regime's single last-token row, Sec. 3.2), over contiguous K/V.
//
// The work is memory-bound (a few query rows per key), so each key/value byte
// is read once per (sequence, kv head) and all rows of the group share it. A
// CTA takes one chunk of keys for one row group and writes an unnormalised
// partial (running max m, sum l, accumulator o); the combine kernel merges
// the chunks with the usual log-sum-exp weights.
//
// Tensor cores (mma.sync m16n8k16, bf16): keys are the M dimension and the
// query rows the N dimension, so 8 rows fill an instruction:
//   S^T[16 keys x 8 rows]  = K[16 x 16 ch] . Q^T[16 ch x 8 rows]
//   O^T[16 ch x 8 rows]   += V^T[16 ch x 16 keys] . P^T[16 keys x 8 rows]
// The affined query is split as q = hi + lo with hi = bf16(q), lo = bf16(q - hi)
// and both halves are multiplied, which keeps the logits as accurate as fp32
// queries. P^T leaves the accumulator in the "row = key" layout; movmatrix
// transposes each 8x8 block into the B-operand layout of the PV product.
// Row-wise softmax reductions run across the 8 lanes that share a row.
#include "internal.cuh"

namespace orthros {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kBlockKeys = 64;  // keys per pipeline stage (16 per warp)
constexpr int kStages = 3;
constexpr int kMaxRows = 16;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

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
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Swizzled [64 keys][D] bf16 tile: 16-byte chunk c of key row k lives at
// chunk (c ^ (k & 7)); rows are D*2 bytes apart.
template <int D> __device__ __forceinline__ uint32_t tile_off(int key, int chunk) {
    return key * (D * 2) + ((chunk ^ (key & 7)) << 4);
}

struct RowInfo {
    int lo, hi;  // key range (inclusive); lo > hi = no keys
};

template <int D, int NT>
__global__ void __launch_bounds__(kThreads) splitkv_kernel(const SplitParams p) {
    constexpr int kTileBytes = kBlockKeys * D * 2;
    constexpr int kChunks = D / 8;  // 16-byte chunks per key row
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *ks = smem;
    uint8_t *vs = smem + kStages * kTileBytes;
    __shared__ RowInfo rows[kMaxRows];
    __shared__ int grp_lo, grp_hi, grp_ok;
    __shared__ int grp_bad;  // a block-table entry of this chunk's keys lay outside the page pool

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g4 = lane >> 2, t4 = lane & 3;  // mma fragment coordinates
    const int chunk_id = blockIdx.x % p.max_chunks;  // consecutive CTAs walk one group's chunks
    const int group = blockIdx.x / p.max_chunks;
    const int gsz = p.Hq / p.Hkv;

    // ---------------- group -> (sequence, kv head, rows) ----------------
    int b, kv, nrows;
    int pos_base = 0;  // prefill: first output row of the group
    if (p.mode == kSplitDecode) {
        b = group / p.Hkv;
        kv = group % p.Hkv;
        nrows = 2 * gsz;
    } else {
        const int gi = p.group_info[3 * group];
        b = gi >> 16;
        kv = gi & 0xffff;
        pos_base = p.group_info[3 * group + 1];
        nrows = p.group_info[3 * group + 2] * gsz;
    }
    int L = 0;
    if (p.mode == kSplitDecode) {
        L = p.cache_lens[b];
    }
    if (tid < kMaxRows) {
        RowInfo ri{1, 0};
        if (tid < nrows) {
            if (p.mode == kSplitDecode) {
                if (L >= 0 && L / p.page_size < p.max_pages) {
                    ri.hi = L;
                    ri.lo = tid < gsz ? max(0, L - p.window + 1) : 0;
                } else if (chunk_id == 0 && tid == 0) {
                    set_status(p.status, ORTHROS_DEV_BAD_LENGTH);
                }
            } else {
                const int t = prefill_row_end(p, p.out_positions[pos_base + tid / gsz]);
                if (t >= 0) {
                    ri.lo = p.key_lo;
                    ri.hi = t;
                } else if (chunk_id == 0 && tid % gsz == 0) {
                    set_status(p.status, ORTHROS_DEV_BAD_POSITION);
                }
            }
        }
        rows[tid] = ri;
    }
    __syncthreads();
    if (tid == 0) {
        int lo = 0x7fffffff, hi = -1;
        for (int r = 0; r < kMaxRows; ++r)
            if (rows[r].lo <= rows[r].hi) {
                lo = min(lo, rows[r].lo);
                hi = max(hi, rows[r].hi);
            }
        const int c0 = chunk_id * p.chunk, c1 = c0 + p.chunk - 1;
        grp_lo = max(lo, c0);
        grp_hi = min(hi, c1);
        grp_ok = grp_lo <= grp_hi;
        grp_bad = 0;
    }
    __syncthreads();
    float *part = p.partial + ((long long)group * p.max_chunks + chunk_id) * kMaxRows * (D + 2);
    if (!grp_ok) {
        // nothing of this chunk is needed by any row: mark it empty
        if (tid < kMaxRows) {
            part[tid * (D + 2) + D] = -INFINITY;
            part[tid * (D + 2) + D + 1] = 0.f;
        }
        return;
    }
    const int key_lo = grp_lo, key_hi = grp_hi;
    const int blk0 = key_lo / kBlockKeys, blk1 = key_hi / kBlockKeys;
    const int nblk = blk1 - blk0 + 1;

    // ---------------- query fragments (affine in fp32, hi/lo bf16 split) ----------------
    // B operand of m16n8k16 (col-major Q^T): b0 = Q[row n=g4][ch 2t4, 2t4+1],
    // b1 = Q[row g4][ch 2t4+8, 2t4+9] of each 16-channel step.
    uint32_t qh[NT][D / 16][2], ql[NT][D / 16][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int r = nt * 8 + g4;
        const bool valid = r < nrows;
        const __nv_bfloat16 *qrow = nullptr;
        const float *al = nullptr, *be = nullptr;
        if (valid) {
            if (p.mode == kSplitDecode) {
                const bool base = r < gsz;
                const int h = kv * gsz + (base ? r : r - gsz);
                const __nv_bfloat16 *src = (!base && p.q_out) ? p.q_out : p.q;
                qrow = src + ((long long)b * p.Hq + h) * D;
                al = (base ? p.alpha_base : p.alpha_out) + h * D;
                be = (base ? p.beta_base : p.beta_out) + h * D;
            } else {
                const int pi = pos_base + r / gsz;
                const int h = kv * gsz + r % gsz;
                const int i = min(max(p.out_positions[pi] - p.q_off, 0), p.Tq - 1);  // query row of the position
                qrow = p.q_out ? p.q_out + ((long long)pi * p.Hq + h) * D
                               : p.q + (((long long)b * p.Tq + i) * p.Hq + h) * D;
                al = p.alpha_out + h * D;
                be = p.beta_out + h * D;
            }
        }
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int ch = ks * 16 + half * 8 + 2 * t4;
                float x0 = 0.f, x1 = 0.f;
                if (valid) {
                    const __nv_bfloat162 raw = *reinterpret_cast<const __nv_bfloat162 *>(qrow + ch);
                    x0 = fmaf(al[ch], __bfloat162float(raw.x), be[ch]);
                    x1 = fmaf(al[ch + 1], __bfloat162float(raw.y), be[ch + 1]);
                }
                const uint32_t hi = pack2(x0, x1);
                const float h0 = __uint_as_float(hi << 16), h1 = __uint_as_float(hi & 0xffff0000u);
                qh[nt][ks][half] = hi;
                ql[nt][ks][half] = pack2(x0 - h0, x1 - h1);
            }
        }
    }
    // row ranges of the 2 rows (2t4, 2t4+1) this thread owns in each n-tile
    int rlo[NT][2], rhi[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            rlo[nt][e] = rows[nt * 8 + 2 * t4 + e].lo;
            rhi[nt][e] = rows[nt * 8 + 2 * t4 + e].hi;
        }

    // ---------------- key/value loads (cp.async, swizzled) ----------------
    const long long tok_stride = (long long)p.Hkv * D;  // elements between consecutive tokens
    const __nv_bfloat16 *kbase = p.k + (long long)kv * D;
    const __nv_bfloat16 *vbase = p.v + (long long)kv * D;
    const int32_t *bt = p.mode == kSplitDecode ? p.block_table + (long long)b * p.max_pages : nullptr;
    const long long seq_off = p.mode == kSplitDecode ? 0 : (long long)b * p.T * tok_stride;
    auto load_block = [&](int bi, int stage) {
        const int key0 = (blk0 + bi) * kBlockKeys;
        constexpr int kPer = kBlockKeys * kChunks / kThreads;  // 16-byte chunks per thread
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int idx = u * kThreads + tid;
            const int kr = idx / kChunks, c = idx % kChunks;
            int j = key0 + kr;
            j = min(max(j, key_lo), key_hi);  // rows outside the range are masked; keep reads in bounds
            long long off;
            if (bt) {
                int pg = bt[j / p.page_size];
                if (pg < 0 || pg >= p.num_pages) {
                    set_status(p.status, ORTHROS_DEV_BAD_PAGE);
                    grp_bad = 1;
                    pg = 0;
                }
                off = ((long long)pg * p.page_size + j % p.page_size) * tok_stride;
            } else {
                off = seq_off + (long long)j * tok_stride;
            }
            cp_async16(smem_u32(ks + stage * kTileBytes + tile_off<D>(kr, c)), kbase + off + c * 8);
            cp_async16(smem_u32(vs + stage * kTileBytes + tile_off<D>(kr, c)), vbase + off + c * 8);
        }
    };

    float m[NT][2], l[NT][2];
    float o[NT][D / 16][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        m[nt][0] = m[nt][1] = -INFINITY;
        l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[nt][mt][e] = 0.f;
    }
    const float c2 = p.scale_log2;

#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
        if (s < nblk) load_block(s, s);
        cp_async_commit();
    }
    for (int bi = 0; bi < nblk; ++bi) {
        const int stage = bi % kStages;
        cp_async_wait<kStages - 2>();
        __syncthreads();
        // refill the stage consumed in the previous iteration
        if (bi + kStages - 1 < nblk) load_block(bi + kStages - 1, (bi + kStages - 1) % kStages);
        cp_async_commit();

        const uint32_t kt = smem_u32(ks + stage * kTileBytes);
        const uint32_t vt = smem_u32(vs + stage * kTileBytes);
        const int krow0 = warp * 16;  // this warp's 16 keys of the block
        const int key_base = (blk0 + bi) * kBlockKeys + krow0;

        // S^T = K Q^T (hi + lo)
        float sacc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) sacc[nt][e] = 0.f;
#pragma unroll
        for (int ksp = 0; ksp < D / 16; ++ksp) {
            // A = K[16 keys][16 ch]: lanes 0-15 rows 0-15 at chunk 2ksp, lanes 16-31 at chunk 2ksp+1
            const int kr = krow0 + (lane & 15);
            const int ck = 2 * ksp + (lane >> 4);
            uint32_t a0, a1, a2, a3;
            ldsm_x4(kt + tile_off<D>(kr, ck), a0, a1, a2, a3);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                mma_bf16(sacc[nt], a0, a1, a2, a3, qh[nt][ksp][0], qh[nt][ksp][1]);
                mma_bf16(sacc[nt], a0, a1, a2, a3, ql[nt][ksp][0], ql[nt][ksp][1]);
            }
        }
        // masks and online softmax; sacc[nt] = {S[key g][row 2t], S[key g][row 2t+1],
        // S[key g+8][row 2t], S[key g+8][row 2t+1]}
        uint32_t pb[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int ja = key_base + g4, jb = ja + 8;
            float sv[4];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                sv[e] = (ja >= rlo[nt][e] && ja <= rhi[nt][e]) ? sacc[nt][e] : -INFINITY;
                sv[2 + e] = (jb >= rlo[nt][e] && jb <= rhi[nt][e]) ? sacc[nt][2 + e] : -INFINITY;
            }
            float pr[4];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float mx = fmaxf(sv[e], sv[2 + e]);
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                const float m_new = fmaxf(m[nt][e], mx);
                const float mb = m_new == -INFINITY ? 0.f : m_new * c2;
                const float alpha = ex2(m[nt][e] * c2 - mb);  // 0 when the old max is -inf
                pr[e] = ex2(fmaf(sv[e], c2, -mb));
                pr[2 + e] = ex2(fmaf(sv[2 + e], c2, -mb));
                float ls = pr[e] + pr[2 + e];
                ls += __shfl_xor_sync(0xffffffffu, ls, 4);
                ls += __shfl_xor_sync(0xffffffffu, ls, 8);
                ls += __shfl_xor_sync(0xffffffffu, ls, 16);
                l[nt][e] = l[nt][e] * alpha + ls;
                m[nt][e] = m_new;
#pragma unroll
                for (int mt = 0; mt < D / 16; ++mt) {
                    o[nt][mt][e] *= alpha;
                    o[nt][mt][2 + e] *= alpha;
                }
            }
            // P^T 8x8 blocks (keys 0-7 / 8-15) -> B fragments via transpose
            pb[nt][0] = movmatrix_t(pack2(pr[0], pr[1]));
            pb[nt][1] = movmatrix_t(pack2(pr[2], pr[3]));
        }
        // O^T += V^T P^T: A = V^T[16 ch][16 keys] through ldmatrix.trans
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
            const int vr = krow0 + (lane & 7) + ((lane >> 4) << 3);
            const int vc = 2 * mt + ((lane >> 3) & 1);
            uint32_t a0, a1, a2, a3;
            ldsm_x4_t(vt + tile_off<D>(vr, vc), a0, a1, a2, a3);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_bf16(o[nt][mt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
        }
    }
    cp_async_wait<0>();
    __syncthreads();

    // ---------------- merge the 4 warps' states, write the chunk partial ----------------
    // o[nt][mt] = {O^T[ch 16mt+g][row 2t], [ch 16mt+g][row 2t+1], [ch 16mt+g+8][row 2t], [..][row 2t+1]}
    float *red = reinterpret_cast<float *>(smem);  // [warps][16 rows][D + 2]
    constexpr int kRowStride = D + 2;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int r = nt * 8 + 2 * t4 + e;
            float *dst = red + (warp * kMaxRows + r) * kRowStride;
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                dst[16 * mt + g4] = o[nt][mt][e];
                dst[16 * mt + g4 + 8] = o[nt][mt][2 + e];
            }
            if (g4 == 0) {
                dst[D] = m[nt][e];
                dst[D + 1] = l[nt][e];
            }
        }
    __syncthreads();
    for (int idx = tid; idx < NT * 8 * (D + 2); idx += kThreads) {
        const int r = idx / (D + 2), c = idx % (D + 2);
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red[(w * kMaxRows + r) * kRowStride + D]);
        float acc = 0.f;
        const float Mb = M == -INFINITY ? 0.f : M * c2;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float *src = red + (w * kMaxRows + r) * kRowStride;
            const float wgt = ex2(src[D] * c2 - Mb);
            if (c < D) acc += wgt * src[c];
            else if (c == D + 1) acc += wgt * src[D + 1];
        }
        // rows that read keys loaded from a substituted page: a NaN row sum
        // makes the combined row NaN
        if (c == D + 1 && grp_bad && rows[r].lo <= key_hi && rows[r].hi >= key_lo) acc = __int_as_float(0x7fc00000);
        part[r * kRowStride + c] = c == D ? M : acc;
    }
}

// One warp per (group, row): merge the chunk partials, normalise, store.
template <int D>
__global__ void __launch_bounds__(256) combine_kernel(const SplitParams p) {
    const int gw = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (gw >= p.n_groups * kMaxRows) return;
    const int group = gw / kMaxRows, r = gw % kMaxRows;
    const int gsz = p.Hq / p.Hkv;
    int b, kv, nrows, pos_base = 0;
    if (p.mode == kSplitDecode) {
        b = group / p.Hkv;
        kv = group % p.Hkv;
        nrows = 2 * gsz;
    } else if (p.mode == kSplitDecodeSplit) {
        b = (group >> 1) / p.Hkv;
        kv = (group >> 1) % p.Hkv;
        nrows = gsz;
    } else if (p.mode == kSplitExtend) {
        const int *e = p.ext_info + 4 * group;
        b = e[0] >> 16;
        kv = e[0] & 0xffff;
        nrows = ((e[3] & 0xffff) + (e[3] >> 16)) * gsz;
    } else {
        const int gi = p.group_info[3 * group];
        b = gi >> 16;
        kv = gi & 0xffff;
        pos_base = p.group_info[3 * group + 1];
        nrows = p.group_info[3 * group + 2] * gsz;
    }
    if (r >= nrows) return;
    int hi;
    __nv_bfloat16 *dst;
    float *dst32 = nullptr;
    float *lse_dst;
    if (p.mode == kSplitExtend) {
        // the same validity rule as the split kernel's rows
        const int h = kv * gsz + r % gsz;
        int kind, idx;
        hi = extend_position(p, group, b, p.cache_lens[b], r / gsz, kind, idx);
        dst = (kind == 0 ? p.o_base : p.o_out) + ((long long)idx * p.Hq + h) * D;
        lse_dst = (kind == 0 ? p.lse_base : p.lse_out) + (long long)idx * p.Hq + h;
    } else if (p.mode == kSplitDecode || p.mode == kSplitDecodeSplit) {
        const int L = p.cache_lens[b];
        hi = (L >= 0 && L / p.page_size < p.max_pages) ? L : -1;
        const bool base = p.mode == kSplitDecode ? r < gsz : (group & 1) == 0;
        const int h = kv * gsz + (r < gsz ? r : r - gsz);
        dst = (base ? p.o_base : p.o_out) + ((long long)b * p.Hq + h) * D;
        lse_dst = (base ? p.lse_base : p.lse_out) + (long long)b * p.Hq + h;
    } else {
        const int pi = pos_base + r / gsz;
        const int h = kv * gsz + r % gsz;
        hi = prefill_row_end(p, p.out_positions[pi]);
        dst = p.o_out + ((long long)pi * p.Hq + h) * D;
        lse_dst = p.lse_out + (long long)pi * p.Hq + h;
        if (p.o_out_f32) {  // float output rows (a shard's partials)
            dst = nullptr;
            dst32 = p.o_out_f32 + ((long long)pi * p.Hq + h) * D;
        }
    }
    const float nanv = __int_as_float(0x7fc00000);
    // a split kernel that gave up on a bounded wait left some partials
    // unwritten (they may hold an earlier call's values): every row is NaN
    if (p.status && (*reinterpret_cast<volatile uint32_t *>(p.status) & ORTHROS_DEV_TIMEOUT)) hi = -1;
    if (hi < 0) {
        for (int c = lane; c < D; c += 32) {
            if (dst32) dst32[c] = nanv;
            else dst[c] = __float2bfloat16_rn(nanv);
        }
        if (lane == 0) *lse_dst = nanv;
        return;
    }
    const int nc = hi / p.chunk + 1;
    const float c2 = p.scale_log2;
    const float *part = p.partial + (long long)group * p.max_chunks * kMaxRows * (D + 2) + r * (D + 2);
    const long long cstride = (long long)kMaxRows * (D + 2);
    float M = -INFINITY;
    for (int c = lane; c < nc; c += 32) M = fmaxf(M, part[c * cstride + D]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float Mb = M * c2;
    constexpr int E = D / 32;
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    float Lsum = 0.f;
    for (int c = 0; c < nc; ++c) {
        const float *src = part + c * cstride;
        const float mc = src[D];
        if (mc == -INFINITY) continue;
        const float w = ex2(mc * c2 - Mb);
        Lsum += w * src[D + 1];
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] += w * src[lane + 32 * e];
    }
    // a row without keys (a shard's row before its first key): o = 0, lse = -inf
    const bool empty = M == -INFINITY;
    const float inv = empty ? 0.f : 1.f / Lsum;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        if (dst32) dst32[lane + 32 * e] = acc[e] * inv;
        else dst[lane + 32 * e] = __float2bfloat16_rn(acc[e] * inv);
    }
    if (lane == 0) *lse_dst = empty ? -INFINITY : M * p.scale + logf(Lsum);
}

template <int D, int NT>
cudaError_t launch_split_t(const SplitParams &p, cudaStream_t stream) {
    constexpr int kSmem = 2 * kStages * kBlockKeys * D * 2;
    static_assert(kSmem >= kWarps * kMaxRows * (D + 2) * 4, "reduction scratch must fit the stage buffers");
    static SmemLimit limit;
    if (cudaError_t e = limit.ensure((const void *)splitkv_kernel<D, NT>, kSmem); e != cudaSuccess) return e;
    const long long ctas = (long long)p.max_chunks * p.n_groups;
    if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    splitkv_kernel<D, NT><<<(unsigned)ctas, kThreads, kSmem, stream>>>(p);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_combine_t(const SplitParams &p, cudaStream_t stream) {
    const int warps = p.n_groups * kMaxRows;
    combine_kernel<D><<<(warps + 7) / 8, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_splitkv_extend(const SplitParams &p, int d, int n_small, cudaStream_t stream) {
    if (p.n_groups == 0 || p.max_chunks == 0) return cudaSuccess;
    if (!splitkv_tma_eligible(p)) return cudaErrorInvalidValue;
    cudaError_t e;
    SplitParams q = p;
    if (n_small > 0) {
        q.group_offset = 0;
        q.n_groups = n_small;
        if ((e = launch_splitkv_tma(q, d, 8, stream)) != cudaSuccess) return e;
    }
    if (p.n_groups > n_small) {
        q.group_offset = n_small;
        q.n_groups = p.n_groups - n_small;
        if ((e = launch_splitkv_tma(q, d, 16, stream)) != cudaSuccess) return e;
    }
    return d == 128 ? launch_combine_t<128>(p, stream) : launch_combine_t<64>(p, stream);
}

size_t split_partial_bytes(int n_groups, int max_chunks, int d) {
    return (size_t)n_groups * max_chunks * kMaxRows * (d + 2) * sizeof(float);
}

cudaError_t launch_splitkv(const SplitParams &p, int d, int rows_per_group, cudaStream_t stream) {
    if (p.n_groups == 0 || p.max_chunks == 0) return cudaSuccess;
    cudaError_t e;
    if (p.mode == kSplitExtend) return cudaErrorInvalidValue;  // launch_splitkv_extend
    if (p.mode == kSplitDecodeSplit && !splitkv_tma_eligible(p)) return cudaErrorInvalidValue;  // TMA kernel only
    if (splitkv_tma_eligible(p)) {
        e = launch_splitkv_tma(p, d, rows_per_group, stream);
    } else {
        const int nt = rows_per_group > 8 ? 2 : 1;
        if (d == 128) e = nt == 2 ? launch_split_t<128, 2>(p, stream) : launch_split_t<128, 1>(p, stream);
        else e = nt == 2 ? launch_split_t<64, 2>(p, stream) : launch_split_t<64, 1>(p, stream);
    }
    if (e != cudaSuccess) return e;
    return d == 128 ? launch_combine_t<128>(p, stream) : launch_combine_t<64>(p, stream);
}

}  // namespace orthros
