// cache.cu -- paged K/V cache writes of the Orthros hot path.
//
// The base stream owns the layer-wise K/V cache; the output stream never
// writes it (Orthros paper Sec. 3.1: the sliding-window stream materialises
// the cache, the cross-attention stream only reads it; Sec. 3.2 "Decoding":
// the base token updates the cache).
//
// Page layout: [num_pages, page_size, Hkv, d], token-major inside a page, so
// one (token, head) row of d elements is contiguous (256 B for bf16, d = 128)
// and every copy below moves whole 16-byte vectors.
#include "internal.cuh"

namespace orthros {
namespace {

// One thread moves one 16-byte vector of one (sequence, kv head) row.
__global__ void decode_append_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                                     uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                                     const int32_t *__restrict__ block_table,
                                     const int32_t *__restrict__ cache_lens, int B, int vec_per_tok,
                                     int max_pages, int page_size, int num_pages, uint32_t *status) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)B * vec_per_tok) return;
    const int b = (int)(i / vec_per_tok);
    const int w = (int)(i % vec_per_tok);
    const int L = cache_lens[b];
    if (L < 0 || L / page_size >= max_pages) {
        if (w == 0) set_status(status, ORTHROS_DEV_BAD_LENGTH);
        return;
    }
    const int pg = block_table[(long long)b * max_pages + L / page_size];
    if (pg < 0 || pg >= num_pages) {
        if (w == 0) set_status(status, ORTHROS_DEV_BAD_PAGE);
        return;
    }
    const long long dst = ((long long)pg * page_size + L % page_size) * vec_per_tok + w;
    k_cache[dst] = k_new[i];
    v_cache[dst] = v_new[i];
}

// Continuous-batching step: new token i of sequence b (rows new_indptr[b] ..)
// goes to position cache_lens[b] + (i - new_indptr[b]).
__global__ void extend_append_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                                     uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                                     const int32_t *__restrict__ block_table,
                                     const int32_t *__restrict__ cache_lens, const int32_t *__restrict__ new_indptr,
                                     int B, int n_new, int vec_per_tok, int max_pages, int page_size, int num_pages,
                                     uint32_t *status) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)n_new * vec_per_tok) return;
    const int row = (int)(i / vec_per_tok);
    const int w = (int)(i % vec_per_tok);
    int lo = 0, hi = B - 1;  // sequence of the row: last b with new_indptr[b] <= row
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (new_indptr[mid] <= row) lo = mid; else hi = mid - 1;
    }
    const int b = lo;
    const int L = cache_lens[b];
    const long long t = (long long)L + (row - new_indptr[b]);
    if (L < 0 || t >= (long long)max_pages * page_size) {
        if (w == 0) set_status(status, ORTHROS_DEV_BAD_LENGTH);
        return;
    }
    const int pg = block_table[(long long)b * max_pages + t / page_size];
    if (pg < 0 || pg >= num_pages) {
        if (w == 0) set_status(status, ORTHROS_DEV_BAD_PAGE);
        return;
    }
    const long long dst = ((long long)pg * page_size + t % page_size) * vec_per_tok + w;
    k_cache[dst] = k_new[i];
    v_cache[dst] = v_new[i];
}

// Prefill: token t of sequence b goes to page block_table[b][t / P], slot t % P.
__global__ void prefill_cache_fill_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                                          uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                                          const int32_t *__restrict__ block_table, int B, int T,
                                          int vec_per_tok, int max_pages, int page_size, int num_pages,
                                          uint32_t *status) {
    const long long n = (long long)B * T * vec_per_tok;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        const long long tok = i / vec_per_tok;
        const int w = (int)(i % vec_per_tok);
        const int b = (int)(tok / T);
        const int t = (int)(tok % T);
        const int pg = block_table[(long long)b * max_pages + t / page_size];
        if (pg < 0 || pg >= num_pages) {
            if (w == 0) set_status(status, ORTHROS_DEV_BAD_PAGE);
            continue;
        }
        const long long dst = ((long long)pg * page_size + t % page_size) * vec_per_tok + w;
        k_cache[dst] = k[i];
        v_cache[dst] = v[i];
    }
}

// One pass over the bf16 keys/values of a prefill: keys -> fp16 copy (exact in
// the fp16 range) while recording the largest |k| of the call, and, when a
// block table is given, both tensors -> their cache pages. Also zeroes the
// tile kernel's n_zero-word bitmap of row blocks to compute again.
__global__ void prefill_prep_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                                    uint4 *__restrict__ k16, uint4 *__restrict__ k_cache,
                                    uint4 *__restrict__ v_cache, const int32_t *__restrict__ block_table, int B,
                                    int T, int vec_per_tok, int max_pages, int page_size, int num_pages,
                                    uint32_t *status, unsigned *kmax_bits, uint32_t *zero_words, int n_zero) {
    const long long n = (long long)B * T * vec_per_tok;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_zero; i += gridDim.x * blockDim.x) zero_words[i] = 0;
    float amax = 0.f;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        const uint4 kx = k[i];
        const uint32_t *w = reinterpret_cast<const uint32_t *>(&kx);
        uint4 h;
        uint32_t *hw = reinterpret_cast<uint32_t *>(&h);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xffff0000u);
            amax = fmaxf(amax, fmaxf(fabsf(lo), fabsf(hi)));
            const __half2 hv = __floats2half2_rn(lo, hi);
            hw[e] = *reinterpret_cast<const uint32_t *>(&hv);
        }
        k16[i] = h;
        if (k_cache) {
            const long long tok = i / vec_per_tok;
            const int wi = (int)(i % vec_per_tok);
            const int b = (int)(tok / T);
            const int t = (int)(tok % T);
            const int pg = block_table[(long long)b * max_pages + t / page_size];
            if (pg < 0 || pg >= num_pages) {
                if (wi == 0) set_status(status, ORTHROS_DEV_BAD_PAGE);
                continue;
            }
            const long long dst = ((long long)pg * page_size + t % page_size) * vec_per_tok + wi;
            k_cache[dst] = kx;
            v_cache[dst] = v[i];
        }
    }
    // largest |k| of the call (non-negative floats order like their bit patterns)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0 && amax > 0.f) atomicMax(kmax_bits, __float_as_uint(amax));
}

// Keys beyond the fp16 range. s = 0 unless the largest |k| of the call
// exceeds 65504; then s is the smallest shift that brings it below 2^15, and
// the fp16 copy is rewritten as k * 2^-s (a power of two: exact for every key
// whose scaled magnitude stays a normal fp16 number). Either way the four query
// affines are copied scaled by 2^s (exact), so the tile kernel's staged
// queries are qa * 2^s and its products are the logits unchanged.
__global__ void prefill_key_rescale_kernel(const uint4 *__restrict__ k, uint4 *__restrict__ k16, long long n,
                                           const unsigned *__restrict__ kmax_bits, AffineSet src,
                                           float *__restrict__ aff, int n_aff) {
    const unsigned bits = *kmax_bits;
    const float kmax = __uint_as_float(bits);
    // in range, or inf / NaN (not scalable): s = 0
    const int sft = (kmax > 65504.f && bits < 0x7f800000u) ? (int)((bits >> 23) & 0xff) - 127 - 14 : 0;
    const float up = __uint_as_float((uint32_t)(127 + sft) << 23);
    const long long stride = (long long)gridDim.x * blockDim.x;
    const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    for (long long i = tid; i < 4LL * n_aff; i += stride) {
        const float *sp = src.p[i / n_aff];
        aff[i] = sp ? sp[i % n_aff] * up : 0.f;
    }
    if (sft == 0) return;  // the common case
    const float down = __uint_as_float((uint32_t)(127 - sft) << 23);
    for (long long i = tid; i < n; i += stride) {
        const uint4 kx = k[i];
        const uint32_t *w = reinterpret_cast<const uint32_t *>(&kx);
        uint4 h;
        uint32_t *hw = reinterpret_cast<uint32_t *>(&h);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const __half2 hv =
                __floats2half2_rn(__uint_as_float(w[e] << 16) * down, __uint_as_float(w[e] & 0xffff0000u) * down);
            hw[e] = *reinterpret_cast<const uint32_t *>(&hv);
        }
        k16[i] = h;
    }
}

int grid_for(long long n, int threads, int per_sm) {
    int sms = 152, dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    long long blocks = (n + threads - 1) / threads;
    const long long cap = (long long)sms * per_sm;
    return (int)(blocks < cap ? blocks : cap);
}

}  // namespace

cudaError_t launch_prefill_prep(const void *k, const void *v, void *k16, void *k_cache, void *v_cache,
                                const int32_t *block_table, int B, int T, int Hkv, int d, int max_pages,
                                int page_size, int num_pages, uint32_t *status, unsigned *kmax_bits,
                                uint32_t *zero_words, int n_zero, cudaStream_t stream) {
    const long long n = (long long)B * T * Hkv * d * 2 / 16;
    if (n == 0 && n_zero == 0) return cudaSuccess;
    prefill_prep_kernel<<<grid_for(n > n_zero ? n : n_zero, 256, 8), 256, 0, stream>>>(
        (const uint4 *)k, (const uint4 *)v, (uint4 *)k16, (uint4 *)k_cache, (uint4 *)v_cache, block_table, B, T,
        Hkv * d * 2 / 16, max_pages, page_size, num_pages, status, kmax_bits, zero_words, n_zero);
    return cudaGetLastError();
}

cudaError_t launch_prefill_key_rescale(const void *k, void *k16, int B, int T, int Hkv, int d,
                                       const unsigned *kmax_bits, AffineSet src, float *aff, int n_aff,
                                       cudaStream_t stream) {
    const long long n = (long long)B * T * Hkv * d * 2 / 16;
    // one block per SM: the affine copies are small, and the key pass (only for
    // keys past the fp16 range) strides over the keys
    prefill_key_rescale_kernel<<<grid_for(n > 4LL * n_aff ? n : 4LL * n_aff, 256, 1), 256, 0, stream>>>(
        (const uint4 *)k, (uint4 *)k16, n, kmax_bits, src, aff, n_aff);
    return cudaGetLastError();
}

cudaError_t launch_decode_append(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                                 const int32_t *block_table, const int32_t *cache_lens, int B, int Hkv,
                                 int d, int max_pages, int page_size, int num_pages, int elem_bytes,
                                 uint32_t *status, cudaStream_t stream) {
    if (B == 0) return cudaSuccess;
    const int vec_per_tok = Hkv * d * elem_bytes / 16;
    const long long n = (long long)B * vec_per_tok;
    const int threads = 256;
    decode_append_kernel<<<(unsigned)((n + threads - 1) / threads), threads, 0, stream>>>(
        (const uint4 *)k_new, (const uint4 *)v_new, (uint4 *)k_cache, (uint4 *)v_cache, block_table,
        cache_lens, B, vec_per_tok, max_pages, page_size, num_pages, status);
    return cudaGetLastError();
}

cudaError_t launch_extend_append(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                                 const int32_t *block_table, const int32_t *cache_lens, const int32_t *new_indptr,
                                 int B, int n_new, int Hkv, int d, int max_pages, int page_size, int num_pages,
                                 int elem_bytes, uint32_t *status, cudaStream_t stream) {
    if (n_new == 0) return cudaSuccess;
    const int vec_per_tok = Hkv * d * elem_bytes / 16;
    const long long n = (long long)n_new * vec_per_tok;
    const int threads = 256;
    if ((n + threads - 1) / threads > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    extend_append_kernel<<<(unsigned)((n + threads - 1) / threads), threads, 0, stream>>>(
        (const uint4 *)k_new, (const uint4 *)v_new, (uint4 *)k_cache, (uint4 *)v_cache, block_table, cache_lens,
        new_indptr, B, n_new, vec_per_tok, max_pages, page_size, num_pages, status);
    return cudaGetLastError();
}

cudaError_t launch_prefill_cache_fill(const void *k, const void *v, void *k_cache, void *v_cache,
                                      const int32_t *block_table, int B, int T, int Hkv, int d,
                                      int max_pages, int page_size, int num_pages, int elem_bytes,
                                      uint32_t *status, cudaStream_t stream) {
    if ((long long)B * T == 0) return cudaSuccess;
    const int vec_per_tok = Hkv * d * elem_bytes / 16;
    const long long n = (long long)B * T * vec_per_tok;
    const int threads = 256;
    int sms = 152;
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    long long blocks = (n + threads - 1) / threads;
    const long long cap = (long long)sms * 8;  // grid-stride: a few resident CTAs per SM
    if (blocks > cap) blocks = cap;
    prefill_cache_fill_kernel<<<(unsigned)blocks, threads, 0, stream>>>(
        (const uint4 *)k, (const uint4 *)v, (uint4 *)k_cache, (uint4 *)v_cache, block_table, B, T,
        vec_per_tok, max_pages, page_size, num_pages, status);
    return cudaGetLastError();
}

// Output-row positions of one chunk of a chunked prefill, in that chunk's
// key-buffer coordinates: global position - off, raised to 0 (a row before the
// chunk's keys, whose buffer starts with at least one halo key, then reads
// nothing).
__global__ void shift_positions_kernel(const int32_t *__restrict__ src, int32_t *__restrict__ dst, int n, int off) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) dst[i] = max(src[i] - off, 0);
}

// dst[0] |= src[k * stride] for k < n: the status words of the calls a
// chunked prefill made, folded into its own.
__global__ void fold_status_kernel(uint32_t *dst, const uint32_t *__restrict__ src, int n, int stride) {
    uint32_t bits = 0;
    for (int k = threadIdx.x; k < n; k += blockDim.x) bits |= src[(long long)k * stride];
    for (int o = 16; o > 0; o >>= 1) bits |= __shfl_xor_sync(0xffffffffu, bits, o);
    if (threadIdx.x == 0 && bits) atomicOr(dst, bits);
}

cudaError_t launch_shift_positions(const int32_t *src, int32_t *dst, int n, int off, cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    shift_positions_kernel<<<(n + 255) / 256, 256, 0, stream>>>(src, dst, n, off);
    return cudaGetLastError();
}

cudaError_t launch_fold_status(uint32_t *dst, const uint32_t *src, int n, int stride_words, cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    fold_status_kernel<<<1, 32, 0, stream>>>(dst, src, n, stride_words);
    return cudaGetLastError();
}

}  // namespace orthros
