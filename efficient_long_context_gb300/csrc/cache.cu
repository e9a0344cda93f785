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
// the fp16 range; out-of-range magnitudes raise ORTHROS_DEV_FP16_RANGE), and,
// when a block table is given, both tensors -> their cache pages.
__global__ void prefill_prep_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                                    uint4 *__restrict__ k16, uint4 *__restrict__ k_cache,
                                    uint4 *__restrict__ v_cache, const int32_t *__restrict__ block_table, int B,
                                    int T, int vec_per_tok, int max_pages, int page_size, int num_pages,
                                    uint32_t *status) {
    const long long n = (long long)B * T * vec_per_tok;
    bool over = false;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        const uint4 kx = k[i];
        const uint32_t *w = reinterpret_cast<const uint32_t *>(&kx);
        uint4 h;
        uint32_t *hw = reinterpret_cast<uint32_t *>(&h);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xffff0000u);
            over |= fabsf(lo) > 65504.f || fabsf(hi) > 65504.f;
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
    if (over) set_status(status, ORTHROS_DEV_FP16_RANGE);
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
                                int page_size, int num_pages, uint32_t *status, cudaStream_t stream) {
    const long long n = (long long)B * T * Hkv * d * 2 / 16;
    if (n == 0) return cudaSuccess;
    prefill_prep_kernel<<<grid_for(n, 256, 8), 256, 0, stream>>>(
        (const uint4 *)k, (const uint4 *)v, (uint4 *)k16, (uint4 *)k_cache, (uint4 *)v_cache, block_table, B, T,
        Hkv * d * 2 / 16, max_pages, page_size, num_pages, status);
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

}  // namespace orthros
