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

}  // namespace

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
