// decode_static.cu -- orthros_decode_static: the decoding step without a
// caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they run a
// decoding step: a host framework whose custom-op interface hands over only
// the input and output tensors, code running under an allocator that must not
// grow during serving, or a caller that has no CUDA allocator of its own at
// all. For them this entry point takes its scratch (the status word and the
// split-KV partials of orthros_decode) from one file-scope device array of a
// fixed size, so it allocates nothing and frees nothing.
//
// Rules of use:
//   * The array holds kStaticScratchBytes (32 MiB). Every GPU that loads this
//     library holds it until the process exits.
//   * Sizes whose workspace would exceed it are rejected with
//     ORTHROS_EWORKSPACE before any launch (orthros_last_error() says by how
//     much).
//   * The first call on a device resolves the array's device address with
//     cudaGetSymbolAddress (once per device, with that device current); make
//     that first call before any stream capture.
//   * All calls share the one array and it keeps the previous call's
//     contents. The status word is cleared at the start of every call and
//     every partial is written before it is read, so back-to-back calls on one
//     stream are fine; calls that overlap on the GPU (different streams or
//     threads without ordering between them) race on the array.
//   * Device-side data errors (bad block-table entries or cache lengths) land
//     in the shared status word, which this entry point does not expose; the
//     affected rows come back as NaN, and so do all rows when a kernel gave
//     up on a bounded wait.
//   * The array's address is resolved once per device and kept for the life
//     of the process, so resetting a device after its first call is not
//     supported.
#include <mutex>

#include "internal.cuh"

namespace orthros {
namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the array on the current device (resolved once per device).
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace orthros

using namespace orthros;

extern "C" {

orthros_status orthros_decode_static(const void *q, const void *q_out, const void *k_new, const void *v_new,
                                     void *k_cache, void *v_cache, const int32_t *block_table, int max_pages,
                                     int page_size, int num_pages, const int32_t *cache_lens,
                                     const float *alpha_base, const float *beta_base, const float *alpha_out,
                                     const float *beta_out, int B, int Hq, int Hkv, int d, int window, float scale,
                                     orthros_dtype dtype, void *o_base, float *lse_base, void *o_out,
                                     float *lse_out, orthros_stream_t stream) {
    const size_t need = orthros_decode_workspace_size(B, Hq, Hkv, d, max_pages, page_size, dtype);
    if (need == 0) {
        // sizes the regular entry point rejects: let it report why (before any launch)
        return orthros_decode(q, q_out, k_new, v_new, k_cache, v_cache, block_table, max_pages, page_size,
                              num_pages, cache_lens, alpha_base, beta_base, alpha_out, beta_out, B, Hq, Hkv, d,
                              window, scale, dtype, o_base, lse_base, o_out, lse_out, nullptr, 0, stream);
    }
    if (need > kStaticScratchBytes)
        return report_error(ORTHROS_EWORKSPACE,
                            "orthros_decode_static: these sizes need %zu bytes of scratch, the static array holds %zu",
                            need, kStaticScratchBytes);
    void *scratch = nullptr;
    const cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess)
        return report_error(ORTHROS_ECUDA, "orthros_decode_static: cudaGetSymbolAddress failed: %s",
                            cudaGetErrorString(e));
    return orthros_decode(q, q_out, k_new, v_new, k_cache, v_cache, block_table, max_pages, page_size, num_pages,
                          cache_lens, alpha_base, beta_base, alpha_out, beta_out, B, Hq, Hkv, d, window, scale,
                          dtype, o_base, lse_base, o_out, lse_out, scratch, kStaticScratchBytes, stream);
}

}  // extern "C"
