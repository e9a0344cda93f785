// selftest.cu -- exercises the failure path that every TMA / tensor-core
// kernel of the library relies on: a bounded mbarrier wait that runs out.
//
// One CTA initialises an mbarrier that nothing ever arrives on. Thread 0
// waits on it with the caller's (short) limit, the other threads with the
// library's normal limit. When thread 0's limit runs out it raises the CTA's
// abort flag and ORTHROS_DEV_TIMEOUT in the status word; the other threads see
// the flag and leave their waits at once, and the kernel returns. Nothing
// faults, traps or hangs; the host reads the outcome with orthros_check().
#include "ptx.cuh"

namespace orthros {
namespace {

__global__ void selftest_wait_kernel(uint32_t *status, long long limit) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar, 1);
        abort_flag = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();
    const bool ok = ptx::mbar_wait(&bar, 0, &abort_flag, status, threadIdx.x == 0 ? limit : ptx::kWaitLimitCycles);
    // a completed wait would mean the barrier was armed: report it as bad data
    if (ok) set_status(status, ORTHROS_DEV_BAD_POSITION);
}

}  // namespace
}  // namespace orthros

using namespace orthros;

extern "C" orthros_status orthros_selftest_wait_timeout(long long limit_cycles, void *workspace,
                                                        size_t workspace_bytes, orthros_stream_t stream_) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (limit_cycles < 1 || limit_cycles > ptx::kWaitLimitCycles)
        return report_error(ORTHROS_EINVAL, "limit_cycles = %lld must lie in [1, %lld]", limit_cycles,
                            ptx::kWaitLimitCycles);
    if (!workspace || workspace_bytes < kStatusBytes)
        return report_error(ORTHROS_EWORKSPACE, "workspace needs %zu bytes", kStatusBytes);
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return report_error(ORTHROS_EINVAL, "workspace must be 256-byte aligned");
    uint32_t *status = static_cast<uint32_t *>(workspace);
    cudaError_t e = cudaMemsetAsync(status, 0, sizeof(uint32_t), stream);
    if (e == cudaSuccess) {
        selftest_wait_kernel<<<1, 128, 0, stream>>>(status, limit_cycles);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) return report_error(ORTHROS_ECUDA, "self-test launch: %s", cudaGetErrorString(e));
    return ORTHROS_OK;
}
