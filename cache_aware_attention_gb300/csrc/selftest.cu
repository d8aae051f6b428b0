// mar_selftest_wait_timeout: the bounded barrier wait of the tensor-core kernels, made to
// run out on purpose, so that the status path can be checked on a device.
//
// One thread initialises a shared-memory barrier expecting one arrival that never comes
// and waits on its first phase with tc5::mbar_wait and the caller's (short) poll limit.
// The wait gives up, records MAR_STATUS_TIMEOUT and returns false; the kernel ends. No
// copy, tensor-core operation or tensor memory is involved, so nothing is left in flight.
#include "marattn.h"
#include "tc5.cuh"

namespace mar {
int record_cuda_error(cudaError_t e);

namespace {

__global__ void wait_timeout_kernel(uint32_t limit, uint32_t *status) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    abort_flag = 0;
    tc5::mbar_init(&bar, 1);
    tc5::mbar_fence_init();
    // phase 0 never completes: nothing arrives on the barrier
    const bool ok = tc5::mbar_wait(&bar, 0, status, &abort_flag, limit);
    if (ok) report(status, 0x80000000u);  // cannot happen; would flag a broken wait
}

}  // namespace
}  // namespace mar

extern "C" int mar_selftest_wait_timeout(uint32_t spin_limit, uint32_t *d_status, mar_stream_t stream) {
    if (!d_status || spin_limit < 1 || spin_limit > (1u << 20)) return MAR_ERR_ARG;
    mar::wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(spin_limit, d_status);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? MAR_OK : mar::record_cuda_error(e);
}
