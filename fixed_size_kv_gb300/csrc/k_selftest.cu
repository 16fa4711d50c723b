// k_selftest.cu -- a self-test of the error path that every kernel's bounded waits
// share (the compression GEMM, the MLA decode pipeline).
//
// One thread waits on an mbarrier that nothing arrives on.  The wait is bounded by
// WAIT_NS of %globaltimer; when it gives up, the kernel records SNAP_ERR_TIMEOUT in the
// cache's status word and exits, as a pipeline kernel does when one of its waits
// expires.  Nothing faults and nothing hangs: the device context stays usable.
#include "kernels.cuh"
#include "tc.cuh"

namespace snap {

namespace {

__global__ void bounded_wait_selftest_kernel(int32_t* status) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    // phase 0 never completes: its one expected arrival never comes
    if (threadIdx.x == 0 && !mbar_wait_bounded(smem_u32(&bar), 0, reinterpret_cast<volatile int*>(&abort_flag)))
        report_error(status, SNAP_ERR_TIMEOUT, 900, 0, 0);
}

}  // namespace

cudaError_t launch_bounded_wait_selftest(int32_t* status, cudaStream_t st) {
    bounded_wait_selftest_kernel<<<1, 32, 0, st>>>(status);
    return cudaGetLastError();
}

}  // namespace snap
