// selftest.cu -- runs the library's bounded mbarrier wait on a barrier that
// nothing completes: the wait gives up after its limit (about two seconds of
// SM clock), records ERR_TIMEOUT in this unit's error word and returns, so
// the context stays usable.  It is how the error path every pipelined kernel
// relies on is tested without faulting or hanging the GPU.

#include "common.cuh"
#include "ptx.cuh"

namespace w4 {

namespace {

__global__ void __launch_bounds__(32) wait_timeout_kernel(int* waited) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_u32(&bar), 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // phase 0 never completes: nobody arrives on the barrier
        const bool done = ptx::mbar_wait(ptx::smem_u32(&bar), 0, &abort_flag);
        *waited = done ? 1 : 0;
    }
}

}  // namespace

w4_status run_selftest_wait_timeout(int* waited, cudaStream_t stream) {
    wait_timeout_kernel<<<1, 32, 0, stream>>>(waited);
    return launch_status(cudaGetLastError());
}

int take_device_error_selftest() { return take_unit_device_error(); }
int set_wait_limit_selftest(long long clocks) { return set_unit_wait_limit(clocks); }

}  // namespace w4
