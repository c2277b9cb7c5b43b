// Self-test of the bounded device-side waits.  The tcgen05 kernels wait on mbarriers with
// the library's bounded poll (tc::mbar_wait): after a fixed number of polls (over a second)
// a wait gives up, raises the CTA's abort flag and records its site in the workspace
// status word, which hla2_workspace_status reports as HLA2_ERR_TIMEOUT.  This kernel runs
// that same wait on an mbarrier that nothing ever arrives at, so the timeout path can be
// exercised without a fault, a trap or a hang: the wait gives up, the kernel returns, and
// the context stays usable.
#include "kernels.h"
#include "tc_common.cuh"

namespace hla2 {

namespace {

constexpr int kSelfTestSite = 90;  // status value the self-test's wait records

__global__ void __launch_bounds__(32) wait_timeout_kernel(int* status) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        *status = 0;
        tc::mbar_init(&bar, 1);  // expects one arrival, which never comes
        abort_flag = 0;
        tc::mbar_fence_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) tc::mbar_wait(&bar, 0, &abort_flag, status, kSelfTestSite);
    __syncthreads();
}

// Debug build only: one failing bounds check that guards no access, so that the recording of
// a check's site can be tested without an out-of-bounds access anywhere.
constexpr int kDebugSelfTestSite = 1;
__global__ void debug_check_kernel(int* sink) {
    if (!HLA2_IN(threadIdx.x > 0, kDebugSelfTestSite)) return;  // thread 0 records the site
    (void)sink;
}

}  // namespace

int launch_wait_timeout_selftest(int* status, cudaStream_t st) {
    wait_timeout_kernel<<<1, 32, 0, st>>>(status);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

int launch_debug_check_selftest(cudaStream_t st) {
    debug_check_kernel<<<1, 32, 0, st>>>(nullptr);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace hla2

HLA2_DEBUG_READER(selftest)
