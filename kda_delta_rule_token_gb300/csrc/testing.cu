// Test hook: a kernel whose bounded wait is made to run out on purpose.
//
// It initialises an mbarrier that nothing ever arrives on (no copy and no MMA
// is issued), waits on it for at most `limit_ns` of wall time, records the
// give-up in the context's error word and returns.  Nothing is in flight
// when it gives up, so the device stays usable; the test then reads the
// error through kda_sync_status and checks that the next call is clean.
#include "kda_internal.cuh"
#include "ptx.cuh"

namespace kda {
namespace {

__global__ void kda_testing_wait_kernel(int* err, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !ptx::mbar_wait_timed(&bar, 0, nullptr, limit_ns))
        atomicOr(err, ptx::kErrTestingWait);
}

}  // namespace

cudaError_t launch_testing_wait(int* err_word, unsigned long long limit_ns, cudaStream_t stream) {
    kda_testing_wait_kernel<<<1, 32, 0, stream>>>(err_word, limit_ns);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace kda
