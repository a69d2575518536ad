// kvc_selftest.cu -- kvc_selftest_wait_timeout: the failure path of the
// pipeline waits, exercised without a fault.
//
// Every wait of the step kernels is an mbarrier wait with a time limit: when
// the phase it waits for never completes (a role that stopped, a copy that
// never landed), the waiting role sets the CTA's abort flag, the other roles
// see it at their next check and return, and the kernel ORs KVC_DEV_TIMEOUT
// into the caller's status word. Here one CTA runs those waits on a barrier
// nothing ever arrives at: warp 0 waits with all lanes (as the consumer and
// softmax warps do), warp 1 with one lane under a short limit (as the
// producer and MMA threads do) and gives up first, which sets the flag that
// ends warp 0's wait. Nothing faults, traps or spins without a limit; the
// context stays usable.
#include <cuda_runtime.h>

#include "kvc.h"
#include "kvc_internal.cuh"
#include "kvc_pipeline.cuh"

namespace kvc {
namespace {

__global__ void __launch_bounds__(64, 1)
    wait_timeout_kernel(int32_t* dev_status, unsigned long long limit_ns) {
    __shared__ __align__(8) unsigned long long bar_word;
    __shared__ int abort_flag;
    const uint32_t bar = smem_addr(&bar_word);
    volatile int* abort = &abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(bar, 1u);  // one arrival that never comes
        *abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5;
    if (warp == 0) {
        // all lanes, the whole-warp form; ends when warp 1 sets the flag
        // (or, failing that, at its own limit of 4 x limit_ns)
        const bool ok = mbar_wait_limit(bar, 0u, abort, 4 * limit_ns);
        __all_sync(0xffffffffu, ok);
    } else if ((threadIdx.x & 31) == 0) {
        mbar_wait_limit(bar, 0u, abort, limit_ns);
    }
    __syncthreads();  // every thread reaches this exactly once
    if (threadIdx.x == 0 && *abort && dev_status) atomicOr(dev_status, KVC_DEV_TIMEOUT);
}

}  // namespace
}  // namespace kvc

int kvc_selftest_wait_timeout(int32_t* dev_status, int64_t limit_ns, void* stream) {
    if (!dev_status) return KVC_E_NULL;
    if (limit_ns < 1000 || limit_ns > 100000000) return KVC_E_SHAPE;
    kvc::wait_timeout_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(
        dev_status, static_cast<unsigned long long>(limit_ns));
    return cudaGetLastError() == cudaSuccess ? KVC_OK : KVC_E_CUDA;
}
