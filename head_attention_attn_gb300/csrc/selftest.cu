// selftest.cu -- device self test exposed through the C ABI: the bounded-wait
// path (a wait that gives up and reports instead of hanging).
#include "kernels.h"

namespace attn {
namespace {

// One block waits on a shared-memory barrier that nothing arrives on; the bounded
// wait gives up, records the time-out in the status word, and the block returns.
__global__ void timeout_selftest_kernel(const WaitCtl wc) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(smem_u32(&bar), 1);
        mbar_fence_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) (void)mbar_wait(smem_u32(&bar), 0, wc, &abort_flag);
    __syncthreads();
}

}  // namespace

cudaError_t launch_timeout_selftest(const WaitCtl& wc, cudaStream_t stream) {
    timeout_selftest_kernel<<<1, 32, 0, stream>>>(wc);
    return cudaGetLastError();
}

}  // namespace attn
