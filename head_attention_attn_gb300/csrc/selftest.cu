// selftest.cu -- device self tests exposed through the C ABI: the bounded-wait
// path (a wait that gives up and reports instead of hanging) and the two 2^x
// routines the softmax uses.
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

__global__ void exp2_selftest_kernel(const float* x, float* y_poly, float* y_unit, int n) {
    const int i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
    if (i >= n) return;
    const float a = x[i];
    const float b = (i + 1 < n) ? x[i + 1] : 0.f;
    const float2 p = ex2_poly2(make_float2(a, b));
    y_poly[i] = p.x;
    y_unit[i] = ex2_approx(a);
    if (i + 1 < n) {
        y_poly[i + 1] = p.y;
        y_unit[i + 1] = ex2_approx(b);
    }
}

}  // namespace

cudaError_t launch_timeout_selftest(const WaitCtl& wc, cudaStream_t stream) {
    timeout_selftest_kernel<<<1, 32, 0, stream>>>(wc);
    return cudaGetLastError();
}

cudaError_t launch_exp2_selftest(const float* x, float* y_poly, float* y_unit, int n, cudaStream_t stream) {
    const int pairs = (n + 1) / 2;
    exp2_selftest_kernel<<<(pairs + 255) / 256, 256, 0, stream>>>(x, y_poly, y_unit, n);
    return cudaGetLastError();
}

}  // namespace attn
