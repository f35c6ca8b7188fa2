// simt_f32.cu -- K3: fp32 attention on the CUDA cores (any head_dim in [1, 256]).
//
// fp32 inputs with a 1e-4 error budget rule out TF32 tensor cores, so this path
// is plain FFMA.  One warp owns one query row:
//   - the row of q sits in shared memory (read as a broadcast);
//   - the visible keys [lo, hi) are walked 32 at a time, one key per lane: the
//     lane forms its scaled dot product, the warp takes the chunk max and the
//     sum of exp(s - max) with xor-shuffle reductions, and the running max /
//     sum / accumulator are rescaled when the max grows (online softmax);
//   - each lane accumulates the head dims lane, lane+32, ... of P V, with the
//     probabilities broadcast by shuffle and V rows read coalesced.
// A row with no visible key is written as zeros.
//
// The stages are the ones of realizar cached/attention.rs (scores times scale,
// causal softmax with max subtraction and a guarded normalisation, weights
// times V), fused into one pass.
#include "kernels.h"

namespace attn {
namespace {

constexpr int kRowsPerBlock = 4;  // one warp per query row
constexpr int kMaxD = 256;

struct SimtParams {
    const float* q;
    const float* k;
    const float* v;
    float* out;
    const int32_t* key_lens;
    int Hq, Hkv, Lq, Lk, D, P, mode, window;
    int out_tok;  // out is [B, Lq, Hq, D] instead of [B, Hq, Lq, D]
    float scale;
};

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, m));
    return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
    return x;
}

__global__ void __launch_bounds__(kRowsPerBlock * 32) simt_f32_kernel(const SimtParams p) {
    __shared__ float qs[kRowsPerBlock][kMaxD];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hq = blockIdx.y, b = blockIdx.z;
    const int i = blockIdx.x * kRowsPerBlock + warp;
    if (i >= p.Lq) return;  // whole warp leaves together; no block-wide sync below
    const int hk = hq / (p.Hq / p.Hkv);
    const int D = p.D;

    const float* qrow = p.q + (((size_t)b * p.Hq + hq) * p.Lq + i) * D;
    for (int d = lane; d < D; d += 32) qs[warp][d] = qrow[d];
    __syncwarp();

    const int klen = valid_keys(p.key_lens, b, p.Lk);
    long long lo, hi;
    const long long qpos = (long long)p.P + i;
    key_interval(p.mode, p.window, klen, qpos, qpos, &lo, &hi);

    const size_t head_off = ((size_t)b * p.Hkv + hk) * (size_t)p.Lk * D;
    const float* kh = p.k + head_off;
    const float* vh = p.v + head_off;

    float m = -INFINITY, l = 0.f;
    float acc[kMaxD / 32];
#pragma unroll
    for (int t = 0; t < kMaxD / 32; ++t) acc[t] = 0.f;

    for (long long j0 = lo; j0 < hi; j0 += 32) {
        const long long j = j0 + lane;
        float s = -INFINITY;
        if (j < hi) {
            const float* kr = kh + j * D;
            float dot = 0.f;
            for (int d = 0; d < D; ++d) dot = fmaf(qs[warp][d], kr[d], dot);
            s = dot * p.scale;
        }
        const float mt = warp_max(s);           // finite: lane 0 always holds a visible key
        const float mn = fmaxf(m, mt);
        const float alpha = (m == -INFINITY) ? 0.f : expf(m - mn);
        const float pj = (j < hi) ? expf(s - mn) : 0.f;
        l = l * alpha + warp_sum(pj);
#pragma unroll
        for (int t = 0; t < kMaxD / 32; ++t) acc[t] *= alpha;
        const int n = (int)min(32LL, hi - j0);
        for (int jj = 0; jj < n; ++jj) {
            const float w = __shfl_sync(0xffffffffu, pj, jj);
            const float* vr = vh + (j0 + jj) * D;
#pragma unroll
            for (int t = 0; t < kMaxD / 32; ++t) {
                const int d = lane + 32 * t;
                if (d < D) acc[t] = fmaf(w, vr[d], acc[t]);
            }
        }
        m = mn;
    }

    const float inv = (l > 0.f) ? 1.f / l : 0.f;
    float* orow = p.out + (p.out_tok ? (((size_t)b * p.Lq + i) * p.Hq + hq) * D : (((size_t)b * p.Hq + hq) * p.Lq + i) * D);
#pragma unroll
    for (int t = 0; t < kMaxD / 32; ++t) {
        const int d = lane + 32 * t;
        if (d < D) orow[d] = acc[t] * inv;
    }
}

}  // namespace

cudaError_t launch_simt_f32(const Problem& pr, const WaitCtl& wc, cudaStream_t stream) {
    (void)wc;  // no device-side waits in this kernel
    SimtParams p;
    p.q = reinterpret_cast<const float*>(pr.q);
    p.k = reinterpret_cast<const float*>(pr.k);
    p.v = reinterpret_cast<const float*>(pr.v);
    p.out = reinterpret_cast<float*>(pr.out);
    p.key_lens = pr.key_lens;
    p.Hq = pr.Hq;
    p.Hkv = pr.Hkv;
    p.Lq = pr.Lq;
    p.Lk = pr.Lk;
    p.D = pr.D;
    p.P = pr.pos_offset;
    p.mode = pr.mode;
    p.window = pr.window;
    p.out_tok = pr.out_tok ? 1 : 0;
    p.scale = pr.scale;
    if (pr.Hq > 65535 || pr.B > 65535) return cudaErrorInvalidConfiguration;
    dim3 grid((unsigned)((pr.Lq + kRowsPerBlock - 1) / kRowsPerBlock), (unsigned)pr.Hq, (unsigned)pr.B);
    simt_f32_kernel<<<grid, kRowsPerBlock * 32, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace attn
