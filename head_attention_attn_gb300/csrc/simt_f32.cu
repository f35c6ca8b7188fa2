// simt_f32.cu -- K3: fp32 attention on the CUDA cores (any head_dim in [1, 256]).
//
// fp32 inputs with a 1e-4 error budget rule out TF32 tensor cores, so this path
// is plain FFMA.  A block of 4 warps owns 4 consecutive query rows of one head, one warp a row:
//   - the rows of q sit in shared memory (read as broadcasts);
//   - the union of the rows' visible keys is walked 32 at a time: the block copies the chunk's
//     K and V rows into shared memory together (coalesced, all loads in flight at once), then
//     each lane forms the scaled dot product of one key with its warp's row, the warp takes the
//     chunk max and the sum of exp(s - max) with xor-shuffle reductions, and the running max /
//     sum / accumulator are rescaled when the max grows (online softmax);
//   - each lane accumulates the head dims lane, lane+32, ... of P V, with the probabilities
//     broadcast by shuffle and V read from shared memory; only the row's own visible keys count.
// A row with no visible key is written as zeros.
//
// The stages are the ones of realizar cached/attention.rs (scores times scale,
// causal softmax with max subtraction and a guarded normalisation, weights
// times V), fused into one pass.
#include "kernels.h"

#include <mutex>

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

// Shared memory: q rows [4][D], the K chunk [32][D + 1] (padded: lane j reads row j), the V
// chunk [32][D].
__host__ __device__ constexpr size_t simt_smem_bytes(int D) {
    return sizeof(float) * ((size_t)kRowsPerBlock * D + 32 * (size_t)(D + 1) + 32 * (size_t)D);
}

__global__ void __launch_bounds__(kRowsPerBlock * 32) simt_f32_kernel(const SimtParams p) {
    extern __shared__ float sm[];
    const int D = p.D;
    float* qs = sm;                                   // [4][D]
    float* ks = qs + kRowsPerBlock * D;               // [32][D + 1]
    float* vs = ks + 32 * (D + 1);                    // [32][D]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hq = blockIdx.y, b = blockIdx.z;
    const int i0 = blockIdx.x * kRowsPerBlock;
    const int i = i0 + warp;
    const bool row_ok = i < p.Lq;  // a warp past the last row still helps copy, and stores nothing
    const int hk = hq / (p.Hq / p.Hkv);

    if (row_ok) {
        const float* qrow = p.q + (((size_t)b * p.Hq + hq) * p.Lq + i) * D;
        for (int d = lane; d < D; d += 32) qs[warp * D + d] = qrow[d];
    }

    const int klen = valid_keys(p.key_lens, b, p.Lk);
    long long lo = 0, hi = 0;
    if (row_ok) key_interval(p.mode, p.window, klen, (long long)p.P + i, (long long)p.P + i, &lo, &hi);
    // the block's chunks: the union of its rows' intervals
    long long blo, bhi;
    const int ilast = min(i0 + kRowsPerBlock, p.Lq) - 1;
    key_interval(p.mode, p.window, klen, (long long)p.P + i0, (long long)p.P + ilast, &blo, &bhi);

    const size_t head_off = ((size_t)b * p.Hkv + hk) * (size_t)p.Lk * D;
    const float* kh = p.k + head_off;
    const float* vh = p.v + head_off;

    float m = -INFINITY, l = 0.f;
    float acc[kMaxD / 32];
#pragma unroll
    for (int t = 0; t < kMaxD / 32; ++t) acc[t] = 0.f;

    for (long long j0 = blo; j0 < bhi; j0 += 32) {
        // the chunk's rows [j0, j0 + n) are contiguous in K and V: one flat coalesced copy each
        const int n = (int)min(32LL, bhi - j0);
        __syncthreads();  // the previous chunk is no longer read
        const float* kc = kh + j0 * D;
        const float* vc = vh + j0 * D;
        for (int x = threadIdx.x; x < n * D; x += kRowsPerBlock * 32) {
            const int r = x / D, d = x - r * D;
            ks[r * (D + 1) + d] = kc[x];
            vs[x] = vc[x];
        }
        __syncthreads();
        // this row's visible keys in the chunk: [c_lo, c_hi)
        const int c_lo = (int)max(0LL, min((long long)n, lo - j0));
        const int c_hi = (int)max(0LL, min((long long)n, hi - j0));
        if (c_lo >= c_hi) continue;  // warp-uniform: nothing of this chunk for this row
        float s = -INFINITY;
        if (lane >= c_lo && lane < c_hi) {
            const float* kr = ks + lane * (D + 1);
            const float* qr = qs + warp * D;
            float dot = 0.f;
#pragma unroll 4
            for (int d = 0; d < D; ++d) dot = fmaf(qr[d], kr[d], dot);
            s = dot * p.scale;
        }
        const float mt = warp_max(s);  // finite: some lane holds a visible key
        const float mn = fmaxf(m, mt);
        const float alpha = (m == -INFINITY) ? 0.f : expf(m - mn);
        const float pj = (lane >= c_lo && lane < c_hi) ? expf(s - mn) : 0.f;
        l = l * alpha + warp_sum(pj);
#pragma unroll
        for (int t = 0; t < kMaxD / 32; ++t) acc[t] *= alpha;
#pragma unroll 4
        for (int jj = c_lo; jj < c_hi; ++jj) {
            const float w = __shfl_sync(0xffffffffu, pj, jj);
            const float* vr = vs + jj * D;
#pragma unroll
            for (int t = 0; t < kMaxD / 32; ++t) {
                const int d = lane + 32 * t;
                if (d < D) acc[t] = fmaf(w, vr[d], acc[t]);
            }
        }
        m = mn;
    }

    if (!row_ok) return;
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
    if (pr.D < 1 || pr.D > kMaxD) return cudaErrorInvalidValue;
    const size_t smem = simt_smem_bytes(pr.D);
    if (smem > 48 * 1024) {  // head_dim above ~96 needs the opt-in shared-memory size
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        static std::mutex mu;
        static bool configured[64] = {};
        std::lock_guard<std::mutex> g(mu);
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        if (!configured[dev]) {
            e = cudaFuncSetAttribute(simt_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)simt_smem_bytes(kMaxD));
            if (e != cudaSuccess) return e;
            configured[dev] = true;
        }
    }
    dim3 grid((unsigned)((pr.Lq + kRowsPerBlock - 1) / kRowsPerBlock), (unsigned)pr.Hq, (unsigned)pr.B);
    simt_f32_kernel<<<grid, kRowsPerBlock * 32, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace attn
