// prelude.cu -- K4: the attention prelude, one pass over the fused QKV projection output.
//
// Reads qkv [tokens, q_heads*hd + 2*kv_heads*hd] (bf16 or fp16) once and writes
//   Q to q_out [q_heads, tokens, hd] (head-major, the layout K1 reads),
//   K and V to k_out/v_out [kv_heads, tokens, hd], or straight into head-major caches
//   [kv_heads, capacity, hd] at rows cache_len .. cache_len + tokens - 1.
// Q and K are transformed by qk_mode: 1 = per-head RMS norm (x / sqrt(mean(x^2) + eps) * w)
// then half-split RoPE, 2 = half-split RoPE, 3 = interleaved RoPE, 0 = none; V is copied.
// A RoPE pair (a, b) at angle index j and position p = pos_offset + t becomes
// (a cos[p][j] - b sin[p][j], b cos[p][j] + a sin[p][j]); half-split pairs element j
// with j + hd/2, interleaved pairs 2j with 2j + 1.
//
// The operation is ferrum-kernels Backend::split_qkv_norm_rope and
// Backend::split_qkv_norm_rope_into_cache (which folds kv_cache_append_head_major
// into the same pass), with Backend::qk_norm_rope's per-head RMS norm and positions.
//
// Layout of the work: a row is one (token, head slot) of hd values, head slots ordered
// Q heads, K heads, V heads as in qkv.  hd/16 threads share a row, 16 values each, all
// loads and stores 16 bytes wide:
//   half-split (and copy): thread c holds values [8c, 8c+8) and [hd/2+8c, hd/2+8c+8),
//   interleaved:           thread c holds values [16c, 16c+16);
// either way its rotation pairs use angle indices [8c, 8c+8).  Arithmetic is fp32; the
// result is rounded to the input type.  Bound: HBM (each byte read once, written once).
#include "kernels.h"

namespace attn {
namespace {

struct PreludeParams {
    const uint16_t* qkv;
    const float* q_norm_w;
    const float* k_norm_w;
    const float* cos;
    const float* sin;
    uint16_t* q_out;
    uint16_t* k_out;
    uint16_t* v_out;
    int tokens, q_heads, kv_heads, pos_offset, qk_mode;
    int cache_len, cache_capacity;  // capacity 0: k_out/v_out are [kv_heads, tokens, hd]
    float eps;
    long long rows;                 // tokens * (q_heads + 2 * kv_heads)
};

__device__ __forceinline__ void load8(const uint16_t* p, float (&f)[8], bool f16) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = f16 ? unpack2<true>(w[i]) : unpack2<false>(w[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

__device__ __forceinline__ void store8(uint16_t* p, const float (&f)[8], bool f16) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = f16 ? pack2<true>(f[2 * i], f[2 * i + 1]) : pack2<false>(f[2 * i], f[2 * i + 1]);
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

template <int HD, bool F16>
__global__ void __launch_bounds__(256) prelude_kernel(const PreludeParams p) {
    constexpr int TPR = HD / 16;  // threads per row
    const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long row = gid / TPR;
    const int c = (int)(gid % TPR);
    const bool live = row < p.rows;
    const int slots = p.q_heads + 2 * p.kv_heads;
    const int t = live ? (int)(row / slots) : 0;
    const int hs = live ? (int)(row % slots) : 0;
    const bool is_q = hs < p.q_heads;
    const bool is_k = !is_q && hs < p.q_heads + p.kv_heads;
    const bool rotate = (is_q || is_k) && p.qk_mode != 0;
    const bool interleaved = p.qk_mode == 3;
    // element offsets of my two 8-value pieces inside the row
    const int o0 = interleaved ? 16 * c : 8 * c;
    const int o1 = interleaved ? 16 * c + 8 : HD / 2 + 8 * c;

    float a[8], b[8];  // a: first piece, b: second piece
    if (live) {
        const uint16_t* src = p.qkv + ((long long)t * slots + hs) * HD;
        load8(src + o0, a, F16);
        load8(src + o1, b, F16);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) a[i] = b[i] = 0.f;
    }

    // per-head RMS norm (qk_mode 1, Q and K): every lane of the row group takes part in the
    // reduction, whatever its row needs, so the shuffles never run with a partial group
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = fmaf(a[i], a[i], fmaf(b[i], b[i], ss));
#pragma unroll
    for (int m = 1; m < TPR; m <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m, TPR);
    if (live && rotate && p.qk_mode == 1) {
        const float r = rsqrtf(ss * (1.f / HD) + p.eps);
        const float* w = is_q ? p.q_norm_w : p.k_norm_w;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            a[i] = a[i] * r * __ldg(w + o0 + i);
            b[i] = b[i] * r * __ldg(w + o1 + i);
        }
    }

    if (live && rotate) {
        const long long pos = (long long)p.pos_offset + t;
        const float4* cp = reinterpret_cast<const float4*>(p.cos + pos * (HD / 2) + 8 * c);
        const float4* sp = reinterpret_cast<const float4*>(p.sin + pos * (HD / 2) + 8 * c);
        const float4 c0 = __ldg(cp), c1 = __ldg(cp + 1), s0 = __ldg(sp), s1 = __ldg(sp + 1);
        const float cs[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        const float sn[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
        if (interleaved) {
            // pairs (a[0], a[1]), ..., (b[6], b[7]): angle indices 8c .. 8c+7
            float x[16];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                x[i] = a[i];
                x[8 + i] = b[i];
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float u = x[2 * j], v = x[2 * j + 1];
                x[2 * j] = u * cs[j] - v * sn[j];
                x[2 * j + 1] = v * cs[j] + u * sn[j];
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                a[i] = x[i];
                b[i] = x[8 + i];
            }
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float u = a[j], v = b[j];
                a[j] = u * cs[j] - v * sn[j];
                b[j] = v * cs[j] + u * sn[j];
            }
        }
    }

    if (!live) return;
    uint16_t* dst;
    if (is_q) {
        dst = p.q_out + ((long long)hs * p.tokens + t) * HD;
    } else {
        const int h = is_k ? hs - p.q_heads : hs - p.q_heads - p.kv_heads;
        uint16_t* base = is_k ? p.k_out : p.v_out;
        dst = p.cache_capacity > 0 ? base + ((long long)h * p.cache_capacity + p.cache_len + t) * HD
                                   : base + ((long long)h * p.tokens + t) * HD;
    }
    store8(dst + o0, a, F16);
    store8(dst + o1, b, F16);
}

template <int HD, bool F16>
cudaError_t launch_t(const PreludeParams& p, cudaStream_t stream) {
    const long long threads = p.rows * (HD / 16);
    const long long blocks = (threads + 255) / 256;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    prelude_kernel<HD, F16><<<(unsigned)blocks, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prelude(const PreludeProblem& pr, cudaStream_t stream) {
    PreludeParams p;
    p.qkv = static_cast<const uint16_t*>(pr.qkv);
    p.q_norm_w = pr.q_norm_w;
    p.k_norm_w = pr.k_norm_w;
    p.cos = pr.cos;
    p.sin = pr.sin;
    p.q_out = static_cast<uint16_t*>(pr.q_out);
    p.k_out = static_cast<uint16_t*>(pr.k_out);
    p.v_out = static_cast<uint16_t*>(pr.v_out);
    p.tokens = pr.tokens;
    p.q_heads = pr.q_heads;
    p.kv_heads = pr.kv_heads;
    p.pos_offset = pr.pos_offset;
    p.qk_mode = pr.qk_mode;
    p.cache_len = pr.cache_len;
    p.cache_capacity = pr.cache_capacity;
    p.eps = pr.eps;
    p.rows = (long long)pr.tokens * (pr.q_heads + 2 * pr.kv_heads);
    if (pr.head_dim == 64) return pr.f16 ? launch_t<64, true>(p, stream) : launch_t<64, false>(p, stream);
    if (pr.head_dim == 128) return pr.f16 ? launch_t<128, true>(p, stream) : launch_t<128, false>(p, stream);
    return cudaErrorInvalidValue;
}

}  // namespace attn
