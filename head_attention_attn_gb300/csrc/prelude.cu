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
// Per-item form (decode): token i is item i, its position is cache_lens[i] (device), Q is
// written item-major [items, q_heads, hd] and K, V go to row cache_lens[i] of item i's own
// caches k_caches[i], v_caches[i] ([kv_heads, capacity, hd]), as ferrum-kernels
// qk_norm_rope_batched_per_item (per-item positions, item-major) and
// kv_cache_append_batched_per_cache (one row per item at its cache length) describe.
//
// Layout of the work: a group of hd/16 threads handles 4 consecutive head slots of one
// token (slots ordered Q heads, K heads, V heads as in qkv), 16 values of each row per
// thread, all loads and stores 16 bytes wide.  A thread issues the loads of its 4 rows
// before any arithmetic and loads the token's rotation angles and the norm weights once
// for the 4 rows:
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
    const void* const* k_caches;  // per-item form: device arrays of `tokens` cache pointers
    const void* const* v_caches;
    const int32_t* cache_lens;    // per-item form: position and cache row of item i
    int tokens, q_heads, kv_heads, pos_offset, qk_mode, rope_positions;
    int cache_len, cache_capacity;  // capacity 0 (contiguous form): k_out/v_out are [kv_heads, tokens, hd]
    float eps;
    WaitCtl wc;                     // only its status word is used
};

__device__ __forceinline__ void store8(uint16_t* p, const float (&f)[8], bool f16) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = f16 ? pack2<true>(f[2 * i], f[2 * i + 1]) : pack2<false>(f[2 * i], f[2 * i + 1]);
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ void load8f(const float* p, float* f) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p)), b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    f[0] = a.x, f[1] = a.y, f[2] = a.z, f[3] = a.w, f[4] = b.x, f[5] = b.y, f[6] = b.z, f[7] = b.w;
}

constexpr int kRowsPerGroup = 4;  // head rows of one token handled by one thread group

template <int HD, bool F16>
__global__ void __launch_bounds__(256, 3) prelude_kernel(const __grid_constant__ PreludeParams p) {
    constexpr int TPR = HD / 16;  // threads per group (and per head row)
    constexpr int R = kRowsPerGroup;
    const int slots = p.q_heads + 2 * p.kv_heads;
    const int groups_per_token = (slots + R - 1) / R;
    const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long group = gid / TPR;
    const int c = (int)(gid % TPR);
    bool valid = group < (long long)p.tokens * groups_per_token;
    const int t = valid ? (int)(group / groups_per_token) : 0;        // token (item)
    const int hs0 = valid ? (int)(group % groups_per_token) * R : 0;  // first head slot of the group
    const bool items = p.cache_lens != nullptr;
    const bool interleaved = p.qk_mode == 3;
    const int o0 = interleaved ? 16 * c : 8 * c;
    const int o1 = interleaved ? 16 * c + 8 : HD / 2 + 8 * c;

    long long pos = (long long)p.pos_offset + t;
    uint16_t* kdst = p.k_out;
    uint16_t* vdst = p.v_out;
    long long kv_row = t, head_stride = p.tokens;  // contiguous form: [kv_heads, tokens, hd]
    if (valid && items) {
        const int len = __ldg(p.cache_lens + t);
        const uintptr_t kp = reinterpret_cast<uintptr_t>(p.k_caches[t]);
        const uintptr_t vp = reinterpret_cast<uintptr_t>(p.v_caches[t]);
        const bool bad_len = len < 0 || len >= p.cache_capacity || (p.qk_mode != 0 && len >= p.rope_positions);
        const bool bad_ptr = kp == 0 || vp == 0 || (kp & 15u) != 0 || (vp & 15u) != 0;
        if (bad_len || bad_ptr) {
            // this item is neither read nor written; the lanes stay for the shuffles below
            if (c == 0 && hs0 == 0) record_status(p.wc.status, bad_len ? kStatusBadSeqlens : kStatusBadPointer);
            valid = false;
        } else {
            pos = len;
            kdst = reinterpret_cast<uint16_t*>(kp);
            vdst = reinterpret_cast<uint16_t*>(vp);
            kv_row = len;
            head_stride = p.cache_capacity;
        }
    } else if (p.cache_capacity > 0) {
        kv_row = (long long)p.cache_len + t;
        head_stride = p.cache_capacity;
    }

    // the group's rows: every load first, so R rows are in flight per thread
    uint4 raw[R][2];
    const uint16_t* src = p.qkv + ((long long)t * slots + hs0) * HD;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        if (valid && hs0 + r < slots) {
            raw[r][0] = *reinterpret_cast<const uint4*>(src + r * HD + o0);
            raw[r][1] = *reinterpret_cast<const uint4*>(src + r * HD + o1);
        } else {
            raw[r][0] = raw[r][1] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    // the token's rotation angles and the norm weights of my 16 value indices, once per group
    float cs[8], sn[8];
    if (valid && p.qk_mode != 0) {
        load8f(p.cos + pos * (HD / 2) + 8 * c, cs);
        load8f(p.sin + pos * (HD / 2) + 8 * c, sn);
    }

#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int hs = hs0 + r;
        const bool live = valid && hs < slots;
        const bool is_q = hs < p.q_heads;
        const bool is_k = !is_q && hs < p.q_heads + p.kv_heads;
        const bool rotate = live && (is_q || is_k) && p.qk_mode != 0;
        float a[8], b[8];
        {
            const uint32_t wa[4] = {raw[r][0].x, raw[r][0].y, raw[r][0].z, raw[r][0].w};
            const uint32_t wb[4] = {raw[r][1].x, raw[r][1].y, raw[r][1].z, raw[r][1].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 x = unpack2<F16>(wa[i]), y = unpack2<F16>(wb[i]);
                a[2 * i] = x.x, a[2 * i + 1] = x.y, b[2 * i] = y.x, b[2 * i + 1] = y.y;
            }
        }
        // per-head RMS norm (qk_mode 1): every lane takes part in the reduction, whatever
        // its row needs, so the shuffles never run with a partial warp
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) ss = fmaf(a[i], a[i], fmaf(b[i], b[i], ss));
#pragma unroll
        for (int m = 1; m < TPR; m <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m, TPR);
        if (rotate && p.qk_mode == 1) {
            const float rs = rsqrtf(ss * (1.f / HD) + p.eps);
            float w[16];  // the row's norm weights of my 16 value indices (cached reads)
            const float* wsrc = is_q ? p.q_norm_w : p.k_norm_w;
            load8f(wsrc + o0, w);
            load8f(wsrc + o1, w + 8);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                a[i] = a[i] * rs * w[i];
                b[i] = b[i] * rs * w[8 + i];
            }
        }
        if (rotate) {
            if (interleaved) {
                // pairs (a[0], a[1]), ..., (b[6], b[7]): angle indices 8c .. 8c+7
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float u = a[2 * j], v = a[2 * j + 1];
                    a[2 * j] = u * cs[j] - v * sn[j];
                    a[2 * j + 1] = v * cs[j] + u * sn[j];
                    const float u2 = b[2 * j], v2 = b[2 * j + 1];
                    b[2 * j] = u2 * cs[4 + j] - v2 * sn[4 + j];
                    b[2 * j + 1] = v2 * cs[4 + j] + u2 * sn[4 + j];
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
        if (!live) continue;
        uint16_t* dst;
        if (is_q) {
            dst = items ? p.q_out + ((long long)t * p.q_heads + hs) * HD : p.q_out + ((long long)hs * p.tokens + t) * HD;
        } else {
            const int h = is_k ? hs - p.q_heads : hs - p.q_heads - p.kv_heads;
            dst = (is_k ? kdst : vdst) + ((long long)h * head_stride + kv_row) * HD;
        }
        store8(dst + o0, a, F16);
        store8(dst + o1, b, F16);
    }
}

template <int HD, bool F16>
cudaError_t launch_t(const PreludeParams& p, cudaStream_t stream) {
    const int slots = p.q_heads + 2 * p.kv_heads;
    const long long groups = (long long)p.tokens * ((slots + kRowsPerGroup - 1) / kRowsPerGroup);
    const long long blocks = (groups * (HD / 16) + 255) / 256;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    prelude_kernel<HD, F16><<<(unsigned)blocks, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prelude(const PreludeProblem& pr, const WaitCtl& wc, cudaStream_t stream) {
    PreludeParams p;
    p.qkv = static_cast<const uint16_t*>(pr.qkv);
    p.q_norm_w = pr.q_norm_w;
    p.k_norm_w = pr.k_norm_w;
    p.cos = pr.cos;
    p.sin = pr.sin;
    p.q_out = static_cast<uint16_t*>(pr.q_out);
    p.k_out = static_cast<uint16_t*>(pr.k_out);
    p.v_out = static_cast<uint16_t*>(pr.v_out);
    p.k_caches = pr.k_caches;
    p.v_caches = pr.v_caches;
    p.cache_lens = pr.cache_lens;
    p.tokens = pr.tokens;
    p.q_heads = pr.q_heads;
    p.kv_heads = pr.kv_heads;
    p.pos_offset = pr.pos_offset;
    p.qk_mode = pr.qk_mode;
    p.rope_positions = pr.rope_positions;
    p.cache_len = pr.cache_len;
    p.cache_capacity = pr.cache_capacity;
    p.eps = pr.eps;
    p.wc = wc;
    if (pr.head_dim == 64) return pr.f16 ? launch_t<64, true>(p, stream) : launch_t<64, false>(p, stream);
    if (pr.head_dim == 128) return pr.f16 ? launch_t<128, true>(p, stream) : launch_t<128, false>(p, stream);
    return cudaErrorInvalidValue;
}

}  // namespace attn
