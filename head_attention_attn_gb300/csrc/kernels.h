// kernels.h -- internal (non-exported) launch interface between the C ABI layer
// and the kernels: the tensor-core prefill (K1), the split-KV decode (K2), the fp32 path
// (K3), the attention prelude (K4), the tensor-core decode (K5) and the head_dim-64
// prefill on 64-key blocks (K6).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "attn.h"
#include "common.cuh"

namespace attn {

// Status code of the paged decode (with those in common.cuh): a page-table entry names no
// page of the pool.
constexpr unsigned kStatusBadPage = 7u;

// One validated attention problem (see attn.h for argument meaning).
struct Problem {
    const void* q;
    const void* k;
    const void* v;
    void* out;
    int B, Hq, Hkv, Lq, Lk, D;
    int pos_offset, mode, window;
    const int32_t* key_lens;
    float scale;
    bool f16;  // 16-bit element type: fp16 (true) or bf16 (false); unused by the fp32 path
    // Packed sequences (K1 only): q/out [total, Hq, D] and k/v [total, Hkv, D] token-major,
    // sequence b is rows [cu_seqlens[b], cu_seqlens[b+1]); Lq = Lk = the longest sequence.
    // Null for the head-major batch layout.
    const int32_t* cu_seqlens;
    int total;
    // Head-major batch only: out is token-major [B, Lq, Hq, D] instead of [B, Hq, Lq, D].
    bool out_tok = false;
    // Paged K/V (K1 only, with packed q/out): k and v are pools [num_pages, Hkv, page_size, D];
    // sequence b's position j is row j % page_size of pool page page_table[b * max_pages +
    // j / page_size]; kv_lens[b] positions are cached and the sequence's queries are the newest
    // of them.  Null when K/V are not paged.
    const int32_t* page_table = nullptr;
    const int32_t* kv_lens = nullptr;
    int page_size = 0, max_pages = 0, num_pages = 0;
};

// Visible key interval [lo, hi) for queries at positions [qpos_lo, qpos_hi]
// (inclusive), given klen valid keys.  The rule per mode is the one attn.h
// states; for a single query position the interval is exact, for a range it is
// the union over the range.
__host__ __device__ __forceinline__ void key_interval(int mode, int window, long long klen, long long qpos_lo,
                                                      long long qpos_hi, long long* lo, long long* hi) {
    long long l = 0, h = klen;
    if (mode == 1) {
        if (qpos_hi + 1 < h) h = qpos_hi + 1;
    } else if (mode == 2) {
        if (window > 0) {
            const long long hw = window / 2;
            if (qpos_lo - hw > l) l = qpos_lo - hw;
            if (qpos_hi + hw + 1 < h) h = qpos_hi + hw + 1;
        }
    } else if (mode == 3) {
        if (qpos_hi + 1 < h) h = qpos_hi + 1;
        if (window > 0 && qpos_lo - window + 1 > l) l = qpos_lo - window + 1;
    }
    *lo = l;
    *hi = h;
}

// Valid key count of sequence b: key_lens[b] clamped to [0, Lk], or Lk.
__device__ __forceinline__ int valid_keys(const int32_t* key_lens, int b, int Lk) {
    if (key_lens == nullptr) return Lk;
    int n = __ldg(key_lens + b);
    return n < 0 ? 0 : (n > Lk ? Lk : n);
}

// K1: tcgen05 + TMA fused prefill, bf16 or fp16, head_dim 64 or 128; head-major, packed, or
// packed queries over paged K/V.
cudaError_t launch_prefill_tc(const Problem& p, const WaitCtl& wc, cudaStream_t stream);

// K6: the head_dim 64 prefill with 64-key blocks and four CTAs per SM (head-major or packed).
bool prefill_narrow_supported(const Problem& p);
cudaError_t launch_prefill_narrow(const Problem& p, const WaitCtl& wc, cudaStream_t stream);

// K2: split-KV decode for q_len == 1, bf16 or fp16, head_dim 64 or 128, group size 1/2/4/8.
bool decode_supported(const Problem& p);
cudaError_t launch_decode_splitkv(const Problem& p, const WaitCtl& wc, cudaStream_t stream, int num_sms);

// K5: tensor-core decode for q_len == 1, head_dim 128, 4 or 8 query heads per kv head.
bool decode_tc_supported(const Problem& p);
cudaError_t launch_decode_tc(const Problem& p, const WaitCtl& wc, cudaStream_t stream, int num_sms);
// K5 over per-item caches (TMA through a K and a V tensor map per item, written on the device
// into a stream-ordered workspace) or paged caches (TMA per page piece where the page size
// allows it, rows gathered otherwise), the same shapes.
bool decode_tc_items_supported(int Hq, int Hkv, int D);
bool decode_tc_paged_tma(int page_size, int num_pages, int Hkv);
struct CachesProblem;
struct PagedProblem;
cudaError_t launch_decode_tc_caches(const CachesProblem& p, const WaitCtl& wc, cudaStream_t stream, int num_sms);
// The same, with the maps in a fixed device table of kStaticMapItems items instead of a per-call
// workspace (allocates nothing; calls that overlap on the GPU race on the table).
constexpr int kStaticMapItems = ATTN_NOALLOC_MAX_ITEMS;
cudaError_t launch_decode_tc_caches_static(const CachesProblem& p, const WaitCtl& wc, cudaStream_t stream,
                                           int num_sms);
cudaError_t launch_decode_tc_paged(const PagedProblem& p, const WaitCtl& wc, cudaStream_t stream, int num_sms);

// K2 over per-item caches: one single-query decode step for m items, item i reading its
// own [Hkv, capacity, D] K and V caches through device pointer arrays.
struct CachesProblem {
    const void* q;
    const void* const* k_caches;
    const void* const* v_caches;
    void* out;
    int m, Hq, Hkv, capacity, D;
    const int32_t* kv_lens;
    int sliding;
    float scale;
    bool f16;  // fp16 (true) or bf16 (false)
};
cudaError_t launch_decode_caches(const CachesProblem& p, const WaitCtl& wc, cudaStream_t stream, int num_sms);

// K2 over paged caches: pools [num_pages, Hkv, page_size, D], item i's position j in pool page
// page_table[i * max_pages + j / page_size], row j % page_size.
struct PagedProblem {
    const void* q;
    const void* k_pool;
    const void* v_pool;
    const int32_t* page_table;  // device [m, max_pages]
    void* out;
    int m, Hq, Hkv, num_pages, page_size, max_pages, D;
    const int32_t* kv_lens;
    int sliding;
    float scale;
    bool f16;
};
cudaError_t launch_decode_paged(const PagedProblem& p, const WaitCtl& wc, cudaStream_t stream, int num_sms);

// K4: the attention prelude (split fused QKV, per-head RMS norm, RoPE, head-major
// transpose, optionally into KV caches), bf16 or fp16, head_dim 64 or 128.
struct PreludeProblem {
    const void* qkv;
    const float* q_norm_w;
    const float* k_norm_w;
    const float* cos;
    const float* sin;
    void* q_out;
    void* k_out;
    void* v_out;
    int tokens, q_heads, kv_heads, head_dim, pos_offset, qk_mode;
    int cache_len, cache_capacity;
    float eps;
    bool f16;
    int rope_positions;
    // Per-item form (null otherwise): item i = token i, position cache_lens[i], Q item-major,
    // K/V into row cache_lens[i] of k_caches[i] / v_caches[i] ([kv_heads, capacity, hd]).
    const void* const* k_caches;
    const void* const* v_caches;
    const int32_t* cache_lens;
};
cudaError_t launch_prelude(const PreludeProblem& p, const WaitCtl& wc, cudaStream_t stream);

// K3: fp32 SIMT attention, any head_dim in [1, 256].
cudaError_t launch_simt_f32(const Problem& p, const WaitCtl& wc, cudaStream_t stream);

// Bounded-wait self test: one block waits on an mbarrier nobody signals.
cudaError_t launch_timeout_selftest(const WaitCtl& wc, cudaStream_t stream);

}  // namespace attn
