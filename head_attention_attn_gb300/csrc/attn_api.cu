// attn_api.cu -- the exported C ABI (attn.h): argument checks, kernel choice,
// the device status word of the bounded waits, and per-thread error messages.
//
// Kernel choice:
//   f32                          -> K3 (SIMT fp32, any head_dim 1..256)
//   bf16/fp16, q_len == 1, head_dim 128, group 4/8 -> K5 (tensor-core split-KV decode);
//                                   per-item caches of that shape (TMA through tensor maps
//                                   written on the device), and paged caches of that shape
//                                   where the measured routing table prefers it
//   bf16/fp16, q_len == 1, group 1/2/4/8 -> K2 (split-KV decode, the other shapes)
//   bf16/fp16, head_dim 64, head-major or packed -> K6 (tcgen05 prefill on 64-key blocks)
//   bf16/fp16 otherwise          -> K1 (tcgen05 + TMA fused prefill; head-major, head_dim 128,
//                                   even group, no key padding: its persistent form, one CTA
//                                   per SM over the query blocks); packed queries over
//                                   paged caches also go to K1, whose producer copies K/V
//                                   by TMA a page piece at a time (page sizes of 8..128 rows
//                                   dividing 128, or multiples of 128) or else gathers the
//                                   rows through the page table
// There is no host fallback: an unsupported shape is refused (ferrum-kernels:
// CUDA ops fail rather than copy data through host memory).
#include <math.h>
#include <stdarg.h>
#include <stdio.h>

#include <mutex>
#include <string>

#include "attn.h"
#include "kernels.h"

// Device status word: a bounded wait that gives up writes its code here.
__device__ unsigned int g_attn_status = 0;

namespace {

constexpr int kMaxDevices = 64;
// A device-side wait gives up after 250 ms: a healthy one lasts microseconds (a copy landing, a
// tensor-core product), and a launch whose waits fail ends after about one limit per wave of blocks.
constexpr unsigned long long kWaitLimitNs = 250000000ull;

thread_local std::string t_last_error;

attn_status fail(attn_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return s;
}

struct DeviceState {
    bool ready = false;
    unsigned* status = nullptr;
    int num_sms = 0;
};
DeviceState g_dev[kMaxDevices];
std::mutex g_dev_mu;

attn_status device_state(DeviceState** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(ATTN_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> g(g_dev_mu);
    DeviceState& st = g_dev[dev];
    if (!st.ready) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_attn_status);
        if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
        st.status = static_cast<unsigned*>(ptr);
        st.num_sms = sms;
        st.ready = true;
    }
    *out = &st;
    return ATTN_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// attn_fwd and attn_fwd_out_token_major: the same checks and kernels, out_tok choosing the
// layout of out.
attn_status fwd(const void* q, const void* k, const void* v, void* out, int batch, int q_heads, int kv_heads,
                int q_len, int kv_len, int head_dim, int pos_offset, int mask_mode, int window,
                const int32_t* key_lens, float scale, int dtype, void* cuda_stream, bool out_tok) {
    t_last_error.clear();
    if (batch < 0 || q_len < 0 || kv_len < 0)
        return fail(ATTN_ERR_INVALID_ARG, "negative size (batch=%d, q_len=%d, kv_len=%d)", batch, q_len, kv_len);
    if (q_heads <= 0 || kv_heads <= 0 || head_dim <= 0)
        return fail(ATTN_ERR_INVALID_ARG, "q_heads, kv_heads and head_dim must be positive (%d, %d, %d)", q_heads,
                    kv_heads, head_dim);
    if (q_heads % kv_heads != 0)
        return fail(ATTN_ERR_INVALID_ARG, "q_heads (%d) is not a multiple of kv_heads (%d)", q_heads, kv_heads);
    if (mask_mode < ATTN_MASK_NONE || mask_mode > ATTN_MASK_CAUSAL_WINDOW)
        return fail(ATTN_ERR_INVALID_ARG, "mask_mode %d out of range", mask_mode);
    if (dtype != ATTN_BF16 && dtype != ATTN_F32 && dtype != ATTN_F16)
        return fail(ATTN_ERR_INVALID_ARG, "dtype %d out of range", dtype);
    if (window < 0) return fail(ATTN_ERR_INVALID_ARG, "negative window %d", window);
    if (pos_offset < 0) return fail(ATTN_ERR_INVALID_ARG, "negative pos_offset %d", pos_offset);
    if (!isfinite(scale)) return fail(ATTN_ERR_INVALID_ARG, "scale is not finite");
    if (dtype != ATTN_F32 && head_dim != 64 && head_dim != 128)
        return fail(ATTN_ERR_UNSUPPORTED, "bf16 and fp16 support head_dim 64 and 128, not %d", head_dim);
    if (dtype == ATTN_F32 && head_dim > 256)
        return fail(ATTN_ERR_UNSUPPORTED, "f32 supports head_dim up to 256, not %d", head_dim);
    if ((long long)batch * q_heads > 0x7fffffffLL || (long long)batch * kv_heads > 0x7fffffffLL)
        return fail(ATTN_ERR_UNSUPPORTED, "batch * heads exceeds 2^31-1");
    if (batch == 0 || q_len == 0) return ATTN_OK;  // nothing to compute

    if (!q || !out) return fail(ATTN_ERR_INVALID_ARG, "null q or out pointer");
    const size_t esize = (dtype == ATTN_F32) ? 4 : 2;
    cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
    if (kv_len == 0) {
        // Every row sees no key: the defined result is all zeros.
        const size_t bytes = (size_t)batch * q_heads * q_len * head_dim * esize;
        cudaError_t e = cudaMemsetAsync(out, 0, bytes, stream);
        if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "cudaMemsetAsync: %s", cudaGetErrorString(e));
        return ATTN_OK;
    }
    if (!k || !v) return fail(ATTN_ERR_INVALID_ARG, "null k or v pointer");
    const uintptr_t align = (dtype == ATTN_F32) ? 4 : 16;
    if (!aligned(q, align) || !aligned(k, align) || !aligned(v, align) || !aligned(out, align))
        return fail(ATTN_ERR_INVALID_ARG, "q, k, v and out must be %u-byte aligned", (unsigned)align);
    if (key_lens && !aligned(key_lens, 4)) return fail(ATTN_ERR_INVALID_ARG, "key_lens must be 4-byte aligned");

    DeviceState* st = nullptr;
    attn_status s = device_state(&st);
    if (s != ATTN_OK) return s;
    attn::WaitCtl wc{st->status, kWaitLimitNs};
    attn::Problem p{q, k, v, out, batch, q_heads, kv_heads, q_len, kv_len, head_dim,
                    pos_offset, mask_mode, window, key_lens, scale, dtype == ATTN_F16};
    p.out_tok = out_tok;  // the decode kernels run only for q_len 1, where both layouts coincide

    cudaError_t e;
    const char* which;
    if (dtype == ATTN_F32) {
        if (q_heads > 65535 || batch > 65535)
            return fail(ATTN_ERR_UNSUPPORTED, "f32 path limits q_heads and batch to 65535");
        which = "simt_f32";
        e = attn::launch_simt_f32(p, wc, stream);
    } else if (attn::decode_tc_supported(p) && kv_heads <= 65535 && batch <= 65535) {
        which = "decode_tc";
        e = attn::launch_decode_tc(p, wc, stream, st->num_sms);
    } else if (attn::decode_supported(p) && kv_heads <= 65535 && batch <= 65535) {
        which = "decode_splitkv";
        e = attn::launch_decode_splitkv(p, wc, stream, st->num_sms);
    } else {
        which = "prefill_tc";
        e = attn::launch_prefill_tc(p, wc, stream);
    }
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "%s launch: %s", which, cudaGetErrorString(e));
    return ATTN_OK;
}

// attn_decode_caches and attn_decode_caches_noalloc: the same checks and kernels; `fixed_maps`
// puts the per-item tensor maps of the tensor-core decode in the fixed device table instead of a
// stream-ordered workspace.
attn_status decode_caches(const void* q, const void* const* k_caches, const void* const* v_caches, void* out, int m,
                          int q_heads, int kv_heads, int capacity, int head_dim, const int32_t* kv_lens,
                          int sliding_window, float scale, int dtype, void* cuda_stream, bool fixed_maps) {
    if (m < 0 || capacity < 0) return fail(ATTN_ERR_INVALID_ARG, "negative size (m=%d, capacity=%d)", m, capacity);
    if (q_heads <= 0 || kv_heads <= 0 || head_dim <= 0)
        return fail(ATTN_ERR_INVALID_ARG, "q_heads, kv_heads and head_dim must be positive (%d, %d, %d)", q_heads,
                    kv_heads, head_dim);
    if (q_heads % kv_heads != 0)
        return fail(ATTN_ERR_INVALID_ARG, "q_heads (%d) is not a multiple of kv_heads (%d)", q_heads, kv_heads);
    if (sliding_window < 0) return fail(ATTN_ERR_INVALID_ARG, "negative sliding_window %d", sliding_window);
    if (!isfinite(scale)) return fail(ATTN_ERR_INVALID_ARG, "scale is not finite");
    if (dtype != ATTN_BF16 && dtype != ATTN_F16)
        return fail(ATTN_ERR_UNSUPPORTED, "per-item caches support bf16 and fp16 only");
    if (head_dim != 64 && head_dim != 128)
        return fail(ATTN_ERR_UNSUPPORTED, "bf16 and fp16 support head_dim 64 and 128, not %d", head_dim);
    const int G = q_heads / kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8)
        return fail(ATTN_ERR_UNSUPPORTED, "per-item caches support 1, 2, 4 or 8 query heads per kv head, not %d", G);
    if (m > 65535 || kv_heads > 65535) return fail(ATTN_ERR_UNSUPPORTED, "m and kv_heads are limited to 65535");
    if (m == 0) return ATTN_OK;
    if (!q || !out || !k_caches || !v_caches || !kv_lens)
        return fail(ATTN_ERR_INVALID_ARG, "null q, out, k_caches, v_caches or kv_lens pointer");
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_caches, 8) || !aligned(v_caches, 8) || !aligned(kv_lens, 4))
        return fail(ATTN_ERR_INVALID_ARG, "q/out must be 16-byte, pointer arrays 8-byte, kv_lens 4-byte aligned");
    cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
    if (capacity == 0) {
        cudaError_t e = cudaMemsetAsync(out, 0, (size_t)m * q_heads * head_dim * 2, stream);
        if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "cudaMemsetAsync: %s", cudaGetErrorString(e));
        return ATTN_OK;
    }
    DeviceState* st = nullptr;
    attn_status s = device_state(&st);
    if (s != ATTN_OK) return s;
    attn::WaitCtl wc{st->status, kWaitLimitNs};
    attn::CachesProblem p{q, k_caches, v_caches, out, m, q_heads, kv_heads, capacity, head_dim,
                          kv_lens, sliding_window, scale, dtype == ATTN_F16};
    // At 4 and 8 query heads per kv head (head_dim 128) the tensor-core decode streams the
    // per-item caches by TMA through tensor maps it builds on the device; other shapes take the
    // CUDA-core decode.
    const bool tc = attn::decode_tc_items_supported(q_heads, kv_heads, head_dim);
    cudaError_t e = !tc        ? attn::launch_decode_caches(p, wc, stream, st->num_sms)
                    : fixed_maps ? attn::launch_decode_tc_caches_static(p, wc, stream, st->num_sms)
                                 : attn::launch_decode_tc_caches(p, wc, stream, st->num_sms);
    if (e != cudaSuccess)
        return fail(ATTN_ERR_CUDA, "%s launch: %s", tc ? "decode_tc (caches)" : "decode_caches", cudaGetErrorString(e));
    return ATTN_OK;
}

}  // namespace

extern "C" {

attn_status attn_fwd(const void* q, const void* k, const void* v, void* out, int batch, int q_heads, int kv_heads,
                     int q_len, int kv_len, int head_dim, int pos_offset, int mask_mode, int window,
                     const int32_t* key_lens, float scale, int dtype, void* cuda_stream) {
    return fwd(q, k, v, out, batch, q_heads, kv_heads, q_len, kv_len, head_dim, pos_offset, mask_mode, window,
               key_lens, scale, dtype, cuda_stream, false);
}

attn_status attn_fwd_out_token_major(const void* q, const void* k, const void* v, void* out, int batch,
                                     int q_heads, int kv_heads, int q_len, int kv_len, int head_dim, int pos_offset,
                                     int mask_mode, int window, const int32_t* key_lens, float scale, int dtype,
                                     void* cuda_stream) {
    return fwd(q, k, v, out, batch, q_heads, kv_heads, q_len, kv_len, head_dim, pos_offset, mask_mode, window,
               key_lens, scale, dtype, cuda_stream, true);
}

attn_status attn_fwd_varlen(const void* q, const void* k, const void* v, void* out, const int32_t* cu_seqlens,
                            int batch, int total, int max_seqlen, int q_heads, int kv_heads, int head_dim,
                            int mask_mode, int window, float scale, int dtype, void* cuda_stream) {
    t_last_error.clear();
    if (batch < 0 || total < 0 || max_seqlen < 0)
        return fail(ATTN_ERR_INVALID_ARG, "negative size (batch=%d, total=%d, max_seqlen=%d)", batch, total,
                    max_seqlen);
    if (q_heads <= 0 || kv_heads <= 0 || head_dim <= 0)
        return fail(ATTN_ERR_INVALID_ARG, "q_heads, kv_heads and head_dim must be positive (%d, %d, %d)", q_heads,
                    kv_heads, head_dim);
    if (q_heads % kv_heads != 0)
        return fail(ATTN_ERR_INVALID_ARG, "q_heads (%d) is not a multiple of kv_heads (%d)", q_heads, kv_heads);
    if (mask_mode < ATTN_MASK_NONE || mask_mode > ATTN_MASK_CAUSAL_WINDOW)
        return fail(ATTN_ERR_INVALID_ARG, "mask_mode %d out of range", mask_mode);
    if (dtype != ATTN_BF16 && dtype != ATTN_F32 && dtype != ATTN_F16)
        return fail(ATTN_ERR_INVALID_ARG, "dtype %d out of range", dtype);
    if (window < 0) return fail(ATTN_ERR_INVALID_ARG, "negative window %d", window);
    if (!isfinite(scale)) return fail(ATTN_ERR_INVALID_ARG, "scale is not finite");
    if (dtype == ATTN_F32) return fail(ATTN_ERR_UNSUPPORTED, "packed sequences support bf16 and fp16");
    if (head_dim != 64 && head_dim != 128)
        return fail(ATTN_ERR_UNSUPPORTED, "bf16 and fp16 support head_dim 64 and 128, not %d", head_dim);
    if (max_seqlen > total) return fail(ATTN_ERR_INVALID_ARG, "max_seqlen %d exceeds total %d", max_seqlen, total);
    if (batch == 0 || max_seqlen == 0) return ATTN_OK;  // nothing to compute
    const long long blocks = ((long long)max_seqlen + 255) / 128;  // upper bound on query blocks per head
    if (blocks * batch * q_heads > 0x7fffffffLL)
        return fail(ATTN_ERR_UNSUPPORTED, "max_seqlen * batch * q_heads is too large for one launch");
    if (!q || !k || !v || !out) return fail(ATTN_ERR_INVALID_ARG, "null q, k, v or out pointer");
    if (!cu_seqlens) return fail(ATTN_ERR_INVALID_ARG, "null cu_seqlens pointer");
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || !aligned(cu_seqlens, 4))
        return fail(ATTN_ERR_INVALID_ARG, "q, k, v and out must be 16-byte aligned, cu_seqlens 4-byte aligned");

    DeviceState* st = nullptr;
    attn_status s = device_state(&st);
    if (s != ATTN_OK) return s;
    attn::WaitCtl wc{st->status, kWaitLimitNs};
    attn::Problem p{q, k, v, out, batch, q_heads, kv_heads, max_seqlen, max_seqlen, head_dim,
                    0, mask_mode, window, nullptr, scale, dtype == ATTN_F16, cu_seqlens, total};
    cudaError_t e = attn::launch_prefill_tc(p, wc, static_cast<cudaStream_t>(cuda_stream));
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "prefill_tc launch: %s", cudaGetErrorString(e));
    return ATTN_OK;
}

attn_status attn_fwd_varlen_paged(const void* q, const void* k_pool, const void* v_pool, const int32_t* page_table,
                                  void* out, const int32_t* cu_seqlens_q, const int32_t* kv_lens, int batch,
                                  int total_q, int max_seqlen_q, int q_heads, int kv_heads, int num_pages,
                                  int page_size, int max_pages, int head_dim, int mask_mode, int window, float scale,
                                  int dtype, void* cuda_stream) {
    t_last_error.clear();
    if (batch < 0 || total_q < 0 || max_seqlen_q < 0 || num_pages < 0 || max_pages < 0)
        return fail(ATTN_ERR_INVALID_ARG, "negative size (batch=%d, total_q=%d, max_seqlen_q=%d, num_pages=%d, "
                    "max_pages=%d)", batch, total_q, max_seqlen_q, num_pages, max_pages);
    if (page_size < 1) return fail(ATTN_ERR_INVALID_ARG, "page_size must be at least 1, not %d", page_size);
    if ((long long)page_size * max_pages > 0x7fffffffLL)
        return fail(ATTN_ERR_INVALID_ARG, "max_pages * page_size exceeds 2^31-1");
    if (q_heads <= 0 || kv_heads <= 0 || head_dim <= 0)
        return fail(ATTN_ERR_INVALID_ARG, "q_heads, kv_heads and head_dim must be positive (%d, %d, %d)", q_heads,
                    kv_heads, head_dim);
    if (q_heads % kv_heads != 0)
        return fail(ATTN_ERR_INVALID_ARG, "q_heads (%d) is not a multiple of kv_heads (%d)", q_heads, kv_heads);
    if (mask_mode < ATTN_MASK_NONE || mask_mode > ATTN_MASK_CAUSAL_WINDOW)
        return fail(ATTN_ERR_INVALID_ARG, "mask_mode %d out of range", mask_mode);
    if (dtype != ATTN_BF16 && dtype != ATTN_F32 && dtype != ATTN_F16)
        return fail(ATTN_ERR_INVALID_ARG, "dtype %d out of range", dtype);
    if (window < 0) return fail(ATTN_ERR_INVALID_ARG, "negative window %d", window);
    if (!isfinite(scale)) return fail(ATTN_ERR_INVALID_ARG, "scale is not finite");
    if (dtype == ATTN_F32) return fail(ATTN_ERR_UNSUPPORTED, "paged caches support bf16 and fp16");
    if (head_dim != 64 && head_dim != 128)
        return fail(ATTN_ERR_UNSUPPORTED, "bf16 and fp16 support head_dim 64 and 128, not %d", head_dim);
    if (max_seqlen_q > total_q)
        return fail(ATTN_ERR_INVALID_ARG, "max_seqlen_q %d exceeds total_q %d", max_seqlen_q, total_q);
    if (batch == 0 || max_seqlen_q == 0) return ATTN_OK;  // nothing to compute
    const long long blocks = ((long long)max_seqlen_q + 255) / 128;  // upper bound on query blocks per head
    if (blocks * batch * q_heads > 0x7fffffffLL)
        return fail(ATTN_ERR_UNSUPPORTED, "max_seqlen_q * batch * q_heads is too large for one launch");
    if (!q || !out || !cu_seqlens_q || !kv_lens)
        return fail(ATTN_ERR_INVALID_ARG, "null q, out, cu_seqlens_q or kv_lens pointer");
    if ((long long)page_size * max_pages > 0 && (!k_pool || !v_pool || !page_table))
        return fail(ATTN_ERR_INVALID_ARG, "null k_pool, v_pool or page_table pointer");
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) ||
        !aligned(page_table, 4) || !aligned(cu_seqlens_q, 4) || !aligned(kv_lens, 4))
        return fail(ATTN_ERR_INVALID_ARG,
                    "q, out and the pools must be 16-byte aligned; page_table, cu_seqlens_q and kv_lens 4-byte aligned");

    DeviceState* st = nullptr;
    attn_status s = device_state(&st);
    if (s != ATTN_OK) return s;
    attn::WaitCtl wc{st->status, kWaitLimitNs};
    attn::Problem p{q, k_pool, v_pool, out, batch, q_heads, kv_heads, max_seqlen_q, 0, head_dim,
                    0, mask_mode, window, nullptr, scale, dtype == ATTN_F16, cu_seqlens_q, total_q};
    p.page_table = page_table;
    p.kv_lens = kv_lens;
    p.page_size = page_size;
    p.max_pages = max_pages;
    p.num_pages = num_pages;
    cudaError_t e = attn::launch_prefill_tc(p, wc, static_cast<cudaStream_t>(cuda_stream));
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "prefill_tc (paged) launch: %s", cudaGetErrorString(e));
    return ATTN_OK;
}

attn_status attn_decode_caches(const void* q, const void* const* k_caches, const void* const* v_caches, void* out,
                               int m, int q_heads, int kv_heads, int capacity, int head_dim, const int32_t* kv_lens,
                               int sliding_window, float scale, int dtype, void* cuda_stream) {
    t_last_error.clear();
    return decode_caches(q, k_caches, v_caches, out, m, q_heads, kv_heads, capacity, head_dim, kv_lens,
                         sliding_window, scale, dtype, cuda_stream, false);
}

attn_status attn_decode_caches_noalloc(const void* q, const void* const* k_caches, const void* const* v_caches,
                                       void* out, int m, int q_heads, int kv_heads, int capacity, int head_dim,
                                       const int32_t* kv_lens, int sliding_window, float scale, int dtype,
                                       void* cuda_stream) {
    t_last_error.clear();
    if (m > attn::kStaticMapItems)
        return fail(ATTN_ERR_INVALID_ARG, "m (%d) exceeds the %d items of the fixed map table", m,
                    attn::kStaticMapItems);
    return decode_caches(q, k_caches, v_caches, out, m, q_heads, kv_heads, capacity, head_dim, kv_lens,
                         sliding_window, scale, dtype, cuda_stream, true);
}

attn_status attn_decode_paged(const void* q, const void* k_pool, const void* v_pool, const int32_t* page_table,
                              void* out, int m, int q_heads, int kv_heads, int num_pages, int page_size,
                              int max_pages, int head_dim, const int32_t* kv_lens, int sliding_window, float scale,
                              int dtype, void* cuda_stream) {
    t_last_error.clear();
    if (m < 0 || num_pages < 0 || max_pages < 0)
        return fail(ATTN_ERR_INVALID_ARG, "negative size (m=%d, num_pages=%d, max_pages=%d)", m, num_pages,
                    max_pages);
    if (page_size < 1) return fail(ATTN_ERR_INVALID_ARG, "page_size must be at least 1, not %d", page_size);
    if ((long long)page_size * max_pages > 0x7fffffffLL)
        return fail(ATTN_ERR_INVALID_ARG, "max_pages * page_size exceeds 2^31-1");
    if (q_heads <= 0 || kv_heads <= 0 || head_dim <= 0)
        return fail(ATTN_ERR_INVALID_ARG, "q_heads, kv_heads and head_dim must be positive (%d, %d, %d)", q_heads,
                    kv_heads, head_dim);
    if (q_heads % kv_heads != 0)
        return fail(ATTN_ERR_INVALID_ARG, "q_heads (%d) is not a multiple of kv_heads (%d)", q_heads, kv_heads);
    if (sliding_window < 0) return fail(ATTN_ERR_INVALID_ARG, "negative sliding_window %d", sliding_window);
    if (!isfinite(scale)) return fail(ATTN_ERR_INVALID_ARG, "scale is not finite");
    if (dtype != ATTN_BF16 && dtype != ATTN_F16)
        return fail(ATTN_ERR_UNSUPPORTED, "paged caches support bf16 and fp16 only");
    if (head_dim != 64 && head_dim != 128)
        return fail(ATTN_ERR_UNSUPPORTED, "bf16 and fp16 support head_dim 64 and 128, not %d", head_dim);
    const int G = q_heads / kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8)
        return fail(ATTN_ERR_UNSUPPORTED, "paged caches support 1, 2, 4 or 8 query heads per kv head, not %d", G);
    if (m > 65535 || kv_heads > 65535) return fail(ATTN_ERR_UNSUPPORTED, "m and kv_heads are limited to 65535");
    if (m == 0) return ATTN_OK;
    if (!q || !out || !kv_lens) return fail(ATTN_ERR_INVALID_ARG, "null q, out or kv_lens pointer");
    cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
    if ((long long)page_size * max_pages == 0) {
        cudaError_t e = cudaMemsetAsync(out, 0, (size_t)m * q_heads * head_dim * 2, stream);
        if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "cudaMemsetAsync: %s", cudaGetErrorString(e));
        return ATTN_OK;
    }
    if (!k_pool || !v_pool || !page_table) return fail(ATTN_ERR_INVALID_ARG, "null k_pool, v_pool or page_table pointer");
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) ||
        !aligned(page_table, 4) || !aligned(kv_lens, 4))
        return fail(ATTN_ERR_INVALID_ARG, "q, out and the pools must be 16-byte, page_table and kv_lens 4-byte aligned");
    DeviceState* st = nullptr;
    attn_status s = device_state(&st);
    if (s != ATTN_OK) return s;
    attn::WaitCtl wc{st->status, kWaitLimitNs};
    attn::PagedProblem p{q, k_pool, v_pool, page_table, out, m, q_heads, kv_heads, num_pages, page_size,
                         max_pages, head_dim, kv_lens, sliding_window, scale, dtype == ATTN_F16};
    // Measured on GB300 (64 items, 8 kv heads, 8192 positions, head_dim 128), GB/s of the tensor-core
    // decode (TMA per page where it can, rows gathered otherwise) against the CUDA-core decode
    // (bulk copy per page piece): page 16: 4184 / 5103 (4 query heads per kv head), 4094 / 2413
    // (8); page 32: 5299 / 5124, 5171 / 2421; page 128: 6176 / 5138, 6012 / 2428; page 7:
    // 2043 / 4637, 2001 / 2390; page 1: 1798 / 1556, 1765 / 995.
    const bool tma_pages = attn::decode_tc_paged_tma(page_size, num_pages, kv_heads);
    const bool tc = attn::decode_tc_items_supported(q_heads, kv_heads, head_dim) &&
                    (G == 4 ? (tma_pages && page_size >= 32) : (tma_pages || page_size < 4));
    cudaError_t e = tc ? attn::launch_decode_tc_paged(p, wc, stream, st->num_sms)
                       : attn::launch_decode_paged(p, wc, stream, st->num_sms);
    if (e != cudaSuccess)
        return fail(ATTN_ERR_CUDA, "%s launch: %s", tc ? "decode_tc (paged)" : "decode_paged", cudaGetErrorString(e));
    return ATTN_OK;
}

attn_status attn_qkv_prelude(const void* qkv, const float* q_norm_w, const float* k_norm_w, const float* cos,
                             const float* sin, int rope_positions, void* q_out, void* k_out, void* v_out, int tokens,
                             int q_heads, int kv_heads, int head_dim, int pos_offset, float eps, int qk_mode,
                             int cache_len, int cache_capacity, int dtype, void* cuda_stream) {
    t_last_error.clear();
    if (tokens < 0 || pos_offset < 0 || cache_len < 0 || cache_capacity < 0 || rope_positions < 0)
        return fail(ATTN_ERR_INVALID_ARG, "negative size or offset (tokens=%d, pos_offset=%d, cache_len=%d, "
                    "cache_capacity=%d, rope_positions=%d)", tokens, pos_offset, cache_len, cache_capacity,
                    rope_positions);
    if (q_heads <= 0 || kv_heads <= 0 || head_dim <= 0)
        return fail(ATTN_ERR_INVALID_ARG, "q_heads, kv_heads and head_dim must be positive (%d, %d, %d)", q_heads,
                    kv_heads, head_dim);
    if (qk_mode < 0 || qk_mode > 3) return fail(ATTN_ERR_INVALID_ARG, "qk_mode %d out of range", qk_mode);
    if (dtype != ATTN_BF16 && dtype != ATTN_F32 && dtype != ATTN_F16)
        return fail(ATTN_ERR_INVALID_ARG, "dtype %d out of range", dtype);
    if (dtype == ATTN_F32) return fail(ATTN_ERR_UNSUPPORTED, "the prelude supports bf16 and fp16");
    if (head_dim != 64 && head_dim != 128)
        return fail(ATTN_ERR_UNSUPPORTED, "the prelude supports head_dim 64 and 128, not %d", head_dim);
    if (qk_mode == 1 && (!isfinite(eps) || eps < 0.f))
        return fail(ATTN_ERR_INVALID_ARG, "eps must be finite and >= 0");
    if (cache_capacity > 0 && (long long)cache_len + tokens > cache_capacity)
        return fail(ATTN_ERR_INVALID_ARG, "cache_len %d + tokens %d exceeds cache_capacity %d", cache_len, tokens,
                    cache_capacity);
    if (qk_mode != 0 && (long long)pos_offset + tokens > rope_positions)
        return fail(ATTN_ERR_INVALID_ARG, "positions up to %lld exceed the %d rows of the cos/sin tables",
                    (long long)pos_offset + tokens, rope_positions);
    if (tokens == 0) return ATTN_OK;
    if (!qkv || !q_out || !k_out || !v_out) return fail(ATTN_ERR_INVALID_ARG, "null qkv, q_out, k_out or v_out");
    if (!aligned(qkv, 16) || !aligned(q_out, 16) || !aligned(k_out, 16) || !aligned(v_out, 16))
        return fail(ATTN_ERR_INVALID_ARG, "qkv, q_out, k_out and v_out must be 16-byte aligned");
    if (qk_mode != 0 && (!cos || !sin || !aligned(cos, 16) || !aligned(sin, 16)))
        return fail(ATTN_ERR_INVALID_ARG, "cos and sin must be non-null and 16-byte aligned");
    if (qk_mode == 1 && (!q_norm_w || !k_norm_w || !aligned(q_norm_w, 4) || !aligned(k_norm_w, 4)))
        return fail(ATTN_ERR_INVALID_ARG, "q_norm_w and k_norm_w must be non-null and 4-byte aligned");
    DeviceState* st = nullptr;
    attn_status s = device_state(&st);
    if (s != ATTN_OK) return s;
    attn::WaitCtl wc{st->status, kWaitLimitNs};
    attn::PreludeProblem p{qkv, q_norm_w, k_norm_w, cos, sin, q_out, k_out, v_out, tokens, q_heads, kv_heads,
                           head_dim, pos_offset, qk_mode, cache_len, cache_capacity, eps, dtype == ATTN_F16,
                           rope_positions, nullptr, nullptr, nullptr};
    cudaError_t e = attn::launch_prelude(p, wc, static_cast<cudaStream_t>(cuda_stream));
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "prelude launch: %s", cudaGetErrorString(e));
    return ATTN_OK;
}

attn_status attn_qkv_prelude_caches(const void* qkv, const float* q_norm_w, const float* k_norm_w, const float* cos,
                                    const float* sin, int rope_positions, void* q_out, const void* const* k_caches,
                                    const void* const* v_caches, const int32_t* cache_lens, int m, int q_heads,
                                    int kv_heads, int head_dim, int capacity, float eps, int qk_mode, int dtype,
                                    void* cuda_stream) {
    t_last_error.clear();
    if (m < 0 || capacity < 0 || rope_positions < 0)
        return fail(ATTN_ERR_INVALID_ARG, "negative size (m=%d, capacity=%d, rope_positions=%d)", m, capacity,
                    rope_positions);
    if (q_heads <= 0 || kv_heads <= 0 || head_dim <= 0)
        return fail(ATTN_ERR_INVALID_ARG, "q_heads, kv_heads and head_dim must be positive (%d, %d, %d)", q_heads,
                    kv_heads, head_dim);
    if (qk_mode < 0 || qk_mode > 3) return fail(ATTN_ERR_INVALID_ARG, "qk_mode %d out of range", qk_mode);
    if (dtype != ATTN_BF16 && dtype != ATTN_F32 && dtype != ATTN_F16)
        return fail(ATTN_ERR_INVALID_ARG, "dtype %d out of range", dtype);
    if (dtype == ATTN_F32) return fail(ATTN_ERR_UNSUPPORTED, "the prelude supports bf16 and fp16");
    if (head_dim != 64 && head_dim != 128)
        return fail(ATTN_ERR_UNSUPPORTED, "the prelude supports head_dim 64 and 128, not %d", head_dim);
    if (qk_mode == 1 && (!isfinite(eps) || eps < 0.f))
        return fail(ATTN_ERR_INVALID_ARG, "eps must be finite and >= 0");
    if (m == 0) return ATTN_OK;
    if (capacity == 0) return fail(ATTN_ERR_INVALID_ARG, "capacity must be positive to append a row");
    if (!qkv || !q_out || !k_caches || !v_caches || !cache_lens)
        return fail(ATTN_ERR_INVALID_ARG, "null qkv, q_out, k_caches, v_caches or cache_lens");
    if (!aligned(qkv, 16) || !aligned(q_out, 16) || !aligned(k_caches, 8) || !aligned(v_caches, 8) ||
        !aligned(cache_lens, 4))
        return fail(ATTN_ERR_INVALID_ARG, "qkv/q_out must be 16-byte, pointer arrays 8-byte, cache_lens 4-byte aligned");
    if (qk_mode != 0 && (!cos || !sin || !aligned(cos, 16) || !aligned(sin, 16)))
        return fail(ATTN_ERR_INVALID_ARG, "cos and sin must be non-null and 16-byte aligned");
    if (qk_mode == 1 && (!q_norm_w || !k_norm_w || !aligned(q_norm_w, 4) || !aligned(k_norm_w, 4)))
        return fail(ATTN_ERR_INVALID_ARG, "q_norm_w and k_norm_w must be non-null and 4-byte aligned");
    DeviceState* st = nullptr;
    attn_status s = device_state(&st);
    if (s != ATTN_OK) return s;
    attn::WaitCtl wc{st->status, kWaitLimitNs};
    attn::PreludeProblem p{qkv, q_norm_w, k_norm_w, cos, sin, q_out, nullptr, nullptr, m, q_heads, kv_heads,
                           head_dim, 0, qk_mode, 0, capacity, eps, dtype == ATTN_F16, rope_positions,
                           k_caches, v_caches, cache_lens};
    cudaError_t e = attn::launch_prelude(p, wc, static_cast<cudaStream_t>(cuda_stream));
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "prelude launch: %s", cudaGetErrorString(e));
    return ATTN_OK;
}

const char* attn_last_error(void) { return t_last_error.c_str(); }

attn_status attn_sync_status(void* cuda_stream) {
    t_last_error.clear();
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream));
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "stream: %s", cudaGetErrorString(e));
    DeviceState* st = nullptr;
    attn_status s = device_state(&st);
    if (s != ATTN_OK) return s;
    unsigned word = 0;
    e = cudaMemcpy(&word, st->status, sizeof word, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "reading the status word: %s", cudaGetErrorString(e));
    if (word != 0) {
        const unsigned zero = 0;
        e = cudaMemcpy(st->status, &zero, sizeof zero, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "clearing the status word: %s", cudaGetErrorString(e));
        if (word == attn::kStatusTimeout) return fail(ATTN_ERR_TIMEOUT, "a device-side wait timed out");
        if (word == attn::kStatusBadPointer)
            return fail(ATTN_ERR_INVALID_ARG, "a per-item cache pointer is null or not 16-byte aligned");
        if (word == attn::kStatusBadPage)
            return fail(ATTN_ERR_INVALID_ARG, "a page-table entry names no page of the pool");
        if (word == attn::kStatusBadSeqlens)
            return fail(ATTN_ERR_INVALID_ARG,
                        "a device-side length is out of range: cu_seqlens not non-decreasing within total and "
                        "max_seqlen, a cache length outside the capacity or the rope tables, or fewer cached "
                        "positions than queries");
        return fail(ATTN_ERR_CUDA, "device status word %u", word);
    }
    return ATTN_OK;
}

attn_status attn_selftest_timeout(int limit_us, void* cuda_stream) {
    t_last_error.clear();
    if (limit_us < 1 || limit_us > 1000000)
        return fail(ATTN_ERR_INVALID_ARG, "limit_us %d outside [1, 1000000]", limit_us);
    DeviceState* st = nullptr;
    attn_status s = device_state(&st);
    if (s != ATTN_OK) return s;
    attn::WaitCtl wc{st->status, (unsigned long long)limit_us * 1000ull};
    cudaError_t e = attn::launch_timeout_selftest(wc, static_cast<cudaStream_t>(cuda_stream));
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "selftest launch: %s", cudaGetErrorString(e));
    return ATTN_OK;
}

int attn_version(void) { return 100; }

}  // extern "C"
