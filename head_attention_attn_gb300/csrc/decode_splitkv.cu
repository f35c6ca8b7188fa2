// decode_splitkv.cu -- K2: single-query (q_len == 1) attention against a KV cache, bf16 or fp16,
// head_dim 64 or 128, bound by HBM bandwidth.
//
// Work unit: (batch b, kv head hk).  Its G = q_heads/kv_heads query heads are
// served together, so every K and V byte is read from HBM once.  The visible key
// range of a decode query is one interval [lo, hi) (causal at pos_offset,
// windows, key padding); a cluster of S CTAs splits it into S contiguous chunks.
//
// Inside a CTA one producer lane streams the CTA's keys in chunks of 32 rows of K
// and of V with bulk asynchronous copies (cp.async.bulk, completing on an mbarrier)
// into a 4-stage shared-memory ring of 48-key stages, so about 100 KB per CTA is in
// flight; six compute warps take 8 keys each of every chunk:
//   - a key row (head_dim 16-bit values) is spread over D/8 lanes, 16 bytes per lane, read
//     from shared memory with 128-bit loads, 2 (D=128) or 4 (D=64) rows per
//     instruction;
//   - q (pre-scaled by scale*log2(e)) lives in registers; the per-lane partial
//     dot products of all (head, key) pairs are summed across the lanes of a
//     row with a shuffle reduce-scatter (each level halves the values a lane
//     keeps), so every lane ends with complete scores for a few pairs;
//   - a lane-group running max and sum per head (base-2 exponent, O rescaled
//     only when the max grows by more than 2^8) and fp32 accumulators of P V
//     for the lane's 8 head dims, with packed f32x2 FMAs.
// Combine: the lane groups of a warp merge with shuffles, the 6 warps merge
// through shared memory, and the S CTAs of the cluster merge through
// distributed shared memory in CTA rank 0, which normalises and stores the input type.
// No global scratch memory is used.
//
// The operation is the q_len = 1 case of ferrum-kernels Backend::flash_attention
// and the per-cache decode of Backend::flash_attention_batched_per_cache (one
// launch for all items, device-side lengths, sliding window = last w positions).
#include "kernels.h"

#include <algorithm>
#include <mutex>

namespace attn {
namespace {

constexpr int kWarps = 6;                  // compute warps
constexpr int kThreads = (kWarps + 1) * 32;  // + one producer warp
constexpr int kMaxSplits = 8;              // portable cluster size
constexpr int kChunk = 8 * kWarps;         // keys per pipeline stage (8 per compute warp)
constexpr int kStages = 4;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;

struct DecodeParams {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;           // contiguous caches [B, Hkv, Lk, D] (k/v), or
    const __nv_bfloat16* v;
    const __nv_bfloat16* const* kc;   // per-item caches: device arrays of B pointers, each
    const __nv_bfloat16* const* vc;   // [Hkv, Lk, D] with Lk the capacity (null: contiguous)
    __nv_bfloat16* out;
    const int32_t* key_lens;          // per-item valid lengths (required with per-item caches)
    int Hq, Hkv, Lk, P, mode, window;
    int sliding;                      // per-item caches: attend to the last `sliding` keys (0: all)
    float scale_log2;
    WaitCtl wc;
    // Paged caches (null: not paged): k/v are pools [num_pages, Hkv, page_size, D]; item b's
    // position j lives in pool page page_table[b * max_pages + j / page_size], row j % page_size.
    const int32_t* page_table = nullptr;
    int page_size = 0, max_pages = 0, num_pages = 0;
};

template <int D, int G>
struct DCfg {
    static constexpr int LPK = D / 8;              // lanes per key row (16 bytes each)
    static constexpr int KPP = 32 / LPK;           // key rows per warp load instruction
    static constexpr int NP = kChunk / kWarps / KPP;  // passes per warp batch
    static constexpr int KB = NP * KPP;            // keys per warp batch (8)
    static constexpr int NV = NP * G;              // partial dot products per lane per batch
    static constexpr int LEVELS = (LPK == 16) ? 4 : 3;
    static constexpr int kRowBytes = D * 2;
    static constexpr int kStageBytes = 2 * kChunk * kRowBytes;  // K rows then V rows
    static constexpr int kSmem = kStages * kStageBytes + 1024;  // ring + 1 KB alignment slack
};

// 8 bf16 or fp16 values (16 bytes) -> 4 float2 pairs (element 2i in .x, 2i+1 in .y).
template <bool F16>
__device__ __forceinline__ void elem8_to_f2(const uint4& u, float2 (&f)[4]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) f[i] = unpack2<F16>(w[i]);
}

__device__ __forceinline__ float safe_ex2_diff(float a, float m) {
    // 2^(a - m) with -inf handling: a == -inf -> 0; m == -inf (nothing seen) -> 0.
    return (m == -INFINITY) ? 0.f : ex2_approx(a - m);
}

// Bulk copy of `bytes` contiguous bytes global -> shared, completing on an mbarrier.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(addr));
    return r;
}

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, const WaitCtl& wc) {
    const unsigned long long t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > wc.limit_ns) {
            record_status(wc.status, kStatusTimeout);
            return;
        }
    }
}

// Two CTAs per SM, except with 8 query heads per kv head: their accumulators need more
// registers than two CTAs leave (the two-CTA build spills about 600 bytes per thread), and
// one CTA per SM without spills measured twice as fast.
template <int D, int G, bool F16>
__global__ void __launch_bounds__(kThreads, (G == 8) ? 1 : 2) decode_splitkv_kernel(const DecodeParams p) {
    using C = DCfg<D, G>;
    constexpr int LPK = C::LPK, KPP = C::KPP, NP = C::NP, KB = C::KB, NV = C::NV;
    static_assert(KB * kWarps == kChunk, "a chunk is split evenly over the compute warps");

    extern __shared__ uint8_t dsmem[];
    __shared__ __align__(8) uint64_t s_full[kStages], s_empty[kStages];
    __shared__ int s_abort;
    __shared__ __align__(16) float s_p[kWarps][KPP][NP][G];  // probabilities of the current batch, [pass][head]
    __shared__ float s_wm[kWarps][G], s_wl[kWarps][G];
    __shared__ __align__(16) float s_wacc[kWarps][G][D];
    __shared__ float s_cm[G], s_cl[G];
    __shared__ __align__(16) float s_cacc[G][D];

    const uint32_t raw = smem_u32(dsmem);
    const uint32_t ring = raw + ((1024u - (raw & 1023u)) & 1023u);
    volatile int* abort_flag = &s_abort;

    const int split = blockIdx.x;          // == rank in the cluster
    const int nsplit = gridDim.x;
    const int hk = blockIdx.y;
    const int b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // Visible interval of the single query, split over the cluster in whole chunks.
    // Contiguous caches: the query sits at position P and the mask mode applies.
    // Per-item caches: the query is the newest of the item's kv_lens[b] positions and
    // sees them all, or the last `sliding` of them.
    const int klen = valid_keys(p.key_lens, b, p.Lk);
    long long lo, hi;
    const __nv_bfloat16* kbase;
    const __nv_bfloat16* vbase;
    const int32_t* pages = nullptr;  // paged: this item's row of the page table
    if (p.page_table != nullptr) {
        // Paged caches: like per-item caches, with the item's positions spread over pool
        // pages.  Every CTA of the cluster checks all of the item's visible pages, so they
        // agree: an item with an entry outside the pool is not read and gets zeros.
        pages = p.page_table + (size_t)b * p.max_pages;
        lo = (p.sliding > 0 && klen > p.sliding) ? (long long)(klen - p.sliding) : 0;
        hi = klen;
        bool bad = false;
        if (hi > lo) {
            for (long long x = lo / p.page_size + threadIdx.x; x <= (hi - 1) / p.page_size; x += blockDim.x) {
                const int id = __ldg(pages + x);
                bad |= (id < 0 || id >= p.num_pages);
            }
        }
        if (__syncthreads_or(bad)) {
            if (threadIdx.x == 0) record_status(p.wc.status, kStatusBadPage);
            lo = hi = 0;
        }
        kbase = p.k;  // pool bases: a chunk's rows are addressed page by page
        vbase = p.v;
    } else if (p.kc != nullptr) {
        kbase = p.kc[b];
        vbase = p.vc[b];
        lo = (p.sliding > 0 && klen > p.sliding) ? (long long)(klen - p.sliding) : 0;
        hi = klen;
        const bool bad = kbase == nullptr || vbase == nullptr ||
                         ((reinterpret_cast<uintptr_t>(kbase) | reinterpret_cast<uintptr_t>(vbase)) & 15u) != 0;
        if (bad) {
            if (threadIdx.x == 0) record_status(p.wc.status, kStatusBadPointer);
            lo = hi = 0;  // nothing is read; the item's output is written as zeros
        }
        kbase += (size_t)hk * (size_t)p.Lk * D;
        vbase += (size_t)hk * (size_t)p.Lk * D;
    } else {
        key_interval(p.mode, p.window, klen, p.P, p.P, &lo, &hi);
        const size_t head_off = ((size_t)b * p.Hkv + hk) * (size_t)p.Lk * D;
        kbase = p.k + head_off;
        vbase = p.v + head_off;
    }
    if (hi < lo) hi = lo;
    const long long span = hi - lo;
    long long per = (span + nsplit - 1) / nsplit;
    per = (per + kChunk - 1) / kChunk * kChunk;
    const long long kbeg = lo + (long long)split * per;
    const long long kend = min(hi, kbeg + per);
    const int nchunks = (kend > kbeg) ? (int)((kend - kbeg + kChunk - 1) / kChunk) : 0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(smem_u32(&s_full[i]), 1);
            mbar_init(smem_u32(&s_empty[i]), kWarps);
        }
        s_abort = 0;
        mbar_fence_init();
    }
    __syncthreads();

    float m_run[G], l_run[G];
    float2 acc[G][4];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        m_run[g] = -INFINITY;
        l_run[g] = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[g][i] = make_float2(0.f, 0.f);
    }

    if (warp == kWarps) {
        // ------------------------------------------------------------ producer
        // Lane 0 copies a contiguous chunk; over paged caches every lane loads the page ids of
        // its own page pieces of the chunk and issues their copies, so the page-table reads and
        // the copies of one chunk proceed in parallel.
        int issued = 0;  // kept by lane 0
        for (int c = 0; c < nchunks; ++c) {
            const int st = c % kStages;
            if (c >= kStages &&
                !__all_sync(0xffffffffu, mbar_wait(smem_u32(&s_empty[st]), (uint32_t)(c / kStages - 1) & 1, p.wc,
                                                   abort_flag)))
                break;
            const long long k0 = kbeg + (long long)c * kChunk;
            const int rows = (int)min((long long)kChunk, kend - k0);
            const uint32_t bytes = (uint32_t)rows * C::kRowBytes;
            const uint32_t dst = ring + st * C::kStageBytes;
            const uint32_t bar = smem_u32(&s_full[st]);
            if (lane == 0) mbar_arrive_expect_tx(bar, 2 * bytes);
            __syncwarp();
            if (pages != nullptr) {
                // the chunk's rows may span pages: one copy per page piece, same bytes in total
                const long long pg0 = k0 / p.page_size;
                const int npieces = (int)((k0 + rows - 1) / p.page_size - pg0 + 1);
                for (int i = lane; i < npieces; i += 32) {
                    const long long pg = pg0 + i;
                    const long long a = max(k0, pg * p.page_size), e = min(k0 + rows, (pg + 1) * p.page_size);
                    const size_t src = (((size_t)__ldg(pages + pg) * p.Hkv + hk) * p.page_size +
                                        (size_t)(a - pg * p.page_size)) * D;
                    const uint32_t off = (uint32_t)(a - k0) * C::kRowBytes, nb = (uint32_t)(e - a) * C::kRowBytes;
                    bulk_load(dst + off, kbase + src, nb, bar);
                    bulk_load(dst + kChunk * C::kRowBytes + off, vbase + src, nb, bar);
                }
            } else if (lane == 0) {
                bulk_load(dst, kbase + k0 * D, bytes, bar);
                bulk_load(dst + kChunk * C::kRowBytes, vbase + k0 * D, bytes, bar);
            }
            issued = c + 1;
        }
        // no copy may still be writing shared memory when the block moves on
        if (lane == 0)
            for (int c = (issued > kStages ? issued - kStages : 0); c < issued; ++c)
                drain_wait(smem_u32(&s_full[c % kStages]), (uint32_t)(c / kStages) & 1, p.wc);
    } else {
        // ------------------------------------------------------------ compute warps
        const int grp = lane / LPK;            // which key row of a load instruction this lane reads
        const int gl = lane % LPK;             // position inside the row: dims [8*gl, 8*gl+8)

        // q of the G heads, my 8 dims, pre-scaled by scale*log2(e).
        float2 qf[G][4];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const __nv_bfloat16* qp = p.q + ((size_t)b * p.Hq + (size_t)hk * G + g) * D + 8 * gl;
            const uint4 u = *reinterpret_cast<const uint4*>(qp);
            elem8_to_f2<F16>(u, qf[g]);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                qf[g][i].x *= p.scale_log2;
                qf[g][i].y *= p.scale_log2;
            }
        }

        // Value index layout of a batch: i = g * NP + pass.  The reduce-scatter
        // halves on the high index bit first (head bits, then pass bits), so after
        // RS levels a lane keeps KEEP consecutive passes of a single head.  Levels
        // beyond RS (when NV < LPK) become all-reduce levels and leave identical
        // copies in the lanes that differ only in those bits.
        constexpr int LOG_NV = (NV >= 32) ? 5 : (NV >= 16) ? 4 : (NV >= 8) ? 3 : (NV >= 4) ? 2 : 1;
        constexpr int RS = (LOG_NV < C::LEVELS) ? LOG_NV : C::LEVELS;
        constexpr int KEEP = NV >> RS;
        constexpr int HEAD_LEVELS = (G >= 8) ? 3 : (G >= 4) ? 2 : (G >= 2) ? 1 : 0;
        static_assert(KEEP >= 1 && NP % KEEP == 0, "values of a lane stay within one head");
        static_assert(HEAD_LEVELS <= RS, "head bits are spread by reduce-scatter levels");

        // Lanes that differ only in all-reduce bits hold copies of the same values; one
        // of them (all-reduce bits zero) owns the row sums of its head.
        int ar_mask = 0;
#pragma unroll
        for (int lev = RS; lev < C::LEVELS; ++lev) ar_mask |= LPK >> (lev + 1);
        const bool owner = (gl & ar_mask) == 0;
        float l_own = 0.f;
        int gh_lane = 0;

        for (int c = 0; c < nchunks; ++c) {
            const int st = c % kStages;
            if (!mbar_wait(smem_u32(&s_full[st]), (uint32_t)(c / kStages) & 1, p.wc, abort_flag)) break;
            const long long kb = kbeg + (long long)c * kChunk + warp * KB;   // this warp's 8 keys
            const uint32_t kst = ring + st * C::kStageBytes + (warp * KB) * C::kRowBytes + 16 * gl;
            const uint32_t vst = kst + kChunk * C::kRowBytes;

            // ---- partial dots over my 8 dims (rows past the range are not read)
            float val[NV];
#pragma unroll
            for (int ps = 0; ps < NP; ++ps) {
                const int r = ps * KPP + grp;
                const bool valid = kb + r < kend;
                const uint4 u = valid ? lds128(kst + r * C::kRowBytes) : make_uint4(0, 0, 0, 0);
                float2 kf[4];
                elem8_to_f2<F16>(u, kf);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float2 t = __fmul2_rn(qf[g][0], kf[0]);
                    t = __ffma2_rn(qf[g][1], kf[1], t);
                    t = __ffma2_rn(qf[g][2], kf[2], t);
                    t = __ffma2_rn(qf[g][3], kf[3], t);
                    val[g * NP + ps] = t.x + t.y;
                }
            }
            // ---- reduce-scatter, then all-reduce, over the LPK lanes of the row
            int base = 0;
#pragma unroll
            for (int lev = 0; lev < RS; ++lev) {
                const int mask = LPK >> (lev + 1);
                const int half = NV >> (lev + 1);
                const bool upper = (gl & mask) != 0;
#pragma unroll
                for (int t = 0; t < half; ++t) {
                    const float send = upper ? val[t] : val[t + half];
                    const float keep = upper ? val[t + half] : val[t];
                    val[t] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
                }
                if (upper) base += half;
            }
#pragma unroll
            for (int lev = RS; lev < C::LEVELS; ++lev) {
                const int mask = LPK >> (lev + 1);
#pragma unroll
                for (int t = 0; t < KEEP; ++t) val[t] += __shfl_xor_sync(0xffffffffu, val[t], mask);
            }
            // ---- this lane's values: head gh, passes p0 .. p0+KEEP-1; mask keys past the range
            const int gh = base / NP;
            const int p0 = base % NP;
            gh_lane = gh;
            float bm = -INFINITY;
#pragma unroll
            for (int t = 0; t < KEEP; ++t) {
                if (kb + (p0 + t) * KPP + grp >= kend) val[t] = -INFINITY;
                bm = fmaxf(bm, val[t]);
            }
#pragma unroll
            for (int lev = HEAD_LEVELS; lev < RS; ++lev)
                bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, LPK >> (lev + 1)));
            float alpha[G];
            bool any_rescale = false;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                int src_gl = 0;  // a lane whose head bits spell g
#pragma unroll
                for (int lev = 0; lev < HEAD_LEVELS; ++lev)
                    if ((g >> (HEAD_LEVELS - 1 - lev)) & 1) src_gl |= LPK >> (lev + 1);
                const float bmg = (G > 1) ? __shfl_sync(0xffffffffu, bm, grp * LPK + src_gl) : bm;
                alpha[g] = 1.f;
                if (bmg != -INFINITY) {
                    if (m_run[g] == -INFINITY) {
                        m_run[g] = bmg;
                    } else if (bmg > m_run[g] + kRescaleThreshold) {
                        alpha[g] = ex2_approx(m_run[g] - bmg);
                        m_run[g] = bmg;
                        any_rescale = true;
                    }
                }
            }
            {
                float mh = m_run[0], ah = alpha[0];
#pragma unroll
                for (int g = 1; g < G; ++g) {
                    mh = (gh == g) ? m_run[g] : mh;
                    ah = (gh == g) ? alpha[g] : ah;
                }
                float ps_sum = 0.f;
#pragma unroll
                for (int t = 0; t < KEEP; ++t) {
                    const float pt = safe_ex2_diff(val[t], mh);
                    s_p[warp][grp][p0 + t][gh] = pt;
                    ps_sum += pt;
                }
                // the lane owning these probabilities (not an all-reduce copy) keeps their sum
                l_own = l_own * ah + (owner ? ps_sum : 0.f);
            }
            __syncwarp();
            if (any_rescale) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float2 a2 = make_float2(alpha[g], alpha[g]);
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[g][i] = __fmul2_rn(acc[g][i], a2);
                }
            }
            // ---- accumulate P V for my 8 dims (value rows past the range read as zeros)
#pragma unroll
            for (int ps = 0; ps < NP; ++ps) {
                const int r = ps * KPP + grp;
                const uint4 u = (kb + r < kend) ? lds128(vst + r * C::kRowBytes) : make_uint4(0, 0, 0, 0);
                float2 vf[4];
                elem8_to_f2<F16>(u, vf);
                float pv[G];
                if constexpr (G % 4 == 0) {
#pragma unroll
                    for (int g = 0; g < G; g += 4) {
                        const float4 p4 = *reinterpret_cast<const float4*>(&s_p[warp][grp][ps][g]);
                        pv[g] = p4.x;
                        pv[g + 1] = p4.y;
                        pv[g + 2] = p4.z;
                        pv[g + 3] = p4.w;
                    }
                } else {
#pragma unroll
                    for (int g = 0; g < G; ++g) pv[g] = s_p[warp][grp][ps][g];
                }
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float2 p2 = make_float2(pv[g], pv[g]);
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[g][i] = __ffma2_rn(p2, vf[i], acc[g][i]);
                }
            }
            __syncwarp();  // s_p is rewritten by the next batch; the stage may be refilled
            if (lane == 0) mbar_arrive(smem_u32(&s_empty[st]));
        }

        // ---------------------------------------------------------------- combine
        // (0) row sums: add the owners' partial sums over the pass-bit and all-reduce
        // lanes of each head, then every lane gathers the sum of every head
        {
            float lsum = l_own;
#pragma unroll
            for (int lev = HEAD_LEVELS; lev < C::LEVELS; ++lev)
                lsum += __shfl_xor_sync(0xffffffffu, lsum, LPK >> (lev + 1));
#pragma unroll
            for (int g = 0; g < G; ++g) {
                int src_gl = 0;
#pragma unroll
                for (int lev = 0; lev < HEAD_LEVELS; ++lev)
                    if ((g >> (HEAD_LEVELS - 1 - lev)) & 1) src_gl |= LPK >> (lev + 1);
                l_run[g] = (G > 1) ? __shfl_sync(0xffffffffu, lsum, grp * LPK + src_gl) : lsum;
            }
            (void)gh_lane;
        }
        // (1) the KPP row groups of the warp (same dims, different keys)
#pragma unroll
        for (int off = LPK; off < 32; off <<= 1) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float mo = __shfl_xor_sync(0xffffffffu, m_run[g], off);
                const float lo_ = __shfl_xor_sync(0xffffffffu, l_run[g], off);
                const float mc = fmaxf(m_run[g], mo);
                const float fa = safe_ex2_diff(m_run[g], mc);
                const float fb = safe_ex2_diff(mo, mc);
                l_run[g] = l_run[g] * fa + lo_ * fb;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float2 other;
                    other.x = __shfl_xor_sync(0xffffffffu, acc[g][i].x, off);
                    other.y = __shfl_xor_sync(0xffffffffu, acc[g][i].y, off);
                    acc[g][i].x = acc[g][i].x * fa + other.x * fb;
                    acc[g][i].y = acc[g][i].y * fa + other.y * fb;
                }
                m_run[g] = mc;
            }
        }
        // (2) the warps of the CTA, through shared memory
        if (lane < LPK) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    *reinterpret_cast<float2*>(&s_wacc[warp][g][8 * gl + 2 * i]) = acc[g][i];
                if (lane == 0) {
                    s_wm[warp][g] = m_run[g];
                    s_wl[warp][g] = l_run[g];
                }
            }
        }
    }
    __syncthreads();
    for (int t = threadIdx.x; t < G * D; t += kThreads) {
        const int g = t / D, d = t % D;
        float mc = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) mc = fmaxf(mc, s_wm[w][g]);
        float o = 0.f, l = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float f = safe_ex2_diff(s_wm[w][g], mc);
            o += f * s_wacc[w][g][d];
            l += f * s_wl[w][g];
        }
        s_cacc[g][d] = o;
        if (d == 0) {
            s_cm[g] = mc;
            s_cl[g] = l;
        }
    }
    // (3) the CTAs of the cluster, through distributed shared memory, in rank 0
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    if (split == 0) {
        for (int t = threadIdx.x; t < G * D; t += kThreads) {
            const int g = t / D, d = t % D;
            float ms[kMaxSplits], ls[kMaxSplits], os[kMaxSplits];
            float mc = -INFINITY;
            for (int r = 0; r < nsplit; ++r) {
                uint32_t a_m, a_l, a_o;
                asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a_m) : "r"(smem_u32(&s_cm[g])), "r"(r));
                asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a_l) : "r"(smem_u32(&s_cl[g])), "r"(r));
                asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a_o) : "r"(smem_u32(&s_cacc[g][d])), "r"(r));
                asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(ms[r]) : "r"(a_m) : "memory");
                asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(ls[r]) : "r"(a_l) : "memory");
                asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(os[r]) : "r"(a_o) : "memory");
                mc = fmaxf(mc, ms[r]);
            }
            float o = 0.f, l = 0.f;
            for (int r = 0; r < nsplit; ++r) {
                const float f = safe_ex2_diff(ms[r], mc);
                o += f * os[r];
                l += f * ls[r];
            }
            const float res = (l > 0.f) ? o / l : 0.f;
            const size_t oi = ((size_t)b * p.Hq + (size_t)hk * G + g) * D + d;
            if constexpr (F16) reinterpret_cast<__half*>(p.out)[oi] = __float2half_rn(res);
            else p.out[oi] = __float2bfloat16_rn(res);
        }
    }
    // keep every CTA's shared memory alive until rank 0 has read it
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <int D, int G, bool F16>
cudaError_t launch_dg(const DecodeParams& p, int B, int nsplit, cudaStream_t stream) {
    using C = DCfg<D, G>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::mutex mu;
    static bool configured[64] = {};
    {
        std::lock_guard<std::mutex> g(mu);
        if (dev < 64 && !configured[dev]) {
            e = cudaFuncSetAttribute(decode_splitkv_kernel<D, G, F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     C::kSmem);
            if (e != cudaSuccess) return e;
            configured[dev] = true;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)nsplit, (unsigned)p.Hkv, (unsigned)B);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)nsplit;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_splitkv_kernel<D, G, F16>, p);
}

template <int D, bool F16>
cudaError_t launch_dt(const DecodeParams& p, int G, int B, int nsplit, cudaStream_t s) {
    switch (G) {
        case 1: return launch_dg<D, 1, F16>(p, B, nsplit, s);
        case 2: return launch_dg<D, 2, F16>(p, B, nsplit, s);
        case 4: return launch_dg<D, 4, F16>(p, B, nsplit, s);
        case 8: return launch_dg<D, 8, F16>(p, B, nsplit, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_any(const DecodeParams& p, int D, bool f16, int G, int B, int nsplit, cudaStream_t s) {
    if (D == 64) return f16 ? launch_dt<64, true>(p, G, B, nsplit, s) : launch_dt<64, false>(p, G, B, nsplit, s);
    return f16 ? launch_dt<128, true>(p, G, B, nsplit, s) : launch_dt<128, false>(p, G, B, nsplit, s);
}

// Split count (cluster size) for `units` (item, kv head) pairs of up to `span` keys each.
// Measured on GB300 over batch 1-64, 512-32768 keys: fewer, longer CTAs win as long as
// there are about 256 of them (their pipeline fill and the cluster combine cost more than
// a partly filled last wave), a split should cover at least 1024 keys, and with 256 or
// more units two splits beat one.
int choose_splits(long long units, long long span, int num_sms) {
    const long long target = num_sms > 0 ? (27LL * num_sms) / 16 : 256;  // about 1.7 CTAs per SM (256 on 152 SMs)
    int n = 1;
    while (n < kMaxSplits && units * n < target) n *= 2;
    if (units >= 256) n = std::max(n, 2);
    const long long by_len = std::max(1LL, span / 1024);
    return (int)std::max(1LL, std::min<long long>(n, by_len));
}

}  // namespace

bool decode_supported(const Problem& p) {
    if (p.Lq != 1 || (p.D != 64 && p.D != 128)) return false;
    const int G = p.Hq / p.Hkv;
    return G == 1 || G == 2 || G == 4 || G == 8;
}

cudaError_t launch_decode_splitkv(const Problem& pr, const WaitCtl& wc, cudaStream_t stream, int num_sms) {
    DecodeParams p;
    p.q = reinterpret_cast<const __nv_bfloat16*>(pr.q);
    p.k = reinterpret_cast<const __nv_bfloat16*>(pr.k);
    p.v = reinterpret_cast<const __nv_bfloat16*>(pr.v);
    p.kc = nullptr;
    p.vc = nullptr;
    p.sliding = 0;
    p.out = reinterpret_cast<__nv_bfloat16*>(pr.out);
    p.key_lens = pr.key_lens;
    p.Hq = pr.Hq;
    p.Hkv = pr.Hkv;
    p.Lk = pr.Lk;
    p.P = pr.pos_offset;
    p.mode = pr.mode;
    p.window = pr.window;
    p.scale_log2 = pr.scale * kLog2e;
    p.wc = wc;
    if (pr.Hkv > 65535 || pr.B > 65535) return cudaErrorInvalidConfiguration;
    const int nsplit = choose_splits((long long)pr.B * pr.Hkv, pr.Lk, num_sms);
    const int G = pr.Hq / pr.Hkv;
    return launch_any(p, pr.D, pr.f16, G, pr.B, nsplit, stream);
}

cudaError_t launch_decode_paged(const PagedProblem& pp, const WaitCtl& wc, cudaStream_t stream, int num_sms) {
    DecodeParams p;
    p.q = reinterpret_cast<const __nv_bfloat16*>(pp.q);
    p.k = reinterpret_cast<const __nv_bfloat16*>(pp.k_pool);
    p.v = reinterpret_cast<const __nv_bfloat16*>(pp.v_pool);
    p.kc = nullptr;
    p.vc = nullptr;
    p.out = reinterpret_cast<__nv_bfloat16*>(pp.out);
    p.key_lens = pp.kv_lens;
    p.Hq = pp.Hq;
    p.Hkv = pp.Hkv;
    p.Lk = pp.page_size * pp.max_pages;  // the item's capacity: kv_lens clamp to it
    p.P = 0;
    p.mode = 0;
    p.window = 0;
    p.sliding = pp.sliding;
    p.scale_log2 = pp.scale * kLog2e;
    p.wc = wc;
    p.page_table = pp.page_table;
    p.page_size = pp.page_size;
    p.max_pages = pp.max_pages;
    p.num_pages = pp.num_pages;
    if (pp.Hkv > 65535 || pp.m > 65535) return cudaErrorInvalidConfiguration;
    const long long span = pp.sliding > 0 ? std::min(pp.sliding, p.Lk) : p.Lk;
    const int nsplit = choose_splits((long long)pp.m * pp.Hkv, span, num_sms);
    const int G = pp.Hq / pp.Hkv;
    return launch_any(p, pp.D, pp.f16, G, pp.m, nsplit, stream);
}

cudaError_t launch_decode_caches(const CachesProblem& cp, const WaitCtl& wc, cudaStream_t stream, int num_sms) {
    DecodeParams p;
    p.q = reinterpret_cast<const __nv_bfloat16*>(cp.q);
    p.k = nullptr;
    p.v = nullptr;
    p.kc = reinterpret_cast<const __nv_bfloat16* const*>(cp.k_caches);
    p.vc = reinterpret_cast<const __nv_bfloat16* const*>(cp.v_caches);
    p.out = reinterpret_cast<__nv_bfloat16*>(cp.out);
    p.key_lens = cp.kv_lens;
    p.Hq = cp.Hq;
    p.Hkv = cp.Hkv;
    p.Lk = cp.capacity;
    p.P = 0;
    p.mode = 0;
    p.window = 0;
    p.sliding = cp.sliding;
    p.scale_log2 = cp.scale * kLog2e;
    p.wc = wc;
    if (cp.Hkv > 65535 || cp.m > 65535) return cudaErrorInvalidConfiguration;
    const long long span = cp.sliding > 0 ? std::min(cp.sliding, cp.capacity) : cp.capacity;
    const int nsplit = choose_splits((long long)cp.m * cp.Hkv, span, num_sms);
    const int G = cp.Hq / cp.Hkv;
    return launch_any(p, cp.D, cp.f16, G, cp.m, nsplit, stream);
}

}  // namespace attn
