// prefill_narrow.cu -- K6: fused attention prefill for head_dim 64 on the 5th-generation tensor
// cores (sm_103a), bf16 or fp16 inputs and outputs, fp32 accumulation.
//
// At head_dim 64 the per-tile chain (S -> softmax -> P -> P V -> next S) is short and its
// latency, not a throughput, sets the pace: the more independent query tiles an SM holds, the
// better.  This kernel keeps each tile's tensor memory at 128 columns (S of a 64-key block: 64
// fp32 columns, P aliasing its first 32; O: 64) and its shared memory near 50 KB, so four CTAs
// of one 128-row query tile each share an SM (the tensor memory's limit), at 80 registers a
// thread.
//   warp 0       TMA producer: the Q tile, then 64-key K and V tiles through 2-stage rings
//                (128-byte swizzle).  With key padding or a band that ends inside the tensor
//                it also zeroes the rows of the last V tile that no query of the sequence sees.
//   warp 1       TMEM owner and single-thread MMA issuer.
//   warps 2-5    softmax, one thread per query row (its TMEM lane): the 64 scores of a block
//                come from one TMEM load, the row maximum needs no partner, the 64
//                probabilities (2^x on the special-function unit, scale*log2(e) folded in)
//                go back into TMEM as packed 16-bit pairs, and the row sum is kept over the
//                rounded values the tensor core multiplies.  O is rescaled only when the row
//                maximum grows by more than 2^8.  A warp whose 32 rows see none of a block's
//                keys skips it and writes zero P.  After the last block each thread normalises
//                and stores its row.
// The MMA order per block j is QK(j) -> softmax(j) -> PV(j) -> QK(j + 1): S and P share
// columns, so a tile's chain is sequential and the other CTAs on the SM fill its gaps.
//   QK(j):  S  = Q K_j^T   (M = 128, N = 64, both operands K-major in shared memory)
//   PV(j):  O += P V_j     (A = P from TMEM, B = V from shared memory, MN-major, N = 64)
// Each query tile visits only the 64-key blocks that intersect its visible band.
//
// What is computed follows ferrum-kernels Backend::flash_attention, ripvec-core
// Driver::fused_scale_mask_softmax (softmax(scores*scale + mask)) and the realizar
// cached/attention.rs causal softmax (a fully masked row gives zeros).
#include "kernels.h"

#include <algorithm>
#include <mutex>

namespace attn {
namespace {

constexpr int D = 64;
constexpr int BM = 128;       // query rows per tile
constexpr int BN = 64;        // keys per block
constexpr int kStages = 2;    // K/V ring depth
constexpr int kThreads = 192;  // producer, MMA issuer, 4 softmax warps
constexpr int kCtasPerSm = 4;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;

constexpr int kQBytes = BM * D * 2;   // 16 KB
constexpr int kKVBytes = BN * D * 2;  // 8 KB
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQBytes;
constexpr int kOffV = kOffK + kStages * kKVBytes;
constexpr int kOffBar = kOffV + kStages * kKVBytes;
constexpr int kSmem = kOffBar + 256 + 1024;  // + realignment slack
constexpr uint32_t kTmemCols = 128;
constexpr uint32_t kColS = 0;   // S (64 fp32 columns); P aliases columns 0..31
constexpr uint32_t kColO = 64;  // O (64 fp32 columns)
static_assert(kCtasPerSm * kSmem <= 232448, "shared memory of the CTAs of one SM");

enum : int {
    kBarQFull = 0,
    kBarKFull = 1,
    kBarVFull = kBarKFull + kStages,
    kBarKEmpty = kBarVFull + kStages,
    kBarVEmpty = kBarKEmpty + kStages,
    kBarSFull = kBarVEmpty + kStages,
    kBarPFull = kBarSFull + 1,   // 4 arrivals, one per softmax warp
    kBarOFull = kBarPFull + 1,   // the tile's last P V product completed
    kBarMmaDone = kBarOFull + 1,
    kBarVLand = kBarMmaDone + 1,  // the tail V tile's copy, before its unseen rows are zeroed
    kNumBars = kBarVLand + 1,
};
static_assert(kNumBars * 8 <= 240, "barrier area");

struct NarrowParams {
    __nv_bfloat16* out;
    const int32_t* key_lens;
    int B, Hq, Hkv, Lq, Lk, P, mode, window;
    int num_m;                  // query tiles per head
    const int32_t* cu_seqlens;  // packed token-major sequences [B + 1], or null (head-major batch)
    int total;                  // packed rows
    int out_tok;                // head-major batch: out is [B, Lq, Hq, D]
    int tma_out;                // out [B, Hq, Lq, D]: the tile is stored by one TMA copy from shared memory
    float scale_log2;
    WaitCtl wc;
};

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, const WaitCtl& wc) {
    const unsigned long long t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > wc.limit_ns) {
            record_status(wc.status, kStatusTimeout);
            return;
        }
    }
}

// D(tmem) (+)= A(tmem) * B(smem), kind::f16.
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ float row_max64(const float* s) {
    float e8[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) e8[q] = fmaxf(s[q], s[8 + q]);
#pragma unroll
    for (int c = 16; c < 64; c += 16) {
#pragma unroll
        for (int q = 0; q < 8; ++q) e8[q] = fmax3(e8[q], s[c + q], s[c + 8 + q]);
    }
    return fmax3(fmax3(e8[0], e8[1], e8[2]), fmax3(e8[3], e8[4], e8[5]), fmaxf(e8[6], e8[7]));
}

__device__ __forceinline__ float row_min64(const float* s) {
    float m = s[0];
#pragma unroll
    for (int c = 1; c < 64; ++c) m = fminf(m, s[c]);
    return m;
}

// TOK: packed token-major sequences.  ZT: some sequence may have key rows inside the tensor
// that none of its queries sees (the host clears it when it can show that none does).
// POS: the scale is positive (known on the host), so the minimum path for negative scales and the
// explicit zeroing for scale 0 are left out of the softmax.
template <bool F16, bool TOK, bool ZT, bool POS>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    prefill_narrow_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                          const NarrowParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + kOffBar;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kOffBar + 240);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffBar + 248);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    int idx = blockIdx.x;
    const int hq = idx % p.Hq;
    idx /= p.Hq;
    const int b = idx % p.B;
    idx /= p.B;
    const int mblk = p.num_m - 1 - idx;  // heaviest tiles first
    const int hk = hq / (p.Hq / p.Hkv);
    const int q0 = mblk * BM;
    int Lq = p.Lq, Lk = p.Lk, row0 = 0;
    if constexpr (TOK) {
        const int s0 = __ldg(p.cu_seqlens + b), s1 = __ldg(p.cu_seqlens + b + 1);
        if (s0 < 0 || s1 < s0 || s1 > p.total || s1 - s0 > p.Lq) {
            // not a prefix sum inside [0, total] with lengths <= max_seqlen: read nothing
            if (threadIdx.x == 0 && mblk == 0) record_status(p.wc.status, kStatusBadSeqlens);
            return;
        }
        row0 = s0;
        Lq = Lk = s1 - s0;
    }
    if (q0 >= Lq) return;  // a packed sequence shorter than this tile (uniform exit)
    const int klen = valid_keys(p.key_lens, b, Lk);

    // visible key interval of the tile, in 64-key blocks from kv0
    long long tlo, thi;
    key_interval(p.mode, p.window, klen, (long long)p.P + q0, (long long)p.P + min(q0 + BM, Lq) - 1, &tlo, &thi);
    const bool any = thi > tlo;
    const long long kv0 = any ? tlo : 0;
    const int nblk = any ? (int)((thi - tlo + BN - 1) / BN) : 0;
    const int kbh = b * p.Hkv + hk;

    // Rows of the last V tile past every key the sequence's queries see (and inside the
    // tensor) are zeroed before its P V product: their weight is 0, but 0 * Inf or 0 * NaN on
    // the tensor core is NaN.
    int zero_lo = 0, zero_hi = 0;
    bool zero_tail = false;
    if constexpr (ZT) {
        long long slo, shi;
        key_interval(p.mode, p.window, klen, (long long)p.P, (long long)p.P + Lq - 1, &slo, &shi);
        const long long tail_row = kv0 + (long long)(nblk - 1) * BN;
        const long long row_limit = TOK ? (long long)p.total - row0 : (long long)Lk;
        zero_lo = (int)max(0LL, shi - tail_row);
        zero_hi = (int)min((long long)BN, row_limit - tail_row);
        zero_tail = nblk > 0 && zero_hi > zero_lo;
    }

    auto load_q = [&]() {
        mbar_arrive_expect_tx(bar0 + 8 * kBarQFull, kQBytes);
        if constexpr (TOK)
            tma_load_3d(sbase + kOffQ, &tmQ, bar0 + 8 * kBarQFull, 0, hq, row0 + q0);
        else
            tma_load_3d(sbase + kOffQ, &tmQ, bar0 + 8 * kBarQFull, 0, q0, b * p.Hq + hq);
    };
    auto load_kv = [&](const CUtensorMap* map, int off, int bar, int j) {
        const int s = j % kStages;
        const int krow = (int)kv0 + j * BN;
        const uint32_t done = (zero_tail && bar == kBarVFull && j == nblk - 1) ? bar0 + 8 * kBarVLand
                                                                               : bar0 + 8 * (bar + s);
        mbar_arrive_expect_tx(done, kKVBytes);
        tma_load_3d(sbase + off + s * kKVBytes, map, done, 0, TOK ? hk : krow, TOK ? row0 + krow : kbh);
    };
    const int nearly = min(kStages, nblk);  // K/V tiles whose copies go out before the CTA barrier

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNumBars; ++i) mbar_init(bar0 + 8 * i, i == kBarPFull ? 4u : 1u);
        *abort_flag = 0;
        mbar_fence_init();
        // the first copies start now and land while TMEM is allocated and the CTA synchronises
        if (nblk > 0) {
            load_q();
            for (int j = 0; j < nearly; ++j) {
                load_kv(&tmK, kOffK, kBarKFull, j);
                load_kv(&tmV, kOffV, kBarVFull, j);
            }
        }
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        int issued = 2 * nearly;  // K and V copies issued so far (kept by lane 0)
        if (lane == 0 && nblk > 0) {
            for (int j = nearly; j < nblk; ++j) {
                const int s = j % kStages;
                const uint32_t n = (uint32_t)(j / kStages);
                if (!mbar_wait(bar0 + 8 * (kBarKEmpty + s), (n - 1) & 1, p.wc, abort_flag)) break;
                load_kv(&tmK, kOffK, kBarKFull, j);
                if (!mbar_wait(bar0 + 8 * (kBarVEmpty + s), (n - 1) & 1, p.wc, abort_flag)) {
                    issued = 2 * j + 1;
                    break;
                }
                load_kv(&tmV, kOffV, kBarVFull, j);
                issued = 2 * j + 2;
            }
            drain_wait(bar0 + 8 * kBarQFull, 0, p.wc);
            const int nk = (issued + 1) / 2, nv = issued / 2;
            for (int j = (nk > kStages ? nk - kStages : 0); j < nk; ++j)
                drain_wait(bar0 + 8 * (kBarKFull + j % kStages), (uint32_t)(j / kStages) & 1, p.wc);
            for (int j = (nv > kStages ? nv - kStages : 0); j < nv; ++j)
                if (!(zero_tail && j == nblk - 1))  // the tail tile is waited for below
                    drain_wait(bar0 + 8 * (kBarVFull + j % kStages), (uint32_t)(j / kStages) & 1, p.wc);
        }
        // The tail V tile: once it has landed the warp zeroes its rows [zero_lo, zero_hi) (128
        // bytes each, whatever the swizzle does inside a row), makes the stores visible to the
        // tensor core and releases the tile.
        if (zero_tail && __shfl_sync(0xffffffffu, issued, 0) >= 2 * nblk) {
            const bool landed = __all_sync(0xffffffffu, mbar_wait(bar0 + 8 * kBarVLand, 0, p.wc, abort_flag));
            if (landed) {
                const int s = (nblk - 1) % kStages;
                uint8_t* vt = smem + kOffV + s * kKVBytes;
                for (int u = lane; u < (zero_hi - zero_lo) * 8; u += 32)
                    *reinterpret_cast<uint4*>(vt + (zero_lo + u / 8) * 128 + (u & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar0 + 8 * (kBarVFull + s));
            } else if (lane == 0) {
                drain_wait(bar0 + 8 * kBarVLand, 0, p.wc);  // gave up: the copy may still be in flight
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && nblk > 0) {
            constexpr uint32_t kIdescQK = idesc_f16kind_f32(BM, BN, 0, 0, F16);
            constexpr uint32_t kIdescPV = idesc_f16kind_f32(BM, D, 0, 1, F16);
            bool ok = mbar_wait(bar0 + 8 * kBarQFull, 0, p.wc, abort_flag);
            const uint64_t qd = smem_desc_sw128(sbase + kOffQ, 16, 1024);
            for (int j = 0; ok && j <= nblk; ++j) {
                if (j > 0) {  // PV(j - 1), once its P is in TMEM
                    const int jp = j - 1, s = jp % kStages;
                    if (!mbar_wait(bar0 + 8 * kBarPFull, (uint32_t)jp & 1, p.wc, abort_flag)) break;
                    if (!mbar_wait(bar0 + 8 * (kBarVFull + s), (uint32_t)(jp / kStages) & 1, p.wc, abort_flag)) break;
                    tc_fence_after();
                    // descriptors: the tile's, plus each step's offset >> 4 in the address field
                    const uint64_t vd = smem_desc_sw128(sbase + kOffV + s * kKVBytes, BN * 128, 1024);
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        tc_mma_ts(tmem + kColO, tmem + kColS + kk * 8, vd + (uint64_t)((kk * 16 * 128) >> 4), kIdescPV,
                                  (jp > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(bar0 + 8 * (kBarVEmpty + s));
                    if (jp == nblk - 1) tc_commit(bar0 + 8 * kBarOFull);
                }
                if (j < nblk) {  // QK(j): overwrites S and P, which PV(j - 1), issued above, reads first
                    const int s = j % kStages;
                    if (!mbar_wait(bar0 + 8 * (kBarKFull + s), (uint32_t)(j / kStages) & 1, p.wc, abort_flag)) break;
                    tc_fence_after();
                    const uint64_t kd = smem_desc_sw128(sbase + kOffK + s * kKVBytes, 16, 1024);
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks)
                        tc_mma_ss(tmem + kColS, qd + (uint64_t)((ks * 32) >> 4), kd + (uint64_t)((ks * 32) >> 4), kIdescQK,
                                  ks > 0 ? 1u : 0u);
                    tc_commit(bar0 + 8 * kBarSFull);
                    tc_commit(bar0 + 8 * (kBarKEmpty + s));
                }
            }
            tc_commit(bar0 + 8 * kBarMmaDone);
            drain_wait(bar0 + 8 * kBarMmaDone, 0, p.wc);
        }
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        const int wq = warp & 3;  // TMEM lane quarter
        const int row = wq * 32 + lane;
        const int qi = q0 + row;
        long long rlo, rhi;
        key_interval(p.mode, p.window, klen, (long long)p.P + qi, (long long)p.P + qi, &rlo, &rhi);
        // the row's visible keys relative to its first column of the first block, clamped to the keys
        // that exist (a band past them is empty either way): 32-bit offsets for the block loop
        const int rlo_rel = (int)(min(max(rlo, 0LL), (long long)klen) - (kv0));
        const int rhi_rel = (int)(min(max(rhi, 0LL), (long long)klen) - (kv0));
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t tS = tmem + lane_off + kColS;
        const uint32_t tO = tmem + lane_off + kColO;
        const float sl = p.scale_log2;
        float m_run = -INFINITY;
        float l_run = 0.f;
        bool ok = true;

        for (int j = 0; j < nblk; ++j) {
            // every lane waits; the warp continues only if all lanes saw the phase, so the
            // warp-collective tcgen05 operations below never run with a partial warp
            if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar0 + 8 * kBarSFull, (uint32_t)j & 1, p.wc, abort_flag));
            if (!ok) break;
            tc_fence_after();
            const int c_lo = min(max(rlo_rel - j * BN, 0), 64);  // my visible columns [c_lo, c_hi)
            const int c_hi = min(max(rhi_rel - j * BN, 0), 64);
            const bool full = (c_lo == 0 && c_hi == 64);
            // every row of the warp sees none of the block's keys: zeros for its P, no exponentials
            const bool skip = __all_sync(0xffffffffu, c_lo >= c_hi);
            float alpha = 1.f;
            bool rescale = false;
            float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
            // P(j) overwrites S(j), which this thread has read into registers; PV(j - 1) completed
            // before S(j) was committed, so O is stable here
            if (skip) {
                uint32_t z[16];
#pragma unroll
                for (int q = 0; q < 16; ++q) z[q] = 0u;
                tmem_st16_async(tS, z);
                tmem_st16_async(tS + 16, z);
            } else {
                float s[64];
                tmem_ld32_async(tS, reinterpret_cast<uint32_t*>(s));
                tmem_ld32_async(tS + 32, reinterpret_cast<uint32_t*>(s) + 32);
                tmem_ld_wait32(reinterpret_cast<uint32_t*>(s));
                tmem_ld_wait32(reinterpret_cast<uint32_t*>(s) + 32);
                float ext;
                if (POS || sl >= 0.f) {
                    if (!full) {
                        mask_scores64(s, range_bits64(c_lo, c_hi), -INFINITY);
                    }
                    ext = row_max64(s);
                } else {
                    if (!full) {
                        mask_scores64(s, range_bits64(c_lo, c_hi), INFINITY);
                    }
                    ext = row_min64(s);
                }
                const bool seen = (POS || sl >= 0.f) ? (ext != -INFINITY) : (ext != INFINITY);
                if (seen) {
                    const float ms = ext * sl;
                    if (m_run == -INFINITY) {
                        m_run = ms;
                    } else if (ms > m_run + kRescaleThreshold) {
                        alpha = ex2_approx(m_run - ms);
                        m_run = ms;
                        rescale = true;
                    }
                }
                const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;
                const float2 sl2 = make_float2(sl, sl), negm2 = make_float2(neg_m, neg_m);
                // two rounds of 32 keys, each stored to TMEM as soon as it is packed
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    uint32_t pk[16];
#pragma unroll
                    for (int c2 = 0; c2 < 32; c2 += 2) {
                        const int c = 32 * k + c2;
                        const float2 x2 = __ffma2_rn(make_float2(s[c], s[c + 1]), sl2, negm2);
                        float p0 = ex2_approx(x2.x);  // special-function unit; 2^-inf = 0
                        float p1 = ex2_approx(x2.y);
                        // masked scores hold -inf (+inf with a negative scale), so their
                        // 2^(s*scale*log2e - m) is already 0; only scale 0 turns them into NaN
                        // (inf * 0) and needs the explicit zero
                        if (!POS && !full && sl == 0.f) {
                            p0 = (c >= c_lo && c < c_hi) ? p0 : 0.f;
                            p1 = (c + 1 >= c_lo && c + 1 < c_hi) ? p1 : 0.f;
                        }
                        const uint32_t wv = pack2<F16>(p0, p1);
                        pk[c2 / 2] = wv;
                        const float2 r2 = unpack2<F16>(wv);
                        if ((c2 / 2) & 1) acc1 = __fadd2_rn(acc1, r2); else acc0 = __fadd2_rn(acc0, r2);
                    }
                    tmem_st16_async(tS + 16 * k, pk);
                }
            }
            tmem_st_wait();
            acc0 = __fadd2_rn(acc0, acc1);
            l_run = l_run * alpha + (acc0.x + acc0.y);
            if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    float o[32];
                    tmem_ld32(tO + 32 * c, o);
#pragma unroll
                    for (int q = 0; q < 32; ++q) o[q] *= alpha;
                    tmem_st32(tO + 32 * c, o);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar0 + 8 * kBarPFull);
        }

        // ------------------------------------------------------------ epilogue
        if (ok && nblk > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar0 + 8 * kBarOFull, 0, p.wc, abort_flag));
            tc_fence_after();
        }
        // (the TMEM loads are warp-collective: every lane runs them, and only rows inside the
        // sequence are stored)
        if (p.tma_out) {
            // head-major output: each thread writes its normalised row into the Q buffer (free
            // once the last product has completed; never loaded without key blocks) in the
            // 128-byte-swizzle layout of a Q tile, and one thread stores the tile with TMA (rows
            // past Lq are clipped by the copy)
            if (ok) {
                const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
                uint8_t* qrow_s = smem + kOffQ + row * 128;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    float o[32];
                    if (nblk > 0) {
                        tmem_ld32(tO + 32 * c, o);
                    } else {
#pragma unroll
                        for (int q = 0; q < 32; ++q) o[q] = 0.f;
                    }
#pragma unroll
                    for (int q = 0; q < 32; q += 8) {
                        const int unit = (32 * c + q) / 8;  // 16-byte unit of the row
                        *reinterpret_cast<uint4*>(qrow_s + ((unit ^ (row & 7)) << 4)) =
                            make_uint4(pack2<F16>(o[q] * inv, o[q + 1] * inv), pack2<F16>(o[q + 2] * inv, o[q + 3] * inv),
                                       pack2<F16>(o[q + 4] * inv, o[q + 5] * inv), pack2<F16>(o[q + 6] * inv, o[q + 7] * inv));
                    }
                }
                fence_proxy_async_smem();
            }
            // the four softmax warps meet (every path reaches this) and agree that all rows are in place
            uint32_t all_ok;
            asm volatile(
                "{\n\t.reg .pred pin, pout;\n\tsetp.ne.u32 pin, %1, 0;\n\t"
                "bar.red.and.pred pout, 1, 128, pin;\n\tselp.u32 %0, 1, 0, pout;\n\t}"
                : "=r"(all_ok)
                : "r"((uint32_t)ok)
                : "memory");
            if (all_ok && warp == 2 && lane == 0) {
                asm volatile(
                    "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                        reinterpret_cast<uint64_t>(&tmO)),
                    "r"(0), "r"(q0), "r"(b * p.Hq + hq), "r"(sbase + kOffQ)
                    : "memory");
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");  // before the CTA may leave
            }
        } else if (ok) {
            const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
            __nv_bfloat16* orow =
                p.out + (TOK        ? ((size_t)(row0 + qi) * p.Hq + hq) * D
                         : p.out_tok ? (((size_t)b * Lq + qi) * p.Hq + hq) * D
                                     : ((size_t)(b * p.Hq + hq) * Lq + qi) * D);
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                float o[32];
                if (nblk > 0) {
                    tmem_ld32(tO + 32 * c, o);
                } else {
#pragma unroll
                    for (int q = 0; q < 32; ++q) o[q] = 0.f;
                }
                if (qi < Lq) {
#pragma unroll
                    for (int q = 0; q < 32; q += 8) {
                        uint4 v4 = make_uint4(pack2<F16>(o[q] * inv, o[q + 1] * inv),
                                              pack2<F16>(o[q + 2] * inv, o[q + 3] * inv),
                                              pack2<F16>(o[q + 4] * inv, o[q + 5] * inv),
                                              pack2<F16>(o[q + 6] * inv, o[q + 7] * inv));
                        *reinterpret_cast<uint4*>(orow + 32 * c + q) = v4;
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult qres;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &qres) ==
                cudaSuccess &&
            qres == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// A 16-bit tensor with rows of 64 values, as 3-D (64, dim1, dim2) with the given byte strides;
// box 64 x box1 x box2, 128-byte swizzle, zero fill outside the tensor.
bool encode(CUtensorMap* map, const void* base, unsigned long long dim1, unsigned long long dim2,
            unsigned long long stride1, unsigned long long stride2, int box1, int box2, bool f16) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)dim1, (cuuint64_t)dim2};
    cuuint64_t strides[2] = {(cuuint64_t)stride1, (cuuint64_t)stride2};
    cuuint32_t box[3] = {64, (cuuint32_t)box1, (cuuint32_t)box2};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base),
              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool F16, bool TOK, bool ZT, bool POS>
cudaError_t launch_impl(const Problem& pr, const WaitCtl& wc, cudaStream_t stream) {
    CUtensorMap tq, tk, tv, to;
    const unsigned long long row = D * 2;
    if (TOK) {
        // [total, H, 64] as (64, H, total): a box is 128 (Q) or 64 (K, V) consecutive rows of one head
        if (!encode(&tq, pr.q, pr.Hq, pr.total, row, row * pr.Hq, 1, BM, F16) ||
            !encode(&tk, pr.k, pr.Hkv, pr.total, row, row * pr.Hkv, 1, BN, F16) ||
            !encode(&tv, pr.v, pr.Hkv, pr.total, row, row * pr.Hkv, 1, BN, F16))
            return cudaErrorInvalidValue;
    } else if (!encode(&tq, pr.q, pr.Lq, (unsigned long long)pr.B * pr.Hq, row, row * pr.Lq, BM, 1, F16) ||
               !encode(&tk, pr.k, pr.Lk, (unsigned long long)pr.B * pr.Hkv, row, row * pr.Lk, BN, 1, F16) ||
               !encode(&tv, pr.v, pr.Lk, (unsigned long long)pr.B * pr.Hkv, row, row * pr.Lk, BN, 1, F16)) {
        return cudaErrorInvalidValue;
    }
    // head-major output [B, Hq, Lq, 64]: stored a tile at a time by TMA, through the map Q uses
    const bool tma_out = !TOK && !pr.out_tok;
    if (tma_out) {
        if (!encode(&to, pr.out, pr.Lq, (unsigned long long)pr.B * pr.Hq, row, row * pr.Lq, BM, 1, F16))
            return cudaErrorInvalidValue;
    } else {
        to = tq;  // not used
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::mutex mu;
    static bool configured[64] = {};
    {
        std::lock_guard<std::mutex> g(mu);
        if (dev < 64 && !configured[dev]) {
            e = cudaFuncSetAttribute(prefill_narrow_kernel<F16, TOK, ZT, POS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kSmem);
            if (e != cudaSuccess) return e;
            configured[dev] = true;
        }
    }
    NarrowParams p = {};
    p.out = reinterpret_cast<__nv_bfloat16*>(pr.out);
    p.key_lens = pr.key_lens;
    p.B = pr.B;
    p.Hq = pr.Hq;
    p.Hkv = pr.Hkv;
    p.Lq = pr.Lq;
    p.Lk = pr.Lk;
    p.P = pr.pos_offset;
    p.mode = pr.mode;
    p.window = pr.window;
    p.num_m = (pr.Lq + BM - 1) / BM;  // pr.Lq is max_seqlen for packed sequences
    p.cu_seqlens = pr.cu_seqlens;
    p.total = pr.total;
    p.out_tok = pr.out_tok ? 1 : 0;
    p.tma_out = tma_out ? 1 : 0;
    p.scale_log2 = pr.scale * kLog2e;
    p.wc = wc;
    const long long grid = (long long)p.num_m * pr.B * pr.Hq;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    prefill_narrow_kernel<F16, TOK, ZT, POS><<<(unsigned)grid, kThreads, kSmem, stream>>>(tq, tk, tv, to, p);
    return cudaGetLastError();
}

// Whether some row inside the tensor can go unseen by every query of its sequence (key padding,
// packed sequences, or a band that ends before kv_len): only then is the tail zeroing compiled in.
bool tail_zero_needed(const Problem& p) {
    if (p.key_lens != nullptr || p.cu_seqlens != nullptr) return true;
    long long slo, shi;
    key_interval(p.mode, p.window, p.Lk, (long long)p.pos_offset, (long long)p.pos_offset + p.Lq - 1, &slo, &shi);
    return shi < p.Lk;
}

template <bool F16, bool POS>
cudaError_t launch_fs(const Problem& p, const WaitCtl& wc, cudaStream_t stream) {
    if (p.cu_seqlens != nullptr) return launch_impl<F16, true, true, POS>(p, wc, stream);
    if (tail_zero_needed(p)) return launch_impl<F16, false, true, POS>(p, wc, stream);
    return launch_impl<F16, false, false, POS>(p, wc, stream);
}

template <bool F16>
cudaError_t launch_f(const Problem& p, const WaitCtl& wc, cudaStream_t stream) {
    return p.scale > 0.f ? launch_fs<F16, true>(p, wc, stream) : launch_fs<F16, false>(p, wc, stream);
}

}  // namespace

bool prefill_narrow_supported(const Problem& p) { return p.D == 64 && p.page_table == nullptr; }

cudaError_t launch_prefill_narrow(const Problem& p, const WaitCtl& wc, cudaStream_t stream) {
    return p.f16 ? launch_f<true>(p, wc, stream) : launch_f<false>(p, wc, stream);
}

}  // namespace attn
