// prefill_tc.cu -- K1: fused attention prefill on the 5th-generation tensor cores (sm_103a).
//
// One CTA computes one 128-row query tile of one (batch, query head):
//   warp 0      TMA producer: the Q tile once, then K and V tiles of 128 keys
//               through a 2-stage shared-memory ring (128-byte swizzle).
//   warp 1      TMEM owner and single-thread MMA issuer:
//               S = Q K^T into TMEM (M=128, N=128, K=head_dim), and
//               O += P V into TMEM (M=128, N=head_dim, K=128).
//   warps 2-5   softmax: one thread per query row reads its S row from TMEM,
//               masks, keeps the running row max and sum (base-2 exponent with
//               scale*log2(e) folded in), writes P as bf16 into shared memory
//               (the A operand of the P V product), rescales O in TMEM when the
//               running max grows by more than 2^8, and finally normalises O by
//               the row sum and stores bf16 rows of out.
// Key tiles start at the first key any row of the tile may see, and only tiles
// that intersect the visible band are visited, so causal and windowed masks
// skip fully masked tiles.  The S buffer is released as soon as the softmax
// warps have copied it to registers, so the tensor core computes the next
// S = Q K^T while the softmax of the current tile runs.
//
// What is computed follows the ferrum-kernels Backend::flash_attention
// statement of the operation, the ripvec-core Driver::fused_scale_mask_softmax
// definition softmax(scores*scale + mask), and the realizar cached/attention.rs
// causal softmax (a fully masked row gives zeros).
#include "kernels.h"

#include <mutex>

namespace attn {
namespace {

constexpr int BM = 128;           // query rows per tile
constexpr int BN = 128;           // keys per tile
constexpr int kThreads = 192;     // 6 warps
constexpr int kStages = 2;        // K/V ring depth
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows by > 2^8

template <int D>
struct Cfg {
    static constexpr int kChunks = D / 64;           // 64-element (128-byte) swizzle atoms per row
    static constexpr int kQBytes = BM * D * 2;
    static constexpr int kKVBytes = BN * D * 2;
    static constexpr int kPBytes = BM * BN * 2;
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kQBytes;
    static constexpr int kOffV = kOffK + kStages * kKVBytes;
    static constexpr int kOffP = kOffV + kStages * kKVBytes;
    static constexpr int kOffBar = kOffP + kPBytes;
    static constexpr int kSmem = kOffBar + 256 + 1024;  // barriers + 1 KB for base alignment
    static constexpr uint32_t kTmemCols = 256;
    static constexpr uint32_t kColS = 0;
    static constexpr uint32_t kColO = 128;
    static constexpr int kMinBlocks = (D == 64) ? 2 : 1;
};

// Barrier slots (8 bytes each) inside the barrier area.
enum : int {
    kBarQFull = 0,
    kBarKFull = 1,                       // + stage
    kBarVFull = kBarKFull + kStages,     // + stage
    kBarKEmpty = kBarVFull + kStages,    // + stage
    kBarVEmpty = kBarKEmpty + kStages,   // + stage
    kBarSFull = kBarVEmpty + kStages,
    kBarSFree = kBarSFull + 1,
    kBarPFull = kBarSFree + 1,
    kBarPVDone = kBarPFull + 1,
    kBarMmaDone = kBarPVDone + 1,        // final commit: every MMA of the block has completed
    kNumBars = kBarMmaDone + 1,
};
static_assert(kNumBars * 8 <= 128, "barrier area");

struct PrefillParams {
    __nv_bfloat16* out;
    const int32_t* key_lens;
    int B, Hq, Hkv, Lq, Lk, P, mode, window;
    int num_m;          // query tiles per head
    float scale_log2;   // scale * log2(e)
    WaitCtl wc;
};

// Wait that ignores the abort flag (used to drain copies still in flight), bounded in time.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, const WaitCtl& wc) {
    const unsigned long long t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > wc.limit_ns) {
            record_status(wc.status, kStatusTimeout);
            return;
        }
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads, Cfg<D>::kMinBlocks)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment of the tile area (required by the 128-byte swizzle pattern).
    const uint32_t raw_s = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + C::kOffBar;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffBar + 128);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffBar + 136);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Work item: heaviest query tiles first (causal tiles near the end see the most keys).
    int idx = blockIdx.x;
    const int hq = idx % p.Hq;
    idx /= p.Hq;
    const int b = idx % p.B;
    idx /= p.B;
    const int mblk = p.num_m - 1 - idx;
    const int hk = hq / (p.Hq / p.Hkv);
    const int q0 = mblk * BM;
    const int q_last = min(q0 + BM, p.Lq) - 1;

    const int klen = valid_keys(p.key_lens, b, p.Lk);
    long long lo, hi;
    key_interval(p.mode, p.window, klen, (long long)p.P + q0, (long long)p.P + q_last, &lo, &hi);
    const int ntiles = (hi > lo) ? (int)((hi - lo + BN - 1) / BN) : 0;
    const int kv0 = (int)lo;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNumBars; ++i) {
            uint32_t count = 1;
            if (i == kBarSFree || i == kBarPFull) count = 4;  // one arrival per softmax warp
            mbar_init(bar0 + 8 * i, count);
        }
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), C::kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && ntiles > 0) {
            const int qbh = b * p.Hq + hq;
            const int kbh = b * p.Hkv + hk;
            mbar_arrive_expect_tx(bar0 + 8 * kBarQFull, C::kQBytes);
            for (int c = 0; c < C::kChunks; ++c)
                tma_load_3d(sbase + C::kOffQ + c * (BM * 128), &tmQ, bar0 + 8 * kBarQFull, c * 64, q0, qbh);
            int issued = 0;
            for (int j = 0; j < ntiles; ++j) {
                const int s = j % kStages;
                const uint32_t n = (uint32_t)(j / kStages);
                const int krow = kv0 + j * BN;
                if (j >= kStages && !mbar_wait(bar0 + 8 * (kBarKEmpty + s), (n - 1) & 1, p.wc, abort_flag)) break;
                mbar_arrive_expect_tx(bar0 + 8 * (kBarKFull + s), C::kKVBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_3d(sbase + C::kOffK + s * C::kKVBytes + c * (BN * 128), &tmK,
                                bar0 + 8 * (kBarKFull + s), c * 64, krow, kbh);
                if (j >= kStages && !mbar_wait(bar0 + 8 * (kBarVEmpty + s), (n - 1) & 1, p.wc, abort_flag)) {
                    issued = 2 * j + 1;
                    break;
                }
                mbar_arrive_expect_tx(bar0 + 8 * (kBarVFull + s), C::kKVBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_3d(sbase + C::kOffV + s * C::kKVBytes + c * (BN * 128), &tmV,
                                bar0 + 8 * (kBarVFull + s), c * 64, krow, kbh);
                issued = 2 * j + 2;
            }
            // Drain: no copy may still be writing shared memory when the block exits.
            drain_wait(bar0 + 8 * kBarQFull, 0, p.wc);
            const int nk = (issued + 1) / 2, nv = issued / 2;
            for (int j = (nk > kStages ? nk - kStages : 0); j < nk; ++j)
                drain_wait(bar0 + 8 * (kBarKFull + j % kStages), (uint32_t)(j / kStages) & 1, p.wc);
            for (int j = (nv > kStages ? nv - kStages : 0); j < nv; ++j)
                drain_wait(bar0 + 8 * (kBarVFull + j % kStages), (uint32_t)(j / kStages) & 1, p.wc);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && ntiles > 0) {
            constexpr uint32_t kIdescQK = idesc_bf16_f32(BM, BN, 0, 0);
            constexpr uint32_t kIdescPV = idesc_bf16_f32(BM, D, 0, 1);
            const uint32_t tS = tmem + C::kColS;
            const uint32_t tO = tmem + C::kColO;
            bool ok = mbar_wait(bar0 + 8 * kBarQFull, 0, p.wc, abort_flag);
            auto issue_qk = [&](int j) -> bool {
                const int s = j % kStages;
                if (!mbar_wait(bar0 + 8 * (kBarKFull + s), (uint32_t)(j / kStages) & 1, p.wc, abort_flag))
                    return false;
                if (j > 0 && !mbar_wait(bar0 + 8 * kBarSFree, (uint32_t)(j - 1) & 1, p.wc, abort_flag))
                    return false;
                tc_fence_after();
                const uint32_t kbase = sbase + C::kOffK + s * C::kKVBytes;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * (BM * 128) + (ks & 3) * 32;
                    const uint64_t a = smem_desc_sw128(sbase + C::kOffQ + off, 16, 1024);
                    const uint64_t bd = smem_desc_sw128(kbase + (ks >> 2) * (BN * 128) + (ks & 3) * 32, 16, 1024);
                    tc_mma_ss(tS, a, bd, kIdescQK, ks > 0 ? 1u : 0u);
                }
                tc_commit(bar0 + 8 * kBarSFull);
                tc_commit(bar0 + 8 * (kBarKEmpty + s));
                return true;
            };
            if (ok) ok = issue_qk(0);
            for (int j = 0; ok && j < ntiles; ++j) {
                if (j + 1 < ntiles && !issue_qk(j + 1)) break;
                const int s = j % kStages;
                if (!mbar_wait(bar0 + 8 * kBarPFull, (uint32_t)j & 1, p.wc, abort_flag)) break;
                if (!mbar_wait(bar0 + 8 * (kBarVFull + s), (uint32_t)(j / kStages) & 1, p.wc, abort_flag)) break;
                tc_fence_after();
                const uint32_t vbase = sbase + C::kOffV + s * C::kKVBytes;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    const uint64_t a =
                        smem_desc_sw128(sbase + C::kOffP + (kk >> 2) * (BM * 128) + (kk & 3) * 32, 16, 1024);
                    // V tile: keys along K (128 B per key row), head dims along N in 64-wide
                    // chunks that are BN*128 bytes apart.
                    const uint64_t bd = smem_desc_sw128(vbase + kk * (16 * 128), BN * 128, 1024);
                    tc_mma_ss(tO, a, bd, kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(bar0 + 8 * (kBarVEmpty + s));
                tc_commit(bar0 + 8 * kBarPVDone);
            }
            // Wait for every MMA issued so far before the block may release TMEM.
            tc_commit(bar0 + 8 * kBarMmaDone);
            drain_wait(bar0 + 8 * kBarMmaDone, 0, p.wc);
        }
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        const int wq = warp & 3;                 // TMEM lane quarter this warp may access
        const int row = wq * 32 + lane;          // query row within the tile
        const int qi = q0 + row;
        const long long qpos = (long long)p.P + qi;
        long long rlo, rhi;
        key_interval(p.mode, p.window, klen, qpos, qpos, &rlo, &rhi);
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t tS = tmem + lane_off + C::kColS;
        const uint32_t tO = tmem + lane_off + C::kColO;
        const float sl = p.scale_log2;
        float m_run = -INFINITY;
        float l_run = 0.f;
        bool ok = true;
        uint8_t* prow = smem + C::kOffP + (row >> 3) * 1024 + (row & 7) * 128;
        const int sw = row & 7;

        for (int j = 0; j < ntiles; ++j) {
            if (!mbar_wait(bar0 + 8 * kBarSFull, (uint32_t)j & 1, p.wc, abort_flag)) { ok = false; break; }
            tc_fence_after();
            float s[BN];
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) tmem_ld32(tS + 32 * c, s + 32 * c);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar0 + 8 * kBarSFree);

            const long long tb = (long long)kv0 + (long long)j * BN;
            const int c_lo = (int)max(0LL, min((long long)BN, rlo - tb));
            const int c_hi = (int)max(0LL, min((long long)BN, rhi - tb));
            const bool full = (c_lo == 0 && c_hi == BN);

            // Extreme of the raw scores over the visible columns: the max when the
            // scale is non-negative, the min when it is negative.
            float ext;
            if (sl >= 0.f) {
                ext = -INFINITY;
                if (full) {
#pragma unroll
                    for (int c = 0; c < BN; ++c) ext = fmaxf(ext, s[c]);
                } else {
#pragma unroll
                    for (int c = 0; c < BN; ++c) ext = (c >= c_lo && c < c_hi) ? fmaxf(ext, s[c]) : ext;
                }
            } else {
                ext = INFINITY;
#pragma unroll
                for (int c = 0; c < BN; ++c) ext = (c >= c_lo && c < c_hi) ? fminf(ext, s[c]) : ext;
            }
            const bool any = c_lo < c_hi;
            float alpha = 1.f;
            bool rescale = false;
            if (any) {
                const float ms = ext * sl;
                if (m_run == -INFINITY) {
                    m_run = ms;  // O holds only zero contributions so far
                } else if (ms > m_run + kRescaleThreshold) {
                    alpha = ex2_approx(m_run - ms);
                    m_run = ms;
                    rescale = true;
                }
            }
            const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;
            float sum = 0.f;
            uint32_t pk[BN / 2];
#pragma unroll
            for (int c = 0; c < BN; c += 2) {
                float p0 = ex2_approx(fmaf(s[c], sl, neg_m));
                float p1 = ex2_approx(fmaf(s[c + 1], sl, neg_m));
                if (!full) {
                    p0 = (c >= c_lo && c < c_hi) ? p0 : 0.f;
                    p1 = (c + 1 >= c_lo && c + 1 < c_hi) ? p1 : 0.f;
                }
                sum += p0 + p1;
                pk[c / 2] = pack_bf16x2(p0, p1);
            }
            l_run = l_run * alpha + sum;

            // P buffer and O are free once the previous P V product has completed.
            if (j > 0) {
                if (!mbar_wait(bar0 + 8 * kBarPVDone, (uint32_t)(j - 1) & 1, p.wc, abort_flag)) { ok = false; break; }
                tc_fence_after();
            }
            if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    float o[32];
                    tmem_ld32(tO + 32 * c, o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] *= alpha;
                    tmem_st32(tO + 32 * c, o);
                }
            }
            // P row -> shared memory, K-major with the 128-byte swizzle: 16-byte chunk cc of
            // the row goes to chunk position cc ^ (row % 8); keys 64..127 in the second atom.
#pragma unroll
            for (int q = 0; q < BN / 8; ++q) {
                const int atom = q >> 3, cc = q & 7;
                uint4 v4 = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                *reinterpret_cast<uint4*>(prow + atom * (BM * 128) + ((cc ^ sw) << 4)) = v4;
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar0 + 8 * kBarPFull);
        }

        // ------------------------------------------------------------ epilogue
        if (ok && ntiles > 0) {
            ok = mbar_wait(bar0 + 8 * kBarPVDone, (uint32_t)(ntiles - 1) & 1, p.wc, abort_flag);
            tc_fence_after();
        }
        if (ok) {
            const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
            __nv_bfloat16* orow = p.out + ((size_t)(b * p.Hq + hq) * p.Lq + qi) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                float o[32];
                if (ntiles > 0) {
                    tmem_ld32(tO + 32 * c, o);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0.f;
                }
                if (qi < p.Lq) {
#pragma unroll
                    for (int i = 0; i < 32; i += 8) {
                        uint4 v4 = make_uint4(pack_bf16x2(o[i] * inv, o[i + 1] * inv),
                                              pack_bf16x2(o[i + 2] * inv, o[i + 3] * inv),
                                              pack_bf16x2(o[i + 4] * inv, o[i + 5] * inv),
                                              pack_bf16x2(o[i + 6] * inv, o[i + 7] * inv));
                        *reinterpret_cast<uint4*>(orow + 32 * c + i) = v4;
                    }
                }
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

// ---------------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
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

// [rows_outer, L, D] bf16 tensor viewed as 3-D (D, L, rows_outer); box 64 x 128 x 1, 128-byte swizzle,
// out-of-range rows read as zeros.
bool encode_bf16_3d(CUtensorMap* map, const void* base, int D, int L, int outer) {
    EncodeTiledFn fn = get_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)L, (cuuint64_t)outer};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)L * D * 2};
    cuuint32_t box[3] = {64, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_impl(const Problem& pr, const WaitCtl& wc, cudaStream_t stream) {
    using C = Cfg<D>;
    CUtensorMap tq, tk, tv;
    if (!encode_bf16_3d(&tq, pr.q, D, pr.Lq, pr.B * pr.Hq) || !encode_bf16_3d(&tk, pr.k, D, pr.Lk, pr.B * pr.Hkv) ||
        !encode_bf16_3d(&tv, pr.v, D, pr.Lk, pr.B * pr.Hkv))
        return cudaErrorInvalidValue;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::mutex mu;
    static bool configured[64] = {};
    {
        std::lock_guard<std::mutex> g(mu);
        if (dev < 64 && !configured[dev]) {
            e = cudaFuncSetAttribute(prefill_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
            if (e != cudaSuccess) return e;
            configured[dev] = true;
        }
    }
    PrefillParams p;
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
    p.num_m = (pr.Lq + BM - 1) / BM;
    p.scale_log2 = pr.scale * kLog2e;
    p.wc = wc;
    const long long grid = (long long)p.num_m * pr.B * pr.Hq;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    prefill_tc_kernel<D><<<(unsigned)grid, kThreads, C::kSmem, stream>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_tc(const Problem& p, const WaitCtl& wc, cudaStream_t stream) {
    if (p.D == 64) return launch_impl<64>(p, wc, stream);
    if (p.D == 128) return launch_impl<128>(p, wc, stream);
    return cudaErrorInvalidValue;
}

}  // namespace attn
