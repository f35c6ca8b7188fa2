// decode_tc.cu -- K5: single-query (q_len == 1) attention against a KV cache on the
// 5th-generation tensor cores, head_dim 128, 4 or 8 query heads per kv head, bf16 or fp16.
//
// With several query heads per kv head the per-key work of a CUDA-core decode (every head
// against every key, then every head's probability into V) outgrows the HBM stream.  Here
// the tensor core does both products for the whole group:
//   S^T [128 keys x 16] = K_j Q^T        (A = the K tile, K-major; B = Q, the group's heads
//                                         padded with zero rows to 16, K-major)
//   O^T [128 dims x 16] += V_j^T P_j^T   (A = the V tile read MN-major; B = P^T, 16 rows of
//                                         128 keys in shared memory, K-major)
// with fp32 accumulators in TMEM (S^T double-buffered, 64 columns in all).
//
// Work unit: (batch b, kv head hk, split); the splits of one unit form a cluster and merge
// their partial results through distributed shared memory in CTA rank 0.
//   warp 0       producer: 128-key K and V tiles through 3-stage rings by TMA, from one
//                contiguous [B, Hkv, Lk, D] cache, from per-item caches through tensor maps
//                built on the device (a small kernel patches each item's cache address into a
//                host-encoded template), or from paged caches one copy per page piece; or, for
//                page sizes TMA cannot copy whole, by 16-byte cp.async copies that all 32 lanes
//                issue row by row into the same swizzled layout, rows past the visible keys
//                written as zeros.
//   warp 1       TMEM owner and single-thread MMA issuer: QK(j) then PV(j-1).
//   warps 2-5    one key per thread: it reads its key's 16 head scores from TMEM, the per-head
//                block maxima come from a shuffle reduce-scatter and a 4-warp exchange,
//                then it writes its key's probabilities (2^x on the special-function unit,
//                scale*log2(e) folded in) into P^T; O^T is rescaled only when a head's
//                maximum grows by more than 2^8.  In the epilogue the same threads own the
//                128 head dims.
//
// The operation is the q_len = 1 case of ferrum-kernels Backend::flash_attention (the
// GQA decode of a KV cache at pos_offset), with the masks of attn.h, and the per-cache
// decode of Backend::flash_attention_batched_per_cache (device kv_lens, the last-w sliding
// window) over per-item or paged caches.
#include "kernels.h"

#include <algorithm>
#include <mutex>

namespace attn {
namespace {

constexpr int D = 128;
constexpr int BN = 128;         // keys per block
constexpr int NH = 16;          // MMA N: the group's query heads, padded
constexpr int kStages = 3;
constexpr int kThreads = 192;        // TMA source: producer, MMA, 4 softmax warps
constexpr int kThreadsGather = 256;  // gather sources: + 2 producer warps (one per ring stage)
constexpr int kMaxSplits = 8;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;

struct L {
    static constexpr int kKVBytes = BN * D * 2;  // one K or V tile
    static constexpr int kQBytes = NH * D * 2;
    static constexpr int kPBytes = NH * BN * 2;
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kOffK + kStages * kKVBytes;
    static constexpr int kOffQ = kOffV + kStages * kKVBytes;
    static constexpr int kOffP = kOffQ + kQBytes;
    static constexpr int kOffX = kOffP + kPBytes;            // [2 parities][4 warps][16] block maxima
    static constexpr int kOffS = kOffX + 2 * 4 * NH * 4;     // [4 warps][16] row-sum parts
    static constexpr int kOffRow = kOffS + 4 * NH * 4;       // [3][128] gather: byte offset of each key row
    static constexpr int kOffBar = kOffRow + kStages * BN * 8;
    static constexpr int kSmem = kOffBar + 256 + 1024;        // + realignment slack
    // after the last P V product the K ring is free; the combine reuses it
    static constexpr int kOffCm = 0;                         // [16] log2-domain maxima
    static constexpr int kOffCl = kOffCm + NH * 4;           // [16] row sums
    static constexpr int kOffCo = kOffCl + NH * 4;           // [16][128] unnormalised outputs
    static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0, "swizzled tiles need 1024-byte alignment");
    static_assert(kSmem <= 232448, "shared memory budget");
};

enum : int {
    kBarKFull = 0,
    kBarKEmpty = kBarKFull + kStages,
    kBarVFull = kBarKEmpty + kStages,
    kBarVEmpty = kBarVFull + kStages,
    kBarSFull = kBarVEmpty + kStages,  // + buffer
    kBarSFree = kBarSFull + 2,         // + buffer, 4 arrivals
    kBarPFull = kBarSFree + 2,         // 4 arrivals
    kBarPVDone = kBarPFull + 1,
    kBarXch = kBarPVDone + 1,          // + parity, 4 arrivals
    kBarSum = kBarXch + 2,             // 4 arrivals
    kBarMmaDone = kBarSum + 1,
    kNumBars = kBarMmaDone + 1,
};
static_assert(kNumBars * 8 <= 240, "barrier area");

constexpr uint32_t kColS = 0;   // + 16 * buffer
constexpr uint32_t kColO = 32;
constexpr uint32_t kTmemCols = 64;

// Where the K and V rows come from.
enum : int {
    kSrcTma = 0,     // one contiguous [B, Hkv, Lk, D] cache per tensor, TMA tensor maps
    kSrcCaches = 1,  // per-item caches [Hkv, capacity, D] through device arrays of pointers, by TMA
                     // through a K and a V tensor map per item built on the device
    kSrcPaged = 2,   // pools [num_pages, Hkv, page_size, D] and a device page table [B, max_pages]
};

struct DecodeTcParams {
    const uint16_t* q;
    uint16_t* out;
    const int32_t* key_lens;  // key_lens (contiguous cache) or kv_lens (per-item and paged caches)
    int Hq, Hkv, Lk, P, mode, window;  // Lk: the capacity of an item's cache (per-item and paged caches)
    float scale_log2;
    WaitCtl wc;
    // per-item and paged caches: the query of item b is its newest position kv_lens[b] - 1 and
    // sees the item's positions, or only the last `sliding` of them
    int sliding;
    const uint16_t* const* kc;  // per-item caches
    const uint16_t* const* vc;
    const uint16_t* kpool;      // paged caches
    const uint16_t* vpool;
    const int32_t* page_table;
    int page_size, max_pages, num_pages;
    int paged_tma;  // paged: the page size lets TMA copy whole pages (else the rows are gathered)
    const CUtensorMap* item_maps;  // per-item caches: [items][2] (K, V) in global memory
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, const WaitCtl& wc) {
    const unsigned long long t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > wc.limit_ns) {
            record_status(wc.status, kStatusTimeout);
            return;
        }
    }
}

// Load 16 consecutive 32-bit columns of this warp's 32 TMEM lanes, then wait.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* r) {
    uint32_t* u = reinterpret_cast<uint32_t*>(r);
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7]),
          "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]), "=r"(u[14]), "=r"(u[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtl& wc, volatile int* abort) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, wc, abort));
}

// Per-head reduction of 16 values over the 32 lanes (max or sum).  A reduce-scatter halves
// the values a lane keeps at each level (16 shuffles in all); afterwards lanes 2m and 2m + 1
// both hold the result for head 8*b4 + 4*b3 + 2*b2 + b1, with b_k bit k of the lane index.
template <bool MAX>
__device__ __forceinline__ float head_reduce(const float (&x)[NH], int lane) {
    const bool b4 = (lane >> 4) & 1, b3 = (lane >> 3) & 1, b2 = (lane >> 2) & 1, b1 = (lane >> 1) & 1;
    float t8[8], t4[4], t2[2], t1;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float keep = b4 ? x[8 + i] : x[i], send = b4 ? x[i] : x[8 + i];
        const float o = __shfl_xor_sync(0xffffffffu, send, 16);
        t8[i] = MAX ? fmaxf(keep, o) : keep + o;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float keep = b3 ? t8[4 + i] : t8[i], send = b3 ? t8[i] : t8[4 + i];
        const float o = __shfl_xor_sync(0xffffffffu, send, 8);
        t4[i] = MAX ? fmaxf(keep, o) : keep + o;
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float keep = b2 ? t4[2 + i] : t4[i], send = b2 ? t4[i] : t4[2 + i];
        const float o = __shfl_xor_sync(0xffffffffu, send, 4);
        t2[i] = MAX ? fmaxf(keep, o) : keep + o;
    }
    {
        const float keep = b1 ? t2[1] : t2[0], send = b1 ? t2[0] : t2[1];
        const float o = __shfl_xor_sync(0xffffffffu, send, 2);
        t1 = MAX ? fmaxf(keep, o) : keep + o;
    }
    const float o = __shfl_xor_sync(0xffffffffu, t1, 1);
    return MAX ? fmaxf(t1, o) : t1 + o;
}

__device__ __forceinline__ int head_of_lane(int lane) {
    return 8 * ((lane >> 4) & 1) + 4 * ((lane >> 3) & 1) + 2 * ((lane >> 2) & 1) + ((lane >> 1) & 1);
}

template <int SRC>
__host__ __device__ constexpr bool has_gather() { return SRC == kSrcPaged; }

// Make a tensor map written through the generic proxy (by another kernel) visible to this
// thread's tensor-map-proxy reads.
__device__ __forceinline__ void tensormap_acquire(const CUtensorMap* map) {
    asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(reinterpret_cast<uint64_t>(map))
                 : "memory");
}

// One warp per map: map w is item w / 2's K (w even) or V (w odd) cache.  The warp stages the
// host-encoded template in shared memory, lane 0 patches the cache's address into it
// (tensormap.replace), and the warp copies it to global memory with a release of the
// tensor-map proxy.  A null or misaligned cache keeps the template's address: the decode reads
// nothing of such an item.
__global__ void __launch_bounds__(128) build_item_maps_kernel(const __grid_constant__ CUtensorMap tmpl,
                                                             const uint16_t* const* kc, const uint16_t* const* vc,
                                                             CUtensorMap* maps, int m) {
    __shared__ __align__(128) CUtensorMap staged[4];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int w = blockIdx.x * 4 + warp;
    if (w >= 2 * m) return;  // whole warps
    CUtensorMap* sm = staged + warp;
    const uint32_t sa = smem_u32(sm);
    if (lane < 16) reinterpret_cast<uint64_t*>(sm)[lane] = reinterpret_cast<const uint64_t*>(&tmpl)[lane];
    __syncwarp();
    if (lane == 0) {
        const uint16_t* base = (w & 1) ? vc[w >> 1] : kc[w >> 1];
        if (base != nullptr && (reinterpret_cast<uintptr_t>(base) & 15u) == 0)
            asm volatile("tensormap.replace.tile.global_address.shared::cta.b1024.b64 [%0], %1;" ::"r"(sa),
                         "l"(reinterpret_cast<uint64_t>(base))
                         : "memory");
    }
    __syncwarp();
    asm volatile(
        "tensormap.cp_fenceproxy.global.shared::cta.tensormap::generic.release.gpu.sync.aligned [%0], [%1], 128;" ::"l"(
            reinterpret_cast<uint64_t>(maps + w)),
        "r"(sa)
        : "memory");
}

template <int G, bool F16, int SRC>
__global__ void __launch_bounds__(has_gather<SRC>() ? kThreadsGather : kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     const DecodeTcParams p) {
    static_assert(G >= 1 && G <= NH, "group size");
    constexpr bool kGather = has_gather<SRC>();  // an instantiation with the gather producers
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + L::kOffBar;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kOffBar + 240);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffBar + 248);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x, nsplit = gridDim.x;
    const int hk = blockIdx.y, b = blockIdx.z;

    // The query's visible interval [lo, hi); this split's share [vbeg, vend), in 128-key blocks
    // from gbeg.  Block j's tile starts at position blk_start(j) and its keys that count are
    // [max(vbeg, gbeg + j BN), min(vend, gbeg + (j + 1) BN)).
    const int klen = valid_keys(p.key_lens, b, p.Lk);
    long long lo, hi;
    const uint16_t* kbase = nullptr;  // per-item caches: the item's K and V caches
    const uint16_t* vbase = nullptr;
    const int32_t* pages = nullptr;
    bool tma = true;  // copies by TMA (else, for page sizes TMA cannot copy, the gather producers)
    if constexpr (SRC == kSrcTma) {
        key_interval(p.mode, p.window, klen, p.P, p.P, &lo, &hi);
    } else {
        lo = (p.sliding > 0 && klen > p.sliding) ? (long long)(klen - p.sliding) : 0;
        hi = klen;
        bool bad = false;
        if constexpr (SRC == kSrcCaches) {
            kbase = p.kc[b];
            vbase = p.vc[b];
            const uintptr_t ka = reinterpret_cast<uintptr_t>(kbase), va = reinterpret_cast<uintptr_t>(vbase);
            bad = kbase == nullptr || vbase == nullptr || ((ka | va) & 15u) != 0;
        } else {
            // every CTA of the cluster checks all of the item's visible page entries, so they agree
            tma = p.paged_tma != 0;
            kbase = static_cast<const uint16_t*>(p.kpool);
            vbase = static_cast<const uint16_t*>(p.vpool);
            pages = p.page_table + (size_t)b * p.max_pages;
            if (hi > lo)
                for (long long x = lo / p.page_size + threadIdx.x; x <= (hi - 1) / p.page_size; x += blockDim.x) {
                    const int id = __ldg(pages + x);
                    bad |= (id < 0 || id >= p.num_pages);
                }
        }
        if (__syncthreads_or(bad)) {
            // nothing of the item is read and its output is zeros
            if (threadIdx.x == 0) record_status(p.wc.status, SRC == kSrcPaged ? kStatusBadPage : kStatusBadPointer);
            lo = hi = 0;
        }
    }
    if (hi < lo) hi = lo;
    // Blocks start on multiples of 128 positions (the positions before lo in the first block do
    // not count): page pieces then land on whole 8-row groups of the swizzled tiles, and every
    // source splits the keys the same way, so the contiguous, per-item and paged decodes of the
    // same cache compute the same numbers in the same order.
    const long long origin = (lo / BN) * BN;
    long long per = (hi - origin + nsplit - 1) / nsplit;
    per = (per + BN - 1) / BN * BN;
    const long long gbeg = origin + (long long)split * per;
    const long long vbeg = max(gbeg, lo);
    const long long vend = min(hi, gbeg + per);
    const int nblk = (vend > vbeg) ? (int)((vend - gbeg + BN - 1) / BN) : 0;
    auto blk_start = [&](int j) -> long long { return gbeg + (long long)j * BN; };
    // the same bounds as offsets from gbeg (all within [-BN, per], so 32-bit)
    const int vb_rel = (int)(vbeg - gbeg), ve_rel = (int)(vend - gbeg);
    const int lo_rel = (int)max(-(long long)BN, lo - gbeg), hi_rel = (int)min(per + BN, hi - gbeg);
    if (threadIdx.x == 0) {
        for (int i = 0; i < kNumBars; ++i) {
            uint32_t count = 1;
            if (i == kBarSFree || i == kBarSFree + 1 || i == kBarPFull || i == kBarXch || i == kBarXch + 1 ||
                i == kBarSum)
                count = 4;  // one arrival per softmax warp
            if (kGather && !tma && ((i >= kBarKFull && i < kBarKFull + kStages) || (i >= kBarVFull && i < kBarVFull + kStages)))
                count = 32;  // one arrival per lane of the stage's producer warp, after its copies landed
            mbar_init(bar0 + 8 * i, count);
        }
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp >= 2 && warp < 6) {
        // Q of the group's heads into a 16-row K-major tile (128-byte swizzle), zero rows past G;
        // 256 16-byte units, two per thread
        const int t = threadIdx.x - 64;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int ui = 2 * t + k;
            const int r = ui >> 4, u = ui & 15;  // row (head) and 16-byte unit of the row
            uint4 val = make_uint4(0u, 0u, 0u, 0u);
            if (r < G) val = *reinterpret_cast<const uint4*>(p.q + ((long long)b * p.Hq + (long long)hk * G + r) * D + 8 * u);
            const uint32_t addr = L::kOffQ + (u >> 3) * (NH * 128) + r * 128 + (((u & 7) ^ (r & 7)) << 4);
            *reinterpret_cast<uint4*>(smem + addr) = val;
        }
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), kTmemCols);
        tmem_relinquish();
    }
    if (tma && warp == 0 && lane == 0) {
        if constexpr (SRC == kSrcCaches) {
            // the item's maps were written by an earlier kernel through the generic proxy: acquire
            // them for the tensor-map proxy before the first copy reads them
            const CUtensorMap* maps = p.item_maps + 2 * b;
            tensormap_acquire(maps);
            tensormap_acquire(maps + 1);
            tma_prefetch_desc(maps);
            tma_prefetch_desc(maps + 1);
        } else {
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    float m_run[NH];    // per head, log2 domain (identical in every softmax thread)
    float l_part[NH];   // per head, this thread's share of the row sum
#pragma unroll
    for (int h = 0; h < NH; ++h) m_run[h] = -INFINITY, l_part[h] = 0.f;
    bool ok = true;

    if (warp >= 6 && tma) {
        // the two extra producer warps of a gather instantiation have nothing to copy when the
        // block's rows come by TMA
    } else if (kGather && !tma && (warp == 0 || warp >= 6)) {
        // ------------------------------------------------------------ gather producers
        // Three warps, one per ring stage (warp 0: stage 0, warps 6 and 7: stages 1 and 2), so
        // each stage is released as soon as its own copies have landed and all three are in
        // flight at once.  For a block the warp writes the byte offset of each of the 128 key
        // rows (or ~0 past the visible keys) to shared memory, then copies 2 rows per
        // instruction, 16 lanes per 256-byte row, each 16-byte unit to its swizzled place in
        // the K or V tile (the layout TMA gives); rows past the visible keys are zeros.  K is
        // released first (wait_group 1), then V; each lane waits for its own copies, fences
        // them for the tensor core and arrives.
        const int st = warp == 0 ? 0 : warp - 5;
        unsigned long long* rowoff = reinterpret_cast<unsigned long long*>(smem + L::kOffRow) + st * BN;
        const int half = lane >> 4, u = lane & 15, c = u >> 3, qd = u & 7;
        const char* kb = reinterpret_cast<const char*>(kbase);
        const char* vb = reinterpret_cast<const char*>(vbase);
        const uint32_t kt = sbase + L::kOffK + st * L::kKVBytes, vt = sbase + L::kOffV + st * L::kKVBytes;
        for (int j = st; j < nblk; j += kStages) {
            const uint32_t n = (uint32_t)(j / kStages);
            if (j >= kStages) {
                if (!warp_wait(bar0 + 8 * (kBarKEmpty + st), (n - 1) & 1, p.wc, abort_flag)) break;
                if (!warp_wait(bar0 + 8 * (kBarVEmpty + st), (n - 1) & 1, p.wc, abort_flag)) break;
            }
            const long long krow0 = gbeg + (long long)j * BN;
            __syncwarp();
            for (int r = lane; r < BN; r += 32) {
                const long long key = krow0 + r;
                unsigned long long off = ~0ull;
                if (key >= vbeg && key < vend) {  // the keys that count; other rows are zeros
                    const long long pg = __ldg(pages + key / p.page_size);
                    off = (((unsigned long long)pg * p.Hkv + hk) * (unsigned long long)p.page_size +
                           (unsigned long long)(key % p.page_size)) * (D * 2);
                }
                rowoff[r] = off;
            }
            __syncwarp();
#pragma unroll 2
            for (int kind = 0; kind < 2; ++kind) {  // K, then V
                const uint32_t tile = kind ? vt : kt;
                const char* src = kind ? vb : kb;
#pragma unroll 8
                for (int i = 0; i < BN / 2; ++i) {
                    const int r = 2 * i + half;
                    const unsigned long long off = rowoff[r];
                    const uint32_t dofs = c * (BN * 128) + r * 128 + ((qd ^ (r & 7)) << 4);
                    if (off != ~0ull) cp_async16(tile + dofs, src + off + u * 16);
                    else *reinterpret_cast<uint4*>(smem + (tile - sbase) + dofs) = make_uint4(0u, 0u, 0u, 0u);
                }
                cp_async_commit();
            }
            cp_async_wait<1>();  // this lane's K copies have landed
            fence_proxy_async_smem();
            mbar_arrive(bar0 + 8 * (kBarKFull + st));
            cp_async_wait<0>();  // and its V copies
            fence_proxy_async_smem();
            mbar_arrive(bar0 + 8 * (kBarVFull + st));
        }
        cp_async_wait<0>();  // nothing stays in flight, whatever happened above
    } else if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        // contiguous cache: one box per 64-column chunk at (chunk, position, b Hkv + hk); per-item
        // caches: the same boxes at (chunk, position, hk) through the item's own maps; paged:
        // one copy per page piece that holds visible keys (whole pages of at most 128 rows, or
        // 128 rows of a longer page), the pool map bounding every coordinate.  Lane 0 issues the
        // copies.
        if (nblk > 0) {
            const int kbh = SRC == kSrcTma ? b * p.Hkv + hk : hk;
            const CUtensorMap* map_k = SRC == kSrcCaches ? p.item_maps + 2 * b : &tmK;
            const CUtensorMap* map_v = SRC == kSrcCaches ? p.item_maps + 2 * b + 1 : &tmV;
            auto load = [&](const CUtensorMap* map, uint32_t tile, uint32_t bar, int j) {
                const long long s0 = blk_start(j);
                if constexpr (SRC == kSrcTma || SRC == kSrcCaches) {
                    mbar_arrive_expect_tx(bar, L::kKVBytes);
                    for (int c = 0; c < D / 64; ++c) tma_load_3d(tile + c * (BN * 128), map, bar, c * 64, (int)s0, kbh);
                } else {
                    const int ps = p.page_size;
                    if (ps >= BN) {  // one 128-row piece of a page
                        const int pg = __ldg(pages + s0 / ps);
                        mbar_arrive_expect_tx(bar, L::kKVBytes);
                        for (int c = 0; c < D / 64; ++c)
                            tma_load_3d(tile + c * (BN * 128), map, bar, c * 64, (int)(s0 % ps), pg * p.Hkv + hk);
                    }
                }
            };
            // paged with pages shorter than a block: whole pages of ps rows (ps divides 128, a
            // multiple of 8), lane i reading the page id of the block's i-th page with keys and
            // copying that page, after lane 0 has posted the bytes of them all
            auto load_pages = [&](const CUtensorMap* map, uint32_t tile, uint32_t bar, int j) {
                const int ps = p.page_size;
                const long long s0 = blk_start(j);
                const long long f = max(s0, lo) / ps, e = (min(s0 + BN, hi) - 1) / ps;  // pages with keys
                if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)((e - f + 1) * ps * (D * 2)));
                __syncwarp();
                for (long long x = f + lane; x <= e; x += 32) {
                    const int pg = __ldg(pages + x);
                    const uint32_t row = (uint32_t)(x * ps - s0);
                    for (int c = 0; c < D / 64; ++c)
                        tma_load_3d(tile + c * (BN * 128) + row * 128, map, bar, c * 64, 0, pg * p.Hkv + hk);
                }
            };
            const bool small_pages = SRC == kSrcPaged && p.page_size < BN;
            // the whole warp runs the loop for small pages, lane 0 alone otherwise
            int issued = 0;  // kept by lane 0
            if (small_pages || lane == 0) {
                auto wait = [&](uint32_t bar, uint32_t parity) {
                    return small_pages ? warp_wait(bar, parity, p.wc, abort_flag)
                                       : mbar_wait(bar, parity, p.wc, abort_flag);
                };
                for (int j = 0; j < nblk; ++j) {
                    const int s = j % kStages;
                    const uint32_t n = (uint32_t)(j / kStages);
                    const uint32_t kt = sbase + L::kOffK + s * L::kKVBytes, vt = sbase + L::kOffV + s * L::kKVBytes;
                    if (j >= kStages && !wait(bar0 + 8 * (kBarKEmpty + s), (n - 1) & 1)) break;
                    if (small_pages) load_pages(&tmK, kt, bar0 + 8 * (kBarKFull + s), j);
                    else load(map_k, kt, bar0 + 8 * (kBarKFull + s), j);
                    if (j >= kStages && !wait(bar0 + 8 * (kBarVEmpty + s), (n - 1) & 1)) {
                        issued = 2 * j + 1;
                        break;
                    }
                    if (small_pages) load_pages(&tmV, vt, bar0 + 8 * (kBarVFull + s), j);
                    else load(map_v, vt, bar0 + 8 * (kBarVFull + s), j);
                    issued = 2 * j + 2;
                }
            }
            if (lane == 0) {
                const int nk = (issued + 1) / 2, nv = issued / 2;
                for (int j = (nk > kStages ? nk - kStages : 0); j < nk; ++j)
                    drain_wait(bar0 + 8 * (kBarKFull + j % kStages), (uint32_t)(j / kStages) & 1, p.wc);
                for (int j = (nv > kStages ? nv - kStages : 0); j < nv; ++j)
                    drain_wait(bar0 + 8 * (kBarVFull + j % kStages), (uint32_t)(j / kStages) & 1, p.wc);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && nblk > 0) {
            constexpr uint32_t kIdescS = idesc_f16kind_f32(BN, NH, 0, 0, F16);  // M = keys, N = heads
            constexpr uint32_t kIdescO = idesc_f16kind_f32(D, NH, 1, 0, F16);   // M = dims (V^T, MN-major)
            bool mok = true;
            auto pv = [&](int i) -> bool {
                const int s = i % kStages;
                if (!mbar_wait(bar0 + 8 * (kBarVFull + s), (uint32_t)(i / kStages) & 1, p.wc, abort_flag)) return false;
                if (!mbar_wait(bar0 + 8 * kBarPFull, (uint32_t)i & 1, p.wc, abort_flag)) return false;
                tc_fence_after();
                const uint32_t vbase = sbase + L::kOffV + s * L::kKVBytes;
                const uint32_t pbase = sbase + L::kOffP;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    const uint64_t a = smem_desc_sw128(vbase + kk * (16 * 128), BN * 128, 1024);
                    const uint64_t bd = smem_desc_sw128(pbase + (kk >> 2) * (NH * 128) + (kk & 3) * 32, 16, 1024);
                    tc_mma_ss(tmem + kColO, a, bd, kIdescO, (i > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(bar0 + 8 * kBarPVDone);
                tc_commit(bar0 + 8 * (kBarVEmpty + s));
                return true;
            };
            for (int j = 0; mok && j < nblk; ++j) {
                const int s = j % kStages;
                if (!mbar_wait(bar0 + 8 * (kBarKFull + s), (uint32_t)(j / kStages) & 1, p.wc, abort_flag)) break;
                if (j >= 2 && !mbar_wait(bar0 + 8 * (kBarSFree + (j & 1)), (uint32_t)((j - 2) >> 1) & 1, p.wc,
                                         abort_flag))
                    break;
                tc_fence_after();
                const uint32_t kbase = sbase + L::kOffK + s * L::kKVBytes;
                const uint32_t qbase = sbase + L::kOffQ;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint64_t a = smem_desc_sw128(kbase + (ks >> 2) * (BN * 128) + (ks & 3) * 32, 16, 1024);
                    const uint64_t bd = smem_desc_sw128(qbase + (ks >> 2) * (NH * 128) + (ks & 3) * 32, 16, 1024);
                    tc_mma_ss(tmem + kColS + NH * (j & 1), a, bd, kIdescS, ks > 0 ? 1u : 0u);
                }
                tc_commit(bar0 + 8 * (kBarSFull + (j & 1)));
                tc_commit(bar0 + 8 * (kBarKEmpty + s));
                if (j >= 1) mok = pv(j - 1);
            }
            if (mok) pv(nblk - 1);
            tc_commit(bar0 + 8 * kBarMmaDone);
            drain_wait(bar0 + 8 * kBarMmaDone, 0, p.wc);
        }
    } else {
        // ------------------------------------------------------------ softmax: one key per thread
        const int sw = warp - 2;                     // softmax warp 0..3
        const int key = 32 * (warp & 3) + lane;      // my TMEM lane: key of the block, later head dim
        const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        const float sl = p.scale_log2;
        float* xch = reinterpret_cast<float*>(smem + L::kOffX);
        uint8_t* pt = smem + L::kOffP;
        // where my key's 16 probabilities go in P^T: chunk, byte in the swizzled row
        const int kc = key >> 6, ku = (key & 63) >> 3, kb = (key & 7) * 2;
        const int my_head = head_of_lane(lane);

        for (int j = 0; j < nblk; ++j) {
            const int par = j & 1;
            if (!warp_wait(bar0 + 8 * (kBarSFull + par), (uint32_t)(j >> 1) & 1, p.wc, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float s[NH];
            tmem_ld16(tmem + lane_off + kColS + NH * par, s);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar0 + 8 * (kBarSFree + par));

            // scores in the log2 domain; keys that do not count in this block and padding heads are -inf
            // (offsets from gbeg: block j holds rel = j BN + key, and the split counts [vb_rel, ve_rel))
            const int rel = j * BN + key;
            const bool vis = rel >= vb_rel && rel < ve_rel;
            float x[NH];
#pragma unroll
            for (int h = 0; h < NH; ++h) x[h] = (vis && h < G) ? s[h] * sl : -INFINITY;
            // per-head block maxima: warp reduce-scatter, then the four warps through shared memory
            const float wmax = head_reduce<true>(x, lane);
            if ((lane & 1) == 0) xch[(par * 4 + sw) * NH + my_head] = wmax;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar0 + 8 * (kBarXch + par));
            if (!warp_wait(bar0 + 8 * (kBarXch + par), (uint32_t)(j >> 1) & 1, p.wc, abort_flag)) {
                ok = false;
                break;
            }
            float alpha[NH];
            bool rescale = false;
#pragma unroll
            for (int h = 0; h < NH; ++h) {
                const float bm = fmaxf(fmaxf(xch[(par * 4 + 0) * NH + h], xch[(par * 4 + 1) * NH + h]),
                                       fmaxf(xch[(par * 4 + 2) * NH + h], xch[(par * 4 + 3) * NH + h]));
                alpha[h] = 1.f;
                if (bm != -INFINITY) {
                    if (m_run[h] == -INFINITY) {
                        m_run[h] = bm;
                    } else if (bm > m_run[h] + kRescaleThreshold) {
                        alpha[h] = ex2_approx(m_run[h] - bm);
                        m_run[h] = bm;
                        rescale = true;
                    }
                }
            }
            // the previous P V product must be done before P^T and O^T are touched
            if (j > 0 && !warp_wait(bar0 + 8 * kBarPVDone, (uint32_t)(j - 1) & 1, p.wc, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int h = 0; h < NH; ++h) {
                const float pr = (x[h] == -INFINITY) ? 0.f : ex2_approx(x[h] - m_run[h]);
                const uint32_t w = pack2<F16>(pr, 0.f);
                *reinterpret_cast<uint16_t*>(pt + kc * (NH * 128) + h * 128 + ((ku ^ (h & 7)) << 4) + kb) =
                    (uint16_t)(w & 0xffffu);
                l_part[h] = l_part[h] * alpha[h] + unpack2<F16>(w & 0xffffu).x;
            }
            if (rescale) {  // identical in every thread: O^T columns of grown heads scale by alpha
                float o[NH];
                tmem_ld16(tmem + lane_off + kColO, o);
#pragma unroll
                for (int h = 0; h < NH; ++h) o[h] *= alpha[h];
                tmem_st16(tmem + lane_off + kColO, reinterpret_cast<const uint32_t*>(o));
            }
            // A V tile row that the query does not see gets weight 0, but the tensor core multiplies
            // that 0 into the row, and 0 * Inf or 0 * NaN is NaN: in a block whose tile reaches
            // outside [lo, hi) (the first or last), once the tile has landed each thread zeroes its
            // row if it lies outside (the gather writes such rows as zeros already).
            if (tma && (j * BN < lo_rel || (j + 1) * BN > hi_rel)) {
                const int s = j % kStages;
                if (!warp_wait(bar0 + 8 * (kBarVFull + s), (uint32_t)(j / kStages) & 1, p.wc, abort_flag)) {
                    ok = false;
                    break;
                }
                if (rel < lo_rel || rel >= hi_rel) {
                    uint8_t* vrow = smem + L::kOffV + s * L::kKVBytes + key * 128;
#pragma unroll
                    for (int c = 0; c < D / 64; ++c)
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            *reinterpret_cast<uint4*>(vrow + c * (BN * 128) + q * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            fence_proxy_async_smem();  // P^T (and zeroed V rows) are read by the tensor core (async proxy)
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar0 + 8 * kBarPFull);
        }

        // ------------------------------------------------------------ epilogue: this split's partial
        if (ok && nblk > 0) {
            ok = warp_wait(bar0 + 8 * kBarPVDone, (uint32_t)(nblk - 1) & 1, p.wc, abort_flag);
            tc_fence_after();
        }
        // row sums over the 128 keys: warp reduce-scatter, then the four warps
        const float wsum = head_reduce<false>(l_part, lane);
        float* sums = reinterpret_cast<float*>(smem + L::kOffS);
        if ((lane & 1) == 0) sums[sw * NH + my_head] = wsum;
        __syncwarp();
        if (lane == 0) mbar_arrive(bar0 + 8 * kBarSum);
        if (ok) ok = warp_wait(bar0 + 8 * kBarSum, 0, p.wc, abort_flag);
        float o[NH];
        if (ok && nblk > 0) {
            tmem_ld16(tmem + lane_off + kColO, o);
        } else {
#pragma unroll
            for (int h = 0; h < NH; ++h) o[h] = 0.f;
        }
        // the partial (m, l, O) of this split into the (now free) K ring, for the combine
        float* cm = reinterpret_cast<float*>(smem + L::kOffCm);
        float* cl = reinterpret_cast<float*>(smem + L::kOffCl);
        float* co = reinterpret_cast<float*>(smem + L::kOffCo);
        if (threadIdx.x == 64) {
#pragma unroll
            for (int h = 0; h < NH; ++h) {
                const bool has = ok && nblk > 0;
                cm[h] = has ? m_run[h] : -INFINITY;
                cl[h] = has ? sums[0 * NH + h] + sums[1 * NH + h] + sums[2 * NH + h] + sums[3 * NH + h] : 0.f;
            }
        }
#pragma unroll
        for (int h = 0; h < G; ++h) co[h * D + key] = o[h];
    }

    // ---------------------------------------------------------------- combine the splits in rank 0
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    if (split == 0 && warp >= 2 && warp < 6) {
        const int dim = 32 * (warp & 3) + lane;
        for (int h = 0; h < G; ++h) {
            float ms[kMaxSplits], ls[kMaxSplits], os[kMaxSplits];
            float mc = -INFINITY;
            for (int r = 0; r < nsplit; ++r) {
                uint32_t a_m, a_l, a_o;
                asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a_m) : "r"(sbase + L::kOffCm + 4 * h), "r"(r));
                asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a_l) : "r"(sbase + L::kOffCl + 4 * h), "r"(r));
                asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a_o)
                             : "r"(sbase + L::kOffCo + 4 * (h * D + dim)), "r"(r));
                asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(ms[r]) : "r"(a_m) : "memory");
                asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(ls[r]) : "r"(a_l) : "memory");
                asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(os[r]) : "r"(a_o) : "memory");
                mc = fmaxf(mc, ms[r]);
            }
            float acc = 0.f, l = 0.f;
            if (mc != -INFINITY) {
                for (int r = 0; r < nsplit; ++r) {
                    const float f = (ms[r] == -INFINITY) ? 0.f : ex2_approx(ms[r] - mc);
                    acc += f * os[r];
                    l += f * ls[r];
                }
            }
            const float res = (l > 0.f) ? acc / l : 0.f;
            const long long oi = ((long long)b * p.Hq + (long long)hk * G + h) * D + dim;
            p.out[oi] = (uint16_t)(pack2<F16>(res, 0.f) & 0xffffu);
        }
    }
    // keep every CTA's shared memory alive until rank 0 has read it
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");

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

// [outer, L, 128] 16-bit tensor as 3-D (128, L, outer); box 64 x rows x 1, 128-byte swizzle, zero
// fill for coordinates outside the tensor.
bool encode_kv(CUtensorMap* map, const void* base, unsigned long long L, unsigned long long outer, int rows, bool f16) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)L, (cuuint64_t)outer};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)L * D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base),
              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int G, bool F16, int SRC>
cudaError_t launch_g(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeTcParams& p, int items, int nsplit,
                     cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::mutex mu;
    static bool configured[64] = {};
    {
        std::lock_guard<std::mutex> g(mu);
        if (dev < 64 && !configured[dev]) {
            e = cudaFuncSetAttribute(decode_tc_kernel<G, F16, SRC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     L::kSmem);
            if (e != cudaSuccess) return e;
            configured[dev] = true;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)nsplit, (unsigned)p.Hkv, (unsigned)items);
    cfg.blockDim = dim3(has_gather<SRC>() ? kThreadsGather : kThreads, 1, 1);
    cfg.dynamicSmemBytes = L::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)nsplit;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_tc_kernel<G, F16, SRC>, tk, tv, p);
}

template <int SRC>
cudaError_t launch_src(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeTcParams& p, int G, bool f16,
                       int items, int nsplit, cudaStream_t stream) {
    if (G == 4) return f16 ? launch_g<4, true, SRC>(tk, tv, p, items, nsplit, stream)
                           : launch_g<4, false, SRC>(tk, tv, p, items, nsplit, stream);
    if (G == 8) return f16 ? launch_g<8, true, SRC>(tk, tv, p, items, nsplit, stream)
                           : launch_g<8, false, SRC>(tk, tv, p, items, nsplit, stream);
    return cudaErrorInvalidValue;
}

// One CTA per SM.  Measured on GB300 (batch 4-64, 2048-8192 keys): the best split count
// reaches about 0.84 CTAs per SM (128 on 152 SMs) and no more; clusters of 8 of these
// 200-KB CTAs schedule poorly (twice slower than 4 at batch 4), and a split should cover at
// least 1024 keys.
int choose_splits(long long units, long long keys, int num_sms) {
    constexpr int kMaxUsedSplits = 4;
    const long long target = num_sms > 0 ? (27LL * num_sms) / 32 : 128;
    int n = 1;
    while (n < kMaxUsedSplits && units * n < target) n *= 2;
    return (int)std::max(1LL, std::min<long long>(n, std::max(1LL, keys / 1024)));
}

DecodeTcParams base_params(const void* q, void* out, const int32_t* lens, int Hq, int Hkv, int Lk, float scale,
                           const WaitCtl& wc) {
    DecodeTcParams p = {};
    p.q = static_cast<const uint16_t*>(q);
    p.out = static_cast<uint16_t*>(out);
    p.key_lens = lens;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.Lk = Lk;
    p.scale_log2 = scale * kLog2e;
    p.wc = wc;
    return p;
}

}  // namespace

bool decode_tc_supported(const Problem& p) {
    if (p.Lq != 1 || p.D != 128) return false;
    const int G = p.Hq / p.Hkv;
    return G == 4 || G == 8;
}

bool decode_tc_items_supported(int Hq, int Hkv, int D) {
    if (D != 128 || Hkv <= 0 || Hq % Hkv != 0) return false;
    const int G = Hq / Hkv;
    return G == 4 || G == 8;
}

bool decode_tc_paged_tma(int page_size, int num_pages, int Hkv) {
    return ((page_size >= 8 && page_size <= BN && BN % page_size == 0) || page_size % BN == 0) &&
           (long long)num_pages * Hkv <= 0x7fffffffLL;
}

cudaError_t launch_decode_tc(const Problem& pr, const WaitCtl& wc, cudaStream_t stream, int num_sms) {
    if (pr.Hkv > 65535 || pr.B > 65535) return cudaErrorInvalidConfiguration;
    DecodeTcParams p = base_params(pr.q, pr.out, pr.key_lens, pr.Hq, pr.Hkv, pr.Lk, pr.scale, wc);
    p.P = pr.pos_offset;
    p.mode = pr.mode;
    p.window = pr.window;
    CUtensorMap tk, tv;
    if (!encode_kv(&tk, pr.k, pr.Lk, (unsigned long long)pr.B * pr.Hkv, BN, pr.f16) ||
        !encode_kv(&tv, pr.v, pr.Lk, (unsigned long long)pr.B * pr.Hkv, BN, pr.f16))
        return cudaErrorInvalidValue;
    const int nsplit = choose_splits((long long)pr.B * pr.Hkv, pr.Lk, num_sms);
    return launch_src<kSrcTma>(tk, tv, p, pr.Hq / pr.Hkv, pr.f16, pr.B, nsplit, stream);
}

namespace {

// The caches' addresses are known only on the device, so a template map of one item's
// [Hkv, capacity, 128] cache is encoded on the host (its address a placeholder: q, 16-byte
// aligned) and a kernel writes each item's K and V maps, with the real addresses, into `maps`
// ([m][2], 128-byte aligned) before the decode reads them.
cudaError_t decode_caches_with_maps(const CachesProblem& cp, const WaitCtl& wc, cudaStream_t stream, int num_sms,
                                    const CUtensorMap& tmpl, CUtensorMap* maps) {
    DecodeTcParams p = base_params(cp.q, cp.out, cp.kv_lens, cp.Hq, cp.Hkv, cp.capacity, cp.scale, wc);
    p.sliding = cp.sliding;
    p.kc = reinterpret_cast<const uint16_t* const*>(cp.k_caches);
    p.vc = reinterpret_cast<const uint16_t* const*>(cp.v_caches);
    const long long span = cp.sliding > 0 ? std::min(cp.sliding, cp.capacity) : cp.capacity;
    const int nsplit = choose_splits((long long)cp.m * cp.Hkv, span, num_sms);
    build_item_maps_kernel<<<(unsigned)((2 * cp.m + 3) / 4), 128, 0, stream>>>(tmpl, p.kc, p.vc, maps, cp.m);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    p.item_maps = maps;
    return launch_src<kSrcCaches>(tmpl, tmpl, p, cp.Hq / cp.Hkv, cp.f16, cp.m, nsplit, stream);
}

}  // namespace

// The fixed map table of attn_decode_caches_noalloc: room for kStaticMapItems items (1 MB).
// Calls that overlap on the GPU share it, so they race.
static __device__ __align__(256) CUtensorMap g_static_item_maps[2 * kStaticMapItems];

cudaError_t launch_decode_tc_caches(const CachesProblem& cp, const WaitCtl& wc, cudaStream_t stream, int num_sms) {
    if (cp.Hkv > 65535 || cp.m > 65535) return cudaErrorInvalidConfiguration;
    CUtensorMap tmpl;
    if (!encode_kv(&tmpl, cp.q, cp.capacity, cp.Hkv, BN, cp.f16)) return cudaErrorInvalidValue;
    // the maps live in a stream-ordered workspace, freed in stream order after the decode
    void* ws = nullptr;
    cudaError_t e = cudaMallocAsync(&ws, (size_t)cp.m * 2 * sizeof(CUtensorMap), stream);
    if (e != cudaSuccess) return e;
    if ((reinterpret_cast<uintptr_t>(ws) & 127u) != 0) {  // a tensor map in global memory is 128-byte aligned
        cudaFreeAsync(ws, stream);
        return cudaErrorMisalignedAddress;
    }
    e = decode_caches_with_maps(cp, wc, stream, num_sms, tmpl, static_cast<CUtensorMap*>(ws));
    const cudaError_t ef = cudaFreeAsync(ws, stream);
    return e != cudaSuccess ? e : ef;
}

cudaError_t launch_decode_tc_caches_static(const CachesProblem& cp, const WaitCtl& wc, cudaStream_t stream,
                                           int num_sms) {
    if (cp.Hkv > 65535 || cp.m > kStaticMapItems) return cudaErrorInvalidConfiguration;
    CUtensorMap tmpl;
    if (!encode_kv(&tmpl, cp.q, cp.capacity, cp.Hkv, BN, cp.f16)) return cudaErrorInvalidValue;
    // the table's address, looked up once per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    static std::mutex mu;
    static CUtensorMap* table[64] = {};
    CUtensorMap* maps = nullptr;
    {
        std::lock_guard<std::mutex> g(mu);
        if (table[dev] == nullptr) {
            void* a = nullptr;
            e = cudaGetSymbolAddress(&a, g_static_item_maps);
            if (e != cudaSuccess) return e;
            if ((reinterpret_cast<uintptr_t>(a) & 127u) != 0) return cudaErrorMisalignedAddress;
            table[dev] = static_cast<CUtensorMap*>(a);
        }
        maps = table[dev];
    }
    // nothing in the table has to start at zero: the kernel writes every map an item uses
    // before the decode reads it
    return decode_caches_with_maps(cp, wc, stream, num_sms, tmpl, maps);
}

cudaError_t launch_decode_tc_paged(const PagedProblem& pp, const WaitCtl& wc, cudaStream_t stream, int num_sms) {
    if (pp.Hkv > 65535 || pp.m > 65535) return cudaErrorInvalidConfiguration;
    const int cap = pp.page_size * pp.max_pages;  // an item's capacity: kv_lens clamp to it
    DecodeTcParams p = base_params(pp.q, pp.out, pp.kv_lens, pp.Hq, pp.Hkv, cap, pp.scale, wc);
    p.sliding = pp.sliding;
    p.kpool = static_cast<const uint16_t*>(pp.k_pool);
    p.vpool = static_cast<const uint16_t*>(pp.v_pool);
    p.page_table = pp.page_table;
    p.page_size = pp.page_size;
    p.max_pages = pp.max_pages;
    p.num_pages = pp.num_pages;
    // TMA copies whole pages of 8 to 128 rows that divide a 128-key block, or 128-row pieces of
    // pages that are multiples of 128 rows, through the pools seen as [num_pages * Hkv,
    // page_size, 128]; other page sizes are gathered row by row
    const int ps = pp.page_size;
    p.paged_tma = (((ps >= 8 && ps <= BN && BN % ps == 0) || ps % BN == 0) &&
                   (long long)pp.num_pages * pp.Hkv <= 0x7fffffffLL) ? 1 : 0;
    CUtensorMap tk = {}, tv = {};
    if (p.paged_tma) {
        const int rows = std::min(ps, BN);
        if (!encode_kv(&tk, pp.k_pool, ps, (unsigned long long)pp.num_pages * pp.Hkv, rows, pp.f16) ||
            !encode_kv(&tv, pp.v_pool, ps, (unsigned long long)pp.num_pages * pp.Hkv, rows, pp.f16))
            return cudaErrorInvalidValue;
    }
    const long long span = pp.sliding > 0 ? std::min(pp.sliding, cap) : cap;
    const int nsplit = choose_splits((long long)pp.m * pp.Hkv, span + BN, num_sms);
    return launch_src<kSrcPaged>(tk, tv, p, pp.Hq / pp.Hkv, pp.f16, pp.m, nsplit, stream);
}

}  // namespace attn
