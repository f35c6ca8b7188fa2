// prefill_tc.cu -- K1: fused attention prefill on the 5th-generation tensor cores (sm_103a),
// bf16 or fp16 inputs and outputs, fp32 accumulation.
//
// One CTA computes NT 128-row query tiles (NT = 2 for head_dim 128, NT = 1 for
// head_dim 64), sharing every K and V tile between them.  With two tiles and an even number
// of query heads per kv head, the tiles are two query heads of one kv group over the same
// rows (both visit exactly the same key tiles, so neither idles at the end); otherwise they
// are two consecutive row blocks of one (batch, query head).
//   warp 0       TMA producer: the Q tiles once, then 128-key K and V tiles
//                through 2-stage shared-memory rings (128-byte swizzle); over paged
//                caches one copy per page piece, or a row gather for other page sizes.
//   warp 1       TMEM owner and single-thread MMA issuer.
//   warps 2..    softmax, 8 warps per query tile: a row of S is split between two
//                threads, one per half of the 128 key columns.  Each thread reads its 64
//                scores from TMEM, the two halves exchange their row maxima through
//                shared memory at a named barrier of the tile's 8 warps (hardware, no
//                polling), and each writes its 64 probabilities (2^x on the
//                special-function unit, scale*log2(e) folded in) back into TMEM as
//                packed 16-bit pairs (the input type: bf16 or fp16).  After the tile's
//                last key block each half normalises and stores its half of the head
//                dims of the row (head-major, token-major or packed rows).
// With one tile per CTA (head_dim 64, two CTAs per SM), thread 0 issues the Q copy and the
// first K/V copies before the CTA barrier, and a softmax warp whose 32 rows see none of its
// 64 key columns skips the mask, the max and the exponentials (it writes zero P).
// TMEM: S_0 .. S_{NT-1} | O_0 .. O_{NT-1}, 128 columns each; P_t aliases the first 64
// columns of S_t.  With two tiles the MMA order is the ping-pong
//   PV0(j-1), QK0(j), PV1(j-1), QK1(j)
// so the tensor core works on one tile while the other tile's softmax runs; with one
// tile per CTA the two CTAs resident on an SM take turns in the same way.  Each tile's P
// is released in two parts, so the first half of PV_t(j) runs while the softmax packs
// the rest.
//   QK_t(j):  S_t  = Q_t K_j^T   (A, B from shared memory, K-major)
//   PV_t(j):  O_t += P_t V_j     (A = P from TMEM, B = V from shared memory, MN-major)
// A commit after QK_t(j) completes only after every earlier MMA, PV_t(j-1)
// included, so when the softmax sees S_t(j) it may also rescale O_t and
// overwrite P_t.  O is rescaled only when the row max grows by more than 2^8.
// Each query tile visits only the key tiles that intersect its visible band.
//
// What is computed follows ferrum-kernels Backend::flash_attention, ripvec-core
// Driver::fused_scale_mask_softmax (softmax(scores*scale + mask)) and the
// realizar cached/attention.rs causal softmax (a fully masked row gives zeros).
#include "kernels.h"

#include <algorithm>
#include <mutex>

namespace attn {
namespace {

constexpr int BM = 128;           // query rows per tile
constexpr int BN = 128;           // keys per tile
// NT query tiles per CTA (1 or 2); 2 + 8 NT warps: producer, MMA, 8 softmax warps per tile
template <int NT>
constexpr int threads_for() { return 64 + 256 * NT; }
constexpr int kStages = 2;        // K/V ring depth
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;

template <int D, int NT>
struct Cfg {
    static constexpr int kTiles = NT;
    static constexpr int kChunks = D / 64;
    static constexpr int kQBytes = BM * D * 2;   // one query tile
    static constexpr int kKVBytes = BN * D * 2;  // one K or V tile
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kTiles * kQBytes;
    static constexpr int kOffV = kOffK + kStages * kKVBytes;
    static constexpr int kOffX = kOffV + kStages * kKVBytes;          // row-extreme exchange
    static constexpr int kOffL = kOffX + kTiles * 2 * BM * 4;         // row-sum exchange
    static constexpr int kOffRow = kOffL + kTiles * 2 * BM * 4;        // paged: byte offset of each key row
    static constexpr int kOffBar = kOffRow + BN * 8;
    static constexpr int kSmem = kOffBar + 256 + 1024;
    static constexpr uint32_t kTmemCols = NT == 2 ? 512 : 256;
    static constexpr uint32_t kColS = 0;    // + 128 * tile
    static constexpr uint32_t kColO = 128 * NT;  // + 128 * tile
};

constexpr int kTiles = 2;  // barrier slots are laid out for the larger configuration
enum : int {
    kBarQFull = 0,
    kBarKFull = 1,
    kBarVFull = kBarKFull + kStages,
    kBarKEmpty = kBarVFull + kStages,
    kBarVEmpty = kBarKEmpty + kStages,
    kBarSFull = kBarVEmpty + kStages,  // + tile
    kBarPFull = kBarSFull + kTiles,    // + tile
    kBarOFull = kBarPFull + kTiles,    // + tile: the tile's last P V product completed
    kBarMmaDone = kBarOFull + kTiles,
    kBarVLand = kBarMmaDone + 1,       // the tail V tile's copy, before its invisible rows are zeroed
    kBarPHalf = kBarVLand + 1,         // + tile: the first 32 keys of both halves of P are in TMEM
    kNumBars = kBarPHalf + kTiles,
};
static_assert(kNumBars * 8 <= 240, "barrier area");

// Where Q, K, V and out live.
enum : int {
    kHeadMajor = 0,  // q/out [B, Hq, Lq, D], k/v [B, Hkv, Lk, D]: TMA
    kPacked = 1,     // packed sequences, token-major q/out [total, Hq, D] and k/v [total, Hkv, D]: TMA
    kPaged = 2,      // packed token-major q/out, K/V in paged pools: Q by TMA, K/V by TMA per page
                     // piece where the page size allows it, else rows gathered
};

struct PrefillParams {
    __nv_bfloat16* out;
    const int32_t* key_lens;
    int B, Hq, Hkv, Lq, Lk, P, mode, window;
    int num_m;          // query blocks (NT tiles each) per head
    const int32_t* cu_seqlens;  // packed token-major sequences [B + 1], or null (head-major batch)
    int total;          // packed rows (token-major)
    int out_tok;        // head-major batch: out is [B, Lq, Hq, D] instead of [B, Hq, Lq, D]
    int tma_out;        // head-major out [B, Hq, Lq, 128]: tiles stored by TMA from shared memory
    float scale_log2;
    WaitCtl wc;
    // kPaged: pools [num_pages, Hkv, page_size, D]; sequence b's position j is row j % page_size of
    // pool page page_table[b * max_pages + j / page_size]; kv_lens[b] positions are cached and the
    // sequence's queries are its newest positions
    const uint8_t* kpool;
    const uint8_t* vpool;
    const int32_t* page_table;
    const int32_t* kv_lens;
    int page_size, max_pages, num_pages;
    // kPaged with a page size TMA can place (8 to 128 rows dividing 128, or a multiple of 128):
    // K/V copied by TMA a page piece at a time through maps of the pools, key tiles starting on
    // multiples of 128 positions
    int paged_tma;
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


// Load 64 consecutive fp32 columns (two 32-column loads, one wait).
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float* r) {
    uint32_t* u = reinterpret_cast<uint32_t*>(r);
    tmem_ld32_async(taddr, u);
    tmem_ld32_async(taddr + 32, u + 32);
    tmem_ld_wait32(u);
    tmem_ld_wait32(u + 32);
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

// Key tiles of one query tile: [jb, je) in units of BN keys from kv0.
struct TileRange {
    int jb, je;
};

// The 8 softmax warps of query tile t meet at named barrier 1 + t.
__device__ __forceinline__ void tile_bar_sync(int t) {
    if (t == 0) named_bar_sync<1, 256>();
    else named_bar_sync<2, 256>();
}

// One key block of a query tile's softmax, for one thread: half a row of S (64 scores at
// TMEM columns 64h of tS), the row extreme exchanged with the other half through xch at the
// tile's named barrier (every warp of the tile meets it once per block on every path, so it
// cannot hang; a thread that gave up, !ok, stops right after it), P for the 64 keys written to
// columns [32h, 32h + 32) of tS in two parts (the first released on bar_phalf, all of it on
// bar_pfull), the running maximum and sum updated and O rescaled in TMEM when the maximum
// jumps.  MAYSKIP: a warp whose rows see none of its keys writes zeros without exponentials.
template <int D, bool F16, bool POS, bool MAYSKIP>
__device__ __forceinline__ void softmax_block(uint32_t tS, uint32_t tO, int h, int row, int lane, int t, float sl,
                                              int rlo_rel, int rhi_rel, int j, float* xch, bool ok, float& m_run,
                                              float& l_run, uint32_t bar_phalf, uint32_t bar_pfull) {
    const int c_lo = min(max(rlo_rel - j * BN, 0), 64);  // my visible columns [c_lo, c_hi)
    const int c_hi = min(max(rhi_rel - j * BN, 0), 64);
    const bool full = (c_lo == 0 && c_hi == 64);
    // every row of my warp sees none of my 64 keys (a band edge on a 32-row boundary):
    // no max and no exponentials, just zeros for my half of P.  Only with one tile per
    // CTA (head_dim 64): there every window key tile has such warps, while at two tiles
    // only diagonal tiles do and the test costs more than it saves.
    const bool skip = MAYSKIP && __all_sync(0xffffffffu, c_lo >= c_hi);

    // My 64 scores stay in registers for both passes: the other half writes P into
    // columns 32..63 after the exchange below, so nothing is read back from TMEM.
    // (after a give-up the load below reads allocated but stale columns; nothing uses them)
    float s[64];
    tmem_ld64(tS + 64 * h, s);
    float hext;
    if (skip) {
        hext = (POS || sl >= 0.f) ? -INFINITY : INFINITY;
    } else if (POS || sl >= 0.f) {
        if (!full) {
            mask_scores64(s, range_bits64(c_lo, c_hi), -INFINITY);
        }
        hext = row_max64(s);
    } else {
        if (!full) {
            mask_scores64(s, range_bits64(c_lo, c_hi), INFINITY);
        }
        hext = row_min64(s);
    }
    // exchange the half extremes of each row between the two halves of the tile; every
    // warp of the tile meets this barrier once per key block on every path, so it
    // cannot hang (the order of S_t(j+1) after every P_t(j) keeps the slots from
    // being overwritten before the partner has read them)
    xch[h * BM + row] = hext;
    tile_bar_sync(t);
    if (!ok) return;
    const float oext = xch[(1 - h) * BM + row];
    const float ext = (POS || sl >= 0.f) ? fmaxf(hext, oext) : fminf(hext, oext);
    const bool any = (POS || sl >= 0.f) ? (ext != -INFINITY) : (ext != INFINITY);

    float alpha = 1.f;
    bool rescale = false;
    if (any) {
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

    // The product over this block's P starts once every warp of the tile has released the
    // first 32 of its keys; a warp that must rescale O first (rare) releases them only
    // after the rescale below, with the rest.
    const bool warp_rescale = __any_sync(0xffffffffu, rescale);
    auto release_first_part = [&]() {
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_phalf);
    };
    // P for my 64 keys -> TMEM columns [32h, 32h + 32) of S_t, as bf16 or fp16 pairs; the row
    // sum adds the rounded values the tensor core will multiply into V.
    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
    if (skip) {
        uint32_t z[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) z[q] = 0u;
        tmem_st16_async(tS + 32 * h, z);
        if (!warp_rescale) release_first_part();
        tmem_st16_async(tS + 32 * h + 16, z);
    } else {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        uint32_t pk[16];
#pragma unroll
        for (int c2 = 0; c2 < 32; c2 += 2) {
            const int c = 32 * k + c2;
            const float2 x2 = __ffma2_rn(make_float2(s[c], s[c + 1]), sl2, negm2);
            float p0 = ex2_approx(x2.x);  // special-function unit; 2^-inf = 0
            float p1 = ex2_approx(x2.y);
            // Masked scores hold -inf (or +inf with a negative scale), so their
            // 2^(s*scale*log2e - m) is already exactly 0; only scale 0 turns them
            // into NaN (inf * 0) and needs the explicit zero.
            if (!POS && !full && sl == 0.f) {
                p0 = (c >= c_lo && c < c_hi) ? p0 : 0.f;
                p1 = (c + 1 >= c_lo && c + 1 < c_hi) ? p1 : 0.f;
            }
            const uint32_t wv = pack2<F16>(p0, p1);
            pk[c2 / 2] = wv;
            const float2 r2 = unpack2<F16>(wv);
            if ((c2 / 2) & 1) acc1 = __fadd2_rn(acc1, r2); else acc0 = __fadd2_rn(acc0, r2);
        }
        tmem_st16_async(tS + 32 * h + 16 * k, pk);
        if (k == 0 && !warp_rescale) release_first_part();
    }
    }
    tmem_st_wait();
    acc0 = __fadd2_rn(acc0, acc1);
    l_run = l_run * alpha + (acc0.x + acc0.y);
    // O_t is stable here: the commit behind S_t(j) covers the earlier P V product, and
    // this block's has not started (this warp has released nothing yet).
    if (warp_rescale) {
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
            float o[32];
            tmem_ld32(tO + (D / 2) * h + 32 * c, o);
#pragma unroll
            for (int q = 0; q < 32; ++q) o[q] *= alpha;
            tmem_st32(tO + (D / 2) * h + 32 * c, o);
        }
        release_first_part();
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_pfull);
}

// PAIR (two tiles, even group size): the tiles are two query heads of one kv group over the
// same 128 query rows, so both visit exactly the same key tiles.  Otherwise the tiles are two
// consecutive 128-row blocks of one query head.
// ZT: some query block may need rows of its last V tile zeroed (the host clears it when it can show
// that none does; the code is then left out, which the heaviest workloads measurably prefer).
// POS: the scale is positive (known on the host), so the minimum path for negative scales and the
// explicit zeroing for scale 0 are left out of the softmax.
template <int D, int NT, bool F16, int LAYOUT, bool PAIR, bool ZT, bool POS>
__global__ void __launch_bounds__(threads_for<NT>(), 3 - NT)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                      const PrefillParams p) {
    using C = Cfg<D, NT>;
    constexpr int kTiles = NT;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + C::kOffBar;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffBar + 240);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffBar + 248);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    constexpr bool TOK = LAYOUT != kHeadMajor;  // packed token-major q/out
    constexpr bool PAGED = LAYOUT == kPaged;

    int idx = blockIdx.x;
    const int nh = PAIR ? p.Hq / 2 : p.Hq;
    const int hq = (idx % nh) * (PAIR ? 2 : 1);  // query head of tile 0
    idx /= nh;
    const int b = idx % p.B;
    idx /= p.B;
    const int mblk = p.num_m - 1 - idx;  // heaviest blocks first
    const int hk = hq / (p.Hq / p.Hkv);
    const int q0 = mblk * (PAIR ? BM : kTiles * BM);  // first query row of tile 0
    // tile t: query head hq + tile_dh(t), rows from q0 + tile_dq(t)
    auto tile_dh = [](int t) { return PAIR ? t : 0; };
    auto tile_dq = [](int t) { return PAIR ? 0 : t * BM; };
    // Rows of this item: the batch entry's Lq queries / Lk keys (head-major), or (TOK) packed
    // sequence b, rows [row0, row0 + len) of the token-major tensors (self-attention).
    constexpr bool tok = TOK;
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
    if (q0 >= Lq) return;  // a packed sequence shorter than this query block (uniform exit)
    int P = p.P;
    int klen;
    bool bad_item = false;
    if constexpr (PAGED) {
        // the sequence's Lq queries are the newest of its kv_lens[b] cached positions
        const long long cap = (long long)p.page_size * p.max_pages;
        long long n = __ldg(p.kv_lens + b);
        n = n < 0 ? 0 : (n > cap ? cap : n);
        klen = (int)n;
        P = klen - Lq;
        bad_item = P < 0;
    } else {
        klen = valid_keys(p.key_lens, b, Lk);
    }

    // Visible key interval of each query tile, and the shared key-tile grid.
    long long tlo[kTiles], thi[kTiles];
    long long kv0 = -1;
#pragma unroll
    for (int t = 0; t < kTiles; ++t) {
        const int qa = q0 + tile_dq(t);
        if (qa >= Lq) {
            tlo[t] = 0;
            thi[t] = 0;
            continue;
        }
        const int qb = min(qa + BM, Lq) - 1;
        key_interval(p.mode, p.window, klen, (long long)P + qa, (long long)P + qb, &tlo[t], &thi[t]);
        if (thi[t] > tlo[t] && (kv0 < 0 || tlo[t] < kv0)) kv0 = tlo[t];
    }
    if constexpr (PAGED) {
        // Every CTA of the sequence checks the page entries of all the keys its queries can
        // see, so they agree: a sequence with an entry outside the pool, or with fewer cached
        // positions than queries, reads nothing and its rows are zeros.
        long long slo, shi;
        key_interval(p.mode, p.window, klen, (long long)P, (long long)P + Lq - 1, &slo, &shi);
        bool bad = false;
        if (!bad_item && shi > slo) {
            const int32_t* pages = p.page_table + (size_t)b * p.max_pages;
            for (long long x = slo / p.page_size + threadIdx.x; x <= (shi - 1) / p.page_size; x += blockDim.x) {
                const int id = __ldg(pages + x);
                bad |= (id < 0 || id >= p.num_pages);
            }
        }
        const bool bad_pages = __syncthreads_or(bad);
        if (bad_item || bad_pages) {
            if (threadIdx.x == 0) record_status(p.wc.status, bad_pages ? kStatusBadPage : kStatusBadSeqlens);
            kv0 = -1;
        }
    }
    // the CTA's visible keys (the union of its tiles' bands); with TMA page copies the key-tile
    // grid starts on a multiple of 128, so that pages never straddle two tiles
    const long long vis_lo = kv0;
    long long vis_hi = 0;
#pragma unroll
    for (int t = 0; t < kTiles; ++t)
        if (thi[t] > tlo[t] && thi[t] > vis_hi) vis_hi = thi[t];
    if (PAGED && p.paged_tma && kv0 > 0) kv0 = (kv0 / BN) * BN;
    TileRange rng[kTiles];
    int ntiles = 0;
#pragma unroll
    for (int t = 0; t < kTiles; ++t) {
        if (kv0 < 0 || thi[t] <= tlo[t]) {
            rng[t] = {0, 0};
        } else {
            rng[t].jb = (int)((tlo[t] - kv0) / BN);
            rng[t].je = (int)((thi[t] - kv0 + BN - 1) / BN);
            ntiles = max(ntiles, rng[t].je);
        }
    }
    if (kv0 < 0) kv0 = 0;
    // Rows of the last key tile that no query of the sequence sees (past the end of the union of
    // its queries' bands: key padding, cache rows past the newest query) get weight 0, and the
    // tensor core multiplies that 0 into the V row: an Inf or NaN there would still make the
    // product NaN.  Such rows [zero_lo, zero_hi) of the tail V tile are zeroed in shared memory
    // before its P V products (rows past the tensor already read as zeros from the copy; the
    // paged gather writes every row past this CTA's keys as zeros).  A row that some query of
    // the sequence sees is finite for its output to be, so it needs nothing.  Only the producer
    // computes this.
    auto tail_rows = [&](int* zlo, int* zhi) -> bool {
        long long slo, shi;
        key_interval(p.mode, p.window, klen, (long long)P, (long long)P + Lq - 1, &slo, &shi);
        const long long tail_row = kv0 + (long long)(ntiles - 1) * BN;
        const long long row_limit = TOK ? (long long)p.total - row0 : (long long)Lk;
        *zlo = (int)max(0LL, shi - tail_row);
        *zhi = (int)min((long long)BN, row_limit - tail_row);
        return ZT && !PAGED && ntiles > 0 && *zhi > *zlo;
    };
    const int kbh = b * p.Hkv + hk;
    // L2 hints: a Q tile is read by this CTA alone, once; K and V tiles are read again by the
    // other query blocks of the kv head, so they are the ones to keep in L2
    auto load_q = [&]() {
        const uint64_t once = l2_policy_evict_first();
        mbar_arrive_expect_tx(bar0 + 8 * kBarQFull, kTiles * C::kQBytes);
        for (int t = 0; t < kTiles; ++t)
            for (int c = 0; c < C::kChunks; ++c)
                if constexpr (TOK)
                    tma_load_3d_hint(sbase + C::kOffQ + t * C::kQBytes + c * (BM * 128), &tmQ, bar0 + 8 * kBarQFull,
                                     c * 64, hq + tile_dh(t), row0 + q0 + tile_dq(t), once);
                else
                    tma_load_3d_hint(sbase + C::kOffQ + t * C::kQBytes + c * (BM * 128), &tmQ, bar0 + 8 * kBarQFull,
                                     c * 64, q0 + tile_dq(t), b * p.Hq + hq + tile_dh(t), once);
    };
    // (the tail V tile lands on its own barrier, land_tail, when some of its rows must be zeroed first)
    auto load_kv = [&](const CUtensorMap* map, int off, int bar, int j, bool land_tail) {
        const int s = j % kStages;
        const int krow = (int)kv0 + j * BN;
        const uint32_t done = (land_tail && bar == kBarVFull && j == ntiles - 1) ? bar0 + 8 * kBarVLand
                                                                                 : bar0 + 8 * (bar + s);
        const uint64_t keep = l2_policy_evict_last();
        mbar_arrive_expect_tx(done, C::kKVBytes);
        for (int c = 0; c < C::kChunks; ++c)
            tma_load_3d_hint(sbase + off + s * C::kKVBytes + c * (BN * 128), map, done, c * 64,
                             TOK ? hk : krow, TOK ? row0 + krow : kbh, keep);
    };
    // With one tile per CTA (two CTAs per SM) the first copies go out before the CTA
    // synchronises; with two tiles (one CTA per SM) that delays the CTA's start more than
    // the copies gain, so the producer starts them after the barrier.
    const int nearly = (kTiles == 1 && !PAGED) ? min(kStages, ntiles) : 0;  // K/V tiles loaded at entry

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNumBars; ++i) {
            uint32_t count = 1;
            if ((i >= kBarPFull && i < kBarPFull + kTiles) || (i >= kBarPHalf && i < kBarPHalf + kTiles))
                count = 8;  // one arrival per softmax warp of the tile
            if (PAGED && !p.paged_tma &&
                ((i >= kBarKFull && i < kBarKFull + kStages) || (i >= kBarVFull && i < kBarVFull + kStages)))
                count = 32;  // gathered rows: one arrival per producer lane, after its copies have landed
            mbar_init(bar0 + 8 * i, count);
        }
        *abort_flag = 0;
        mbar_fence_init();
        // Thread 0 is the producer: its first copies start now and land while TMEM is
        // allocated and the CTA synchronises.
        if (kTiles == 1 && !PAGED && ntiles > 0) {
            int zlo, zhi;
            const bool zt = tail_rows(&zlo, &zhi);
            load_q();
            for (int j = 0; j < nearly; ++j) {
                load_kv(&tmK, C::kOffK, kBarKFull, j, false);
                load_kv(&tmV, C::kOffV, kBarVFull, j, zt);
            }
        }
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), C::kTmemCols);
        tmem_relinquish();
    }
    if (kTiles == 2 && warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        if (!PAGED || p.paged_tma) {
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (PAGED && p.paged_tma && warp == 0) {
        // ------------------------------------------------------------ TMA page producer (paged K/V)
        // Tile j holds keys [kv0 + 128 j, +128); with kv0 a multiple of 128, no page straddles
        // two tiles.  Lane 0 posts the tile's bytes, then lane i copies the i-th of the tile's pages
        // that hold visible keys (one box per 64-column chunk; a page of 128 rows or more gives
        // its 128-row piece).  V rows outside the CTA's visible keys [vis_lo, vis_hi) -- before
        // the band in the first tile, past it in the last, never copied or copied from cache rows
        // no query here sees -- would meet P = 0 on the tensor core, where 0 * NaN is NaN: such
        // a tile lands on its own barrier, the warp zeroes those rows, and only then releases it.
        const int ps = p.page_size;
        const int32_t* pages = p.page_table + (size_t)b * p.max_pages;
        const uint64_t keep = l2_policy_evict_last();
        if (lane == 0 && ntiles > 0) load_q();
        int issued = 0;      // K and V tiles issued
        int land_uses = 0;   // phases of the landing barrier used
        bool land_failed = false;
        for (int j = 0; j < ntiles; ++j) {
            const int s = j % kStages;
            const uint32_t n = (uint32_t)(j / kStages);
            const long long s0 = kv0 + (long long)j * BN;
            const long long clo = max(s0, vis_lo), chi = min(s0 + BN, vis_hi);  // the tile's visible keys
            const int zlo = (int)(clo - s0), zhi = (int)(chi - s0);             // V rows kept: [zlo, zhi)
            const bool zero = zlo > 0 || zhi < BN;
            const long long f = clo / ps, e = (chi - 1) / ps;                   // pages with visible keys
            const int npages = (int)(e - f + 1);
            const uint32_t bytes = (uint32_t)(ps < BN ? npages * ps : BN) * (D * 2);
            bool ok = true;
            for (int kind = 0; kind < 2; ++kind) {
                const int empty = kind ? kBarVEmpty : kBarKEmpty;
                if (j >= kStages &&
                    !__all_sync(0xffffffffu, mbar_wait(bar0 + 8 * (empty + s), (n - 1) & 1, p.wc, abort_flag))) {
                    ok = false;
                    break;
                }
                const uint32_t tile = sbase + (kind ? C::kOffV : C::kOffK) + s * C::kKVBytes;
                const bool land = kind && zero;
                const uint32_t done = land ? bar0 + 8 * kBarVLand : bar0 + 8 * ((kind ? kBarVFull : kBarKFull) + s);
                const CUtensorMap* map = kind ? &tmV : &tmK;
                if (lane == 0) mbar_arrive_expect_tx(done, bytes);
                __syncwarp();
                if (ps < BN) {
                    for (int x = lane; x < npages; x += 32) {
                        const long long pgi = f + x;
                        const int pg = __ldg(pages + pgi);
                        const uint32_t r = (uint32_t)(pgi * ps - s0);  // a multiple of the page size
#pragma unroll
                        for (int c = 0; c < C::kChunks; ++c)
                            tma_load_3d_hint(tile + c * (BN * 128) + r * 128, map, done, c * 64, 0, pg * p.Hkv + hk, keep);
                    }
                } else if (lane == 0) {
                    const int pg = __ldg(pages + s0 / ps);
#pragma unroll
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_3d_hint(tile + c * (BN * 128), map, done, c * 64, (int)(s0 % ps), pg * p.Hkv + hk, keep);
                }
                ++issued;
                if (land) {
                    const uint32_t par = (uint32_t)land_uses & 1;
                    ++land_uses;
                    if (!__all_sync(0xffffffffu, mbar_wait(bar0 + 8 * kBarVLand, par, p.wc, abort_flag))) {
                        if (lane == 0) drain_wait(bar0 + 8 * kBarVLand, par, p.wc);  // the copies may still be in flight
                        land_failed = true;
                        ok = false;
                        break;
                    }
                    uint8_t* vt = smem + C::kOffV + s * C::kKVBytes;
                    constexpr int kUnits = C::kChunks * 8;  // 16-byte units of a row
                    const int nz = zlo + (BN - zhi);        // rows to zero: [0, zlo) and [zhi, BN)
                    for (int u = lane; u < nz * kUnits; u += 32) {
                        const int i = u / kUnits;
                        const int r = i < zlo ? i : zhi + (i - zlo);
                        const int c = (u / 8) % C::kChunks, q = u & 7;
                        *reinterpret_cast<uint4*>(vt + c * (BN * 128) + r * 128 + q * 16) = make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar0 + 8 * (kBarVFull + s));
                }
            }
            if (!ok) break;
        }
        // nothing of this CTA's stays in flight when it leaves, whatever happened above
        if (lane == 0 && ntiles > 0) {
            drain_wait(bar0 + 8 * kBarQFull, 0, p.wc);
            // a V tile whose landing wait gave up was drained above and never released
            const int nk = (issued + 1) / 2, nv = issued / 2 - (land_failed ? 1 : 0);
            for (int j = (nk > kStages ? nk - kStages : 0); j < nk; ++j)
                drain_wait(bar0 + 8 * (kBarKFull + j % kStages), (uint32_t)(j / kStages) & 1, p.wc);
            for (int j = (nv > kStages ? nv - kStages : 0); j < nv; ++j)
                drain_wait(bar0 + 8 * (kBarVFull + j % kStages), (uint32_t)(j / kStages) & 1, p.wc);
        }
    } else if (PAGED && warp == 0) {
        // ------------------------------------------------------------ gather producer (paged K/V)
        // Q comes by TMA.  For every key tile the lanes write the byte offset of each of its
        // 128 rows in the pools (or ~0 past the visible keys) to shared memory, then copy whole
        // rows, 16 bytes per lane, each unit to its swizzled place (the layout TMA would give).
        // The copies of K(j) and V(j) are separate items in that order; an item is released to
        // the MMA issuer once the next one has been issued and its own copies have landed and
        // are fenced for the tensor core.  One item of lag never waits on itself: K(j) is
        // released before V(j) needs the V slot freed by PV(j - 2), and V(j) before K(j + 1)
        // needs the K slot freed by QK(j - 1), while the issuer runs PV(j - 1) before QK(j).
        if (lane == 0 && ntiles > 0) load_q();
        if (ntiles > 0) {
            long long hi_all = 0;  // rows from here on are zeros
#pragma unroll
            for (int t = 0; t < kTiles; ++t)
                if (thi[t] > tlo[t] && thi[t] > hi_all) hi_all = thi[t];
            unsigned long long* rowoff = reinterpret_cast<unsigned long long*>(smem + C::kOffRow);
            constexpr int kUnits = C::kChunks * 8;  // 16-byte units of one row
            constexpr int kRowsPerStep = 32 / kUnits;
            const int rsub = lane / kUnits, u = lane % kUnits, c = u >> 3, qd = u & 7;
            const int32_t* pages = p.page_table + (size_t)b * p.max_pages;
            int items = 0;
            bool ok = true;
            for (int j = 0; ok && j < ntiles; ++j) {
                const int s = j % kStages;
                const uint32_t n = (uint32_t)(j / kStages);
                const long long krow0 = kv0 + (long long)j * BN;
                __syncwarp();
                for (int r = lane; r < BN; r += 32) {
                    const long long key = krow0 + r;
                    unsigned long long off = ~0ull;
                    if (key < hi_all) {
                        const long long pg = __ldg(pages + key / p.page_size);
                        off = (((unsigned long long)pg * p.Hkv + hk) * (unsigned long long)p.page_size +
                               (unsigned long long)(key % p.page_size)) * (D * 2);
                    }
                    rowoff[r] = off;
                }
                __syncwarp();
                for (int kind = 0; kind < 2; ++kind) {  // K(j), then V(j)
                    const int empty = kind ? kBarVEmpty : kBarKEmpty;
                    if (j >= kStages &&
                        !__all_sync(0xffffffffu, mbar_wait(bar0 + 8 * (empty + s), (n - 1) & 1, p.wc, abort_flag))) {
                        ok = false;
                        break;
                    }
                    const int off_tile = (kind ? C::kOffV : C::kOffK) + s * C::kKVBytes;
                    const uint8_t* src = kind ? p.vpool : p.kpool;
#pragma unroll 4
                    for (int i = 0; i < BN / kRowsPerStep; ++i) {
                        const int r = kRowsPerStep * i + rsub;
                        const unsigned long long off = rowoff[r];
                        const uint32_t dofs = off_tile + c * (BN * 128) + r * 128 + ((qd ^ (r & 7)) << 4);
                        if (off != ~0ull) cp_async16(sbase + dofs, src + off + u * 16);
                        else *reinterpret_cast<uint4*>(smem + dofs) = make_uint4(0u, 0u, 0u, 0u);
                    }
                    cp_async_commit();
                    ++items;
                    if (items >= 2) {  // the item before this one has landed: release it
                        const int x = items - 2;
                        cp_async_wait<1>();
                        fence_proxy_async_smem();
                        mbar_arrive(bar0 + 8 * (((x & 1) ? kBarVFull : kBarKFull) + (x >> 1) % kStages));
                    }
                }
            }
            cp_async_wait<0>();  // nothing stays in flight, whatever happened above
            if (ok) {
                const int x = items - 1;
                fence_proxy_async_smem();
                mbar_arrive(bar0 + 8 * (((x & 1) ? kBarVFull : kBarKFull) + (x >> 1) % kStages));
            }
            if (lane == 0) drain_wait(bar0 + 8 * kBarQFull, 0, p.wc);
        }
    } else if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        int issued = 2 * nearly;  // K and V copies issued so far (kept by lane 0)
        int zero_lo, zero_hi;
        const bool zero_tail = tail_rows(&zero_lo, &zero_hi);
        if (lane == 0 && ntiles > 0) {
            if (kTiles == 2) load_q();
            for (int j = nearly; j < ntiles; ++j) {
                const int s = j % kStages;
                const uint32_t n = (uint32_t)(j / kStages);
                if (j >= kStages && !mbar_wait(bar0 + 8 * (kBarKEmpty + s), (n - 1) & 1, p.wc, abort_flag)) break;
                load_kv(&tmK, C::kOffK, kBarKFull, j, false);
                if (j >= kStages && !mbar_wait(bar0 + 8 * (kBarVEmpty + s), (n - 1) & 1, p.wc, abort_flag)) {
                    issued = 2 * j + 1;
                    break;
                }
                load_kv(&tmV, C::kOffV, kBarVFull, j, zero_tail);
                issued = 2 * j + 2;
            }
            drain_wait(bar0 + 8 * kBarQFull, 0, p.wc);
            const int nk = (issued + 1) / 2, nv = issued / 2;
            for (int j = (nk > kStages ? nk - kStages : 0); j < nk; ++j)
                drain_wait(bar0 + 8 * (kBarKFull + j % kStages), (uint32_t)(j / kStages) & 1, p.wc);
            for (int j = (nv > kStages ? nv - kStages : 0); j < nv; ++j)
                if (!(zero_tail && j == ntiles - 1))  // the tail tile is waited for below
                    drain_wait(bar0 + 8 * (kBarVFull + j % kStages), (uint32_t)(j / kStages) & 1, p.wc);
        }
        // The tail V tile: once it has landed, the whole warp zeroes its rows [zero_lo, zero_hi)
        // (a row is 128 bytes per 64-column chunk, whatever the swizzle does inside it), makes the
        // stores visible to the tensor core and releases the tile to the MMA issuer.
        if (zero_tail && __shfl_sync(0xffffffffu, issued, 0) >= 2 * ntiles) {
            const bool landed = __all_sync(0xffffffffu, mbar_wait(bar0 + 8 * kBarVLand, 0, p.wc, abort_flag));
            if (landed) {
                const int s = (ntiles - 1) % kStages;
                uint8_t* vt = smem + C::kOffV + s * C::kKVBytes;
                const int units = (zero_hi - zero_lo) * C::kChunks * 8;  // 16-byte stores
                for (int u = lane; u < units; u += 32) {
                    const int r = zero_lo + u / (C::kChunks * 8), c = (u / 8) % C::kChunks, q = u & 7;
                    *reinterpret_cast<uint4*>(vt + c * (BN * 128) + r * 128 + q * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar0 + 8 * (kBarVFull + s));
            } else if (lane == 0) {
                drain_wait(bar0 + 8 * kBarVLand, 0, p.wc);  // gave up: the copy may still be in flight
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && ntiles > 0) {
            constexpr uint32_t kIdescQK = idesc_f16kind_f32(BM, BN, 0, 0, F16);
            constexpr uint32_t kIdescPV = idesc_f16kind_f32(BM, D, 0, 1, F16);
            bool ok = mbar_wait(bar0 + 8 * kBarQFull, 0, p.wc, abort_flag);
            int it[kTiles] = {};  // local iteration (P phases consumed) per tile
            for (int j = 0; ok && j <= ntiles; ++j) {
                // PV_t(j-1) then QK_t(j), tile by tile
                bool v_waited = false, k_waited = false;
                bool used_v = false, used_k = false;
#pragma unroll
                for (int t = 0; t < kTiles; ++t) {
                    const int jp = j - 1;
                    if (jp >= 0 && jp >= rng[t].jb && jp < rng[t].je) {
                        const int s = jp % kStages;
                        // P_t arrives in two parts: keys [0, 32) and [64, 96) first, then the rest;
                        // the product over the first part runs while the softmax packs the second
                        if (!mbar_wait(bar0 + 8 * (kBarPHalf + t), (uint32_t)it[t] & 1, p.wc, abort_flag)) { ok = false; break; }
                        if (!v_waited) {
                            if (!mbar_wait(bar0 + 8 * (kBarVFull + s), (uint32_t)(jp / kStages) & 1, p.wc, abort_flag)) { ok = false; break; }
                            v_waited = true;
                        }
                        tc_fence_after();
                        // descriptors: the tile's, plus each step's offset >> 4 in the address field
                        const uint64_t vd = smem_desc_sw128(sbase + C::kOffV + s * C::kKVBytes, BN * 128, 1024);
                        const uint32_t tP = tmem + C::kColS + 128 * t;
                        const uint32_t tO = tmem + C::kColO + 128 * t;
#pragma unroll
                        for (int part = 0; part < 2; ++part) {
                            if (part == 1) {
                                if (!mbar_wait(bar0 + 8 * (kBarPFull + t), (uint32_t)it[t] & 1, p.wc, abort_flag)) { ok = false; break; }
                                tc_fence_after();
                            }
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                // 16-key steps kk: part 0 takes 0, 1, 4, 5 and part 1 takes 2, 3, 6, 7
                                const int kk = (u >> 1) * 4 + part * 2 + (u & 1);
                                tc_mma_ts(tO, tP + kk * 8, vd + (uint64_t)((kk * 16 * 128) >> 4), kIdescPV,
                                          (jp > rng[t].jb || kk > 0) ? 1u : 0u);
                            }
                        }
                        if (!ok) break;
                        it[t] += 1;
                        used_v = true;
                        if (jp == rng[t].je - 1) tc_commit(bar0 + 8 * (kBarOFull + t));
                    }
                    if (j < ntiles && j >= rng[t].jb && j < rng[t].je) {
                        const int s = j % kStages;
                        if (!k_waited) {
                            if (!mbar_wait(bar0 + 8 * (kBarKFull + s), (uint32_t)(j / kStages) & 1, p.wc, abort_flag)) { ok = false; break; }
                            k_waited = true;
                            tc_fence_after();
                        }
                        const uint64_t kd = smem_desc_sw128(sbase + C::kOffK + s * C::kKVBytes, 16, 1024);
                        const uint64_t qd = smem_desc_sw128(sbase + C::kOffQ + t * C::kQBytes, 16, 1024);
                        const uint32_t tS = tmem + C::kColS + 128 * t;
#pragma unroll
                        for (int ks = 0; ks < D / 16; ++ks) {
                            const uint64_t off = (uint64_t)((((ks >> 2) * (BM * 128)) + (ks & 3) * 32) >> 4);
                            tc_mma_ss(tS, qd + off, kd + off, kIdescQK, ks > 0 ? 1u : 0u);
                        }
                        tc_commit(bar0 + 8 * (kBarSFull + t));
                        used_k = true;
                    }
                }
                if (!ok) break;
                if (used_v) tc_commit(bar0 + 8 * (kBarVEmpty + (j - 1) % kStages));
                if (used_k) tc_commit(bar0 + 8 * (kBarKEmpty + j % kStages));
            }
            tc_commit(bar0 + 8 * kBarMmaDone);
            drain_wait(bar0 + 8 * kBarMmaDone, 0, p.wc);
        }
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        // 16 warps: tile t = sw / 8; half h = (sw / 4) % 2 takes key columns [64h, 64h + 64)
        // of every S row and the head dims [h D/2, (h+1) D/2) of O.
        const int sw = warp - 2;
        const int t = sw >> 3;
        const int h = (sw >> 2) & 1;
        const int wq = warp & 3;                 // TMEM lane quarter
        const int row = wq * 32 + lane;
        const int qi = q0 + tile_dq(t) + row;
        const int hqt = hq + tile_dh(t);
        const long long qpos = (long long)P + qi;
        long long rlo, rhi;
        key_interval(p.mode, p.window, klen, qpos, qpos, &rlo, &rhi);
        // the row's visible keys relative to its first column of the first block, clamped to the keys
        // that exist (a band past them is empty either way): 32-bit offsets for the block loop
        const int rlo_rel = (int)(min(max(rlo, 0LL), (long long)klen) - (kv0 + 64 * h));
        const int rhi_rel = (int)(min(max(rhi, 0LL), (long long)klen) - (kv0 + 64 * h));
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t tS = tmem + lane_off + C::kColS + 128 * t;
        const uint32_t tO = tmem + lane_off + C::kColO + 128 * t;
        const float sl = p.scale_log2;
        float m_run = -INFINITY;
        float l_run = 0.f;  // this half's share of the row sum
        bool ok = true;
        const int jb = rng[t].jb, je = rng[t].je;
        float* xch = reinterpret_cast<float*>(smem + C::kOffX) + (t * 2) * BM;  // [2 halves][128 rows]

        for (int j = jb; j < je; ++j) {
            const int i = j - jb;
            // every lane waits; the warp continues only if all lanes saw the phase, so the
            // warp-collective tcgen05 operations below never run with a partial warp
            // A warp that gave up stays in the loop and keeps meeting the tile's named barrier
            // once per key block, so the other warps of the tile never wait for it.
            if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar0 + 8 * (kBarSFull + t), (uint32_t)i & 1, p.wc, abort_flag));
            tc_fence_after();
            softmax_block<D, F16, POS, kTiles == 1>(tS, tO, h, row, lane, t, sl, rlo_rel, rhi_rel, j, xch, ok, m_run,
                                                    l_run, bar0 + 8 * (kBarPHalf + t), bar0 + 8 * (kBarPFull + t));
        }

        // ------------------------------------------------------------ epilogue
        // row sum = both halves' shares; each half stores its D/2 head dims of the row
        float* lch = reinterpret_cast<float*>(smem + C::kOffL) + (t * 2) * BM;
        float l_tot = l_run;
        if (ok) lch[h * BM + row] = l_run;
        tile_bar_sync(t);
        if (ok) l_tot += lch[(1 - h) * BM + row];
        const bool has = je > jb;
        if (ok && has) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar0 + 8 * (kBarOFull + t), 0, p.wc, abort_flag));
            tc_fence_after();
        }
        if (D == 128 && LAYOUT == kHeadMajor && p.tma_out) {
            // head-major output: each half writes its 64 head dims of the row (one 128-byte chunk)
            // into the tile's Q buffer in the layout of a Q tile (free once the tile's last product
            // has completed; without key blocks its copy is waited for), and one thread of the tile
            // stores both chunks with TMA (rows past Lq are clipped by the copy)
            if (ok && !has && ntiles > 0) {
                ok = __all_sync(0xffffffffu, mbar_wait(bar0 + 8 * kBarQFull, 0, p.wc, abort_flag));
            }
            if (ok) {
                const float inv = (l_tot > 0.f) ? 1.f / l_tot : 0.f;
                uint8_t* srow = smem + C::kOffQ + t * C::kQBytes + h * (BM * 128) + row * 128;
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    float o[32];
                    if (has) {
                        tmem_ld32(tO + (D / 2) * h + 32 * c, o);
                    } else {
#pragma unroll
                        for (int q = 0; q < 32; ++q) o[q] = 0.f;
                    }
#pragma unroll
                    for (int q = 0; q < 32; q += 8) {
                        const int unit = (32 * c + q) / 8;  // 16-byte unit of the 128-byte chunk row
                        *reinterpret_cast<uint4*>(srow + ((unit ^ (row & 7)) << 4)) =
                            make_uint4(pack2<F16>(o[q] * inv, o[q + 1] * inv), pack2<F16>(o[q + 2] * inv, o[q + 3] * inv),
                                       pack2<F16>(o[q + 4] * inv, o[q + 5] * inv), pack2<F16>(o[q + 6] * inv, o[q + 7] * inv));
                    }
                }
                fence_proxy_async_smem();
            }
            // the tile's 8 warps meet (every path reaches this) and agree that all rows are in place
            uint32_t all_ok;
            asm volatile(
                "{\n\t.reg .pred pin, pout;\n\tsetp.ne.u32 pin, %1, 0;\n\t"
                "bar.red.and.pred pout, %2, 256, pin;\n\tselp.u32 %0, 1, 0, pout;\n\t}"
                : "=r"(all_ok)
                : "r"((uint32_t)ok), "r"(1 + t)
                : "memory");
            if (all_ok && (sw & 7) == 0 && lane == 0 && q0 + tile_dq(t) < Lq) {
                const uint64_t once = l2_policy_evict_first();  // nothing in this launch reads it back
#pragma unroll
                for (int c = 0; c < 2; ++c)
                    asm volatile(
                        "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%1, %2, %3}], [%4], %5;" ::"l"(
                            reinterpret_cast<uint64_t>(&tmO)),
                        "r"(c * 64), "r"(q0 + tile_dq(t)), "r"(b * p.Hq + hqt),
                        "r"(sbase + C::kOffQ + t * C::kQBytes + c * (BM * 128)), "l"(once)
                        : "memory");
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");  // before the CTA may leave
            }
        } else if (ok && q0 + tile_dq(t) < Lq) {
            const float inv = (l_tot > 0.f) ? 1.f / l_tot : 0.f;
            __nv_bfloat16* orow =
                p.out + (tok        ? ((size_t)(row0 + qi) * p.Hq + hqt) * D
                         : p.out_tok ? (((size_t)b * Lq + qi) * p.Hq + hqt) * D
                                     : ((size_t)(b * p.Hq + hqt) * Lq + qi) * D) +
                (D / 2) * h;
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                float o[32];
                if (has) {
                    tmem_ld32(tO + (D / 2) * h + 32 * c, o);
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
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

// ---------------------------------------------------------------------- persistent form
// Head-major inputs at head_dim 128 with an even group size and no key row that every query
// misses (no tail zeroing): one CTA per SM walks the query blocks blockIdx.x, blockIdx.x +
// gridDim.x, ... of the heaviest-first order (serpentine), each block two query heads of one kv group over
// the same 128 rows (so both tiles visit the same key tiles).  The next block's Q loads once the
// last QK^T of the current one has completed, its first K/V tiles as soon as ring slots free up,
// and its first QK^T runs while the current block's epilogue reads O; the epilogue stores with
// per-thread 16-byte writes, leaving the Q buffers to the next block.  Every barrier phase
// counts across blocks.
enum : int {
    kPQFull = 0,
    kPQFree = 1,                   // the block's last QK^T completed: the Q buffers may be refilled
    kPKFull = 2,                   // + stage
    kPVFull = kPKFull + kStages,   // + stage
    kPKEmpty = kPVFull + kStages,  // + stage
    kPVEmpty = kPKEmpty + kStages, // + stage
    kPSFull = kPVEmpty + kStages,  // + tile
    kPPHalf = kPSFull + 2,         // + tile, 8 arrivals
    kPPFull = kPPHalf + 2,         // + tile, 8 arrivals
    kPOFull = kPPFull + 2,         // + tile: the block's last P V product completed
    kPOFree = kPOFull + 2,         // + tile, 8 arrivals: the epilogue has read O_t
    kPMmaDone = kPOFree + 2,
    kPNumBars = kPMmaDone + 1,
};
static_assert(kPNumBars * 8 <= 240, "barrier area");

template <bool F16, bool POS>
__global__ void __launch_bounds__(threads_for<2>(), 1)
    prefill_persist_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
    constexpr int D = 128;
    using C = Cfg<D, 2>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + C::kOffBar;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffBar + 240);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffBar + 248);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nh = p.Hq / 2;
    const int num_items = p.num_m * p.B * nh;
    const int G = p.Hq / p.Hkv;

    // This CTA's k-th query block: the items are in heaviest-first order, taken forwards in even
    // rounds and backwards in odd ones, so that every CTA's total comes out about the same.
    const int grid = (int)gridDim.x;
    const int rounds = (num_items + grid - 1) / grid;
    auto item_index = [&](int k) { return k * grid + ((k & 1) ? grid - 1 - (int)blockIdx.x : (int)blockIdx.x); };
    // one query block: heads hq, hq + 1 of batch entry b, rows [q0, q0 + 128); keys from kv0 in
    // ntiles tiles of 128
    struct Item {
        int hq, b, q0, ntiles;
        long long kv0;
    };
    auto item_of = [&](int idx) {
        Item it;
        it.hq = (idx % nh) * 2;
        idx /= nh;
        it.b = idx % p.B;
        idx /= p.B;
        it.q0 = (p.num_m - 1 - idx) * BM;  // heaviest blocks first
        long long tlo, thi;
        key_interval(p.mode, p.window, p.Lk, (long long)p.P + it.q0, (long long)p.P + min(it.q0 + BM, p.Lq) - 1, &tlo,
                     &thi);
        it.kv0 = thi > tlo ? tlo : 0;
        it.ntiles = thi > tlo ? (int)((thi - tlo + BN - 1) / BN) : 0;
        return it;
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < kPNumBars; ++i) {
            const bool eight = (i >= kPPHalf && i < kPPHalf + 2) || (i >= kPPFull && i < kPPFull + 2) ||
                               (i >= kPOFree && i < kPOFree + 2);
            mbar_init(bar0 + 8 * i, eight ? 8u : 1u);
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
        if (lane == 0) {
            const uint64_t once = l2_policy_evict_first(), keep = l2_policy_evict_last();
            long long g = 0;     // K/V tiles issued (one global count over the CTA's blocks)
            long long gv = 0;    // V tiles issued
            int nq = 0;          // Q pairs issued
            bool ok = true;
            for (int k = 0; ok && k < rounds; ++k) {
                const int idx = item_index(k);
                if (idx >= num_items) continue;
                const Item it = item_of(idx);
                const int kbh = it.b * p.Hkv + it.hq / G;
                for (int j = 0; j < it.ntiles; ++j) {
                    const int s = (int)(g & 1);
                    const uint32_t n = (uint32_t)(g >> 1);
                    const int krow = (int)it.kv0 + j * BN;
                    if (g >= kStages && !mbar_wait(bar0 + 8 * (kPKEmpty + s), (n - 1) & 1, p.wc, abort_flag)) { ok = false; break; }
                    mbar_arrive_expect_tx(bar0 + 8 * (kPKFull + s), C::kKVBytes);
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_3d_hint(sbase + C::kOffK + s * C::kKVBytes + c * (BN * 128), &tmK, bar0 + 8 * (kPKFull + s),
                                         c * 64, krow, kbh, keep);
                    ++g;
                    if (j == 0) {
                        // the previous block's last QK^T has read its Q
                        if (nq > 0 && !mbar_wait(bar0 + 8 * kPQFree, (uint32_t)(nq - 1) & 1, p.wc, abort_flag)) { ok = false; break; }
                        mbar_arrive_expect_tx(bar0 + 8 * kPQFull, 2 * C::kQBytes);
                        for (int t = 0; t < 2; ++t)
                            for (int c = 0; c < C::kChunks; ++c)
                                tma_load_3d_hint(sbase + C::kOffQ + t * C::kQBytes + c * (BM * 128), &tmQ, bar0 + 8 * kPQFull,
                                                 c * 64, it.q0, it.b * p.Hq + it.hq + t, once);
                        ++nq;
                    }
                    if (gv >= kStages && !mbar_wait(bar0 + 8 * (kPVEmpty + s), (n - 1) & 1, p.wc, abort_flag)) { ok = false; break; }
                    mbar_arrive_expect_tx(bar0 + 8 * (kPVFull + s), C::kKVBytes);
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_3d_hint(sbase + C::kOffV + s * C::kKVBytes + c * (BN * 128), &tmV, bar0 + 8 * (kPVFull + s),
                                         c * 64, krow, kbh, keep);
                    ++gv;
                }
            }
            // nothing of this CTA's stays in flight when it leaves, whatever happened above
            if (nq > 0) drain_wait(bar0 + 8 * kPQFull, (uint32_t)(nq - 1) & 1, p.wc);
            for (long long j = (g > kStages ? g - kStages : 0); j < g; ++j)
                drain_wait(bar0 + 8 * (kPKFull + (int)(j & 1)), (uint32_t)(j >> 1) & 1, p.wc);
            for (long long j = (gv > kStages ? gv - kStages : 0); j < gv; ++j)
                drain_wait(bar0 + 8 * (kPVFull + (int)(j & 1)), (uint32_t)(j >> 1) & 1, p.wc);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t kIdescQK = idesc_f16kind_f32(BM, BN, 0, 0, F16);
            constexpr uint32_t kIdescPV = idesc_f16kind_f32(BM, D, 0, 1, F16);
            bool ok = true;
            long long g0 = 0;  // global index of the block's first key tile
            int nq = 0;        // blocks with key tiles done
            for (int k = 0; ok && k < rounds; ++k) {
                const int idx = item_index(k);
                if (idx >= num_items) continue;
                const Item it = item_of(idx);
                if (it.ntiles == 0) continue;
                if (!mbar_wait(bar0 + 8 * kPQFull, (uint32_t)nq & 1, p.wc, abort_flag)) break;
                for (int j = 0; ok && j <= it.ntiles; ++j) {
                    bool v_waited = false, k_waited = false;
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        if (j >= 1) {  // PV_t(j - 1), in two parts as P arrives
                            const long long gp = g0 + j - 1;
                            const int s = (int)(gp & 1);
                            if (!mbar_wait(bar0 + 8 * (kPPHalf + t), (uint32_t)gp & 1, p.wc, abort_flag)) { ok = false; break; }
                            // the first product of a block overwrites O_t: the previous epilogue has read it
                            if (j == 1 && nq > 0 &&
                                !mbar_wait(bar0 + 8 * (kPOFree + t), (uint32_t)(nq - 1) & 1, p.wc, abort_flag)) { ok = false; break; }
                            if (!v_waited) {
                                if (!mbar_wait(bar0 + 8 * (kPVFull + s), (uint32_t)(gp >> 1) & 1, p.wc, abort_flag)) { ok = false; break; }
                                v_waited = true;
                            }
                            tc_fence_after();
                            const uint64_t vd = smem_desc_sw128(sbase + C::kOffV + s * C::kKVBytes, BN * 128, 1024);
                            const uint32_t tP = tmem + C::kColS + 128 * t;
                            const uint32_t tO = tmem + C::kColO + 128 * t;
                            for (int part = 0; part < 2; ++part) {
                                if (part == 1) {
                                    if (!mbar_wait(bar0 + 8 * (kPPFull + t), (uint32_t)gp & 1, p.wc, abort_flag)) { ok = false; break; }
                                    tc_fence_after();
                                }
#pragma unroll
                                for (int u = 0; u < 4; ++u) {
                                    const int kk = (u >> 1) * 4 + part * 2 + (u & 1);
                                    tc_mma_ts(tO, tP + kk * 8, vd + (uint64_t)((kk * 16 * 128) >> 4), kIdescPV,
                                              (j > 1 || kk > 0) ? 1u : 0u);
                                }
                            }
                            if (!ok) break;
                            if (j == it.ntiles) tc_commit(bar0 + 8 * (kPOFull + t));
                        }
                        if (j < it.ntiles) {  // QK_t(j)
                            const long long gk = g0 + j;
                            const int s = (int)(gk & 1);
                            if (!k_waited) {
                                if (!mbar_wait(bar0 + 8 * (kPKFull + s), (uint32_t)(gk >> 1) & 1, p.wc, abort_flag)) { ok = false; break; }
                                k_waited = true;
                                tc_fence_after();
                            }
                            const uint64_t kd = smem_desc_sw128(sbase + C::kOffK + s * C::kKVBytes, 16, 1024);
                            const uint64_t qd = smem_desc_sw128(sbase + C::kOffQ + t * C::kQBytes, 16, 1024);
                            const uint32_t tS = tmem + C::kColS + 128 * t;
#pragma unroll
                            for (int ks = 0; ks < D / 16; ++ks) {
                                const uint64_t off = (uint64_t)((((ks >> 2) * (BM * 128)) + (ks & 3) * 32) >> 4);
                                tc_mma_ss(tS, qd + off, kd + off, kIdescQK, ks > 0 ? 1u : 0u);
                            }
                            tc_commit(bar0 + 8 * (kPSFull + t));
                        }
                    }
                    if (!ok) break;
                    if (j == it.ntiles - 1) tc_commit(bar0 + 8 * kPQFree);
                    if (j >= 1) tc_commit(bar0 + 8 * (kPVEmpty + (int)((g0 + j - 1) & 1)));
                    if (j < it.ntiles) tc_commit(bar0 + 8 * (kPKEmpty + (int)((g0 + j) & 1)));
                }
                g0 += it.ntiles;
                ++nq;
            }
            tc_commit(bar0 + 8 * kPMmaDone);
            drain_wait(bar0 + 8 * kPMmaDone, 0, p.wc);
        }
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        const int sw = warp - 2;
        const int t = sw >> 3;
        const int h = (sw >> 2) & 1;
        const int wq = warp & 3;
        const int row = wq * 32 + lane;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t tS = tmem + lane_off + C::kColS + 128 * t;
        const uint32_t tO = tmem + lane_off + C::kColO + 128 * t;
        const float sl = p.scale_log2;
        float* xch = reinterpret_cast<float*>(smem + C::kOffX) + (t * 2) * BM;
        float* lch = reinterpret_cast<float*>(smem + C::kOffL) + (t * 2) * BM;
        bool ok = true;
        long long g0 = 0;
        int nq = 0;
        for (int k = 0; k < rounds; ++k) {
            const int idx = item_index(k);
            if (idx >= num_items) continue;
            const Item it = item_of(idx);
            const int qi = it.q0 + row;
            const int hqt = it.hq + t;
            __nv_bfloat16* orow = p.out + (D / 2) * h +
                                  (p.out_tok ? (((size_t)it.b * p.Lq + qi) * p.Hq + hqt) * D   // [B, Lq, Hq, D]
                                             : ((size_t)(it.b * p.Hq + hqt) * p.Lq + qi) * D); // [B, Hq, Lq, D]
            if (it.ntiles == 0) {  // no visible key: zeros (every warp of the tile takes this path)
                if (qi < p.Lq)
#pragma unroll
                    for (int q = 0; q < D / 2; q += 8) *reinterpret_cast<uint4*>(orow + q) = make_uint4(0u, 0u, 0u, 0u);
                continue;
            }
            long long rlo, rhi;
            key_interval(p.mode, p.window, p.Lk, (long long)p.P + qi, (long long)p.P + qi, &rlo, &rhi);
            const int rlo_rel = (int)(min(max(rlo, 0LL), (long long)p.Lk) - (it.kv0 + 64 * h));
            const int rhi_rel = (int)(min(max(rhi, 0LL), (long long)p.Lk) - (it.kv0 + 64 * h));
            float m_run = -INFINITY;
            float l_run = 0.f;
            for (int j = 0; j < it.ntiles; ++j) {
                const long long g = g0 + j;
                if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar0 + 8 * (kPSFull + t), (uint32_t)g & 1, p.wc, abort_flag));
                tc_fence_after();
                softmax_block<D, F16, POS, false>(tS, tO, h, row, lane, t, sl, rlo_rel, rhi_rel, j, xch, ok, m_run, l_run,
                                                  bar0 + 8 * (kPPHalf + t), bar0 + 8 * (kPPFull + t));
            }
            // ------------------------------------------------------------ epilogue of the block
            if (ok) lch[h * BM + row] = l_run;
            tile_bar_sync(t);
            float l_tot = l_run;
            if (ok) l_tot += lch[(1 - h) * BM + row];
            if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar0 + 8 * (kPOFull + t), (uint32_t)nq & 1, p.wc, abort_flag));
            tc_fence_after();
            const float inv = (l_tot > 0.f) ? 1.f / l_tot : 0.f;
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                float o[32];
                tmem_ld32(tO + (D / 2) * h + 32 * c, o);  // (warp-collective; stale after a give-up, then unused)
                if (ok && qi < p.Lq) {
#pragma unroll
                    for (int q = 0; q < 32; q += 8)
                        *reinterpret_cast<uint4*>(orow + 32 * c + q) =
                            make_uint4(pack2<F16>(o[q] * inv, o[q + 1] * inv), pack2<F16>(o[q + 2] * inv, o[q + 3] * inv),
                                       pack2<F16>(o[q + 4] * inv, o[q + 5] * inv), pack2<F16>(o[q + 6] * inv, o[q + 7] * inv));
                }
            }
            // O_t has been read: the next block's first product may overwrite it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar0 + 8 * (kPOFree + t));
            g0 += it.ntiles;
            ++nq;
        }
    }

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

// [rows_outer, L, D] 16-bit tensor (bf16 or fp16) viewed as 3-D (D, L, rows_outer); box 64 x rows x 1
// (128 unless given), 128-byte swizzle, out-of-range rows read as zeros.
bool encode_16bit_3d(CUtensorMap* map, const void* base, int D, int L, long long outer, bool f16, int rows = 128) {
    EncodeTiledFn fn = get_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)L, (cuuint64_t)outer};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)L * D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// [total, H, D] 16-bit tensor (packed token-major rows) viewed as 3-D (D, H, total); box 64 x 1 x 128,
// so one box is 128 consecutive rows of one head, laid out in shared memory exactly like the
// head-major box above.  Rows past total read as zeros.
bool encode_16bit_3d_tok(CUtensorMap* map, const void* base, int D, int H, int total, bool f16) {
    EncodeTiledFn fn = get_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)total};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
    cuuint32_t box[3] = {64, 1, 128};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                    const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int D, int NT, bool F16, int LAYOUT, bool PAIR, bool ZT, bool POS>
cudaError_t launch_impl(const Problem& pr, const WaitCtl& wc, cudaStream_t stream) {
    using C = Cfg<D, NT>;
    constexpr int kTiles = NT;
    CUtensorMap tq, tk, tv, to;
    // paged K/V by TMA: page sizes of 8 to 128 rows that divide a 128-key tile, or multiples of 128
    // rows, through the pools seen as [num_pages * Hkv, page_size, D]; other page sizes are gathered
    const int ps = pr.page_size;
    const bool paged_tma = LAYOUT == kPaged && ((ps >= 8 && ps <= BN && BN % ps == 0) || (ps > 0 && ps % BN == 0)) &&
                           (long long)pr.num_pages * pr.Hkv <= 0x7fffffffLL;
    if (LAYOUT == kPaged) {
        if (!encode_16bit_3d_tok(&tq, pr.q, D, pr.Hq, pr.total, F16)) return cudaErrorInvalidValue;
        if (paged_tma) {
            const long long outer = (long long)pr.num_pages * pr.Hkv;
            if (!encode_16bit_3d(&tk, pr.k, D, ps, outer, F16, ps < BN ? ps : BN) ||
                !encode_16bit_3d(&tv, pr.v, D, ps, outer, F16, ps < BN ? ps : BN))
                return cudaErrorInvalidValue;
        } else {
            tk = tq;  // the K and V rows are gathered through the page table
            tv = tq;
        }
    } else if (LAYOUT == kPacked) {
        if (!encode_16bit_3d_tok(&tq, pr.q, D, pr.Hq, pr.total, F16) ||
            !encode_16bit_3d_tok(&tk, pr.k, D, pr.Hkv, pr.total, F16) ||
            !encode_16bit_3d_tok(&tv, pr.v, D, pr.Hkv, pr.total, F16))
            return cudaErrorInvalidValue;
    } else if (!encode_16bit_3d(&tq, pr.q, D, pr.Lq, pr.B * pr.Hq, F16) ||
               !encode_16bit_3d(&tk, pr.k, D, pr.Lk, pr.B * pr.Hkv, F16) ||
               !encode_16bit_3d(&tv, pr.v, D, pr.Lk, pr.B * pr.Hkv, F16)) {
        return cudaErrorInvalidValue;
    }
    // head-major output [B, Hq, Lq, 128]: tiles stored by TMA through a map shaped like Q's
    const bool tma_out = D == 128 && LAYOUT == kHeadMajor && !pr.out_tok;
    if (tma_out) {
        if (!encode_16bit_3d(&to, pr.out, D, pr.Lq, pr.B * pr.Hq, F16)) return cudaErrorInvalidValue;
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
            e = cudaFuncSetAttribute(prefill_tc_kernel<D, NT, F16, LAYOUT, PAIR, ZT, POS>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
            if (e != cudaSuccess) return e;
            configured[dev] = true;
        }
    }
    PrefillParams p = {};
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
    constexpr int rows = PAIR ? BM : kTiles * BM;  // query rows per work item
    p.num_m = (pr.Lq + rows - 1) / rows;  // pr.Lq is max_seqlen for packed sequences
    p.cu_seqlens = pr.cu_seqlens;
    p.total = pr.total;
    p.out_tok = pr.out_tok ? 1 : 0;
    p.tma_out = tma_out ? 1 : 0;
    p.scale_log2 = pr.scale * kLog2e;
    p.wc = wc;
    if (LAYOUT == kPaged) {
        p.kpool = static_cast<const uint8_t*>(pr.k);
        p.vpool = static_cast<const uint8_t*>(pr.v);
        p.page_table = pr.page_table;
        p.kv_lens = pr.kv_lens;
        p.page_size = pr.page_size;
        p.max_pages = pr.max_pages;
        p.num_pages = pr.num_pages;
        p.paged_tma = paged_tma ? 1 : 0;
    }
    const long long grid = (long long)p.num_m * pr.B * (PAIR ? pr.Hq / 2 : pr.Hq);
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    prefill_tc_kernel<D, NT, F16, LAYOUT, PAIR, ZT, POS><<<(unsigned)grid, threads_for<NT>(), C::kSmem, stream>>>(tq, tk, tv, to, p);
    return cudaGetLastError();
}

// Whether the tail zeroing can matter for a head-major call: only key padding, or a mask whose
// band (the union over all queries) ends before kv_len, leaves rows inside the tensor that no
// query sees.
// SMs of the current device (looked up once per device); 0 if unknown.
int sm_count() {
    static std::mutex mu;
    static int count[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> g(mu);
    if (count[dev] == 0 && cudaDeviceGetAttribute(&count[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        count[dev] = 0;
    return count[dev];
}

// The persistent paired-head kernel: head-major q/k/v, out head-major or token-major, head_dim
// 128, even group size, no key padding and no key row past every query's band.  One CTA per SM
// (at most one per block).
template <bool F16, bool POS>
cudaError_t launch_persist(const Problem& pr, const WaitCtl& wc, cudaStream_t stream) {
    using C = Cfg<128, 2>;
    CUtensorMap tq, tk, tv;
    if (!encode_16bit_3d(&tq, pr.q, 128, pr.Lq, pr.B * pr.Hq, F16) ||
        !encode_16bit_3d(&tk, pr.k, 128, pr.Lk, pr.B * pr.Hkv, F16) ||
        !encode_16bit_3d(&tv, pr.v, 128, pr.Lk, pr.B * pr.Hkv, F16))
        return cudaErrorInvalidValue;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::mutex mu;
    static bool configured[64] = {};
    {
        std::lock_guard<std::mutex> g(mu);
        if (dev < 64 && !configured[dev]) {
            e = cudaFuncSetAttribute(prefill_persist_kernel<F16, POS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     C::kSmem);
            if (e != cudaSuccess) return e;
            configured[dev] = true;
        }
    }
    PrefillParams p = {};
    p.out = reinterpret_cast<__nv_bfloat16*>(pr.out);
    p.B = pr.B;
    p.Hq = pr.Hq;
    p.Hkv = pr.Hkv;
    p.Lq = pr.Lq;
    p.Lk = pr.Lk;
    p.P = pr.pos_offset;
    p.mode = pr.mode;
    p.window = pr.window;
    p.num_m = (pr.Lq + BM - 1) / BM;
    p.out_tok = pr.out_tok ? 1 : 0;
    p.scale_log2 = pr.scale * kLog2e;
    p.wc = wc;
    const long long items = (long long)p.num_m * pr.B * (pr.Hq / 2);
    if (items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const int sms = sm_count();
    const long long grid = std::min(items, (long long)(sms > 0 ? sms : 1));
    if (grid <= 0) return cudaSuccess;
    prefill_persist_kernel<F16, POS><<<(unsigned)grid, threads_for<2>(), C::kSmem, stream>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

bool tail_zero_needed(const Problem& p) {
    if (p.key_lens != nullptr || p.cu_seqlens != nullptr) return true;
    long long slo, shi;
    key_interval(p.mode, p.window, p.Lk, (long long)p.pos_offset, (long long)p.pos_offset + p.Lq - 1, &slo, &shi);
    return shi < p.Lk;
}

template <int D, int NT, bool F16, int LAYOUT, bool PAIR>
cudaError_t launch_zt(const Problem& p, const WaitCtl& wc, cudaStream_t stream) {
    if constexpr (LAYOUT == kHeadMajor) {
        if (!tail_zero_needed(p))
            return p.scale > 0.f ? launch_impl<D, NT, F16, LAYOUT, PAIR, false, true>(p, wc, stream)
                                 : launch_impl<D, NT, F16, LAYOUT, PAIR, false, false>(p, wc, stream);
    }
    return p.scale > 0.f ? launch_impl<D, NT, F16, LAYOUT, PAIR, LAYOUT != kPaged, true>(p, wc, stream)
                         : launch_impl<D, NT, F16, LAYOUT, PAIR, LAYOUT != kPaged, false>(p, wc, stream);
}

template <int LAYOUT>
cudaError_t launch_layout(const Problem& p, const WaitCtl& wc, cudaStream_t stream) {
    // head_dim 64: one query tile per CTA, so two CTAs share an SM (256 TMEM columns and
    // about 83 KB of shared memory each) and hide each other's set-up and epilogue.
    // head_dim 128: two tiles per CTA (512 TMEM columns, one CTA per SM), ping-pong inside;
    // an even group size pairs two query heads of one kv group over the same rows.
    if (p.D == 64) {  // head-major and packed layouts take the narrow-block kernel
        if constexpr (LAYOUT == kPaged)
            return p.f16 ? launch_zt<64, 1, true, LAYOUT, false>(p, wc, stream)
                         : launch_zt<64, 1, false, LAYOUT, false>(p, wc, stream);
        return cudaErrorInvalidValue;
    }
    if (p.D == 128) {
        if constexpr (LAYOUT == kHeadMajor) {
            if ((p.Hq / p.Hkv) % 2 == 0 && !tail_zero_needed(p)) {
                if (p.f16) return p.scale > 0.f ? launch_persist<true, true>(p, wc, stream)
                                                : launch_persist<true, false>(p, wc, stream);
                return p.scale > 0.f ? launch_persist<false, true>(p, wc, stream)
                                     : launch_persist<false, false>(p, wc, stream);
            }
        }
        if ((p.Hq / p.Hkv) % 2 == 0)
            return p.f16 ? launch_zt<128, 2, true, LAYOUT, true>(p, wc, stream)
                         : launch_zt<128, 2, false, LAYOUT, true>(p, wc, stream);
        return p.f16 ? launch_zt<128, 2, true, LAYOUT, false>(p, wc, stream)
                     : launch_zt<128, 2, false, LAYOUT, false>(p, wc, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_prefill_tc(const Problem& p, const WaitCtl& wc, cudaStream_t stream) {
    if (prefill_narrow_supported(p)) return launch_prefill_narrow(p, wc, stream);
    if (p.page_table != nullptr) return launch_layout<kPaged>(p, wc, stream);
    if (p.cu_seqlens != nullptr) return launch_layout<kPacked>(p, wc, stream);
    return launch_layout<kHeadMajor>(p, wc, stream);
}

}  // namespace attn
