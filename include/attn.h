/*
 * attn.h -- C ABI of the GB300 (sm_103a) multi-head scaled-dot-product attention library.
 *
 * The library is libattn.so.  Every entry point takes plain device pointers and
 * sizes; no framework types cross this boundary.
 *
 * What attn_fwd computes, for every batch b, query head h and query row i:
 *
 *   out[b,h,i,:] = sum_j w_j * V[b, h/G, j, :]
 *   w_j = exp(s_j - max) / sum_k exp(s_k - max)    over the keys j allowed for (b, i)
 *   s_j = scale * <Q[b,h,i,:], K[b, h/G, j, :]>
 *
 * with G = q_heads / kv_heads.  A disallowed key has weight exactly 0, and a row
 * with no allowed key is all zeros.
 *
 * Sources (web pages on attention back ends):
 *   - ferrum-kernels Backend::flash_attention: the statement of the operation, taking
 *     (q, k, v, out, batch, q_len, kv_len, pos_offset, cfg).  The cfg struct is not
 *     given there; its fields are the flat arguments below.
 *   - ripvec-core Driver::fused_scale_mask_softmax: softmax(scores * scale + mask).
 *   - ripvec-core Driver::fused_scale_mask_softmax_windowed: the symmetric window.
 *   - ripvec-core Driver::build_attn_mask: the key-padding mask.
 *   - ferrum-kernels Backend::flash_attention_batched_per_cache: the device kv_lens
 *     and the decode sliding window.
 *   - realizar cached/attention.rs, parallel_multihead_attention_gpu_cached and
 *     batched_causal_softmax: the three stages and the causal softmax.
 */
#ifndef ATTN_H
#define ATTN_H

#include <stdint.h>

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes.  Every entry point returns one of these. */
typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1, /* argument check failed; nothing was launched */
    ATTN_ERR_UNSUPPORTED = 2, /* valid, but no kernel for this head_dim / dtype; nothing launched */
    ATTN_ERR_CUDA = 3,        /* a CUDA runtime or driver call failed */
    ATTN_ERR_TIMEOUT = 4      /* a bounded device-side wait gave up (see attn_sync_status) */
} attn_status;

/*
 * Mask modes.  A query row i sits at absolute position pos_offset + i.  Keys sit
 * at positions 0 .. kv_len-1.  Key padding (key_lens) applies in every mode.
 */
typedef enum {
    /* Every key is visible: bidirectional encoder attention. */
    ATTN_MASK_NONE = 0,

    /* Key j is visible when j <= pos_offset + i.
     * Source: realizar batched_causal_softmax, where row i sees 0..=i;
     * ferrum-kernels Backend::qk_norm_rope, where token i has position pos_offset + i. */
    ATTN_MASK_CAUSAL = 1,

    /* Key j is visible when |pos_offset + i - j| <= window/2, with window/2 rounded down.
     * window == 0 means no window.
     * Source: ripvec-core Driver::fused_scale_mask_softmax_windowed. */
    ATTN_MASK_WINDOW = 2,

    /* Key j is visible when pos_offset + i - window < j <= pos_offset + i.
     * window == 0 means plain causal.
     * Source: ferrum-kernels flash_attention_batched_per_cache, sliding_window
     * (the last w valid positions). */
    ATTN_MASK_CAUSAL_WINDOW = 3
} attn_mask_mode;

/* Element type of q, k, v and out.  Accumulation is always fp32.
 * ATTN_F16 follows the pages' CUDA activation type (ferrum-kernels
 * activation_elem_size_bytes: fp16 on CUDA; ripvec-core's _f16 kernels with fp32
 * reductions).  bf16 and fp16 take the same kernels and the same shape rules. */
typedef enum { ATTN_BF16 = 0, ATTN_F32 = 1, ATTN_F16 = 2 } attn_dtype;

/*
 * attn_fwd -- enqueue one attention forward pass on cuda_stream and return.
 *
 * Layout.  All tensors are contiguous, row-major, head-major, in caller-owned
 * device memory:
 *   q, out   [batch, q_heads, q_len, head_dim]
 *   k, v     [batch, kv_heads, kv_len, head_dim]
 *   key_lens [batch] int32, or NULL.  key_lens[b] keys of sequence b are valid
 *            (values outside [0, kv_len] are clamped to that range).  NULL means
 *            all kv_len keys are valid.
 *
 * Query head h reads key/value head h / (q_heads / kv_heads), so each kv head
 * serves a contiguous group of query heads (grouped-query attention).
 *
 * Arguments:
 *   scale       The multiplier applied to the raw dot products.  Any finite
 *               value is accepted; 0 gives uniform weights over the visible keys.
 *               The usual value is 1/sqrt(head_dim).
 *   dtype       An attn_dtype.
 *   cuda_stream A cudaStream_t.  NULL means the legacy default stream.
 *
 * Supported shapes:
 *   - bf16 and fp16 need head_dim 64 or 128, and the base addresses of q, k, v and out
 *     aligned to 16 bytes.
 *   - f32 accepts any head_dim from 1 to 256, with 4-byte alignment.
 *   - batch or q_len 0: nothing is launched and ATTN_OK is returned.
 *   - kv_len 0: no row sees a key, so out is zero-filled (cudaMemsetAsync on the stream).
 *
 * Ownership and lifetime.  The library keeps no pointer after the call returns,
 * and allocates no device memory.  The buffers must stay valid until the stream
 * work completes.  out must not alias q, k or v.
 *
 * Non-finite values.  Key and value rows that no query of the call can see (rows at
 * or past key_lens[b], and rows outside every query's mask band, e.g. cache rows
 * past pos_offset + q_len - 1 under a causal mask) never influence out, whatever
 * they hold: the kernels zero such value rows in shared memory before the
 * tensor-core product, since 0 * Inf and 0 * NaN are NaN there.  A row that some
 * query sees takes part in the products of its neighbours' rows with weight 0, so
 * an Inf or NaN in it also reaches rows that do not see it.
 *
 * Errors.  Arguments are checked before any launch:
 *   - null pointers, negative sizes, q_heads % kv_heads != 0, a mask_mode or dtype
 *     out of range, a negative window or pos_offset, a non-finite scale, or a
 *     misaligned pointer give ATTN_ERR_INVALID_ARG;
 *   - an unsupported head_dim for the dtype gives ATTN_ERR_UNSUPPORTED;
 *   - a failed launch gives ATTN_ERR_CUDA.
 * After any non-OK status, attn_last_error() describes it.
 *
 * The call is asynchronous; errors inside the kernels are reported by
 * attn_sync_status().  There is no host or CPU fallback: a shape with no kernel
 * is refused.  Source: ferrum-kernels, the CUDA ops that fail rather than copy
 * through host memory.
 */
ATTN_API attn_status attn_fwd(const void* q, const void* k, const void* v, void* out,
                     int batch, int q_heads, int kv_heads, int q_len, int kv_len, int head_dim,
                     int pos_offset, int mask_mode, int window, const int32_t* key_lens,
                     float scale, int dtype, void* cuda_stream);

/*
 * attn_fwd_out_token_major -- attn_fwd with the output written token-major.
 *
 * Source: ferrum-kernels Backend::transpose_head_to_token, which turns the head-major
 * attention output [heads, tokens, head_dim] into [tokens, heads * head_dim] for the output
 * projection; here that transposition is part of the kernels' store, so no extra pass exists.
 *
 * Every argument, check and status is the one attn_fwd has, except the layout of out:
 *   out  [batch, q_len, q_heads, head_dim]   (row (b, i) holds all heads of query i)
 * and the same value out_token_major[b][i][h][:] == out_head_major[b][h][i][:].  For
 * q_len 1 the two layouts are the same bytes.  kv_len 0 zero-fills out.
 */
ATTN_API attn_status attn_fwd_out_token_major(const void* q, const void* k, const void* v, void* out,
                     int batch, int q_heads, int kv_heads, int q_len, int kv_len, int head_dim,
                     int pos_offset, int mask_mode, int window, const int32_t* key_lens,
                     float scale, int dtype, void* cuda_stream);

/*
 * attn_fwd_varlen -- attention over a batch of packed (unpadded) sequences.
 *
 * Source: ripvec-core Driver::prepare_batch_unpadded, which concatenates all tokens flat
 * and returns cu_seqlens for the attention boundaries; there attention pads around the
 * per-head operations (fused_pad_qkv_split_f16: [total_tokens, 3*hidden] to
 * [batch*heads, max_seq, head_dim]) and unpads afterwards (fused_reshape_unpad_f16).
 * Here attention works on the flat layout directly, so neither copy exists and no
 * padded query row is computed.
 *
 * Layout (caller-owned device memory, contiguous, token-major):
 *   q, out      [total, q_heads, head_dim]   (hidden = q_heads * head_dim per token)
 *   k, v        [total, kv_heads, head_dim]
 *   cu_seqlens  [batch + 1] int32 in device memory: sequence b is rows
 *               [cu_seqlens[b], cu_seqlens[b+1]) of every tensor.
 *
 * Each sequence attends to itself: query row i of sequence b sees key rows of the same
 * sequence by mask_mode and window exactly as attn_fwd does with pos_offset 0 and no
 * key padding (causal: j <= i; window modes as in attn_mask_mode).  Query head h reads
 * kv head h / (q_heads / kv_heads).  Rows of out outside every sequence are not written.
 *
 * Arguments:
 *   batch       number of sequences.
 *   total       rows of q, k, v and out.
 *   max_seqlen  an upper bound on every sequence length; it sizes the launch.
 *   scale, dtype, cuda_stream: as for attn_fwd.  dtype must be ATTN_BF16 or ATTN_F16.
 *
 * Supported: head_dim 64 or 128, 16-byte aligned q, k, v, out, 4-byte aligned
 * cu_seqlens; otherwise ATTN_ERR_UNSUPPORTED (fp32, other head_dim) or
 * ATTN_ERR_INVALID_ARG.  batch 0 or max_seqlen 0 launches nothing.
 *
 * Errors: host-visible arguments are checked before the launch (max_seqlen > total is
 * ATTN_ERR_INVALID_ARG).  cu_seqlens lives on the device and is checked there: a
 * sequence with cu_seqlens[b] < 0, cu_seqlens[b+1] < cu_seqlens[b], cu_seqlens[b+1] >
 * total or a length above max_seqlen is not read and its rows are not written, and
 * attn_sync_status() reports ATTN_ERR_INVALID_ARG.
 *
 * The library allocates nothing and keeps no pointer after the call.
 */
ATTN_API attn_status attn_fwd_varlen(const void* q, const void* k, const void* v, void* out,
                                     const int32_t* cu_seqlens, int batch, int total, int max_seqlen,
                                     int q_heads, int kv_heads, int head_dim, int mask_mode, int window,
                                     float scale, int dtype, void* cuda_stream);

/* qk_mode of attn_qkv_prelude (ferrum-kernels Backend::split_qkv_norm_rope). */
typedef enum {
    ATTN_QK_COPY = 0,              /* Q and K are only split and transposed, like V */
    ATTN_QK_NORM_ROPE = 1,         /* per-head RMS norm, then half-split RoPE (QK-norm models) */
    ATTN_QK_ROPE = 2,              /* half-split RoPE only: element j pairs with j + head_dim/2 */
    ATTN_QK_ROPE_INTERLEAVED = 3   /* interleaved RoPE only: element 2j pairs with 2j + 1 */
} attn_qk_mode;

/*
 * attn_qkv_prelude -- the step before attention, in one pass: split the fused QKV
 * projection, apply the per-head RMS norm and RoPE to Q and K, and write Q, K and V
 * head-major, K and V optionally straight into KV caches.
 *
 * Source: ferrum-kernels Backend::split_qkv_norm_rope (fused split-QKV + QK-norm + RoPE +
 * head-major transpose) and Backend::split_qkv_norm_rope_into_cache (the same, writing K
 * and V into pre-allocated head-major caches at rows cache_len .. cache_len + tokens - 1,
 * in place of kv_cache_append_head_major); Backend::qk_norm_rope for the per-head RMS norm
 * and the positions pos_offset + i.
 *
 * Layout (caller-owned device memory, contiguous):
 *   qkv       [tokens, q_heads*head_dim + 2*kv_heads*head_dim]: Q, then K, then V per token
 *   q_out     [q_heads, tokens, head_dim]
 *   k_out, v_out
 *             cache_capacity == 0: [kv_heads, tokens, head_dim];
 *             cache_capacity  > 0: caches [kv_heads, cache_capacity, head_dim], rows
 *             cache_len .. cache_len + tokens - 1 written, every other row untouched.
 *   cos, sin  fp32 [rope_positions, head_dim/2]: row p holds cos and sin of the angles of
 *             position p, column j the angle of rotation pair j.  Read for qk_mode != 0.
 *   q_norm_w, k_norm_w
 *             fp32 [head_dim]: RMS-norm weights shared by every head.  Read for qk_mode 1.
 *
 * Per token t (position p = pos_offset + t) and head of Q or K:
 *   qk_mode 1: x <- x / sqrt(mean(x^2) + eps) * w, then half-split rotation;
 *   qk_mode 2: half-split rotation; qk_mode 3: interleaved rotation; qk_mode 0: none.
 * A rotation pair (a, b) with angle index j becomes (a cos[p][j] - b sin[p][j],
 * b cos[p][j] + a sin[p][j]).  V is always copied.  Arithmetic is fp32; results are
 * rounded to the input type.
 *
 * Arguments: dtype is ATTN_BF16 or ATTN_F16 (for qkv and every output).  head_dim 64 or
 * 128; otherwise ATTN_ERR_UNSUPPORTED.  tokens 0 launches nothing.
 *
 * Errors (checked before the launch, ATTN_ERR_INVALID_ARG): negative sizes or offsets,
 * qk_mode outside 0..3, pos_offset + tokens > rope_positions when a rotation is applied,
 * cache_len + tokens > cache_capacity, eps negative or not finite (qk_mode 1), null or
 * misaligned pointers (16 bytes for qkv, the outputs, cos and sin; 4 bytes for the norm
 * weights).  The outputs must not overlap qkv.
 *
 * The library allocates nothing and keeps no pointer after the call.
 */
ATTN_API attn_status attn_qkv_prelude(const void* qkv, const float* q_norm_w, const float* k_norm_w,
                                      const float* cos, const float* sin, int rope_positions, void* q_out,
                                      void* k_out, void* v_out, int tokens, int q_heads, int kv_heads,
                                      int head_dim, int pos_offset, float eps, int qk_mode, int cache_len,
                                      int cache_capacity, int dtype, void* cuda_stream);

/*
 * attn_qkv_prelude_caches -- the decode-step prelude for m items with per-item KV caches,
 * in one launch: item i's single token is row i of qkv, its position is cache_lens[i], its
 * Q goes to q_out item-major and its K and V are appended at row cache_lens[i] of its own
 * caches.  The output feeds attn_decode_caches (with kv_lens[i] = cache_lens[i] + 1).
 *
 * Source: ferrum-kernels Backend::split_qkv_norm_rope_into_cache (split, QK norm, RoPE,
 * K/V straight into the cache), Backend::qk_norm_rope_batched_per_item (per-item
 * positions from a device buffer, item-major Q) and
 * Backend::kv_cache_append_batched_per_cache (each item writes its row into its own cache
 * at the offset read from cache_lens[i]).
 *
 * Layout: qkv [m, q_heads*head_dim + 2*kv_heads*head_dim]; q_out [m, q_heads, head_dim];
 * k_caches, v_caches device arrays of m device pointers to [kv_heads, capacity, head_dim]
 * caches (16-byte aligned); cache_lens device int32 [m].  cos, sin, q_norm_w, k_norm_w,
 * qk_mode, eps and dtype as for attn_qkv_prelude.
 *
 * Errors: host-visible arguments as for attn_qkv_prelude (capacity must be positive).
 * Items are checked on the device: an item whose cache_lens[i] is outside [0, capacity),
 * or (with a rotation) at or past rope_positions, or whose cache pointer is null or
 * misaligned, is neither read nor written, and attn_sync_status() reports
 * ATTN_ERR_INVALID_ARG.
 *
 * The library allocates nothing and keeps no pointer after the call.
 */
ATTN_API attn_status attn_qkv_prelude_caches(const void* qkv, const float* q_norm_w, const float* k_norm_w,
                                             const float* cos, const float* sin, int rope_positions, void* q_out,
                                             const void* const* k_caches, const void* const* v_caches,
                                             const int32_t* cache_lens, int m, int q_heads, int kv_heads,
                                             int head_dim, int capacity, float eps, int qk_mode, int dtype,
                                             void* cuda_stream);

/*
 * attn_fwd_varlen_paged -- attention of packed multi-token query chunks against paged KV
 * caches: chunked prefill and multi-token verification over the caches of attn_decode_paged.
 *
 * Source: ferrum-kernels Backend::transpose_token_to_head names the CUDA paged-KV path,
 * paged_varlen_attention, whose output is token-major, and paged_decode_attention built on
 * it; the pages give no layout.  The reading taken here: the queries are packed as in
 * attn_fwd_varlen (ripvec-core Driver::prepare_batch_unpadded, cu_seqlens), the caches are
 * the pages of attn_decode_paged, and a sequence's queries are the newest positions of its
 * cache (its tokens were appended before the call, as ferrum-kernels
 * Backend::split_qkv_norm_rope_into_cache does).
 *
 * Layout (caller-owned device memory, contiguous):
 *   q, out        [total_q, q_heads, head_dim], token-major; sequence b's queries are rows
 *                 [cu_seqlens_q[b], cu_seqlens_q[b+1]).
 *   k_pool, v_pool
 *                 [num_pages, kv_heads, page_size, head_dim]; sequence b's cached position j is
 *                 row j % page_size of pool page page_table[b][j / page_size].
 *   page_table    device int32 [batch, max_pages].  Pages may be shared.
 *   cu_seqlens_q  device int32 [batch + 1].
 *   kv_lens       device int32 [batch]: the cached positions of sequence b, clamped to
 *                 [0, max_pages * page_size], its len_b = cu_seqlens_q[b+1] - cu_seqlens_q[b]
 *                 queries included.
 *
 * Query i of sequence b sits at position kv_lens[b] - len_b + i and sees the cached
 * positions that mask_mode and window allow at that position (attn_mask_mode): causal for
 * chunked prefill, the causal window for a sliding-window model.  Query head h reads kv head
 * h / (q_heads / kv_heads).  Rows of out outside every sequence are not written.
 *
 * Arguments: batch (sequences), total_q (rows of q and out), max_seqlen_q (an upper bound on
 * every len_b; it sizes the launch), num_pages, page_size (>= 1), max_pages, mask_mode,
 * window, scale, dtype (ATTN_BF16 or ATTN_F16), cuda_stream as for attn_fwd.
 *
 * Supported: head_dim 64 or 128; otherwise ATTN_ERR_UNSUPPORTED.  batch 0 or max_seqlen_q 0
 * launches nothing.  Key rows no query sees never reach out, whatever they hold.  Pages of 8
 * to 128 rows that divide 128, or of a multiple of 128 rows, are copied a page piece at a time
 * by TMA; other page sizes are gathered row by row, at about a third of the speed.
 *
 * Errors: host-visible arguments are checked before the launch (ATTN_ERR_INVALID_ARG for
 * negative sizes, page_size < 1, max_pages * page_size above 2^31-1, max_seqlen_q >
 * total_q, null or misaligned pointers: 16 bytes for q, out and the pools, 4 bytes for the
 * int32 arrays).  Device-side values are checked on the device and reported by
 * attn_sync_status() as ATTN_ERR_INVALID_ARG:
 *   - a sequence whose cu_seqlens_q bounds are not inside [0, total_q], run backwards or
 *     exceed max_seqlen_q is not read and its rows are not written;
 *   - a sequence with fewer cached positions than queries, or with a page-table entry
 *     outside [0, num_pages) among the positions its queries see, reads nothing and its rows
 *     are written as zeros.
 *
 * The result equals attn_fwd per sequence over the gathered cache (q_len len_b, pos_offset
 * kv_lens[b] - len_b, key_lens kv_lens[b]).  At head_dim 128 both run the same prefill kernel;
 * where they also split the keys into the same 128-key tiles (a causal mask, or a page size
 * that is gathered row by row: not 8..128 dividing 128, nor a multiple of 128) they agree bit
 * for bit, otherwise to rounding.
 * The library allocates nothing and keeps no pointer after the call.
 */
ATTN_API attn_status attn_fwd_varlen_paged(const void* q, const void* k_pool, const void* v_pool,
                                           const int32_t* page_table, void* out, const int32_t* cu_seqlens_q,
                                           const int32_t* kv_lens, int batch, int total_q, int max_seqlen_q,
                                           int q_heads, int kv_heads, int num_pages, int page_size,
                                           int max_pages, int head_dim, int mask_mode, int window, float scale,
                                           int dtype, void* cuda_stream);

/*
 * attn_decode_caches -- one decode step for m items, each against its own KV cache, in
 * one launch.
 *
 * Source: ferrum-kernels Backend::flash_attention_batched_per_cache, the batched decode
 * across M per-request caches that replaces the per-item flash_attention(q_len=1) loop.
 *
 * Arguments:
 *   q, out     [m, q_heads, head_dim] bf16 or fp16, item-major, contiguous, 16-byte aligned.
 *   k_caches, v_caches
 *              Device arrays of m device pointers.  Item i's K (and V) cache is
 *              [kv_heads, capacity, head_dim] of the same type, head-major and contiguous; each
 *              pointer must be 16-byte aligned.
 *   kv_lens    Device int32 [m]: the valid cached positions of item i.  The value is
 *              clamped to [0, capacity].  It is read on the device, so a captured launch
 *              replays with new lengths written between launches.
 *   sliding_window
 *              0: item i's query, the newest position kv_lens[i]-1, sees positions
 *              0 .. kv_lens[i]-1.  w > 0: it sees only the last w of them.
 *   scale      Finite multiplier of the raw dot products.
 *   dtype      ATTN_BF16 or ATTN_F16.
 *
 * Query head h reads kv head h / (q_heads / kv_heads).
 *
 * Supported: head_dim 64 or 128, and q_heads / kv_heads in {1, 2, 4, 8}; otherwise
 * ATTN_ERR_UNSUPPORTED.  An item with kv_lens[i] == 0 gets zeros.  capacity 0 zero-fills
 * out.
 *
 * Errors: host-visible arguments are checked as for attn_fwd.  A null or misaligned
 * pointer inside the device arrays is found on the device: that item is not read,
 * its output is zeros, and attn_sync_status() reports ATTN_ERR_INVALID_ARG.
 *
 * Workspace: at head_dim 128 with 4 or 8 query heads per kv head the caches are copied by
 * TMA through one K and one V tensor map per item, which a kernel writes on the device
 * (only the device holds the caches' addresses).  The call takes m * 256 bytes for them
 * with cudaMallocAsync on cuda_stream and gives them back with cudaFreeAsync on the same
 * stream after the launch; an allocation failure returns ATTN_ERR_CUDA.  Other shapes
 * allocate nothing.  The library keeps no pointer after the call.
 */
ATTN_API attn_status attn_decode_caches(const void* q, const void* const* k_caches, const void* const* v_caches,
                                        void* out, int m, int q_heads, int kv_heads, int capacity, int head_dim,
                                        const int32_t* kv_lens, int sliding_window, float scale, int dtype,
                                        void* cuda_stream);

/*
 * attn_decode_caches_noalloc -- attn_decode_caches without any allocation.
 *
 * Source: none.  The pages have no counterpart; this is a deployment variant of
 * attn_decode_caches (same arguments, same results bit for bit).
 *
 * Where attn_decode_caches takes a stream-ordered workspace for the per-item tensor maps
 * (head_dim 128, 4 or 8 query heads per kv head), this call writes them into a fixed table
 * in the library's device memory, room for ATTN_NOALLOC_MAX_ITEMS items (1 MB).  It calls no
 * allocation routine.  The table's address is looked up once per device
 * (cudaGetSymbolAddress; a failure returns ATTN_ERR_CUDA).  Nothing in it has to start at
 * zero: every map an item uses is written, on cuda_stream, before the decode reads it.
 *
 * Calls whose launches overlap on the GPU (different streams, or devices' work not ordered
 * by the caller) share the table and race: order them, for example on one stream.
 *
 * Errors: as attn_decode_caches, and ATTN_ERR_INVALID_ARG for m > ATTN_NOALLOC_MAX_ITEMS.
 */
#define ATTN_NOALLOC_MAX_ITEMS 4096
ATTN_API attn_status attn_decode_caches_noalloc(const void* q, const void* const* k_caches,
                                                const void* const* v_caches, void* out, int m, int q_heads,
                                                int kv_heads, int capacity, int head_dim, const int32_t* kv_lens,
                                                int sliding_window, float scale, int dtype, void* cuda_stream);

/*
 * attn_decode_paged -- attn_decode_caches over paged KV caches: every item's cache lives in
 * fixed-size pages of two shared pools, addressed through a per-item page table.
 *
 * Source: the pages name ferrum-kernels' paged decode path (paged_decode_attention over
 * paged_varlen_attention) without giving its layout.  The reading taken here keeps the
 * per-item cache form of flash_attention_batched_per_cache, [kv_heads, capacity, head_dim],
 * and cuts it into pages of page_size positions: a page is [kv_heads, page_size, head_dim].
 *
 * Arguments:
 *   q, out      [m, q_heads, head_dim] bf16 or fp16, item-major, contiguous, 16-byte aligned.
 *   k_pool, v_pool
 *               [num_pages, kv_heads, page_size, head_dim] of the same type, contiguous,
 *               16-byte aligned.
 *   page_table  Device int32 [m, max_pages]: item i's positions j*page_size .. (j+1)*page_size-1
 *               are rows 0 .. page_size-1 of pool page page_table[i][j].  Pages may be shared
 *               between items.  Only the entries of an item's visible positions are read.
 *   kv_lens     Device int32 [m]: the valid positions of item i, clamped to
 *               [0, max_pages * page_size].
 *   sliding_window, scale, dtype
 *               As attn_decode_caches: item i's query is the newest position kv_lens[i]-1 and
 *               sees all of its positions, or only the last sliding_window of them.
 *
 * Query head h reads kv head h / (q_heads / kv_heads).  The result equals
 * attn_decode_caches over caches gathered from the pages, bit for bit.
 *
 * Supported: as attn_decode_caches (head_dim 64 or 128, q_heads / kv_heads in {1, 2, 4, 8});
 * page_size >= 1.  An item with kv_lens[i] == 0 gets zeros.  max_pages * page_size == 0
 * zero-fills out.
 *
 * Errors: host-visible arguments are checked as for attn_decode_caches (null or misaligned
 * pointers, negative sizes, page_size < 1, max_pages * page_size above 2^31-1).  A visible
 * page-table entry outside [0, num_pages) is found on the device: that item is not read, its
 * output is zeros, and attn_sync_status() reports ATTN_ERR_INVALID_ARG.
 *
 * The library allocates nothing and keeps no pointer after the call.
 */
ATTN_API attn_status attn_decode_paged(const void* q, const void* k_pool, const void* v_pool,
                                       const int32_t* page_table, void* out, int m, int q_heads, int kv_heads,
                                       int num_pages, int page_size, int max_pages, int head_dim,
                                       const int32_t* kv_lens, int sliding_window, float scale, int dtype,
                                       void* cuda_stream);

/*
 * attn_last_error -- message for the last non-OK status returned on this host thread.
 * The string belongs to the library and stays valid until the next call on this
 * thread.  The result is "" when there has been no error.
 */
ATTN_API const char* attn_last_error(void);

/*
 * attn_sync_status -- wait for cuda_stream, then read and clear the library's
 * device status word on the current device.
 *
 * Every wait of a kernel on a shared-memory barrier (data arriving, the tensor
 * core finishing, another warp's result) is bounded: it gives up after 250 ms (a
 * healthy wait lasts microseconds), so a launch whose waits fail ends after about
 * that long per wave of blocks.  A wait that gives up
 * records a code in this word, waits (again bounded) for its own copies and
 * products in flight, releases its tensor memory and exits its block.  The
 * hardware barriers (a block's __syncthreads, the decode kernels' cluster
 * barrier, and the prefill kernel's barrier between the two halves of a row) are
 * not bounded; every thread meets each of them on every path, including a path
 * that gave up.
 *
 * The word is one per device, shared by every call and every stream on it; the
 * first code recorded wins until this call clears it.  This call synchronises only
 * cuda_stream: a caller that uses several streams should synchronise all of them
 * (or the device) before it trusts the code, which may come from a kernel on any
 * of them.
 *
 * Returns:
 *   - ATTN_ERR_TIMEOUT when a wait gave up;
 *   - ATTN_ERR_INVALID_ARG when a kernel found a bad device-side argument
 *     (a per-item cache pointer, a page-table entry, cu_seqlens or a cache length);
 *   - ATTN_ERR_CUDA when the stream reported an error;
 *   - ATTN_OK otherwise.
 * Source: ferrum-kernels Backend::sync, where sync is separate from the launch.
 */
ATTN_API attn_status attn_sync_status(void* cuda_stream);

/*
 * attn_selftest_timeout -- exercise the bounded-wait path on the device.
 *
 * Launches one block that waits on a shared-memory barrier that nothing
 * signals, with a wait limit of limit_us microseconds (1 to 1,000,000).  The
 * wait gives up, records ATTN_ERR_TIMEOUT in the status word, and the block
 * exits normally.  The caller then reads the code with attn_sync_status().
 * This never faults or hangs the device.
 * Returns ATTN_ERR_INVALID_ARG for a limit out of range, ATTN_ERR_CUDA on a
 * launch failure, and ATTN_OK once enqueued.
 */
ATTN_API attn_status attn_selftest_timeout(int limit_us, void* cuda_stream);

/*
 * attn_version -- library version as major*10000 + minor*100 + patch.
 */
ATTN_API int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H */
