/*
 * dflash_attn.h -- C ABI of libdflash_attn: DFlash block attention on one GPU.
 *
 * The operation. In DFlash speculative decoding every request contributes a
 * block of T = 1 + num_speculative_tokens queries (the bonus token plus the
 * mask tokens; kenforever1 "dflash-gemma4-31b-notes", section "why non-causal
 * attention": "num_query_per_req = 1 + num_speculative_tokens"). The block is
 * processed as a whole: in the draft pass the queries come from the query
 * embeddings and the context K/V from the target's hidden states; in the
 * verify pass the block attends to the target's paged KV cache (same page,
 * code comment "DFlash cross-attention"). Attention is non-causal by default
 * ("DFlash verify/block attention needs causal=False", same page, PR #52
 * table) with a causal switch (prhub report on vLLM PR #43445 "Allow causal
 * DFlash", implementation steps 1-3: causal defaults to False). head_dim goes
 * up to 512 (Gemma 4 31B global layers, same page, section "Global head_dim
 * 512"), and sliding-window layers are supported (same page, hybrid attention).
 *
 * Definition computed (exact attention, fp32 accumulation on the GPU):
 *   request b has L_b = seq_lens[b] keys, the block's own T keys being the
 *   last T of them; block query i sits at position p_i = L_b - T + i.
 *   Query head h reads KV head g = h / (Hq / Hkv).
 *   Key j is visible to query i iff lo_i <= j <= hi_i with
 *     hi_i = causal ? p_i : L_b - 1
 *     lo_i = window > 0 ? max(0, p_i - window + 1) : 0
 *   s_j = scale * <q_i, k_j>; out_i = sum_j softmax(s)_j v_j;
 *   lse_i = log(sum_j exp(s_j))  (natural log).
 *   Key j of request b is slot j % page_size of page page_table[b][j / page_size].
 *
 * Split-KV (flash-decoding style; cf. the FlashAttention "split-KV combine"
 * of the prhub report on vLLM PR #52816 "DFlash2", review highlights). The
 * union key range of request b, [lo_b, L_b) with lo_b = window > 0 ?
 * max(0, L_b - T - window + 1) : 0, is cut into S chunks: base_b =
 * lo_b rounded down to a multiple of page_size, chunk_b = ceil(ceil((L_b -
 * base_b) / S) / page_size) * page_size, chunk c = [base_b + c*chunk_b,
 * base_b + (c+1)*chunk_b) clipped to [lo_b, L_b). Each chunk yields a partial
 * (o_c, lse_c) over its visible keys (o_c normalised; lse_c = -inf and o_c = 0
 * when the chunk holds no visible key), and the combine is
 *   m = max_c lse_c, w_c = exp(lse_c - m), out = sum_c w_c o_c / sum_c w_c,
 *   lse = m + log(sum_c w_c).
 *
 * Conventions for every call:
 *   - All pointers named "device" are CUDA device pointers owned by the
 *     caller; the library allocates nothing, never synchronises the stream and
 *     keeps no state between calls (re-entrant).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).
 *   - Arguments are validated on the host before anything is launched; an
 *     invalid argument returns an error code and launches nothing. The text of
 *     the last error of the calling thread is available from
 *     dflash_last_error_message().
 *   - Values the host cannot see (page ids, seq_lens) are checked on the
 *     device: an out-of-range page id is never dereferenced (its keys read as
 *     zero) and a seq_len outside [T, min(max_seq_len, max_pages*page_size)]
 *     makes the request produce zeros; both set bits in the error word of the
 *     workspace, read with dflash_read_error(). An unsupported combination
 *     returns DFLASH_ERR_UNSUPPORTED; the library never falls back to a
 *     different mask.
 */
#ifndef DFLASH_ATTN_H
#define DFLASH_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define DFLASH_API __attribute__((visibility("default")))
#else
#define DFLASH_API
#endif

#define DFLASH_ABI_VERSION 2
#define DFLASH_MAX_HEAD_DIM 512
#define DFLASH_MAX_BLOCK_LEN 64
#define DFLASH_MAX_SPLITS 256

typedef enum dflash_status {
    DFLASH_OK = 0,
    DFLASH_ERR_INVALID_ARG = 1,  /* bad pointer, size, stride, dtype or scalar */
    DFLASH_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. head_dim not a multiple of 16) */
    DFLASH_ERR_CUDA = 3,         /* a CUDA runtime call or kernel launch failed */
    DFLASH_ERR_DEVICE_CHECK = 4, /* the device saw a bad page id / seq_len (dflash_read_error) */
    DFLASH_ERR_WORKSPACE = 5     /* workspace missing, misaligned or too small */
} dflash_status;

typedef enum dflash_dtype {
    DFLASH_BF16 = 0, /* q, k_cache, v_cache, out in bfloat16 */
    DFLASH_FP32 = 1  /* q, k_cache, v_cache, out in float32 */
} dflash_dtype;

/* Which kernel computes the attention. For bf16, AUTO packs each KV head's
   query heads x block positions into tensor-core tiles: one CTA per tile
   (TC, up to 80 rows) or, when that would split the rows into more groups
   that each read all of the K/V (e.g. 8 heads x 16 positions at head_dim
   512), a CTA pair sharing 2-SM MMAs (TC_PAIR, up to 128 rows, head_dim
   256/512, uniform split plans). fp32, and shapes neither covers, run on the
   CUDA-core kernel (SIMT). SIMT, TC and TC_PAIR force that kernel; TC and
   TC_PAIR are bf16 only and return DFLASH_ERR_UNSUPPORTED for shapes they do
   not cover (page size 16/32/64; TC: head_dim 128/256/512). All kernels
   compute the same definition. */
typedef enum dflash_kernel {
    DFLASH_KERNEL_AUTO = 0,
    DFLASH_KERNEL_SIMT = 1,
    DFLASH_KERNEL_TC = 2,
    DFLASH_KERNEL_TC_PAIR = 3
} dflash_kernel;

/* Device-side error bits accumulated (bitwise OR) in the workspace error word. */
#define DFLASH_DEVERR_PAGE_ID 1u     /* page_table entry outside [0, num_pages) */
#define DFLASH_DEVERR_SEQ_LEN 2u     /* seq_lens[b] < T or above the stated bounds */
#define DFLASH_DEVERR_TIMEOUT 4u     /* a bounded pipeline wait gave up (kernel returned early) */
#define DFLASH_DEVERR_TOKEN_ID 8u    /* a token id outside [0, vocab) (read as token 0) */

/* Sizes and layout of one call. All counts are elements, not bytes. */
typedef struct dflash_dims {
    int32_t batch;          /* B, requests (>= 1) */
    int32_t num_q_heads;    /* Hq (>= 1) */
    int32_t num_kv_heads;   /* Hkv, divides Hq; query head h reads KV head h / (Hq/Hkv) */
    int32_t head_dim;       /* D, multiple of 16, <= 512 */
    int32_t page_size;      /* tokens per page, multiple of 8, <= 256 */
    int32_t num_pages;      /* pages in the K/V pool (first extent of k_cache) */
    int32_t max_pages;      /* columns of page_table (row stride of page_table) */
    int32_t max_seq_len;    /* host-known upper bound on every seq_lens[b]; <= max_pages*page_size.
                               Only used to plan the split count; 0 = max_pages*page_size */
    dflash_dtype dtype;     /* element type of q, k_cache, v_cache and out */
    int64_t kv_stride_page; /* k_cache/v_cache element stride between pages */
    int64_t kv_stride_slot; /* ... between token slots of one page */
    int64_t kv_stride_head; /* ... between KV heads; head_dim is contiguous (stride 1) */
} dflash_dims;

/* Per-call options; pass NULL for the defaults (auto splits, auto kernel, no
   workspace -- only valid when the plan needs none, see dflash_workspace_bytes). */
typedef struct dflash_opts {
    int32_t num_splits;     /* 0 = auto (from the SM count and sizes); n >= 1 = exactly n chunks */
    int32_t kernel;         /* a dflash_kernel value */
    void* workspace;        /* device memory, 256-byte aligned, dflash_workspace_bytes() long.
                               Holds the error word and the split partials. Must be zeroed
                               (e.g. cudaMemset) once before its first use; the library keeps
                               its counters at zero between calls. */
    size_t workspace_bytes; /* size of workspace in bytes */
    void* stream;           /* cudaStream_t; NULL = legacy default stream */
    uint32_t wait_limit_us; /* bound of every device-side wait of the tensor-core kernels
                               (pipeline hand-offs and the in-kernel split combine's arrival
                               wait), in microseconds; 0 = the default of 2 s. A wait that
                               runs out sets DFLASH_DEVERR_TIMEOUT and the kernel returns. */
} dflash_opts;

/*
 * Block attention for a batch of DFlash blocks over a paged KV cache.
 *
 *   q          device, [B*T, Hq, D] contiguous, dims->dtype. Rows b*T .. b*T+T-1
 *              are request b's block (query i at row b*T+i).
 *   k_cache    device, element (page, slot, head, d) at
 *              page*kv_stride_page + slot*kv_stride_slot + head*kv_stride_head + d,
 *              dims->dtype; 16-byte aligned base, strides multiples of 8 elements.
 *   v_cache    device, same layout and dtype as k_cache.
 *   page_table device, int32 [B, max_pages] row-major; entries past
 *              ceil(L_b/page_size) are never read.
 *   seq_lens   device, int32 [B]; L_b counts the block's own T keys (L_b >= T).
 *   block_len  T, 1 <= T <= DFLASH_MAX_BLOCK_LEN.
 *   causal     0 (default, non-causal: every block query sees every block key)
 *              or 1 (query i sees keys up to its own position).
 *   window     0 = global layer; W > 0 = sliding window of W keys ending at each
 *              query's position. W < T is rejected (a non-causal block must see
 *              all of its own keys).
 *   scale      finite and > 0 (usually 1/sqrt(D)).
 *   out        device, [B*T, Hq, D] contiguous, dims->dtype (written).
 *   lse        device, float32 [B*T, Hq] (written) or NULL.
 *   opts       NULL or options above.
 * Returns DFLASH_OK once the work is enqueued on the stream.
 */
DFLASH_API dflash_status dflash_block_attn(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* page_table, const int32_t* seq_lens,
                                const dflash_dims* dims, int32_t block_len, int32_t causal,
                                int32_t window, float scale, void* out, float* lse,
                                const dflash_opts* opts);

/*
 * Log-sum-exp combine of split partials (the formula in the file header).
 *
 *   partial_out  device, float32 [num_splits, num_rows, head_dim] contiguous.
 *   partial_lse  device, float32 [num_splits, num_rows]; -inf marks an empty chunk.
 *   num_splits   1 .. DFLASH_MAX_SPLITS; num_rows >= 1; head_dim multiple of 4, <= 512.
 *   out          device, [num_rows, head_dim] of out_dtype (written; 16-byte aligned for
 *                float32, 8-byte aligned for bfloat16); a row whose
 *                chunks are all empty gets zeros.
 *   lse          device, float32 [num_rows] (written) or NULL; -inf for all-empty rows.
 *   stream       cudaStream_t or NULL.
 */
DFLASH_API dflash_status dflash_split_combine(const float* partial_out, const float* partial_lse,
                                   int32_t num_splits, int64_t num_rows, int32_t head_dim,
                                   dflash_dtype out_dtype, void* out, float* lse, void* stream);

/* Number of chunks dflash_block_attn uses for these sizes when
   opts->num_splits == requested (0 = auto), or a negative dflash_status code
   for invalid dims. Host-only arithmetic (no CUDA call except a cached
   device-attribute query for auto). */
DFLASH_API int32_t dflash_plan_splits(const dflash_dims* dims, int32_t block_len, int32_t window,
                           int32_t requested, int32_t kernel);

/* What a dflash_block_attn call with these sizes and options runs: the split
   count, the kernel the selector resolves to, whether the splits are dealt to
   the requests by length (partials sized for one request), the CTAs of the
   attention launch and the number of kernel launches per call (the attention
   kernel, plus the split combine unless the attention kernel combines in-kernel).
   Assumes a workspace is passed. Host arithmetic plus cached device-attribute
   and occupancy queries for the current device; no launch. */
typedef struct dflash_plan {
    int32_t num_splits; /* chunks per request, or chunk slots in all when balanced */
    int32_t kernel;     /* dflash_kernel value actually run (never AUTO) */
    int32_t balanced;   /* 1: length-balanced slots */
    int32_t launches;   /* kernel launches per call */
    int64_t ctas;       /* CTAs of the attention launch */
} dflash_plan;
DFLASH_API dflash_status dflash_plan_call(const dflash_dims* dims, int32_t block_len, int32_t window,
                                          int32_t num_splits, int32_t kernel, dflash_plan* plan);

/* Workspace bytes a call with these sizes and split count needs (split count
   as returned by dflash_plan_splits). Layout, each part 256-byte aligned: the
   error word (256 bytes), an 8 KB counter block (the arrival counters of the
   tensor-core kernel's in-kernel split combine; fixed size, zero between
   calls; a call whose combine wait timed out resets its counters too, and
   dflash_read_error clears the whole block when it reports
   DFLASH_DEVERR_TIMEOUT), then -- only when
   splits > 1 --
   partial lse float32 [splits, B*T, Hq] and partial out float32
   [splits, B*T, Hq, D]. Returns 0 for invalid dims. */
DFLASH_API size_t dflash_workspace_bytes(const dflash_dims* dims, int32_t block_len, int32_t num_splits);

/* Copy the workspace error word to *device_error (device->host copy on
   `stream`, then a stream synchronisation; not for the hot path). With clear
   != 0 the word is reset to zero afterwards. When the word carries
   DFLASH_DEVERR_TIMEOUT the counter block is zeroed as well (whatever `clear`
   says), so a workspace whose split combine gave up never feeds a later call
   stale arrivals. Returns DFLASH_ERR_DEVICE_CHECK when the word is non-zero,
   DFLASH_OK when it is zero. */
DFLASH_API dflash_status dflash_read_error(const void* workspace, void* stream, uint32_t* device_error,
                                int32_t clear);

/* Static text for a status code. */
DFLASH_API const char* dflash_status_string(dflash_status status);

/* Detail of the last failing call on the calling thread ("" if none). */
DFLASH_API const char* dflash_last_error_message(void);

/*
 * The pages have no counterpart of this entry point; it exists for callers
 * that cannot allocate device memory: code that runs inside a custom
 * allocator's own hooks (where calling back into the allocator would
 * recurse), or in a runtime that owns all device memory and forbids
 * cudaMalloc. dflash_block_attn needs a caller-made
 * workspace whenever it splits the keys; this variant keeps that scratch (the
 * error word, counters and split partials) in a fixed array of
 * DFLASH_NOALLOC_SCRATCH_BYTES bytes inside the library's device image,
 * reserved on each GPU when the library's device code is loaded there and
 * held until the process exits. It allocates nothing.
 *
 * Arguments as in dflash_block_attn, with num_splits (0 = auto), kernel (a
 * dflash_kernel value) and stream (cudaStream_t or NULL) passed directly.
 * An explicit num_splits whose workspace would exceed the array returns
 * DFLASH_ERR_WORKSPACE (request fewer splits). With num_splits = 0 the call takes the auto
 * plan if it fits, else the one-wave length-balanced plan (partials sized for one request)
 * if that fits, else the most uniform chunks that fit. The first call on a device resolves
 * the array's device address (cudaGetSymbolAddress) with that device current, once, and
 * caches it. Every call clears the error word and
 * counters on `stream`, then reuses the array, which keeps the last call's
 * contents: calls that can overlap on the GPU (different streams, or
 * different host threads on the same device) race on it and must be ordered
 * by the caller. Device-side check bits land in the array's error word and are
 * not reported by this entry point (the checks still keep every access in
 * bounds: a bad page id is never dereferenced and its keys read as zero).
 * The split plan may differ from dflash_block_attn's when the auto plan does
 * not fit; the results then differ only by the fp32 summation order.
 */
#define DFLASH_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
DFLASH_API dflash_status dflash_block_attn_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                                   const int32_t* page_table, const int32_t* seq_lens,
                                                   const dflash_dims* dims, int32_t block_len, int32_t causal,
                                                   int32_t window, float scale, void* out, float* lse,
                                                   int32_t num_splits, int32_t kernel, void* stream);

/*
 * Longest-prefix acceptance: the verify step after the target has scored a drafted
 * block. The pages describe the loop as guess a block, verify it in parallel, accept the
 * longest correct prefix, repeat (kenforever1 "dflash-gemma4-31b-notes", relation
 * diagram steps 3-4).
 *
 * A block is [x_0, d_1, ..., d_K] with K = block_len - 1 drafted tokens. For request b and
 * block position j the target token is t_j = argmax_v logits[b, j, v] (the smallest index
 * among equal maxima; logits must be finite). Draft d_i is correct when d_i == t_{i-1}.
 *   accepted_len[b] = the largest a in [0, K] with d_i == t_{i-1} for all i <= a
 *   next_token[b]   = t_a  (the target's token at the first mismatch, or after the block)
 *   target_argmax[b, j] = t_j when target_argmax is not NULL
 *
 *   logits        device, [batch, block_len, vocab] of dtype (bf16 or fp32), row j of request
 *                 b at (b * block_len + j) * row_stride elements, row_stride >= vocab; aligned
 *                 to its element size (rows are read with 16-byte loads between their
 *                 16-byte boundaries).
 *   draft         device int32 [batch, block_len - 1] (may be NULL when block_len == 1).
 *   accepted_len, next_token   device int32 [batch], written.
 *   target_argmax device int32 [batch, block_len] or NULL.
 *   workspace     device, 256-byte aligned, dflash_accept_workspace_bytes() long, zeroed once
 *                 before its first use; the call leaves it zeroed (it holds one 64-bit key
 *                 per row and one arrival counter per request).
 * Limits: batch * block_len <= 65535, 1 <= vocab < 2^31. Invalid arguments are reported
 * before any launch. Asynchronous on `stream`; calls that share a workspace must not overlap.
 */
DFLASH_API size_t dflash_accept_workspace_bytes(int32_t batch, int32_t block_len);
DFLASH_API dflash_status dflash_accept_prefix(const void* logits, dflash_dtype dtype, int32_t batch,
                                              int32_t block_len, int32_t vocab, int64_t row_stride,
                                              const int32_t* draft, int32_t* accepted_len, int32_t* next_token,
                                              int32_t* target_argmax, void* workspace, size_t workspace_bytes,
                                              void* stream);

/*
 * Context K/V projection for the draft pass, fused with the paged-cache write. The
 * drafter's cross-attention takes its context K/V from the target's hidden states
 * (kenforever1 "dflash-gemma4-31b-notes", the code lines under "why non-causal
 * attention"); the vLLM DFlash review's risk list names this precompute as a bare linear
 * layer, so no bias, normalisation or rotary embedding is applied. For every token t
 * whose slot_mapping[t] = s >= 0:
 *   k_cache[s / page_size, s % page_size, h, d] = bf16( sum_k hidden[t, k] * w_k[h*D + d, k] )
 *   v_cache[s / page_size, s % page_size, h, d] = bf16( sum_k hidden[t, k] * w_v[h*D + d, k] )
 * with fp32 accumulation on the tensor cores (a bf16 rounding of the fp32 sum). Tokens
 * with s < 0 are skipped (padding); s >= num_pages * page_size sets
 * DFLASH_DEVERR_PAGE_ID in *device_error and is skipped.
 *
 *   hidden        device bf16 [num_tokens, hidden_size], row t at t * hidden_stride
 *                 elements; 16-byte aligned, hidden_stride >= hidden_size, both
 *                 multiples of 8.
 *   w_k, w_v      device bf16 [num_kv_heads * head_dim, hidden_size], contiguous
 *                 (the out x in layout of a linear layer's weight); 16-byte aligned.
 *   slot_mapping  device int32 [num_tokens]: page * page_size + position in page.
 *   k_cache, v_cache  device bf16, the layout of dflash_block_attn (dims->kv_stride_*,
 *                 multiples of 8 elements, head_dim contiguous); written.
 *   dims          num_kv_heads, head_dim (a multiple of 16, <= 512), page_size,
 *                 num_pages, dtype (DFLASH_BF16) and the three strides are read; the
 *                 other fields are ignored.
 *   device_error  device uint32 word (bits OR-ed in; DFLASH_DEVERR_TIMEOUT if a bounded
 *                 pipeline wait gave up) or NULL.
 *   workspace     device, 256-byte aligned, zeroed once before its first use, or NULL. With
 *                 at least dflash_project_kv_workspace_bytes() bytes, the tiles of a partial
 *                 last round of the persistent grid are split in two along the hidden
 *                 dimension, and the halves meet in the workspace: an 8 KB block of counters
 *                 (left at zero by every call, unless a device timeout was reported), then
 *                 fp32 partial tiles. NULL (or too small) computes every tile whole. Results
 *                 differ only in the fp32 summation order.
 * Limits: 0 <= num_tokens <= DFLASH_PROJECT_MAX_TOKENS (0 is a no-op),
 * num_kv_heads * head_dim <= 65536. Invalid arguments are reported before any launch.
 * Asynchronous on `stream`; allocates nothing. Calls that share a workspace must not overlap.
 */
#define DFLASH_PROJECT_MAX_TOKENS (1 << 24)
DFLASH_API size_t dflash_project_kv_workspace_bytes(void); /* for the current device */
DFLASH_API dflash_status dflash_project_kv(const void* hidden, int32_t num_tokens, int32_t hidden_size,
                                           int64_t hidden_stride, const void* w_k, const void* w_v,
                                           const int32_t* slot_mapping, void* k_cache, void* v_cache,
                                           const dflash_dims* dims, uint32_t* device_error, void* workspace,
                                           size_t workspace_bytes, void* stream);

/*
 * DFlash2 grouped dynamic depthwise convolution inside a drafted block (prhub report on vLLM
 * PR #52816 "DFlash2", the motivation paragraph and change 1: proposal positions see earlier
 * positions of the same block without another backbone pass). For request b, block
 * position i and channel c:
 *   out[b, i, c] = sum over t < num_taps with t <= i of
 *                  (base[t, c] + delta[b, i, t, g(c)]) * x[b, i - t, c]
 * with g(c) = c / (channels / num_groups): contiguous channel groups. Taps that reach past the
 * start of the request's block contribute zero. fp32 accumulation; out is rounded to dtype.
 *
 *   x, out     device, [batch, block_len, channels] contiguous, dtype (bf16 or fp32), aligned to
 *              the element size; out must not overlap x.
 *   base       device float32 [num_taps, channels]: the static per-channel taps.
 *   delta      device float32 [batch, block_len, num_taps, num_groups]: the dynamic taps of each
 *              position and group (what the module's "prepare" step projects from its input).
 * Limits: 1 <= batch <= 65535, 1 <= block_len, num_taps <= DFLASH_MAX_BLOCK_LEN, channels a
 * positive multiple of num_groups. Invalid arguments are reported before any launch.
 * Asynchronous on `stream`; needs no workspace.
 */
DFLASH_API dflash_status dflash_grouped_conv(const void* x, void* out, dflash_dtype dtype, int32_t batch,
                                             int32_t block_len, int32_t channels, int32_t num_taps,
                                             int32_t num_groups, const float* base, const float* delta,
                                             void* stream);

/*
 * DFlash2 candidate-selector walk (prhub report on vLLM PR #52816 "DFlash2", the motivation
 * paragraph and changes 1-2). The head keeps num_candidates = K tokens per draft slot. The
 * transition from token p to candidate k of slot s of request r scores
 *   edge(p -> k) = sum_e A[p, e] * proj[r, s, e] * B[cand[r, s, k], e] + unary[r, s, k]
 * (A: predecessor codebook, B: successor codebook, proj: the projected hidden state of the
 * slot). From p = anchor[r], slot by slot: with temperature 0 the walk takes the first k of
 * maximal edge; with temperature T > 0 it forms q = softmax(edge / T) over the K candidates and
 * takes the smallest k whose running sum of q exceeds uniforms[r, s] (K - 1 if rounding leaves
 * none). The chosen token becomes the next slot's p.
 *
 *   pred_codebook, succ_codebook  device bf16 [vocab, dim], 16-byte aligned; dim a multiple of 8.
 *   proj          device float32 [R, S, dim], 16-byte aligned.
 *   candidates    device int32 [R, S, K]; unary device float32 [R, S, K] (finite).
 *   anchor        device int32 [R]: the verified token each walk starts from.
 *   uniforms      device float32 [R, S] in [0, 1); needed when temperature > 0, else ignored.
 *   tokens        device int32 [R, S], written: the walk's token per slot.
 *   chosen        device int32 [R, S] or NULL: the chosen candidate index per slot.
 *   path_scores   device float32 [R, S, K] or NULL: the K edges from the walk's predecessor.
 *   q             device float32 [R, S, K] or NULL: the sampling distribution (T > 0 only).
 *   device_error  device uint32 word or NULL: DFLASH_DEVERR_TOKEN_ID for ids outside [0, vocab).
 *   workspace     device, 256-byte aligned, dflash_selector_workspace_bytes() long, zeroed once
 *                 before its first use. Layout: a fixed 256 KB block of per-request arrival
 *                 counters (left at zero by every call, so one zeroed workspace serves calls of
 *                 any size), then the R x S x K x K edge tables.
 * fp32 arithmetic (bf16 codebooks widened exactly). Limits: 1 <= R, S <= 65535, 1 <= K <= 64,
 * K * dim * 6 bytes <= 200 KB. Asynchronous on `stream`; calls sharing a workspace must not
 * overlap.
 */
DFLASH_API size_t dflash_selector_workspace_bytes(int32_t num_requests, int32_t num_slots, int32_t num_candidates);
DFLASH_API dflash_status dflash_selector_walk(const void* pred_codebook, const void* succ_codebook, int32_t vocab,
                                              int32_t dim, const float* proj, const int32_t* candidates,
                                              const float* unary, const int32_t* anchor, int32_t num_requests,
                                              int32_t num_slots, int32_t num_candidates, float temperature,
                                              const float* uniforms, int32_t* tokens, int32_t* chosen,
                                              float* path_scores, float* q, uint32_t* device_error,
                                              void* workspace, size_t workspace_bytes, void* stream);

/* DFLASH_ABI_VERSION of the loaded library. */
DFLASH_API int32_t dflash_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH_ATTN_H */
