// C-ABI front end of libdflash_attn: host-side validation, split planning,
// workspace carve-up and kernel launches. See include/dflash_attn.h for the
// contract of each entry point.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "dflash_internal.h"

namespace dflash {
namespace {

thread_local std::string g_last_error;

dflash_status fail(dflash_status s, const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

dflash_status cuda_fail(cudaError_t e, const char* what)
{
    return fail(DFLASH_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

size_t elem_size(int32_t dtype) { return dtype == DFLASH_BF16 ? 2 : 4; }

// Validation of the sizes and layout (no pointers).
dflash_status check_dims(const dflash_dims* d, int32_t T)
{
    if (!d) return fail(DFLASH_ERR_INVALID_ARG, "dims is NULL");
    if (d->batch < 1 || d->batch > 65535) return fail(DFLASH_ERR_INVALID_ARG, "batch %d outside [1, 65535]", d->batch);
    if (d->num_q_heads < 1 || d->num_kv_heads < 1)
        return fail(DFLASH_ERR_INVALID_ARG, "head counts must be >= 1 (Hq=%d, Hkv=%d)", d->num_q_heads,
                    d->num_kv_heads);
    if (d->num_q_heads % d->num_kv_heads != 0)
        return fail(DFLASH_ERR_INVALID_ARG, "num_q_heads %d is not a multiple of num_kv_heads %d",
                    d->num_q_heads, d->num_kv_heads);
    if (d->num_q_heads > 1024) return fail(DFLASH_ERR_INVALID_ARG, "num_q_heads %d > 1024", d->num_q_heads);
    if (d->head_dim < 1 || d->head_dim > DFLASH_MAX_HEAD_DIM)
        return fail(DFLASH_ERR_INVALID_ARG, "head_dim %d outside [1, %d]", d->head_dim, DFLASH_MAX_HEAD_DIM);
    if (d->head_dim % 16 != 0)
        return fail(DFLASH_ERR_UNSUPPORTED, "head_dim %d is not a multiple of 16", d->head_dim);
    if (d->page_size < 8 || d->page_size > 256 || d->page_size % 8 != 0)
        return fail(DFLASH_ERR_INVALID_ARG, "page_size %d must be a multiple of 8 in [8, 256]", d->page_size);
    if (d->num_pages < 1) return fail(DFLASH_ERR_INVALID_ARG, "num_pages %d < 1", d->num_pages);
    if (d->max_pages < 1) return fail(DFLASH_ERR_INVALID_ARG, "max_pages %d < 1", d->max_pages);
    const int64_t cap = (int64_t)d->max_pages * d->page_size;
    if (cap > (int64_t)(1 << 30)) return fail(DFLASH_ERR_INVALID_ARG, "max_pages*page_size too large");
    if (d->max_seq_len < 0 || d->max_seq_len > cap)
        return fail(DFLASH_ERR_INVALID_ARG, "max_seq_len %d outside [0, max_pages*page_size=%lld]", d->max_seq_len,
                    (long long)cap);
    if (d->dtype != DFLASH_BF16 && d->dtype != DFLASH_FP32)
        return fail(DFLASH_ERR_INVALID_ARG, "dtype %d is not DFLASH_BF16 or DFLASH_FP32", (int)d->dtype);
    if (T < 1 || T > DFLASH_MAX_BLOCK_LEN)
        return fail(DFLASH_ERR_INVALID_ARG, "block_len %d outside [1, %d]", T, DFLASH_MAX_BLOCK_LEN);
    const int32_t maxL = d->max_seq_len ? d->max_seq_len : (int32_t)cap;
    if (maxL < T) return fail(DFLASH_ERR_INVALID_ARG, "max_seq_len %d < block_len %d", maxL, T);
    const int64_t es = (int64_t)elem_size(d->dtype);
    if (d->kv_stride_page < 0 || d->kv_stride_slot < 0 || d->kv_stride_head < 0)
        return fail(DFLASH_ERR_INVALID_ARG, "negative K/V stride");
    if ((d->kv_stride_page * es) % 16 || (d->kv_stride_slot * es) % 16 || (d->kv_stride_head * es) % 16)
        return fail(DFLASH_ERR_INVALID_ARG, "K/V strides must be multiples of 16 bytes");
    if (d->kv_stride_head < d->head_dim && d->num_kv_heads > 1)
        return fail(DFLASH_ERR_INVALID_ARG, "kv_stride_head %lld < head_dim %d", (long long)d->kv_stride_head,
                    d->head_dim);
    return DFLASH_OK;
}

int32_t max_len_of(const dflash_dims* d)
{
    return d->max_seq_len ? d->max_seq_len : d->max_pages * d->page_size;
}

std::mutex g_sm_mutex;
int g_sm_count[64] = {0};

}  // namespace

dflash_status report_error(dflash_status s, const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

int device_sm_count()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (dev >= 0 && dev < 64) {
        std::lock_guard<std::mutex> lk(g_sm_mutex);
        if (g_sm_count[dev] == 0) {
            int n = 0;
            if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
            g_sm_count[dev] = n;
        }
        return g_sm_count[dev];
    }
    return 148;
}

WorkspaceLayout workspace_layout(int32_t B, int32_t T, int32_t Hq, int32_t D, int32_t splits)
{
    WorkspaceLayout w;
    w.err_off = 0;
    w.counters_off = 256;
    size_t off = w.counters_off + DFLASH_COUNTER_BYTES;
    w.part_lse_off = off;
    w.part_out_off = off;
    if (splits > 1) {
        const size_t rows = (size_t)B * T * Hq;
        w.part_lse_off = off;
        off += round_up(sizeof(float) * rows * splits, 256);
        w.part_out_off = off;
        off += round_up(sizeof(float) * rows * (size_t)splits * D, 256);
    }
    w.total = off;
    return w;
}

}  // namespace dflash

using namespace dflash;

namespace {

// Kernel the call will use: 1 = SIMT, 2 = tensor-core, or a negative status.
int choose_kernel(const dflash_dims* d, int32_t T, int32_t window, int32_t requested)
{
    AttnParams p{};
    p.B = d->batch;
    p.T = T;
    p.Hq = d->num_q_heads;
    p.Hkv = d->num_kv_heads;
    p.G = d->num_q_heads / d->num_kv_heads;
    p.D = d->head_dim;
    p.page_size = d->page_size;
    p.window = window;
    p.dtype = d->dtype;
    p.sp = d->kv_stride_page;
    p.ss = d->kv_stride_slot;
    p.sh = d->kv_stride_head;
    p.num_pages = d->num_pages;
    if (requested == DFLASH_KERNEL_SIMT) return DFLASH_KERNEL_SIMT;
    if (requested == DFLASH_KERNEL_TC) {
        if (d->dtype != DFLASH_BF16 || !tc_supports(p)) return -DFLASH_ERR_UNSUPPORTED;
        return DFLASH_KERNEL_TC;
    }
    if (requested == DFLASH_KERNEL_TC_PAIR) {
        if (d->dtype != DFLASH_BF16 || !tc_pair_supports(p)) return -DFLASH_ERR_UNSUPPORTED;
        return DFLASH_KERNEL_TC_PAIR;
    }
    if (requested != DFLASH_KERNEL_AUTO) return -DFLASH_ERR_INVALID_ARG;
    if (d->dtype != DFLASH_BF16) return DFLASH_KERNEL_SIMT;
    // The packed rows of a KV head's query heads x block positions go to one CTA when they fit
    // its tile; when one CTA would need several row groups (each reading all of the K/V), the
    // CTA pair takes them with fewer groups (8 heads x 16 positions at head_dim 512: one pair,
    // every K/V byte read once, against two CTAs that each read it all).
    const bool tc = tc_supports(p);
    const bool pair = tc_pair_supports(p);
    if (pair && (!tc || tc_pair_row_groups(p) < tc_row_groups(p))) return DFLASH_KERNEL_TC_PAIR;
    if (tc) return DFLASH_KERNEL_TC;
    return DFLASH_KERNEL_SIMT;
}

// Work units (CTAs per split) of the chosen kernel.
int64_t work_units(const dflash_dims* d, int32_t T, int kernel)
{
    if (kernel == DFLASH_KERNEL_TC) {
        AttnParams p{};
        p.B = d->batch;
        p.T = T;
        p.Hkv = d->num_kv_heads;
        p.G = d->num_q_heads / d->num_kv_heads;
        return tc_ctas_per_split(p);
    }
    if (kernel == DFLASH_KERNEL_TC_PAIR) {
        AttnParams p{};
        p.B = d->batch;
        p.T = T;
        p.Hkv = d->num_kv_heads;
        p.G = d->num_q_heads / d->num_kv_heads;
        return tc_pair_ctas_per_split(p);
    }
    return (int64_t)d->batch * d->num_q_heads * ((T + 15) / 16);
}

// Chunks longer than kLongChunkKeys run better as many uniform waves of about
// kTargetChunkKeys keys than as one wave of long streams (measured on 8 requests of 131072
// keys: 19 chunks of 6.9k keys, 8 waves, 3659 us; one balanced wave, 4245 us; 12 or 24
// chunks, 4280 and 3978 us).
constexpr int64_t kLongChunkKeys = 16384;
constexpr int64_t kTargetChunkKeys = 7168;

int32_t plan_splits_impl(const dflash_dims* d, int32_t T, int32_t window, int32_t requested, int kernel)
{
    if (requested > 0) return requested > DFLASH_MAX_SPLITS ? -DFLASH_ERR_INVALID_ARG : requested;
    if (requested < 0) return -DFLASH_ERR_INVALID_ARG;
    // Several requests on the tensor-core path: one wave of chunk slots dealt to the requests
    // in proportion to their key spans (the kernel reads seq_lens), so a long request does
    // not leave most SMs idle while its equal-count chunks finish.
    const int32_t bal = balanced_slots(d, T, window, kernel);
    if (bal > 0) return bal;
    // Longest union key range any request can have.
    int64_t span = max_len_of(d);
    if (window > 0) span = std::min<int64_t>(span, (int64_t)window + T - 1 + d->page_size);
    // Keep at least 128 keys (one tensor-core tile) per chunk; fill at most one wave over the
    // SMs (a partial second wave would cost a whole extra round of the longest chunks).
    const int64_t max_by_len = std::max<int64_t>(1, span / 128);
    const int64_t units = work_units(d, T, kernel);
    const int64_t sms = device_sm_count();
    int64_t s = sms / units;
    // one wave would leave very long chunks: take more, shorter chunks over several waves
    if (span / std::max<int64_t>(1, s) > kLongChunkKeys) s = (span + kTargetChunkKeys - 1) / kTargetChunkKeys;
    s = std::min<int64_t>(s, max_by_len);
    s = std::min<int64_t>(s, DFLASH_MAX_SPLITS);
    s = std::max<int64_t>(1, s);
    // Whole 128-key tiles per chunk: a chunk of 1.75 tiles costs its CTA a second, mostly
    // empty tile (global_verify: 38 chunks of 224 keys against 32 of 256, which ran faster).
    if (kernel == DFLASH_KERNEL_TC && s > 1) {
        const int64_t chunk = ((span + s - 1) / s + 127) / 128 * 128;
        s = std::max<int64_t>(1, (span + chunk - 1) / chunk);
    }
    return (int32_t)s;
}

}  // namespace

namespace dflash {

int32_t balanced_slots(const dflash_dims* d, int32_t T, int32_t window, int kernel, bool allow_long)
{
    if (kernel != DFLASH_KERNEL_TC || d->batch < 2) return 0;
    AttnParams p{};
    p.B = 1;
    p.T = T;
    p.Hkv = d->num_kv_heads;
    p.G = d->num_q_heads / d->num_kv_heads;
    const int64_t per_req = tc_ctas_per_split(p);  // CTAs of one (request, chunk)
    if (per_req <= 0) return 0;
    if ((int64_t)d->batch * per_req > DFLASH_MAX_COMBINE_GROUPS) return 0;
    int64_t span = max_len_of(d);
    if (window > 0) span = std::min<int64_t>(span, (int64_t)window + T - 1 + d->page_size);
    int64_t c = device_sm_count() / per_req;                            // one wave
    c = std::min<int64_t>(c, (int64_t)d->batch * std::max<int64_t>(1, span / 128));  // >= a tile each
    c = std::min<int64_t>(c, DFLASH_MAX_SPLITS);
    if (c < d->batch || c < 2) return 0;
    // one wave of slots over long requests gives long streams: the uniform plan's several
    // waves of shorter chunks do better (the in-kernel combine needs the grid resident, so the
    // balanced plan cannot spread wider)
    if (!allow_long && (int64_t)d->batch * span / c > kLongChunkKeys) return 0;
    return (int32_t)c;
}

int resolve_kernel(const dflash_dims* d, int32_t T, int32_t window, int32_t requested)
{
    return choose_kernel(d, T, window, requested);
}

}  // namespace dflash

extern "C" {

int32_t dflash_abi_version(void) { return DFLASH_ABI_VERSION; }

const char* dflash_status_string(dflash_status s)
{
    switch (s) {
    case DFLASH_OK: return "ok";
    case DFLASH_ERR_INVALID_ARG: return "invalid argument";
    case DFLASH_ERR_UNSUPPORTED: return "unsupported combination";
    case DFLASH_ERR_CUDA: return "CUDA error";
    case DFLASH_ERR_DEVICE_CHECK: return "device-side check failed (bad page id or seq_len)";
    case DFLASH_ERR_WORKSPACE: return "workspace missing or too small";
    }
    return "unknown status";
}

const char* dflash_last_error_message(void) { return g_last_error.c_str(); }

int32_t dflash_plan_splits(const dflash_dims* dims, int32_t block_len, int32_t window, int32_t requested,
                           int32_t kernel)
{
    const dflash_status s = check_dims(dims, block_len);
    if (s != DFLASH_OK) return -(int32_t)s;
    const int k = choose_kernel(dims, block_len, window, kernel);
    if (k < 0) return k;
    return plan_splits_impl(dims, block_len, window, requested, k);
}

dflash_status dflash_plan_call(const dflash_dims* dims, int32_t block_len, int32_t window, int32_t num_splits,
                               int32_t kernel, dflash_plan* plan)
{
    g_last_error.clear();
    if (!plan) return fail(DFLASH_ERR_INVALID_ARG, "plan is NULL");
    const dflash_status s = check_dims(dims, block_len);
    if (s != DFLASH_OK) return s;
    const int k = choose_kernel(dims, block_len, window, kernel);
    if (k < 0) return fail((dflash_status)(-k), "the requested kernel does not cover these sizes/dtype");
    const int32_t splits = plan_splits_impl(dims, block_len, window, num_splits, k);
    if (splits < 1) return fail(DFLASH_ERR_INVALID_ARG, "num_splits %d outside [0, %d]", num_splits, DFLASH_MAX_SPLITS);
    const bool balanced = num_splits == 0 && splits > 1 && balanced_slots(dims, block_len, window, k) == splits;
    plan->num_splits = splits;
    plan->kernel = k;
    plan->balanced = balanced ? 1 : 0;
    AttnParams p{};
    p.B = dims->batch;
    p.T = block_len;
    p.Hq = dims->num_q_heads;
    p.Hkv = dims->num_kv_heads;
    p.G = dims->num_q_heads / dims->num_kv_heads;
    p.D = dims->head_dim;
    p.page_size = dims->page_size;
    p.window = window;
    p.dtype = dims->dtype;
    p.sp = dims->kv_stride_page;
    p.ss = dims->kv_stride_slot;
    p.sh = dims->kv_stride_head;
    p.num_pages = dims->num_pages;
    p.splits = splits;
    p.balanced = plan->balanced;
    if (k == DFLASH_KERNEL_TC) {
        bool fused = false;
        const cudaError_t e = tc_grid_info(p, &plan->ctas, &fused);
        if (e != cudaSuccess) return cuda_fail(e, "tensor-core grid query");
        plan->launches = (splits == 1 || fused) ? 1 : 2;
    } else if (k == DFLASH_KERNEL_TC_PAIR) {
        p.T = block_len;
        const cudaError_t e = tc_pair_grid_ctas(p, &plan->ctas);
        if (e != cudaSuccess) return cuda_fail(e, "CTA-pair grid query");
        plan->launches = splits == 1 ? 1 : 2;
    } else {
        plan->ctas = work_units(dims, block_len, k) * splits;
        plan->launches = splits == 1 ? 1 : 2;
    }
    return DFLASH_OK;
}

size_t dflash_workspace_bytes(const dflash_dims* dims, int32_t block_len, int32_t num_splits)
{
    if (check_dims(dims, block_len) != DFLASH_OK || num_splits < 1 || num_splits > DFLASH_MAX_SPLITS) return 0;
    return workspace_layout(dims->batch, block_len, dims->num_q_heads, dims->head_dim, num_splits).total;
}

dflash_status dflash_block_attn(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* page_table, const int32_t* seq_lens, const dflash_dims* dims,
                                int32_t block_len, int32_t causal, int32_t window, float scale, void* out,
                                float* lse, const dflash_opts* opts)
{
    return dflash::block_attn_planned(q, k_cache, v_cache, page_table, seq_lens, dims, block_len, causal, window,
                                      scale, out, lse, opts, 0, false);
}

}  // extern "C"

dflash_status dflash::block_attn_planned(const void* q, const void* k_cache, const void* v_cache,
                                         const int32_t* page_table, const int32_t* seq_lens, const dflash_dims* dims,
                                         int32_t block_len, int32_t causal, int32_t window, float scale, void* out,
                                         float* lse, const dflash_opts* opts, int32_t forced_splits,
                                         bool forced_balanced)
{
    g_last_error.clear();
    dflash_status s = check_dims(dims, block_len);
    if (s != DFLASH_OK) return s;
    if (!q || !k_cache || !v_cache || !page_table || !seq_lens || !out)
        return fail(DFLASH_ERR_INVALID_ARG, "NULL tensor pointer");
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16))
        return fail(DFLASH_ERR_INVALID_ARG, "q, k_cache, v_cache and out must be 16-byte aligned");
    if (!aligned(page_table, 4) || !aligned(seq_lens, 4) || (lse && !aligned(lse, 4)))
        return fail(DFLASH_ERR_INVALID_ARG, "page_table, seq_lens and lse must be 4-byte aligned");
    if (causal != 0 && causal != 1) return fail(DFLASH_ERR_INVALID_ARG, "causal must be 0 or 1 (got %d)", causal);
    if (window < 0) return fail(DFLASH_ERR_INVALID_ARG, "window %d < 0", window);
    if (window > 0 && window < block_len)
        return fail(DFLASH_ERR_INVALID_ARG, "window %d < block_len %d: the block would not see its own keys", window,
                    block_len);
    if (!std::isfinite(scale) || !(scale > 0.f))
        return fail(DFLASH_ERR_INVALID_ARG, "scale must be finite and > 0");

    const int32_t requested = opts ? opts->num_splits : 0;
    const int32_t kreq = opts ? opts->kernel : DFLASH_KERNEL_AUTO;
    const int kernel = choose_kernel(dims, block_len, window, kreq);
    if (kernel < 0)
        return fail((dflash_status)(-kernel), kernel == -DFLASH_ERR_UNSUPPORTED
                                                  ? "the tensor-core kernel does not cover these sizes/dtype"
                                                  : "unknown kernel selector %d",
                    kreq);
    int32_t splits = forced_splits;
    bool balanced = forced_balanced;
    if (splits < 1) {
        splits = plan_splits_impl(dims, block_len, window, requested, kernel);
        if (splits < 1)
            return fail(DFLASH_ERR_INVALID_ARG, "num_splits %d outside [0, %d]", requested, DFLASH_MAX_SPLITS);
        // Length-balanced plan: partials are [slot][T][Hq][D], so the layout is sized for one request.
        balanced = requested == 0 && splits > 1 && balanced_slots(dims, block_len, window, kernel) == splits;
    }
    if (balanced && kernel != DFLASH_KERNEL_TC) return fail(DFLASH_ERR_INVALID_ARG, "balanced plan needs the TC kernel");
    const WorkspaceLayout wl =
        workspace_layout(balanced ? 1 : dims->batch, block_len, dims->num_q_heads, dims->head_dim, splits);
    void* ws = opts ? opts->workspace : nullptr;
    const size_t ws_bytes = opts ? opts->workspace_bytes : 0;
    if (ws) {
        if (!aligned(ws, 256)) return fail(DFLASH_ERR_WORKSPACE, "workspace must be 256-byte aligned");
        if (ws_bytes < wl.total)
            return fail(DFLASH_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed for %d splits", ws_bytes, wl.total,
                        splits);
    } else if (splits > 1) {
        return fail(DFLASH_ERR_WORKSPACE, "%d splits need a workspace of %zu bytes", splits, wl.total);
    }

    AttnParams p{};
    p.q = q;
    p.k = k_cache;
    p.v = v_cache;
    p.page_table = page_table;
    p.seq_lens = seq_lens;
    p.out = out;
    p.lse = lse;
    char* wsb = static_cast<char*>(ws);
    p.err = ws ? reinterpret_cast<uint32_t*>(wsb + wl.err_off) : nullptr;
    p.counters = ws ? reinterpret_cast<int32_t*>(wsb + wl.counters_off) : nullptr;
    p.part_lse = splits > 1 ? reinterpret_cast<float*>(wsb + wl.part_lse_off) : nullptr;
    p.part_out = splits > 1 ? reinterpret_cast<float*>(wsb + wl.part_out_off) : nullptr;
    p.B = dims->batch;
    p.T = block_len;
    p.Hq = dims->num_q_heads;
    p.Hkv = dims->num_kv_heads;
    p.G = dims->num_q_heads / dims->num_kv_heads;
    p.D = dims->head_dim;
    p.page_size = dims->page_size;
    p.num_pages = dims->num_pages;
    p.max_pages = dims->max_pages;
    p.max_seq_len = max_len_of(dims);
    p.sp = dims->kv_stride_page;
    p.ss = dims->kv_stride_slot;
    p.sh = dims->kv_stride_head;
    p.causal = causal;
    p.window = window;
    p.scale = scale;
    p.splits = splits;
    p.dtype = dims->dtype;
    p.balanced = balanced ? 1 : 0;
    p.wait_ns = (opts && opts->wait_limit_us) ? (unsigned long long)opts->wait_limit_us * 1000ull
                                              : DFLASH_DEFAULT_WAIT_NS;

    cudaStream_t stream = opts ? static_cast<cudaStream_t>(opts->stream) : nullptr;
    cudaError_t e = (kernel == DFLASH_KERNEL_TC)        ? launch_tc_attn(p, stream)
                    : (kernel == DFLASH_KERNEL_TC_PAIR) ? launch_tc_pair_attn(p, stream)
                                                        : launch_simt_attn(p, stream);
    if (e != cudaSuccess) return cuda_fail(e, "attention kernel launch");
    if (splits > 1 && kernel == DFLASH_KERNEL_SIMT) {
        e = launch_combine(p.part_out, p.part_lse, splits, (int64_t)p.B * p.T * p.Hq, p.D, p.dtype, out, lse, stream);
        if (e != cudaSuccess) return cuda_fail(e, "combine kernel launch");
    }
    return DFLASH_OK;
}

extern "C" {

size_t dflash_accept_workspace_bytes(int32_t batch, int32_t block_len)
{
    if (batch < 1 || block_len < 1 || (int64_t)batch * block_len > 65535) return 0;
    return round_up(sizeof(unsigned long long) * (size_t)batch * block_len, 256) +
           round_up(sizeof(int32_t) * (size_t)batch, 256);
}

dflash_status dflash_accept_prefix(const void* logits, dflash_dtype dtype, int32_t batch, int32_t block_len,
                                   int32_t vocab, int64_t row_stride, const int32_t* draft, int32_t* accepted_len,
                                   int32_t* next_token, int32_t* target_argmax, void* workspace,
                                   size_t workspace_bytes, void* stream)
{
    g_last_error.clear();
    if (dtype != DFLASH_BF16 && dtype != DFLASH_FP32) return fail(DFLASH_ERR_INVALID_ARG, "dtype must be bf16 or fp32");
    if (batch < 1 || block_len < 1 || (int64_t)batch * block_len > 65535)
        return fail(DFLASH_ERR_INVALID_ARG, "batch %d x block_len %d outside [1, 65535]", batch, block_len);
    if (vocab < 1) return fail(DFLASH_ERR_INVALID_ARG, "vocab %d < 1", vocab);
    const int64_t es = dtype == DFLASH_BF16 ? 2 : 4;
    if (row_stride < vocab) return fail(DFLASH_ERR_INVALID_ARG, "row_stride %lld < vocab", (long long)row_stride);
    if (!logits || !accepted_len || !next_token || (block_len > 1 && !draft))
        return fail(DFLASH_ERR_INVALID_ARG, "NULL pointer");
    if (!aligned(logits, (size_t)es) || (draft && !aligned(draft, 4)) || !aligned(accepted_len, 4) ||
        !aligned(next_token, 4) || (target_argmax && !aligned(target_argmax, 4)))
        return fail(DFLASH_ERR_INVALID_ARG, "misaligned pointer (logits to their element size, int32 arrays 4 bytes)");
    const size_t need = dflash_accept_workspace_bytes(batch, block_len);
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < need)
        return fail(DFLASH_ERR_WORKSPACE, "acceptance needs a 256-byte aligned workspace of %zu bytes", need);
    char* wsb = static_cast<char*>(workspace);
    auto* keys = reinterpret_cast<unsigned long long*>(wsb);
    auto* counters = reinterpret_cast<int32_t*>(wsb + round_up(sizeof(unsigned long long) * (size_t)batch * block_len, 256));
    const cudaError_t e = launch_accept(logits, dtype, batch, block_len, vocab, row_stride, draft, accepted_len,
                                        next_token, target_argmax, keys, counters, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "acceptance kernel launch");
    return DFLASH_OK;
}

size_t dflash_project_kv_workspace_bytes(void) { return project_kv_workspace_bytes(); }

dflash_status dflash_project_kv(const void* hidden, int32_t num_tokens, int32_t hidden_size, int64_t hidden_stride,
                                const void* w_k, const void* w_v, const int32_t* slot_mapping, void* k_cache,
                                void* v_cache, const dflash_dims* dims, uint32_t* device_error, void* workspace,
                                size_t workspace_bytes, void* stream)
{
    g_last_error.clear();
    if (!dims) return fail(DFLASH_ERR_INVALID_ARG, "NULL dims");
    if (dims->dtype != DFLASH_BF16) return fail(DFLASH_ERR_UNSUPPORTED, "the projection is bf16 only");
    if (num_tokens < 0 || num_tokens > DFLASH_PROJECT_MAX_TOKENS)
        return fail(DFLASH_ERR_INVALID_ARG, "num_tokens %d outside [0, %d]", num_tokens, DFLASH_PROJECT_MAX_TOKENS);
    if (hidden_size < 8 || hidden_size % 8 != 0)
        return fail(DFLASH_ERR_INVALID_ARG, "hidden_size %d must be a positive multiple of 8", hidden_size);
    if (hidden_stride < hidden_size || hidden_stride % 8 != 0)
        return fail(DFLASH_ERR_INVALID_ARG, "hidden_stride %lld must be >= hidden_size and a multiple of 8",
                    (long long)hidden_stride);
    const int32_t Hkv = dims->num_kv_heads, D = dims->head_dim;
    if (Hkv < 1 || D < 16 || D > DFLASH_MAX_HEAD_DIM || D % 16 != 0)
        return fail(DFLASH_ERR_INVALID_ARG, "num_kv_heads %d / head_dim %d (a multiple of 16 in [16, %d])", Hkv, D,
                    DFLASH_MAX_HEAD_DIM);
    if ((int64_t)Hkv * D > 65536) return fail(DFLASH_ERR_INVALID_ARG, "num_kv_heads * head_dim above 65536");
    if (dims->page_size < 1 || dims->num_pages < 1)
        return fail(DFLASH_ERR_INVALID_ARG, "page_size %d / num_pages %d must be >= 1", dims->page_size,
                    dims->num_pages);
    const int64_t sp = dims->kv_stride_page, ss = dims->kv_stride_slot, sh = dims->kv_stride_head;
    if (sp < 0 || ss < 0 || sh < 0 || sp % 8 || ss % 8 || sh % 8)
        return fail(DFLASH_ERR_INVALID_ARG, "cache strides must be non-negative multiples of 8 elements");
    if (num_tokens == 0) return DFLASH_OK;
    if (!hidden || !w_k || !w_v || !slot_mapping || !k_cache || !v_cache)
        return fail(DFLASH_ERR_INVALID_ARG, "NULL pointer");
    if (!aligned(hidden, 16) || !aligned(w_k, 16) || !aligned(w_v, 16) || !aligned(k_cache, 16) ||
        !aligned(v_cache, 16) || !aligned(slot_mapping, 4) || (device_error && !aligned(device_error, 4)))
        return fail(DFLASH_ERR_INVALID_ARG, "misaligned pointer (16 bytes; slot_mapping and device_error 4)");
    if (workspace && !aligned(workspace, 256))
        return fail(DFLASH_ERR_WORKSPACE, "the projection workspace must be 256-byte aligned");
    const cudaError_t e = launch_project_kv(hidden, num_tokens, hidden_size, hidden_stride, w_k, w_v, slot_mapping,
                                            k_cache, v_cache, Hkv, D, dims->page_size, dims->num_pages, sp, ss, sh,
                                            device_error, workspace, workspace ? workspace_bytes : 0,
                                            static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "projection kernel launch");
    return DFLASH_OK;
}

dflash_status dflash_grouped_conv(const void* x, void* out, dflash_dtype dtype, int32_t batch, int32_t block_len,
                                  int32_t channels, int32_t num_taps, int32_t num_groups, const float* base,
                                  const float* delta, void* stream)
{
    g_last_error.clear();
    if (dtype != DFLASH_BF16 && dtype != DFLASH_FP32) return fail(DFLASH_ERR_INVALID_ARG, "dtype must be bf16 or fp32");
    if (batch < 1 || batch > 65535) return fail(DFLASH_ERR_INVALID_ARG, "batch %d outside [1, 65535]", batch);
    if (block_len < 1 || block_len > DFLASH_MAX_BLOCK_LEN)
        return fail(DFLASH_ERR_INVALID_ARG, "block_len %d outside [1, %d]", block_len, DFLASH_MAX_BLOCK_LEN);
    if (num_taps < 1 || num_taps > DFLASH_MAX_BLOCK_LEN)
        return fail(DFLASH_ERR_INVALID_ARG, "num_taps %d outside [1, %d]", num_taps, DFLASH_MAX_BLOCK_LEN);
    if (channels < 1 || num_groups < 1 || channels % num_groups != 0)
        return fail(DFLASH_ERR_INVALID_ARG, "channels %d must be a positive multiple of num_groups %d", channels,
                    num_groups);
    if (!x || !out || !base || !delta) return fail(DFLASH_ERR_INVALID_ARG, "NULL pointer");
    if (x == out) return fail(DFLASH_ERR_INVALID_ARG, "out must not alias x");
    const size_t es = dtype == DFLASH_BF16 ? 2 : 4;
    if (!aligned(x, es) || !aligned(out, es) || !aligned(base, 4) || !aligned(delta, 4))
        return fail(DFLASH_ERR_INVALID_ARG, "misaligned pointer (x and out to their element size, base and delta 4)");
    const cudaError_t e = launch_grouped_conv(x, out, dtype, batch, block_len, channels, num_taps, num_groups, base,
                                              delta, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "grouped convolution kernel launch");
    return DFLASH_OK;
}

constexpr size_t kSelectorCounterBytes = 65536 * sizeof(int32_t);  // one counter per possible request

size_t dflash_selector_workspace_bytes(int32_t num_requests, int32_t num_slots, int32_t num_candidates)
{
    if (num_requests < 1 || num_requests > 65535 || num_slots < 1 || num_slots > 65535 || num_candidates < 1 ||
        num_candidates > 64)
        return 0;
    // a fixed counter block first, so that a workspace zeroed once stays valid for calls of any
    // size (a counter never lands where an earlier call left its edge table), then the tables
    const size_t tab = sizeof(float) * (size_t)num_requests * num_slots * num_candidates * num_candidates;
    return kSelectorCounterBytes + round_up(tab, 256);
}

dflash_status dflash_selector_walk(const void* pred_codebook, const void* succ_codebook, int32_t vocab, int32_t dim,
                                   const float* proj, const int32_t* candidates, const float* unary,
                                   const int32_t* anchor, int32_t num_requests, int32_t num_slots,
                                   int32_t num_candidates, float temperature, const float* uniforms, int32_t* tokens,
                                   int32_t* chosen, float* path_scores, float* q, uint32_t* device_error,
                                   void* workspace, size_t workspace_bytes, void* stream)
{
    g_last_error.clear();
    const int32_t R = num_requests, S = num_slots, K = num_candidates, E = dim;
    if (R < 1 || R > 65535 || S < 1 || S > 65535)
        return fail(DFLASH_ERR_INVALID_ARG, "num_requests %d / num_slots %d outside [1, 65535]", R, S);
    if (K < 1 || K > 64) return fail(DFLASH_ERR_INVALID_ARG, "num_candidates %d outside [1, 64]", K);
    if (vocab < 1) return fail(DFLASH_ERR_INVALID_ARG, "vocab %d < 1", vocab);
    if (E < 8 || E % 8 != 0) return fail(DFLASH_ERR_INVALID_ARG, "dim %d must be a positive multiple of 8", E);
    if (selector_smem_bytes(K, E) > 200 * 1024)
        return fail(DFLASH_ERR_UNSUPPORTED, "num_candidates * dim = %lld above %d", (long long)K * E,
                    200 * 1024 / 6);
    if (!(temperature >= 0.f) || !std::isfinite(temperature))
        return fail(DFLASH_ERR_INVALID_ARG, "temperature must be finite and >= 0");
    if (!pred_codebook || !succ_codebook || !proj || !candidates || !unary || !anchor || !tokens)
        return fail(DFLASH_ERR_INVALID_ARG, "NULL pointer");
    if (temperature > 0.f && !uniforms) return fail(DFLASH_ERR_INVALID_ARG, "temperature > 0 needs uniforms");
    if (!aligned(pred_codebook, 16) || !aligned(succ_codebook, 16) || !aligned(proj, 16) || !aligned(candidates, 4) ||
        !aligned(unary, 4) || !aligned(anchor, 4) || !aligned(tokens, 4) || (uniforms && !aligned(uniforms, 4)) ||
        (chosen && !aligned(chosen, 4)) || (path_scores && !aligned(path_scores, 4)) || (q && !aligned(q, 4)) ||
        (device_error && !aligned(device_error, 4)))
        return fail(DFLASH_ERR_INVALID_ARG, "misaligned pointer (codebooks and proj 16 bytes, the rest 4)");
    const size_t need = dflash_selector_workspace_bytes(R, S, K);
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < need)
        return fail(DFLASH_ERR_WORKSPACE, "the selector needs a 256-byte aligned workspace of %zu bytes", need);
    char* wsb = static_cast<char*>(workspace);
    int32_t* counters = reinterpret_cast<int32_t*>(wsb);
    float* tab = reinterpret_cast<float*>(wsb + kSelectorCounterBytes);
    const cudaError_t e = launch_selector(pred_codebook, succ_codebook, vocab, E, proj, candidates, unary, anchor, R,
                                          S, K, temperature, uniforms, tokens, chosen, path_scores, q, device_error,
                                          tab, counters, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "selector kernel launch");
    return DFLASH_OK;
}

dflash_status dflash_split_combine(const float* partial_out, const float* partial_lse, int32_t num_splits,
                                   int64_t num_rows, int32_t head_dim, dflash_dtype out_dtype, void* out, float* lse,
                                   void* stream)
{
    g_last_error.clear();
    if (!partial_out || !partial_lse || !out) return fail(DFLASH_ERR_INVALID_ARG, "NULL pointer");
    if (num_splits < 1 || num_splits > DFLASH_MAX_SPLITS)
        return fail(DFLASH_ERR_INVALID_ARG, "num_splits %d outside [1, %d]", num_splits, DFLASH_MAX_SPLITS);
    if (num_rows < 1 || num_rows > 0x7fffffffLL)
        return fail(DFLASH_ERR_INVALID_ARG, "num_rows %lld outside [1, 2^31-1]", (long long)num_rows);
    if (head_dim < 4 || head_dim > DFLASH_MAX_HEAD_DIM || head_dim % 4 != 0)
        return fail(DFLASH_ERR_INVALID_ARG, "head_dim %d must be a multiple of 4 in [4, 512]", head_dim);
    if (out_dtype != DFLASH_BF16 && out_dtype != DFLASH_FP32)
        return fail(DFLASH_ERR_INVALID_ARG, "out_dtype %d invalid", (int)out_dtype);
    if (!aligned(partial_out, 16) || !aligned(partial_lse, 4) || !aligned(out, out_dtype == DFLASH_FP32 ? 16 : 8) ||
        (lse && !aligned(lse, 4)))
        return fail(DFLASH_ERR_INVALID_ARG, "misaligned pointer");
    cudaError_t e = launch_combine(partial_out, partial_lse, num_splits, num_rows, head_dim, out_dtype, out, lse,
                                   static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "combine kernel launch");
    return DFLASH_OK;
}

dflash_status dflash_read_error(const void* workspace, void* stream, uint32_t* device_error, int32_t clear)
{
    g_last_error.clear();
    if (!workspace || !device_error) return fail(DFLASH_ERR_INVALID_ARG, "NULL pointer");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "reading the error word");
    if (clear && word) {
        e = cudaMemsetAsync(const_cast<void*>(workspace), 0, sizeof(word), st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        if (e != cudaSuccess) return cuda_fail(e, "clearing the error word");
    }
    if (word & DFLASH_DEVERR_TIMEOUT) {
        // a split combine that gave up may have left arrivals behind: start the counters afresh
        const WorkspaceLayout wl = workspace_layout(1, 1, 1, 16, 1);
        e = cudaMemsetAsync(static_cast<char*>(const_cast<void*>(workspace)) + wl.counters_off, 0,
                            DFLASH_COUNTER_BYTES, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        if (e != cudaSuccess) return cuda_fail(e, "clearing the counter block");
    }
    *device_error = word;
    return word ? DFLASH_ERR_DEVICE_CHECK : DFLASH_OK;
}

}  // extern "C"
