// dflash_block_attn_noalloc: block attention for callers that cannot allocate
// device memory (for example code running inside a custom allocator's own
// hooks, where calling back into the allocator would recurse, or an embedding
// runtime that owns all device memory and forbids cudaMalloc). The split-KV
// partials and the error word normally live in a caller-provided workspace;
// here they live in a fixed-size scratch array that is part of this library's
// device image.
#include <mutex>

#include "dflash_internal.h"

namespace dflash {
namespace {

// Scratch shared by every call of dflash_block_attn_noalloc on a device. It is
// reserved when the library's device code is loaded on that GPU and held until
// the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[DFLASH_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mutex;
void* g_scratch_ptr[64] = {nullptr};

// Device address of the scratch array on the current device (resolved once per
// device with that device current). The host-side symbol is only a stand-in and
// must never be handed to a kernel.
cudaError_t scratch_address(void** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace dflash

using namespace dflash;

extern "C" DFLASH_API dflash_status dflash_block_attn_noalloc(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* page_table, const int32_t* seq_lens,
    const dflash_dims* dims, int32_t block_len, int32_t causal, int32_t window, float scale, void* out, float* lse,
    int32_t num_splits, int32_t kernel, void* stream)
{
    int32_t splits = dflash_plan_splits(dims, block_len, window, num_splits, kernel);
    if (splits < 1) {
        // invalid sizes: let the main entry point report the precise reason
        dflash_opts o{};
        o.num_splits = num_splits;
        o.kernel = kernel;
        o.stream = stream;
        return dflash_block_attn(q, k_cache, v_cache, page_table, seq_lens, dims, block_len, causal, window, scale,
                                 out, lse, &o);
    }
    const int kres = resolve_kernel(dims, block_len, window, kernel);
    bool balanced = num_splits == 0 && splits > 1 && balanced_slots(dims, block_len, window, kres) == splits;
    auto need_of = [&](int32_t s, bool bal) {
        return workspace_layout(bal ? 1 : dims->batch, block_len, dims->num_q_heads, dims->head_dim, s).total;
    };
    size_t need = need_of(splits, balanced);
    if (num_splits == 0 && need > (size_t)DFLASH_NOALLOC_SCRATCH_BYTES) {
        // The auto plan's partials do not fit the scratch (many uniform waves over very long
        // requests): take the one-wave length-balanced plan, whose partials are sized for one
        // request, if it fits; else the most uniform chunks that fit.
        const int32_t bal = balanced_slots(dims, block_len, window, kres, /*allow_long=*/true);
        if (bal > 1 && need_of(bal, true) <= (size_t)DFLASH_NOALLOC_SCRATCH_BYTES) {
            splits = bal;
            balanced = true;
        } else {
            while (splits > 1 && need_of(splits, false) > (size_t)DFLASH_NOALLOC_SCRATCH_BYTES) --splits;
            balanced = false;
        }
        need = need_of(splits, balanced);
    }
    if (need > (size_t)DFLASH_NOALLOC_SCRATCH_BYTES)
        return report_error(DFLASH_ERR_WORKSPACE,
                            "dflash_block_attn_noalloc: %d splits need %zu bytes of scratch, more than the %u bytes "
                            "it holds; request fewer splits",
                            splits, need, (unsigned)DFLASH_NOALLOC_SCRATCH_BYTES);
    void* ws = nullptr;
    cudaError_t e = scratch_address(&ws);
    if (e != cudaSuccess) return report_error(DFLASH_ERR_CUDA, "resolving the scratch address: %s", cudaGetErrorString(e));
    // the error word and the counters must start at zero; the rest is overwritten before it is read
    const WorkspaceLayout wl =
        workspace_layout(balanced ? 1 : dims->batch, block_len, dims->num_q_heads, dims->head_dim, splits);
    e = cudaMemsetAsync(ws, 0, wl.part_lse_off, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return report_error(DFLASH_ERR_CUDA, "clearing the scratch header: %s", cudaGetErrorString(e));
    dflash_opts o{};
    o.num_splits = num_splits;
    o.kernel = kernel;
    o.workspace = ws;
    o.workspace_bytes = DFLASH_NOALLOC_SCRATCH_BYTES;
    o.stream = stream;
    // the plan chosen above (it may differ from the auto plan when that would not fit)
    return block_attn_planned(q, k_cache, v_cache, page_table, seq_lens, dims, block_len, causal, window, scale, out,
                              lse, &o, splits, balanced);
}
