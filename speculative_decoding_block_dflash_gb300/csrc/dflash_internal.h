// Internal interface between the C-ABI front end (api.cpp) and the kernels.
// Not installed; not part of the ABI.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "dflash_attn.h"

namespace dflash {

// Everything a kernel needs for one dflash_block_attn call. Validated on the host.
struct AttnParams {
    const void* q;
    const void* k;
    const void* v;
    const int32_t* page_table;
    const int32_t* seq_lens;
    void* out;            // [B*T, Hq, D] dtype (nullptr when only partials are produced)
    float* lse;           // [B*T, Hq] or nullptr
    float* part_out;      // [S, B*T, Hq, D] when S > 1
    float* part_lse;      // [S, B*T, Hq]    when S > 1
    uint32_t* err;        // device error word or nullptr
    int32_t* counters;    // [B*Hq] zero-initialised counters or nullptr
    int32_t B, T, Hq, Hkv, G, D;
    int32_t page_size, num_pages, max_pages, max_seq_len;
    int64_t sp, ss, sh;   // K/V element strides: page, slot, head
    int32_t causal, window;
    float scale;
    int32_t splits;       // uniform: chunks per request; balanced: chunk slots in total
    int32_t dtype;        // dflash_dtype
    int32_t balanced;     // 1: the tensor-core kernel deals its `splits` slots to the requests in
                          // proportion to their key spans (partials laid out [slot][T][Hq][D])
    unsigned long long wait_ns;  // bound of every device-side wait (pipeline and combine)
};

// Default bound of a device-side wait (dflash_opts.wait_limit_us == 0).
constexpr unsigned long long DFLASH_DEFAULT_WAIT_NS = 2000000000ull;

// Workspace carve-up (offsets in bytes from the workspace base). The counter block has a
// fixed size, so a workspace zeroed once stays valid for calls of any size: two int32
// counters per (request, row group) of an in-kernel split combine, which only runs when the
// whole grid is resident (at most a few hundred groups).
constexpr size_t DFLASH_COUNTER_BYTES = 8192;
constexpr int DFLASH_MAX_COMBINE_GROUPS = (int)(DFLASH_COUNTER_BYTES / 8);
struct WorkspaceLayout {
    size_t err_off, counters_off, part_lse_off, part_out_off, total;
};
WorkspaceLayout workspace_layout(int32_t B, int32_t T, int32_t Hq, int32_t D, int32_t splits);

// Longest-prefix acceptance (csrc/accept.cu).
int32_t accept_chunks(int32_t B, int32_t T, int32_t V);
cudaError_t launch_accept(const void* logits, int32_t dtype, int32_t B, int32_t T, int32_t V, int64_t row_stride,
                          const int32_t* draft, int32_t* accepted, int32_t* next_token, int32_t* target_argmax,
                          unsigned long long* keys, int32_t* counters, cudaStream_t stream);

// DFlash2 candidate-selector walk (csrc/selector.cu).
size_t selector_smem_bytes(int32_t K, int32_t E);
cudaError_t launch_selector(const void* A, const void* B, int32_t V, int32_t E, const float* proj, const int32_t* cand,
                            const float* unary, const int32_t* anchor, int32_t R, int32_t S, int32_t K,
                            float temperature, const float* uniforms, int32_t* tokens, int32_t* chosen,
                            float* path_scores, float* q, uint32_t* err, float* tab, int32_t* counters,
                            cudaStream_t stream);

// DFlash2 grouped dynamic depthwise convolution (csrc/grouped_conv.cu).
cudaError_t launch_grouped_conv(const void* x, void* out, int32_t dtype, int32_t B, int32_t T, int32_t C,
                                int32_t taps, int32_t G, const float* base, const float* delta, cudaStream_t stream);

// Context K/V projection (csrc/project_kv.cu): persistent CTAs (at most one per SM).
int32_t project_kv_grid(int32_t L, int32_t N);
size_t project_kv_workspace_bytes();
cudaError_t launch_project_kv(const void* hidden, int32_t L, int32_t H, int64_t hidden_stride, const void* w_k,
                              const void* w_v, const int32_t* slot_mapping, void* k_cache, void* v_cache,
                              int32_t Hkv, int32_t D, int32_t page_size, int32_t num_pages, int64_t sp, int64_t ss,
                              int64_t sh, uint32_t* err, void* workspace, size_t workspace_bytes,
                              cudaStream_t stream);

// Slots of the tensor-core kernel's length-balanced split plan for these sizes (auto split
// count, B > 1, whole grid resident), or 0 when the plan is uniform. The auto plan leaves it
// for very long key spans (allow_long = false); the no-alloc entry point may still take it.
int32_t balanced_slots(const dflash_dims* d, int32_t T, int32_t window, int kernel, bool allow_long = false);
// dflash_block_attn with the split plan given (forced_splits >= 1) or planned (forced_splits < 1).
dflash_status block_attn_planned(const void* q, const void* k_cache, const void* v_cache, const int32_t* page_table,
                                 const int32_t* seq_lens, const dflash_dims* dims, int32_t block_len, int32_t causal,
                                 int32_t window, float scale, void* out, float* lse, const dflash_opts* opts,
                                 int32_t forced_splits, bool forced_balanced);
// Kernel a selector resolves to for these sizes (a dflash_kernel value), or -status.
int resolve_kernel(const dflash_dims* d, int32_t T, int32_t window, int32_t requested);

// Kernel launchers (return cudaSuccess or the launch error).
cudaError_t launch_simt_attn(const AttnParams& p, cudaStream_t stream);
cudaError_t launch_combine(const float* part_out, const float* part_lse, int32_t splits,
                           int64_t rows, int32_t D, int32_t out_dtype, void* out, float* lse,
                           cudaStream_t stream);

// Tensor-core kernel: whether it covers these sizes, and its launcher.
bool tc_supports(const AttnParams& p);
int tc_ctas_per_split(const AttnParams& p);  // CTAs per split chunk (B * Hkv * row groups)
cudaError_t launch_tc_attn(const AttnParams& p, cudaStream_t stream);
// Grid of a launch_tc_attn call and whether it combines the splits in-kernel (the whole grid
// resident: a cooperative launch). Assumes a workspace (counters) is given.
cudaError_t tc_grid_info(const AttnParams& p, int64_t* ctas, bool* fused);

int tc_row_groups(const AttnParams& p);       // CTAs per (request, KV head, chunk)

// CTA-pair tensor-core kernel (tcgen05 cta_group::2 over a 2-CTA cluster; up to 128 packed rows
// at head_dim 256/512, every K/V byte read by one SM). Uniform split plans only.
bool tc_pair_supports(const AttnParams& p);
int tc_pair_ctas_per_split(const AttnParams& p);  // CTAs per split chunk (2 * B * Hkv * row groups)
int tc_pair_row_groups(const AttnParams& p);      // pairs per (request, KV head, chunk)
cudaError_t tc_pair_grid_ctas(const AttnParams& p, int64_t* ctas);  // CTAs of the persistent launch
cudaError_t launch_tc_pair_attn(const AttnParams& p, cudaStream_t stream);

// SM count of the current device (cached per device).
int device_sm_count();

// Records the text returned by dflash_last_error_message() and returns s.
dflash_status report_error(dflash_status s, const char* fmt, ...);

}  // namespace dflash
