// Log-sum-exp combine of split-KV partials (flash-decoding style; the
// "split-KV combine" step named in the prhub report on vLLM PR #52816
// "DFlash2", review highlights):
//   m = max_c lse_c, w_c = exp(lse_c - m), out = sum_c w_c o_c / sum_c w_c,
//   lse = m + log(sum_c w_c); chunks with lse_c = -inf weigh nothing.
//
// One thread per float4 of an output row: head_dim / 4 threads cover a row, so a 128-thread
// CTA holds 128 / (head_dim / 4) rows (1 at head_dim 512). Every thread reads the row's chunk
// lse values itself (the row's threads share them through L1), forms the weights in
// registers, and keeps eight partial-row loads in flight per round, with no block barrier.
#include <cmath>

#include "dflash_device.cuh"

namespace dflash {
namespace {

constexpr int kThreads = 128;

__global__ void __launch_bounds__(kThreads)
    combine_kernel(const float* __restrict__ part_out, const float* __restrict__ part_lse, int32_t S,
                   int64_t rows, int32_t D, int32_t out_dtype, void* __restrict__ out,
                   float* __restrict__ lse)
{
    const int lanes = D / 4;                   // threads per output row
    const int per_cta = kThreads / lanes;      // rows per CTA
    const int sub = threadIdx.x / lanes;
    const int d0 = (threadIdx.x - sub * lanes) * 4;
    const int64_t row = (int64_t)blockIdx.x * per_cta + sub;
    // Launched as a programmatic dependent of the attention kernel: wait until
    // that grid has completed and its partials are visible.
    cudaGridDependencySynchronize();
    if (sub >= per_cta || row >= rows) return;
    const float* lrow = part_lse + row;
    // max over chunks
    float m = -INFINITY;
    for (int c0 = 0; c0 < S; c0 += 8) {
        float l[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) l[k] = c0 + k < S ? __ldg(lrow + (int64_t)(c0 + k) * rows) : -INFINITY;
#pragma unroll
        for (int k = 0; k < 8; ++k) m = fmaxf(m, l[k]);
    }
    // weighted sum; empty chunks (lse = -inf) weigh nothing and their partials are not read
    float t = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (m != -INFINITY) {
        const float* base = part_out + row * D + d0;
        const int64_t cstride = rows * D;
        for (int c0 = 0; c0 < S; c0 += 8) {
            float w[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float l = c0 + k < S ? __ldg(lrow + (int64_t)(c0 + k) * rows) : -INFINITY;
                w[k] = (l == -INFINITY) ? 0.f : expf(l - m);
            }
            float4 v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                v[k] = w[k] > 0.f ? __ldg(reinterpret_cast<const float4*>(base + (int64_t)(c0 + k) * cstride))
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                t += w[k];
                acc.x = fmaf(w[k], v[k].x, acc.x);
                acc.y = fmaf(w[k], v[k].y, acc.y);
                acc.z = fmaf(w[k], v[k].z, acc.z);
                acc.w = fmaf(w[k], v[k].w, acc.w);
            }
        }
    }
    const bool empty = (m == -INFINITY) || !(t > 0.f);
    const float inv = empty ? 0.f : 1.f / t;
    const int64_t o = row * D + d0;
    if (out_dtype == DFLASH_BF16) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
        uint2 pk;
        pk.x = *reinterpret_cast<const uint32_t*>(&lo);
        pk.y = *reinterpret_cast<const uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(out) + o) = pk;
    } else {
        *reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + o) =
            make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    }
    if (d0 == 0 && lse) lse[row] = empty ? -INFINITY : m + logf(t);
}

}  // namespace

cudaError_t launch_combine(const float* part_out, const float* part_lse, int32_t splits, int64_t rows,
                           int32_t D, int32_t out_dtype, void* out, float* lse, cudaStream_t stream)
{
    if (rows <= 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    const int64_t per_cta = kThreads / (D / 4);
    cfg.gridDim = dim3((unsigned)((rows + per_cta - 1) / per_cta));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, combine_kernel, part_out, part_lse, splits, rows, D, out_dtype, out, lse);
}

}  // namespace dflash
