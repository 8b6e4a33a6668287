// Log-sum-exp combine of split-KV partials (flash-decoding style; the
// "split-KV combine" step named in the prhub report on vLLM PR #52816
// "DFlash2", review highlights):
//   m = max_c lse_c, w_c = exp(lse_c - m), out = sum_c w_c o_c / sum_c w_c,
//   lse = m + log(sum_c w_c); chunks with lse_c = -inf weigh nothing.
//
// One CTA per output row (query row x head), 512 threads. D/4 threads cover
// one partial row with float4 loads (D <= 512), so the CTA holds 512 / (D/4)
// such groups; group g sums the chunks c = g, g + groups, ... and the groups
// meet in shared memory. The chunk weights are computed once per CTA; each
// thread keeps eight partial-row loads in flight, so at D = 512 a 32-chunk
// combine costs one L2 round trip instead of eight.
#include <cmath>

#include "dflash_device.cuh"

namespace dflash {
namespace {

constexpr int kThreads = 512;

__global__ void __launch_bounds__(kThreads)
    combine_kernel(const float* __restrict__ part_out, const float* __restrict__ part_lse, int32_t S,
                   int64_t rows, int32_t D, int32_t out_dtype, void* __restrict__ out,
                   float* __restrict__ lse)
{
    __shared__ float w_s[DFLASH_MAX_SPLITS];
    __shared__ float red[kThreads / 32];
    __shared__ float m_sh, inv_sh, lse_sh;
    __shared__ float4 acc_s[kThreads];
    const int64_t row = blockIdx.x;
    const int tid = threadIdx.x;
    // Launched as a programmatic dependent of the attention kernel: wait until
    // that grid has completed and its partials are visible.
    cudaGridDependencySynchronize();

    // max over chunks
    float m = -INFINITY;
    for (int c = tid; c < S; c += kThreads) m = fmaxf(m, part_lse[(int64_t)c * rows + row]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if ((tid & 31) == 0) red[tid >> 5] = m;
    __syncthreads();
    if (tid == 0) {
        float mm = red[0];
        for (int w = 1; w < kThreads / 32; ++w) mm = fmaxf(mm, red[w]);
        m_sh = mm;
    }
    __syncthreads();
    m = m_sh;

    float ws = 0.f;
    for (int c = tid; c < S; c += kThreads) {
        const float l = part_lse[(int64_t)c * rows + row];
        const float w = (l == -INFINITY) ? 0.f : expf(l - m);
        w_s[c] = w;
        ws += w;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, off);
    __syncthreads();
    if ((tid & 31) == 0) red[tid >> 5] = ws;
    __syncthreads();
    if (tid == 0) {
        float t = 0.f;
        for (int w = 0; w < kThreads / 32; ++w) t += red[w];
        const bool empty = (m == -INFINITY) || !(t > 0.f);
        inv_sh = empty ? 0.f : 1.f / t;
        lse_sh = empty ? -INFINITY : m + logf(t);
    }
    __syncthreads();
    const float inv = inv_sh;

    const int lanes = D / 4;              // threads per partial row
    const int groups = kThreads / lanes;  // chunk groups
    const int gi = tid / lanes;
    const int d0 = (tid - gi * lanes) * 4;
    // empty chunks carry weight 0 and zero partials
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (inv > 0.f && gi < groups) {
        const float* base = part_out + row * D + d0;
        const int64_t cstride = rows * D;
        for (int c0 = gi; c0 < S; c0 += 8 * groups) {
            float4 v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int c = c0 + k * groups;
                v[k] = c < S ? __ldg(reinterpret_cast<const float4*>(base + c * cstride))
                             : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int c = c0 + k * groups;
                const float w = c < S ? w_s[c] : 0.f;
                acc.x = fmaf(w, v[k].x, acc.x);
                acc.y = fmaf(w, v[k].y, acc.y);
                acc.z = fmaf(w, v[k].z, acc.z);
                acc.w = fmaf(w, v[k].w, acc.w);
            }
        }
    }
    acc_s[tid] = acc;
    __syncthreads();
    if (tid < lanes) {
        for (int g = 1; g < groups; ++g) {
            const float4 o = acc_s[g * lanes + tid];
            acc.x += o.x;
            acc.y += o.y;
            acc.z += o.z;
            acc.w += o.w;
        }
        const int64_t o = row * D + d0;
        if (out_dtype == DFLASH_BF16) {
            __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
            __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
            uint2 pk;
            pk.x = *reinterpret_cast<uint32_t*>(&lo);
            pk.y = *reinterpret_cast<uint32_t*>(&hi);
            *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(out) + o) = pk;
        } else {
            *reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + o) =
                make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        }
    }
    if (tid == 0 && lse) lse[row] = lse_sh;
}

}  // namespace

cudaError_t launch_combine(const float* part_out, const float* part_lse, int32_t splits, int64_t rows,
                           int32_t D, int32_t out_dtype, void* out, float* lse, cudaStream_t stream)
{
    if (rows <= 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)rows);
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
