// DFlash2 grouped dynamic depthwise convolution inside a drafted block (prhub report on vLLM
// PR #52816 "DFlash2", the motivation paragraph and change 1):
//   out[b, i, c] = sum_{t < taps, t <= i} (base[t, c] + delta[b, i, t, g(c)]) * x[b, i - t, c]
// with g(c) = c / (C / G) (contiguous channel groups). Taps that reach past the start of the
// request's own block contribute zero.
//
// The operation is a short per-channel recurrence over a block of at most 64 positions: a few
// MB per call, no contraction worth a tensor core, so the time goes to latency. One CTA takes
// 256 channels of one request (thread = channel). It first stages, with every load in flight
// at once, the request's block of those channels, their static taps and (when it fits in
// 32 KB) the request's whole delta block in shared memory. Each thread then walks the
// positions, summing up to `taps` products in fp32 from shared memory only.
//
// With an even channel count (and x, out aligned to two elements) a thread takes a pair of
// adjacent channels (512 channels a CTA): paired loads and stores, and a tap loop unrolled
// to a compile-time bound (4, 8, 16 or 64) with a guard per tap, so the instruction count
// per output stays near the handful of loads and FMAs it needs. Other shapes take the
// one-channel kernel.
#include <algorithm>

#include "dflash_device.cuh"

namespace dflash {
namespace {

constexpr int kThreads = 256;
constexpr int kDeltaSmemMax = 32 * 1024;  // bytes of delta[b] staged in shared memory

__host__ __device__ inline size_t conv_smem_bytes(int T, int taps, int G, bool* stage_delta)
{
    const size_t delta_bytes = (size_t)T * taps * G * sizeof(float);
    const bool sd = delta_bytes <= (size_t)kDeltaSmemMax;
    if (stage_delta) *stage_delta = sd;
    return ((size_t)T + taps) * kThreads * sizeof(float) + (sd ? delta_bytes : 0);
}

__global__ void __launch_bounds__(kThreads)
    grouped_conv_kernel(const void* __restrict__ x, void* __restrict__ out, int32_t dtype, int32_t T, int32_t C,
                        int32_t taps, int32_t G, const float* __restrict__ base, const float* __restrict__ delta,
                        int32_t stage_delta)
{
    extern __shared__ float sm[];
    float* xs = sm;                       // [T][kThreads]: x of this CTA's channels
    float* bs = xs + T * kThreads;        // [taps][kThreads]: base of this CTA's channels
    float* ds = bs + taps * kThreads;     // [T][taps][G]: delta[b] when staged
    const int b = blockIdx.y;
    const int tid = threadIdx.x;
    const int c = blockIdx.x * kThreads + tid;
    const bool live = c < C;
    const int64_t row0 = (int64_t)b * T;
    const float* db = delta + row0 * taps * G;  // delta[b]
    if (dtype == DFLASH_BF16) {
        const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x) + row0 * C + c;
#pragma unroll 8
        for (int j = 0; j < T; ++j) xs[j * kThreads + tid] = live ? __bfloat162float(xb[(int64_t)j * C]) : 0.f;
    } else {
        const float* xb = static_cast<const float*>(x) + row0 * C + c;
#pragma unroll 8
        for (int j = 0; j < T; ++j) xs[j * kThreads + tid] = live ? __ldg(xb + (int64_t)j * C) : 0.f;
    }
#pragma unroll 4
    for (int t = 0; t < taps; ++t) bs[t * kThreads + tid] = live ? __ldg(base + (int64_t)t * C + c) : 0.f;
    if (stage_delta) {
        const int n = T * taps * G;
        for (int k = tid; k < n; k += kThreads) ds[k] = __ldg(db + k);
    }
    __syncthreads();
    if (!live) return;
    const int g = c / (C / G);
    const int nt = min(taps, T);
    const float* dsrc = stage_delta ? ds : db;
    const int64_t row_stride = (int64_t)taps * G;  // delta elements per position
    for (int i = 0; i < T; ++i) {
        const float* d = dsrc + i * row_stride + g;  // delta[b, i, 0, g]
        float acc = 0.f;
        const int tmax = min(i, nt - 1);
        for (int t = 0; t <= tmax; ++t)
            acc = fmaf(bs[t * kThreads + tid] + d[(int64_t)t * G], xs[(i - t) * kThreads + tid], acc);
        store_elem(out, (row0 + i) * C + c, acc, dtype);
    }
}

// Pair kernel: thread = channels (c, c + 1), c even; NT >= taps.
template <int NT>
__global__ void __launch_bounds__(kThreads)
    grouped_conv_pair_kernel(const void* __restrict__ x, void* __restrict__ out, int32_t dtype, int32_t T, int32_t C,
                             int32_t taps, int32_t G, const float* __restrict__ base,
                             const float* __restrict__ delta, int32_t stage_delta)
{
    extern __shared__ float sm[];
    float2* xs = reinterpret_cast<float2*>(sm);  // [T][kThreads]
    float2* bs = xs + T * kThreads;              // [taps][kThreads]
    float* ds = reinterpret_cast<float*>(bs + taps * kThreads);
    const int b = blockIdx.y;
    const int tid = threadIdx.x;
    const int c = 2 * (blockIdx.x * kThreads + tid);
    const bool live = c < C;  // C is even, so c + 1 < C too
    const int64_t row0 = (int64_t)b * T;
    const float* db = delta + row0 * taps * G;
    const int64_t step = C / 2;  // pairs per row
    if (dtype == DFLASH_BF16) {
        const __nv_bfloat162* xb = reinterpret_cast<const __nv_bfloat162*>(static_cast<const __nv_bfloat16*>(x) +
                                                                             row0 * C + c);
#pragma unroll 8
        for (int j = 0; j < T; ++j) xs[j * kThreads + tid] = live ? __bfloat1622float2(xb[j * step]) : make_float2(0.f, 0.f);
    } else {
        const float2* xb = reinterpret_cast<const float2*>(static_cast<const float*>(x) + row0 * C + c);
#pragma unroll 8
        for (int j = 0; j < T; ++j) xs[j * kThreads + tid] = live ? __ldg(xb + j * step) : make_float2(0.f, 0.f);
    }
    for (int t = 0; t < taps; ++t)
        bs[t * kThreads + tid] = live ? __ldg(reinterpret_cast<const float2*>(base + (int64_t)t * C + c))
                                      : make_float2(0.f, 0.f);
    if (stage_delta) {
        const int n = T * taps * G;
        for (int k = tid; k < n; k += kThreads) ds[k] = __ldg(db + k);
    }
    __syncthreads();
    if (!live) return;
    const int gs = C / G;
    const int g0 = c / gs, g1 = (c + 1) / gs;
    const float* dsrc = stage_delta ? ds : db;
    const int64_t row_stride = (int64_t)taps * G;
    float2 bt[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) bt[t] = t < taps ? bs[t * kThreads + tid] : make_float2(0.f, 0.f);
    for (int i = 0; i < T; ++i) {
        const float* d = dsrc + i * row_stride;  // delta[b, i, 0, 0]
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            if (t < taps && t <= i) {
                const float2 xv = xs[(i - t) * kThreads + tid];
                a0 = fmaf(bt[t].x + d[(int64_t)t * G + g0], xv.x, a0);
                a1 = fmaf(bt[t].y + d[(int64_t)t * G + g1], xv.y, a1);
            }
        }
        const int64_t o = (row0 + i) * C + c;
        if (dtype == DFLASH_BF16)
            *reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(out) + o) = __floats2bfloat162_rn(a0, a1);
        else
            *reinterpret_cast<float2*>(static_cast<float*>(out) + o) = make_float2(a0, a1);
    }
}

}  // namespace

cudaError_t launch_grouped_conv(const void* x, void* out, int32_t dtype, int32_t B, int32_t T, int32_t C,
                                int32_t taps, int32_t G, const float* base, const float* delta, cudaStream_t stream)
{
    bool stage_delta = false;
    const size_t smem = conv_smem_bytes(T, taps, G, &stage_delta);  // pair layout: 2x the x and base rows
    const size_t es = dtype == DFLASH_BF16 ? 2 : 4;
    const size_t psmem = ((size_t)T + taps) * kThreads * sizeof(float2) + (stage_delta ? (size_t)T * taps * G * 4 : 0);
    const bool pair = C % 2 == 0 && reinterpret_cast<uintptr_t>(x) % (2 * es) == 0 &&
                      reinterpret_cast<uintptr_t>(out) % (2 * es) == 0 && reinterpret_cast<uintptr_t>(base) % 8 == 0 &&
                      psmem <= 200 * 1024;
    if (pair) {
        const dim3 grid((C / 2 + kThreads - 1) / kThreads, B);
        auto run = [&](auto kern) -> cudaError_t {
            if (psmem > 48 * 1024) {
                const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)psmem);
                if (e != cudaSuccess) return e;
            }
            kern<<<grid, kThreads, psmem, stream>>>(x, out, dtype, T, C, taps, G, base, delta, stage_delta ? 1 : 0);
            return cudaGetLastError();
        };
        if (taps <= 4) return run(grouped_conv_pair_kernel<4>);
        if (taps <= 8) return run(grouped_conv_pair_kernel<8>);
        if (taps <= 16) return run(grouped_conv_pair_kernel<16>);
        return run(grouped_conv_pair_kernel<64>);
    }
    if (smem > 48 * 1024) {
        const cudaError_t e =
            cudaFuncSetAttribute(grouped_conv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    grouped_conv_kernel<<<dim3((C + kThreads - 1) / kThreads, B), kThreads, smem, stream>>>(
        x, out, dtype, T, C, taps, G, base, delta, stage_delta ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace dflash
