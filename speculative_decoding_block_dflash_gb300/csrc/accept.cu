// Longest-prefix acceptance of a drafted block (the verify step that follows the block
// attention; kenforever1 "dflash-gemma4-31b-notes", relation diagram steps 3-4: the target
// verifies the block in parallel and the longest correct prefix is accepted).
//
// For each request b and block position j the target's token is the argmax of its logits
// row (smallest index among equal maxima); draft d_i is correct when it equals the target
// token at position i-1; the accepted length a is the longest run of correct drafts and
// the emitted token is the target token at position a.
//
// The argmax is a pure HBM stream over B*T rows of V logits. Each row is cut into `chunks`
// slices, one CTA per slice (one wave of four CTAs per SM), so a batch of a few dozen rows
// still fills the GPU. A thread reads its part of a slice with 16-byte loads, eight in flight, and
// keeps a running (maximum, first index). It then forms one 64-bit key: the maximum mapped
// to an order-preserving unsigned integer in the high word and (2^32 - 1 - index) in the
// low word, so that the largest key is the largest logit with the smallest index. The warp
// and then the CTA reduce their keys and one thread merges the CTA's key into the row's key
// with a 64-bit atomicMax. The last CTA of a request (an atomic arrival counter,
// no waiting) reads the request's T row keys, applies the prefix rule, writes the results
// and resets the keys and the counter to zero for the next call.
#include <algorithm>

#include "dflash_device.cuh"

namespace dflash {
namespace {

constexpr int kThreads = 256;
constexpr int kBatch = 8;        // 16-byte loads in flight per thread
constexpr int kCtasPerSm = 4;    // resident CTAs per SM: 64 registers leave room for kBatch loads

__device__ __forceinline__ unsigned long long make_key(float x, int32_t idx)
{
    uint32_t u = __float_as_uint(x);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);  // order-preserving for non-NaN floats
    return ((unsigned long long)u << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)idx);
}

__device__ __forceinline__ unsigned long long key_max(unsigned long long a, unsigned long long b)
{
    return a > b ? a : b;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    accept_kernel(const void* __restrict__ logits, int32_t dtype, int32_t T, int32_t V, int64_t row_stride,
                  int32_t chunks, const int32_t* __restrict__ draft, int32_t* __restrict__ accepted,
                  int32_t* __restrict__ next_token, int32_t* __restrict__ target_argmax,
                  unsigned long long* keys, int32_t* counters)
{
    __shared__ unsigned long long warp_best[kThreads / 32];
    __shared__ int last;
    const int row = blockIdx.y;  // b * T + j
    const int b = row / T;
    const int tid = threadIdx.x;
    const int per = (((V + chunks - 1) / chunks) + 7) & ~7;  // slice length, a multiple of 8
    const int v0 = blockIdx.x * per;
    const int v1 = min(V, v0 + per);

    // Per thread: the running maximum and its index. Indices are visited in increasing order
    // and replaced only on a strictly larger value, so among equal maxima the first is kept;
    // the index starts at the slice's first element so that a slice of -inf logits yields it.
    float bv = -INFINITY;
    int bi = v0;
    auto take = [&](float x, int v) {
        const bool p = x > bv;
        bv = p ? x : bv;
        bi = p ? v : bi;
    };
    // Each slice is read as a scalar head up to the first 16-byte boundary, a body of 16-byte
    // vectors (kBatch in flight per thread) and a scalar tail, so rows of any stride and offset
    // are covered.
    if (dtype == DFLASH_BF16) {
        const __nv_bfloat16* r = static_cast<const __nv_bfloat16*>(logits) + row * row_stride;
        const int mis = (int)((reinterpret_cast<uintptr_t>(r + v0) & 15) >> 1);  // elements past a boundary
        const int vb = min(v1, v0 + (mis ? 8 - mis : 0));
        const int vend = vb + ((max(v1 - vb, 0)) & ~7);  // 8-element (16-byte) body
        for (int v = v0 + tid; v < vb; v += kThreads) take(__bfloat162float(r[v]), v);
        int v = vb + tid * 8;
        for (; v + (kBatch - 1) * kThreads * 8 < vend; v += kBatch * kThreads * 8) {
            uint4 w[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) w[u] = __ldcs(reinterpret_cast<const uint4*>(r + v + u * kThreads * 8));
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int base = v + u * kThreads * 8;
                take(bf16_lo(w[u].x), base + 0);
                take(bf16_hi(w[u].x), base + 1);
                take(bf16_lo(w[u].y), base + 2);
                take(bf16_hi(w[u].y), base + 3);
                take(bf16_lo(w[u].z), base + 4);
                take(bf16_hi(w[u].z), base + 5);
                take(bf16_lo(w[u].w), base + 6);
                take(bf16_hi(w[u].w), base + 7);
            }
        }
        for (; v < vend; v += kThreads * 8) {
            const uint4 w = __ldcs(reinterpret_cast<const uint4*>(r + v));
            take(bf16_lo(w.x), v + 0);
            take(bf16_hi(w.x), v + 1);
            take(bf16_lo(w.y), v + 2);
            take(bf16_hi(w.y), v + 3);
            take(bf16_lo(w.z), v + 4);
            take(bf16_hi(w.z), v + 5);
            take(bf16_lo(w.w), v + 6);
            take(bf16_hi(w.w), v + 7);
        }
        for (int t = vend + tid; t < v1; t += kThreads) take(__bfloat162float(r[t]), t);
    } else {
        const float* r = static_cast<const float*>(logits) + row * row_stride;
        const int mis = (int)((reinterpret_cast<uintptr_t>(r + v0) & 15) >> 2);
        const int vb = min(v1, v0 + (mis ? 4 - mis : 0));
        const int vend = vb + ((max(v1 - vb, 0)) & ~3);  // 4-element (16-byte) body
        for (int v = v0 + tid; v < vb; v += kThreads) take(r[v], v);
        int v = vb + tid * 4;
        for (; v + (kBatch - 1) * kThreads * 4 < vend; v += kBatch * kThreads * 4) {
            float4 f[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) f[u] = __ldcs(reinterpret_cast<const float4*>(r + v + u * kThreads * 4));
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int base = v + u * kThreads * 4;
                take(f[u].x, base + 0);
                take(f[u].y, base + 1);
                take(f[u].z, base + 2);
                take(f[u].w, base + 3);
            }
        }
        for (; v < vend; v += kThreads * 4) {
            const float4 f = __ldcs(reinterpret_cast<const float4*>(r + v));
            take(f.x, v + 0);
            take(f.y, v + 1);
            take(f.z, v + 2);
            take(f.w, v + 3);
        }
        for (int t = vend + tid; t < v1; t += kThreads) take(r[t], t);
    }
    unsigned long long best = (v0 < v1) ? make_key(bv, bi) : 0ull;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) best = key_max(best, __shfl_xor_sync(0xffffffffu, best, off));
    if ((tid & 31) == 0) warp_best[tid >> 5] = best;
    __syncthreads();
    if (tid == 0) {
        for (int w = 1; w < kThreads / 32; ++w) best = key_max(best, warp_best[w]);
        if (best) atomicMax(keys + row, best);
        __threadfence();
        last = atomicAdd(counters + b, 1) == chunks * T - 1;
    }
    __syncthreads();
    if (!last || tid != 0) return;

    // last CTA of request b: every slice of its T rows has been merged
    __threadfence();
    unsigned long long* k = keys + (int64_t)b * T;
    int a = 0;
    bool run = true;
    int32_t tok_a = 0;
    for (int j = 0; j < T; ++j) {
        const unsigned long long key = atomicAdd(k + j, 0ull);  // coherent read of the merged key
        const int32_t tok = (int32_t)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
        if (target_argmax) target_argmax[(int64_t)b * T + j] = tok;
        if (run) {
            if (j < T - 1 && draft[(int64_t)b * (T - 1) + j] == tok) {
                ++a;
            } else {
                tok_a = tok;
                run = false;
            }
        }
        k[j] = 0ull;
    }
    accepted[b] = a;
    next_token[b] = tok_a;
    counters[b] = 0;
}

}  // namespace

int32_t accept_chunks(int32_t B, int32_t T, int32_t V)
{
    const int64_t rows = (int64_t)B * T;
    // one full wave: a partial second wave would add a whole round trip for a few CTAs
    const int64_t want = (int64_t)kCtasPerSm * device_sm_count() / rows;
    const int64_t most = std::max<int64_t>(1, ((int64_t)V + 4095) / 4096);  // >= 4096 logits a slice
    return (int32_t)std::max<int64_t>(1, std::min(want, most));
}

cudaError_t launch_accept(const void* logits, int32_t dtype, int32_t B, int32_t T, int32_t V, int64_t row_stride,
                          const int32_t* draft, int32_t* accepted, int32_t* next_token, int32_t* target_argmax,
                          unsigned long long* keys, int32_t* counters, cudaStream_t stream)
{
    const int32_t chunks = accept_chunks(B, T, V);
    accept_kernel<<<dim3(chunks, B * T), kThreads, 0, stream>>>(logits, dtype, T, V, row_stride, chunks, draft,
                                                                 accepted, next_token, target_argmax, keys, counters);
    return cudaGetLastError();
}

}  // namespace dflash
