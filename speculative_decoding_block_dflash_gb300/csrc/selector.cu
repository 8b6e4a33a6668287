// DFlash2 candidate-selector walk (prhub report on vLLM PR #52816 "DFlash2", the motivation
// paragraph and changes 1-2). The head keeps K candidate tokens per draft slot. The transition
// from token p to candidate c of slot s scores
//   edge_s(p -> c) = < A[p] * proj[s], B[c] > + unary[s, c]
// (A, B: predecessor and successor codebooks [V, E]; proj[s]: the projected hidden state of
// slot s). Starting from the verified anchor, the walk takes per slot the best edge from the
// previous choice (temperature 0), or with T > 0 samples it by the inverse CDF of
// q = softmax(edge / T) with a given uniform, and reports q.
//
// The dependence between slots only selects which predecessor row is used, so the kernel
// first scores every (predecessor candidate, candidate) pair of every slot in parallel: one CTA
// per (request, slot) stages A[p] * proj[s] (fp32) for its P predecessors (the anchor for slot
// 0, the previous slot's K candidates otherwise) and B[c] (bf16) for its K candidates in
// shared memory, and its warps form the P x K dot products (lane-strided partial sums, then a
// shuffle tree). The tables go to the workspace. The last CTA of a request (an arrival
// counter, no waiting) copies the request's tables on chip when they fit and walks the slots
// with one warp: argmax with the first index on ties, or a warp softmax and a warp scan for the
// inverse CDF. It writes the tokens, the chosen indices, the path's edge scores and q, and
// resets its counter.
#include "dflash_device.cuh"

namespace dflash {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

// token id checked against the vocabulary; a bad id reads row 0 and sets an error bit
__device__ __forceinline__ int32_t checked_token(int32_t tok, int32_t V, uint32_t* err)
{
    if (tok < 0 || tok >= V) {
        raise_error(err, DFLASH_DEVERR_TOKEN_ID);
        return 0;
    }
    return tok;
}

__global__ void __launch_bounds__(kThreads)
    selector_kernel(const __nv_bfloat16* __restrict__ A, const __nv_bfloat16* __restrict__ B, int32_t V, int32_t E,
                    const float* __restrict__ proj, const int32_t* __restrict__ cand, const float* __restrict__ unary,
                    const int32_t* __restrict__ anchor, int32_t S, int32_t K, float temperature,
                    const float* __restrict__ uniforms, int32_t* __restrict__ tokens, int32_t* __restrict__ chosen,
                    float* __restrict__ path_scores, float* __restrict__ q, uint32_t* err, float* tab,
                    int32_t* counters)
{
    extern __shared__ float sm[];
    const int s = blockIdx.x;
    const int r = blockIdx.y;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int P = s == 0 ? 1 : K;
    const int64_t rs = (int64_t)r * S + s;
    float* a_s = sm;                                                      // [P][E] fp32: A[p] * proj[s]
    __nv_bfloat16* b_s = reinterpret_cast<__nv_bfloat16*>(a_s + P * E);  // [K][E] bf16: B[c]
    __shared__ int32_t pred_tok[64], cand_tok[64];
    __shared__ float unary_s[64];
    __shared__ int last;
    if (tid < P) pred_tok[tid] = checked_token(s == 0 ? anchor[r] : cand[(rs - 1) * K + tid], V, err);
    if (tid < K) {
        cand_tok[tid] = checked_token(cand[rs * K + tid], V, err);
        unary_s[tid] = unary[rs * K + tid];
    }
    __syncthreads();

    // stage the rows with 16-byte loads (E is a multiple of 8)
    const int E8 = E / 8;
    const float* pj = proj + rs * E;
    for (int idx = tid; idx < P * E8; idx += kThreads) {
        const int j = idx / E8, e = (idx - j * E8) * 8;
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(A + (int64_t)pred_tok[j] * E + e));
        const float4 p0 = __ldg(reinterpret_cast<const float4*>(pj + e));
        const float4 p1 = __ldg(reinterpret_cast<const float4*>(pj + e + 4));
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
        const float2 f0 = __bfloat1622float2(h[0]), f1 = __bfloat1622float2(h[1]);
        const float2 f2 = __bfloat1622float2(h[2]), f3 = __bfloat1622float2(h[3]);
        float4* dst = reinterpret_cast<float4*>(a_s + j * E + e);
        dst[0] = make_float4(f0.x * p0.x, f0.y * p0.y, f1.x * p0.z, f1.y * p0.w);
        dst[1] = make_float4(f2.x * p1.x, f2.y * p1.y, f3.x * p1.z, f3.y * p1.w);
    }
    for (int idx = tid; idx < K * E8; idx += kThreads) {
        const int k = idx / E8, e = (idx - k * E8) * 8;
        *reinterpret_cast<uint4*>(b_s + k * E + e) = __ldg(reinterpret_cast<const uint4*>(B + (int64_t)cand_tok[k] * E + e));
    }
    __syncthreads();

    // the P x K edge table of this slot
    float* t_out = tab + rs * K * K;  // [P][K] rows used
    for (int pair = warp; pair < P * K; pair += kWarps) {
        const int j = pair / K, k = pair - j * K;
        const float* a = a_s + j * E;
        const __nv_bfloat16* bb = b_s + k * E;
        float acc = 0.f;
        for (int e = lane; e < E; e += 32) acc = fmaf(a[e], __bfloat162float(bb[e]), acc);
        acc = warp_sum(acc);
        if (lane == 0) t_out[j * K + k] = acc + unary_s[k];
    }

    // the last CTA of the request walks its slots
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        last = atomicAdd(counters + r, 1) == S - 1;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    // When the request's S x K x K tables, its S x K candidate ids and S uniforms fit in the
    // staging area, the CTA copies them to shared memory in one round of loads, so that no read
    // on the walk's serial chain leaves the SM; otherwise the walk reads them from L2, issuing
    // each slot's loads together.
    const float* req_tab = tab + (int64_t)r * S * K * K;
    const int32_t* req_cand = cand + (int64_t)r * S * K;
    const float* req_u = uniforms ? uniforms + (int64_t)r * S : nullptr;
    const bool on_chip = (int64_t)S * (K * K + K + 1) <= (int64_t)K * E * 3 / 2;
    int32_t* cand_c = reinterpret_cast<int32_t*>(a_s + S * K * K);  // [S][K] when on chip
    float* u_c = reinterpret_cast<float*>(cand_c + S * K);          // [S] when on chip
    if (on_chip) {
        for (int idx = tid; idx < S * K * K; idx += kThreads) a_s[idx] = __ldcg(req_tab + idx);
        for (int idx = tid; idx < S * K; idx += kThreads) cand_c[idx] = req_cand[idx];
        if (req_u)
            for (int idx = tid; idx < S; idx += kThreads) u_c[idx] = req_u[idx];
        __syncthreads();
    }
    if (warp != 0) return;
    int j = 0;  // row of the previous choice in the current slot's table
    for (int ss = 0; ss < S; ++ss) {
        const int64_t rss = (int64_t)r * S + ss;
        const bool h0 = lane < K, h1 = lane + 32 < K;
        float v0, v1, uu = 0.f;
        int32_t t0, t1;
        if (on_chip) {
            const float* row = a_s + (ss * K + j) * K;
            v0 = h0 ? row[lane] : -INFINITY;
            v1 = h1 ? row[lane + 32] : -INFINITY;
            t0 = h0 ? cand_c[ss * K + lane] : 0;
            t1 = h1 ? cand_c[ss * K + lane + 32] : 0;
            if (req_u) uu = u_c[ss];
        } else {
            const float* row = req_tab + ((int64_t)ss * K + j) * K;
            v0 = h0 ? __ldcg(row + lane) : -INFINITY;
            v1 = h1 ? __ldcg(row + lane + 32) : -INFINITY;
            t0 = h0 ? req_cand[ss * K + lane] : 0;
            t1 = h1 ? req_cand[ss * K + lane + 32] : 0;
            if (req_u) uu = req_u[ss];
        }
        if (path_scores) {
            if (h0) path_scores[rss * K + lane] = v0;
            if (h1) path_scores[rss * K + lane + 32] = v1;
        }
        int kstar;
        if (temperature > 0.f) {
            const float m = warp_max(fmaxf(v0, v1));
            const float x0 = h0 ? expf((v0 - m) / temperature) : 0.f;
            const float x1 = h1 ? expf((v1 - m) / temperature) : 0.f;
            const float inv = 1.f / warp_sum(x0 + x1);
            const float q0 = x0 * inv, q1 = x1 * inv;
            if (q) {
                if (h0) q[rss * K + lane] = q0;
                if (h1) q[rss * K + lane + 32] = q1;
            }
            // inclusive running sums in candidate order: lanes hold k = lane, then k = 32 + lane
            float c0 = q0, c1 = q1;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y0 = __shfl_up_sync(0xffffffffu, c0, off);
                const float y1 = __shfl_up_sync(0xffffffffu, c1, off);
                if (lane >= off) {
                    c0 += y0;
                    c1 += y1;
                }
            }
            c1 += __shfl_sync(0xffffffffu, c0, 31);
            const unsigned m0 = __ballot_sync(0xffffffffu, h0 && c0 > uu);
            const unsigned m1 = __ballot_sync(0xffffffffu, h1 && c1 > uu);
            kstar = m0 ? __ffs(m0) - 1 : (m1 ? 32 + __ffs(m1) - 1 : K - 1);
        } else {
            // argmax, first index on ties
            float bv = v0;
            int bk = lane;
            if (v1 > bv) {
                bv = v1;
                bk = lane + 32;
            }
            if (!h0) bk = 1 << 30;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                const int ok = __shfl_xor_sync(0xffffffffu, bk, off);
                if (ov > bv || (ov == bv && ok < bk)) {
                    bv = ov;
                    bk = ok;
                }
            }
            kstar = bk;
        }
        const int32_t tok = __shfl_sync(0xffffffffu, kstar < 32 ? t0 : t1, kstar & 31);
        if (lane == 0) {
            tokens[rss] = tok;
            if (chosen) chosen[rss] = kstar;
        }
        j = kstar;
    }
    if (lane == 0) counters[r] = 0;
}

}  // namespace

size_t selector_smem_bytes(int32_t K, int32_t E)
{
    return (size_t)K * E * sizeof(float) + (size_t)K * E * sizeof(__nv_bfloat16);
}

cudaError_t launch_selector(const void* A, const void* B, int32_t V, int32_t E, const float* proj, const int32_t* cand,
                            const float* unary, const int32_t* anchor, int32_t R, int32_t S, int32_t K,
                            float temperature, const float* uniforms, int32_t* tokens, int32_t* chosen,
                            float* path_scores, float* q, uint32_t* err, float* tab, int32_t* counters,
                            cudaStream_t stream)
{
    const size_t smem = selector_smem_bytes(K, E);
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(selector_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    selector_kernel<<<dim3(S, R), kThreads, smem, stream>>>(
        static_cast<const __nv_bfloat16*>(A), static_cast<const __nv_bfloat16*>(B), V, E, proj, cand, unary, anchor, S, K,
        temperature, uniforms, tokens, chosen, path_scores, q, err, tab, counters);
    return cudaGetLastError();
}

}  // namespace dflash
