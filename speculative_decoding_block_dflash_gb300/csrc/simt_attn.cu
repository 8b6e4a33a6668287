// CUDA-core (SIMT) block attention: the fp32 path and the portable bf16 path.
//
// One CTA handles up to 16 block queries of one query head of one request and
// one split chunk of its keys. Keys are streamed in tiles of 16 through shared
// memory (converted to fp32), scores are per-thread dot products, the softmax
// is online (running max m and sum l per row, rescale by exp(m_old - m_new)),
// and the output accumulators live in registers (thread owns head-dim columns
// tid and tid + 256 for all 16 rows). Everything accumulates in fp32.
//
// Mask semantics follow the DFlash block definition: the block's queries are
// the last T positions of the request; non-causal rows see every key up to
// L - 1 (kenforever1 "dflash-gemma4-31b-notes", "why non-causal attention"),
// causal rows see keys up to their own position (vLLM PR #43445 "Allow causal
// DFlash"), and a window W keeps the last W keys ending at the query.
#include <cmath>

#include "dflash_device.cuh"

namespace dflash {
namespace {

constexpr int kRows = 16;     // block queries per CTA
constexpr int kKeys = 16;     // keys per tile
constexpr int kThreads = 256;
constexpr int kColsPerThread = DFLASH_MAX_HEAD_DIM / kThreads;  // 2

struct SimtSmem {
    static size_t bytes(int D)
    {
        const int ld = D + 1;
        return sizeof(float) * ((size_t)kRows * ld + (size_t)kKeys * ld + (size_t)kKeys * D +
                                kRows * kKeys + 3 * kRows) +
               sizeof(int32_t) * kKeys;
    }
};

__global__ void __launch_bounds__(kThreads) simt_attn_kernel(const AttnParams p)
{
    extern __shared__ float smem[];
    const int D = p.D;
    const int ld = D + 1;
    float* Qs = smem;                       // [kRows][ld]
    float* Ks = Qs + kRows * ld;            // [kKeys][ld]
    float* Vs = Ks + kKeys * ld;            // [kKeys][D]
    float* Ps = Vs + kKeys * D;             // [kRows][kKeys] scores, then probabilities
    float* m_s = Ps + kRows * kKeys;        // [kRows] running max
    float* l_s = m_s + kRows;               // [kRows] running sum
    float* a_s = l_s + kRows;               // [kRows] rescale factor of this tile
    int32_t* pg = reinterpret_cast<int32_t*>(a_s + kRows);  // [kKeys] element offsets base (page)

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int c = blockIdx.x;
    const int n_row_chunks = (p.T + kRows - 1) / kRows;
    const int h = blockIdx.y / n_row_chunks;
    const int i0 = (blockIdx.y % n_row_chunks) * kRows;
    const int b = blockIdx.z;
    const int nrows = min(kRows, p.T - i0);
    const int g = h / p.G;

    const int32_t L = __ldg(p.seq_lens + b);
    const bool len_ok = seq_len_ok(p, L);
    if (!len_ok && tid == 0) raise_error(p.err, DFLASH_DEVERR_SEQ_LEN);

    Chunk ch;
    ch.kb = 0;
    ch.ke = 0;
    if (len_ok) ch = split_chunk(L, p.T, p.window, p.page_size, p.splits, c);

    // Q rows -> shared (fp32); rows past the block are zero.
    for (int idx = tid; idx < kRows * D; idx += kThreads) {
        const int r = idx / D, d = idx - r * D;
        float v = 0.f;
        if (r < nrows) v = load_elem(p.q, ((int64_t)(b * p.T + i0 + r) * p.Hq + h) * D + d, p.dtype);
        Qs[r * ld + d] = v;
    }
    if (tid < kRows) {
        m_s[tid] = -INFINITY;
        l_s[tid] = 0.f;
    }

    float o[kRows][kColsPerThread];
#pragma unroll
    for (int r = 0; r < kRows; ++r)
#pragma unroll
        for (int k = 0; k < kColsPerThread; ++k) o[r][k] = 0.f;

    // Row ranges of this CTA's queries.
    const int my_r = tid >> 4;      // score mapping: row
    const int my_k = tid & 15;      // score mapping: key in tile
    KeyRange rr = row_range(L, p.T, i0 + my_r, p.causal, p.window);

    for (int kt = ch.kb; kt < ch.ke; kt += kKeys) {
        __syncthreads();  // previous tile fully consumed
        if (tid < kKeys) {
            const int j = kt + tid;
            int32_t base = -1;
            if (j < ch.ke) base = lookup_page(p, b, j);
            pg[tid] = base;
        }
        __syncthreads();
        for (int idx = tid; idx < kKeys * D; idx += kThreads) {
            const int kk = idx / D, d = idx - kk * D;
            const int j = kt + kk;
            float kv = 0.f, vv = 0.f;
            const int32_t page = pg[kk];
            if (page >= 0) {
                const int64_t off = (int64_t)page * p.sp + (int64_t)(j % p.page_size) * p.ss +
                                    (int64_t)g * p.sh + d;
                kv = load_elem(p.k, off, p.dtype);
                vv = load_elem(p.v, off, p.dtype);
            }
            Ks[kk * ld + d] = kv;
            Vs[kk * D + d] = vv;
        }
        __syncthreads();

        // Scores: thread (my_r, my_k).
        {
            const int j = kt + my_k;
            float acc = 0.f;
            const float* qr = Qs + my_r * ld;
            const float* kr = Ks + my_k * ld;
            for (int d = 0; d < D; ++d) acc = fmaf(qr[d], kr[d], acc);
            const bool vis = (my_r < nrows) && (j < ch.ke) && (pg[my_k] >= 0) && (j >= rr.lo) &&
                             (j <= rr.hi);
            Ps[my_r * kKeys + my_k] = vis ? acc * p.scale : -INFINITY;
        }
        __syncthreads();

        // Online softmax: warp w owns rows w and w + 8; lanes 0..15 hold the tile's keys.
        for (int r = warp; r < kRows; r += kThreads / 32) {
            const float s = (lane < kKeys) ? Ps[r * kKeys + lane] : -INFINITY;
            float tmax = s;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
            const float m_old = m_s[r];
            const float m_new = fmaxf(m_old, tmax);
            const float pr = (s == -INFINITY) ? 0.f : expf(s - m_new);
            float psum = pr;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
            const float alpha = (m_old == -INFINITY) ? 0.f : expf(m_old - m_new);
            __syncwarp();
            if (lane < kKeys) Ps[r * kKeys + lane] = pr;
            if (lane == 0) {
                l_s[r] = l_s[r] * alpha + psum;
                m_s[r] = m_new;
                a_s[r] = alpha;
            }
        }
        __syncthreads();

        // O = O * alpha + P V.
#pragma unroll
        for (int k = 0; k < kColsPerThread; ++k) {
            const int d = tid + k * kThreads;
            if (d < D) {
                float vcol[kKeys];
#pragma unroll
                for (int kk = 0; kk < kKeys; ++kk) vcol[kk] = Vs[kk * D + d];
#pragma unroll
                for (int r = 0; r < kRows; ++r) {
                    float acc = o[r][k] * a_s[r];
#pragma unroll
                    for (int kk = 0; kk < kKeys; ++kk) acc = fmaf(Ps[r * kKeys + kk], vcol[kk], acc);
                    o[r][k] = acc;
                }
            }
        }
    }
    __syncthreads();

    // Epilogue: normalise; final output when unsplit, else this chunk's partial.
    const int64_t rows_total = (int64_t)p.B * p.T;
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
        if (r >= nrows) break;
        const float l = l_s[r];
        const float inv = (l > 0.f) ? 1.f / l : 0.f;
        const float lse_v = (l > 0.f) ? m_s[r] + logf(l) : -INFINITY;
        const int64_t row = (int64_t)(b * p.T + i0 + r) * p.Hq + h;
#pragma unroll
        for (int k = 0; k < kColsPerThread; ++k) {
            const int d = tid + k * kThreads;
            if (d < D) {
                if (p.splits == 1)
                    store_elem(p.out, row * D + d, o[r][k] * inv, p.dtype);
                else
                    p.part_out[((int64_t)c * rows_total * p.Hq + row) * D + d] = o[r][k] * inv;
            }
        }
        if (tid == 0) {
            if (p.splits == 1) {
                if (p.lse) p.lse[row] = lse_v;
            } else {
                p.part_lse[(int64_t)c * rows_total * p.Hq + row] = lse_v;
            }
        }
    }
}

}  // namespace

cudaError_t launch_simt_attn(const AttnParams& p, cudaStream_t stream)
{
    const size_t smem = SimtSmem::bytes(p.D);
    cudaError_t e = cudaFuncSetAttribute(simt_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    const int n_row_chunks = (p.T + kRows - 1) / kRows;
    dim3 grid(p.splits, p.Hq * n_row_chunks, p.B);
    simt_attn_kernel<<<grid, kThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace dflash
