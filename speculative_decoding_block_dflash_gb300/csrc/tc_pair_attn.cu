// Tensor-core block attention for bf16 on sm_103a, CTA-pair form (tcgen05 cta_group::2).
//
// Same mathematics as tc_attn.cu (transposed S^T = K.Q^T and O^T += V^T.P^T on the tensor
// cores, TMEM accumulators, lazily rescaled running maxima). This
// form serves blocks whose packed rows do not fit one CTA. DFlash2 drafts 15 tokens by default
// (prhub report on vLLM PR #52816 "DFlash2", risks), so a request's block is T = 16 queries
// ("num_query_per_req = 1 + num_speculative_tokens", kenforever1 "dflash-gemma4-31b-notes"),
// and the 8 query heads of a KV head at head_dim 512 make 128 rows. Their fp32 O^T alone is
// 128 x 512 x 4 B = all of one SM's TMEM, so one CTA cannot hold it; two CTAs that each took
// half of the heads would each read every K/V byte.
//
// Here two CTAs of a cluster share one (request, KV head, key chunk) and every K/V byte
// enters exactly one SM. The grid is persistent: one pair per cluster slot the device holds
// at once, each running its share of the (request, KV head, row group, chunk) units back to
// back with its ring, barriers and TMEM carried over (see PairPlan for how units are dealt;
// a pair's consecutive chunks of one group run as one piece, with one epilogue).
// A "pair tile" is 256 keys. The even CTA issues 2-SM MMAs:
//   S^T [256 keys x 128 rows]  = K [256 x D] . Q^T          A = K: each CTA streams its own
//                                                            128 keys; B = Q^T: each CTA holds
//                                                            its 64 rows of Q
//   O^T [256 dims x 128 rows] += V^T [256 x 256 keys] . P^T  per 256-dim output chunk: each CTA
//                                                            streams V of all 256 keys for its
//                                                            128 dims; B = P^T: each CTA holds
//                                                            the P of its 64 rows
// so CTA r's TMEM holds two S^T buffers of its 128 keys for all rows (S of tile j+1 is computed
// while the softmax of tile j runs) and O^T of its 128 dims of every chunk for all rows:
// 2*128 + (D/256)*128 = 512 columns at D = 512. The row sums l do not fit TMEM as well, so
// the softmax forms them on the CUDA cores from the same bf16-rounded P the MMA reads: per
// tile and 16 columns, a transposing shuffle reduction over the warp's 32 keys, kept in four
// registers per lane; the warps' and the two CTAs' partial sums are added once at the end.
//
// Per pair tile each CTA's softmax (thread = key lane) turns its 128 keys x 128 rows into P.
// The row maxima must agree across the pair: each CTA sends its 128 column maxima to the
// other with asynchronous stores that count their bytes on the receiver's mbarrier, and both
// take the same lazy update. Each CTA writes the P of rows 0-63 into the even CTA's P^T
// buffer and of rows 64-127 into the odd CTA's (one half local, one half remote). P^T has two
// buffers, so the softmax of tile j does not wait for PV(j-1): a single buffer left 7 ring
// stages instead of 5, but each tile's V stages then sat in the ring through the next
// softmax, and two buffers measured faster.
//
// Roles (384 threads): warps 0-7 softmax (warps w and w+4 share TMEM lanes 32(w%4).., and take
// the rows 0-63 and 64-127), then the epilogue; warps 8-10 TMA producers (whole 16 KB ring
// stages dealt round-robin); warp 11 the MMA issuer in the even CTA. Every role's loops are
// rolled: fully unrolled stage loops made the kernel 230 KB of code, and its steady state then
// stalled on instruction fetch (an SM instruction cache hit rate near 47 %). Both CTAs fill
// their rings in the same order K(0) K(1) V(0) K(2) V(1) ... so a stage sits at the same
// offset in both, as the pair MMA needs, and both CTAs' copies of a stage count their bytes on
// one barrier in the even CTA (the 2-CTA form of the tensor copy), which alone waits on it.
//
// After a piece's last tile the softmax warps exchange the row sums with the peer, write the
// lse, and read O^T out to the output or the split partials; the next unit's copies and S
// MMAs run meanwhile, and its first PV waits for the read-out (it overwrites O^T).
//
// Every wait is bounded (p.wait_ns); on expiry the kernel records DFLASH_DEVERR_TIMEOUT,
// drains its own copies and MMAs, and both CTAs still meet at the final cluster barrier
// before TMEM is freed, so neither exits while the other may still touch its memory.
#include <cuda.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "dflash_device.cuh"
#include "tc_ptx.cuh"

namespace dflash {
namespace {

using namespace ptx;

constexpr int kThreads = 384;
constexpr int kSoftmaxThreads = 256;
constexpr int kProducerWarp = 8;
constexpr int kNumProducers = 3;
constexpr int kMmaWarp = 11;
constexpr int kPBufs = 2;       // P^T buffers: softmax j writes while PV(j-1) still reads
constexpr int kPairKeys = 256;  // keys per pair tile
constexpr int kOwnKeys = 128;   // keys of a pair tile whose K this CTA streams
constexpr int kHalf = 64;       // Q / P rows held per CTA
constexpr int kN = 128;         // columns (packed rows) of S^T and O^T
constexpr int kStageBytes = 16384;
constexpr int kMaxPids = 128;
constexpr unsigned long long kCopyGraceNs = 200000ull;  // after an abort: time for copies in flight to land
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThresh = 8.0f;

struct PairExtra {
    int32_t Gc;     // query heads per pair
    int32_t n_rg;   // row groups per KV head (G / Gc)
    int32_t Tb;     // block positions per CTA (ceil(T / 2)); CTA r holds positions [r*Tb, r*Tb + Tb)
    int32_t units;  // (request, KV head, row group, chunk) units: splits * Hkv * n_rg * B
};

// Unit u of the work is chunk u mod splits of row-group slot (u / splits) mod (Hkv n_rg) of
// request u / (splits Hkv n_rg); the units of one (request, row group) form group u / splits.
// What a pair streams at a time, called a unit in the roles' loops below, is a run of n_run
// consecutive units of one group (usually one): its chunks' keys as one range, with one
// epilogue and the partial slot of its first chunk.
struct PairUnit {
    int32_t b, g, c_split, n_run, h0;
    int32_t L;
    bool len_ok;
    Chunk ch;
    int32_t t0, ntiles, chunk_pages, first_page;
};

// How units are dealt to the P pairs of the persistent grid. With U = qP + r units and r > 0,
// dealing them round-robin leaves P - r pairs idle for the last round. With split chunks
// (splits > 1) the chunks are instead sized by who runs them: r "small" pairs take q + 1 units
// each and P - r "large" pairs q units, and within every group the chunks of large pairs get
// q + 1 tiles for every q of the small pairs' chunks, so every pair streams about U/P units of
// keys. The large pairs' (P - r) q chunks are spread evenly over the groups, as the first
// chunks of each group. (Uniform chunks on long_draft's 512 units over 76 pairs left 20 pairs
// idle for one unit of the seven.) Either way a pair's consecutive items that are consecutive
// chunks of one group form a run, which the pair streams as one piece with one epilogue: its
// partial goes to the slot of the run's first chunk, and the other slots get an lse of -inf,
// which the split combine skips.
struct PairPlan {
    int32_t npairs, q, r, groups, large;
    bool balanced;
};

__device__ __forceinline__ PairPlan pair_plan(const AttnParams& p, const PairExtra& x)
{
    PairPlan pp;
    pp.npairs = (int32_t)(gridDim.x >> 1);
    pp.q = x.units / pp.npairs;
    pp.r = x.units % pp.npairs;
    pp.groups = x.units / p.splits;
    pp.balanced = p.splits > 1 && pp.r != 0 && pp.q >= 1;
    pp.large = (pp.npairs - pp.r) * pp.q;
    return pp;
}

// chunks of group gr dealt to large pairs (the group's first ones)
__device__ __forceinline__ int32_t pair_large_in_group(const PairPlan& pp, int32_t gr)
{
    return (int32_t)(((int64_t)(gr + 1) * pp.large) / pp.groups - ((int64_t)gr * pp.large) / pp.groups);
}

// The k-th unit of pair `pr`, or -1 past its last.
__device__ __forceinline__ int32_t pair_item(const AttnParams& p, const PairExtra& x, const PairPlan& pp, int32_t pr,
                                             int32_t k)
{
    if (!pp.balanced) {
        const int64_t u = (int64_t)pr + (int64_t)k * pp.npairs;
        return u < x.units ? (int32_t)u : -1;
    }
    const int32_t S = p.splits;
    if (pr >= pp.r) {
        // large pair: large chunk i = (pr - r) q + k, in group order; group gr holds large
        // chunks [floor(gr L / G), floor((gr + 1) L / G))
        if (k >= pp.q) return -1;
        const int64_t i = (int64_t)(pr - pp.r) * pp.q + k;
        const int32_t gr = (int32_t)(((i + 1) * pp.groups + pp.large - 1) / pp.large) - 1;
        const int32_t c = (int32_t)(i - ((int64_t)gr * pp.large) / pp.groups);
        return c + S * gr;
    }
    // small pair: small chunk i = pr (q + 1) + k; group gr holds small chunks
    // [gr S - floor(gr L / G), ...): the last group whose start is <= i, by bisection
    if (k > pp.q) return -1;
    const int64_t i = (int64_t)pr * (pp.q + 1) + k;
    int32_t lo = 0, hi = pp.groups - 1;
    while (lo < hi) {
        const int32_t mid = (lo + hi + 1) >> 1;
        const int64_t start = (int64_t)mid * S - ((int64_t)mid * pp.large) / pp.groups;
        if (start <= i)
            lo = mid;
        else
            hi = mid - 1;
    }
    const int64_t start = (int64_t)lo * S - ((int64_t)lo * pp.large) / pp.groups;
    const int32_t c = pair_large_in_group(pp, lo) + (int32_t)(i - start);
    return c + S * lo;
}

// The run of the pair's items that starts at its k-th: the first unit, or -1 past the last,
// and in n the number of items that continue it with the next chunks of the same group. A run
// is one piece of work: its chunks' keys are one contiguous range, streamed and accumulated
// in TMEM as one, with one epilogue.
__device__ __forceinline__ int32_t pair_run(const AttnParams& p, const PairExtra& x, const PairPlan& pp, int32_t pr,
                                            int32_t k, int32_t& n)
{
    n = 0;
    const int32_t u = pair_item(p, x, pp, pr, k);
    if (u < 0) return -1;
    n = 1;
    while (true) {
        const int32_t v = pair_item(p, x, pp, pr, k + n);
        if (v != u + n || v / p.splits != u / p.splits) break;
        ++n;
    }
    return u;
}

// Unit u with the n - 1 chunks after it in its group (a run): the keys of chunks
// [u mod splits, u mod splits + n) of the group, the partial slot of the first.
__device__ __forceinline__ PairUnit pair_unit(const AttnParams& p, const PairExtra& x, const PairPlan& pp, int u,
                                              int n)
{
    PairUnit U;
    const int ys = p.Hkv * x.n_rg;
    U.c_split = u % p.splits;
    U.n_run = n;
    const int y = (u / p.splits) % ys;
    U.b = u / (p.splits * ys);
    U.g = y / x.n_rg;
    const int rg = y % x.n_rg;
    U.h0 = U.g * p.G + rg * x.Gc;
    U.L = __ldg(p.seq_lens + U.b);
    U.len_ok = seq_len_ok(p, U.L);
    U.ch.kb = 0;
    U.ch.ke = 0;
    if (U.len_ok) {
        if (!pp.balanced) {
            U.ch = split_chunk(U.L, p.T, p.window, p.page_size, p.splits, U.c_split);
            U.ch.ke = split_chunk(U.L, p.T, p.window, p.page_size, p.splits, U.c_split + n - 1).ke;
            if (U.ch.ke < U.ch.kb) U.ch.ke = U.ch.kb;
        } else {
            // the request's union key range [lo, L), cut at whole pair tiles from the page
            // boundary below lo, in proportion to the chunks' weights (q + 1 for the group's
            // first `nl` chunks, which large pairs run, and q for the rest)
            int32_t lo = 0;
            if (p.window > 0) {
                lo = U.L - p.T - p.window + 1;
                if (lo < 0) lo = 0;
            }
            const int32_t base = (lo / p.page_size) * p.page_size;
            const int64_t ntot = (U.L - base + kPairKeys - 1) / kPairKeys;
            const int32_t nl = pair_large_in_group(pp, u / p.splits);
            const int64_t wq1 = pp.q + 1, wq = pp.q;
            const int64_t wt = nl * wq1 + (int64_t)(p.splits - nl) * wq;
            auto cum = [&](int32_t c) -> int64_t {
                return c <= nl ? c * wq1 : nl * wq1 + (int64_t)(c - nl) * wq;
            };
            const int64_t t_b = (2 * ntot * cum(U.c_split) + wt) / (2 * wt);
            const int64_t t_e = (2 * ntot * cum(U.c_split + n) + wt) / (2 * wt);
            int64_t kb = base + t_b * kPairKeys, ke = base + t_e * kPairKeys;
            if (kb < lo) kb = lo;
            if (ke > U.L) ke = U.L;
            if (kb > U.L) kb = U.L;
            U.ch.kb = (int32_t)kb;
            U.ch.ke = (int32_t)ke;
        }
    }
    U.t0 = (U.ch.kb / p.page_size) * p.page_size;
    U.ntiles = (U.ch.kb < U.ch.ke) ? (U.ch.ke - U.t0 + kPairKeys - 1) / kPairKeys : 0;
    U.chunk_pages = U.ntiles * (kPairKeys / p.page_size);
    U.first_page = U.t0 / p.page_size;
    return U;
}

__host__ __device__ constexpr int pair_pow2ceil(int x)
{
    int p = 32;
    while (p < x) p <<= 1;
    return p;
}

template <int D>
struct PairLayout {
    static constexpr int KC = D / 64;       // K stages per pair tile (64 dims each, own 128 keys)
    static constexpr int VC2 = D / 256;     // output chunks of 256 dims (128 per CTA)
    static constexpr int kQBytes = KC * kHalf * 128;
    static constexpr int kPQuarter = kHalf * 128;           // P^T of 64 keys x 64 rows
    static constexpr int kPBuf = 4 * kPQuarter;             // one pair tile
    static constexpr int kQOff = 0;
    static constexpr int kPOff = kQOff + kQBytes;           // [kPBufs][4 quarters][4 atoms][2 KB]
    static constexpr int kRingOff = kPOff + kPBufs * kPBuf;
    static constexpr int kSmallBytes = 12288;               // barriers, tables
    static constexpr int kStagesFit = (227 * 1024 - 1024 - kRingOff - kSmallBytes) / kStageBytes;
    static constexpr int kStages = kStagesFit > 10 ? 10 : kStagesFit;
    static constexpr int kBarOff = kRingOff + kStages * kStageBytes;
    // barriers: full[S] empty[S] s_full[2] p_full p_free[kPBufs] nf_full[2] px_full[2] lx_full[2] drain
    static constexpr int kNumBars = 2 * kStages + 10 + kPBufs;
    static constexpr int kMiscOff = (kBarOff + kNumBars * 8 + 15) / 16 * 16;  // tmem base, abort flag
    static constexpr int kMOff = kMiscOff + 16;             // float m_s[128]
    static constexpr int kAOff = kMOff + kN * 4;            // float a_s[128] (1/l at the end)
    static constexpr int kRedOff = kAOff + kN * 4;          // float red[8 warps][64]: column maxima
    static constexpr int kSumOff = kRedOff + 8 * 64 * 4;    // float red2[8 warps][64]: column sums of P
    static constexpr int kLaccOff = kSumOff + 8 * 64 * 4;   // float l_acc[128]: this CTA's keys' row sums
    static constexpr int kPxOff = kLaccOff + kN * 4;        // float px[2][128]: the peer's maxima
    static constexpr int kNfOff = kPxOff + 2 * kN * 4;      // float nflag[2] (16 B): the peer's flags
    static constexpr int kLxOff = kNfOff + 16;              // float lx[2][128]: the peer's row sums
    static constexpr int kLoOff = kLxOff + 2 * kN * 4;      // int lo_s[128]
    static constexpr int kHiOff = kLoOff + kN * 4;          // int hi_s[128]
    static constexpr int kRowOff = kHiOff + kN * 4;         // int64 orow_s[128]
    static constexpr int kPidOff = kRowOff + kN * 8;        // int pid_s[4][kMaxPids]
    static constexpr int kTotal = kPidOff + kNumProducers * kMaxPids * 4;
    static constexpr int kAlloc = kTotal + 1024;
    static constexpr int kTmemUsed = 2 * kN + VC2 * kN;     // S^T x 2, O^T chunks
    static constexpr int kTmemCols = pair_pow2ceil(kTmemUsed);
    // each producer warp fills every kNumProducers-th stage; with fewer slots than producers
    // a warp could pass a slot two phases ahead (the parity wait cannot tell them apart)
    static_assert(kStages >= kNumProducers, "ring too shallow for the producer warps");
    static_assert(kTotal - kBarOff <= kSmallBytes, "small tables");
    static_assert(kTotal + 1024 <= 227 * 1024, "shared memory budget");
    static_assert(kTmemUsed <= 512, "TMEM budget");
};

// The k-th unit (0 <= k < 2n) of the ring sequence K(0) K(1) V(0) K(2) V(1) ... V(n-1).
__device__ __forceinline__ void pair_ring_unit(int k, int n, bool& is_k, int& tile)
{
    if (k == 0) {
        is_k = true;
        tile = 0;
    } else if (k & 1) {
        const int m = (k + 1) >> 1;
        is_k = m < n;
        tile = is_k ? m : n - 1;
    } else {
        is_k = false;
        tile = (k - 2) >> 1;
    }
}

// Column reductions over a warp: v holds 16 consecutive columns of this lane's key. Each step
// swaps half of the live columns with the partner lane and keeps the combination of the half
// it owns; after four steps lane l holds its 16-lane half's result for column l mod 16, and one
// exchange across the halves completes it (16 shuffles for 16 columns).
__device__ __forceinline__ float pair_transpose_max16(float (&v)[16], int lane)
{
#pragma unroll
    for (int off = 8; off >= 1; off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < off; ++i) {
            const float send = upper ? v[i] : v[i + off];
            const float keep = upper ? v[i + off] : v[i];
            v[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, off));
        }
    }
    return fmaxf(v[0], __shfl_xor_sync(0xffffffffu, v[0], 16));
}

__device__ __forceinline__ float pair_transpose_sum16(float (&v)[16], int lane)
{
#pragma unroll
    for (int off = 8; off >= 1; off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < off; ++i) {
            const float send = upper ? v[i] : v[i + off];
            const float keep = upper ? v[i + off] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
    return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 16);
}

// Named barrier 1 over the 256 softmax threads (warps 0-7), with an OR of a predicate.
__device__ __forceinline__ bool bar_or_256(bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, 1, 256, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(r)
        : "r"((uint32_t)pred)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void bar_sync_256() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    tc_pair_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const AttnParams p, const PairExtra x)
{
    using Lay = PairLayout<D>;
    constexpr int S = Lay::kStages;
    constexpr int KC = Lay::KC;
    constexpr int VC2 = Lay::VC2;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* q_s = smem + Lay::kQOff;
    uint8_t* ring = smem + Lay::kRingOff;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kBarOff);
    uint64_t* full = bars;            // [S] even CTA: both CTAs' copies of the stage have landed
    uint64_t* empty = bars + S;       // [S] the pair MMAs reading the slot are done (both CTAs)
    uint64_t* s_full = bars + 2 * S;  // [2] S^T of tile j is in TMEM buffer j mod 2 (both CTAs)
    uint64_t* p_full = s_full + 2;    // even CTA: both CTAs wrote P (one arrival each)
    uint64_t* p_free = s_full + 3;    // [kPBufs] PV of tile j done: P^T buffer j mod kPBufs is free
    uint64_t* nf_full = p_free + kPBufs;  // [2] the peer's "raise the maxima" flag of the tile (4 bytes)
    uint64_t* px_full = nf_full + 2;  // [2] the peer's 128 column maxima have landed (512 bytes)
    uint64_t* lx_full = nf_full + 4;  // [2] the peer's 128 row sums of a unit have landed (512 bytes)
    uint64_t* drain = nf_full + 6;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lay::kMiscOff + 4);
    float* m_s = reinterpret_cast<float*>(smem + Lay::kMOff);
    float* a_s = reinterpret_cast<float*>(smem + Lay::kAOff);
    float* red = reinterpret_cast<float*>(smem + Lay::kRedOff);
    float* red2 = reinterpret_cast<float*>(smem + Lay::kSumOff);
    float* l_acc = reinterpret_cast<float*>(smem + Lay::kLaccOff);
    float* px = reinterpret_cast<float*>(smem + Lay::kPxOff);
    float* lx = reinterpret_cast<float*>(smem + Lay::kLxOff);
    float* nflag = reinterpret_cast<float*>(smem + Lay::kNfOff);
    int32_t* lo_s = reinterpret_cast<int32_t*>(smem + Lay::kLoOff);
    int32_t* hi_s = reinterpret_cast<int32_t*>(smem + Lay::kHiOff);
    int64_t* orow_s = reinterpret_cast<int64_t*>(smem + Lay::kRowOff);
    int32_t* pid_s = reinterpret_cast<int32_t*>(smem + Lay::kPidOff);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const uint32_t peer = rank ^ 1u;
    const bool leader = (rank == 0);
    const int pair_id = blockIdx.x >> 1;
    const PairPlan pp = pair_plan(p, x);
    const int T = p.T;
    const int Psz = p.page_size;
    const int rows_mine = x.Gc * x.Tb;  // Q rows this CTA loads (of its kHalf)
    const int pages_per_tile = kPairKeys / Psz;

    const int pw = warp - kProducerWarp;
    int32_t* pid_w = pid_s + (pw >= 0 && pw < kNumProducers ? pw : 0) * kMaxPids;
    // page ids of the unit's relative pages [base, base + kMaxPids) -> this producer warp's pid_w;
    // pages past the chunk and invalid ids map to the out-of-bounds coordinate num_pages
    auto load_window = [&](const PairUnit& U, int base) {
        for (int k = lane; k < kMaxPids; k += 32) {
            const int pr = base + k;
            int32_t id = p.num_pages;  // out-of-bounds coordinate: the copy fills zeros
            if (pr < U.chunk_pages && U.t0 + pr * Psz < U.ch.ke) {
                const int32_t v = __ldg(p.page_table + (int64_t)U.b * p.max_pages + U.first_page + pr);
                if (v >= 0 && v < p.num_pages)
                    id = v;
                else
                    raise_error(p.err, DFLASH_DEVERR_PAGE_ID);
            }
            pid_w[k] = id;
        }
        __syncwarp();
    };

    // ---------------------------------------------------------------- set-up
    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(full + i, 1);
            mbar_init(empty + i, 1);
        }
        mbar_init(s_full, 1);
        mbar_init(s_full + 1, 1);
        mbar_init(p_full, 2);
        for (int i = 0; i < kPBufs; ++i) mbar_init(p_free + i, 1);
        mbar_init(nf_full, 1);
        mbar_init(nf_full + 1, 1);
        mbar_init(px_full, 1);
        mbar_init(px_full + 1, 1);
        mbar_init(lx_full, 1);
        mbar_init(lx_full + 1, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        // the exchange barriers of tiles 0 and 1, and of the row sums of units 0 and 1, expect
        // the peer's bytes
        mbar_expect_tx(nf_full, 4);
        mbar_expect_tx(nf_full + 1, 4);
        mbar_expect_tx(px_full, kN * 4);
        mbar_expect_tx(px_full + 1, kN * 4);
        mbar_expect_tx(lx_full, kN * 4);
        mbar_expect_tx(lx_full + 1, kN * 4);
    }
    if (warp == kMmaWarp) {
        tmem_alloc2(tmem_slot, Lay::kTmemCols);
        tmem_relinquish2();
    } else if (tid >= kN && tid < kSoftmaxThreads) {
        // zero this CTA's Q rows [rows_mine, kHalf) of every 64-dim chunk, once: every unit's
        // copy writes the same rows [0, rows_mine)
        const int pad = kHalf - rows_mine;
        for (int idx = tid - kN; idx < KC * pad * 8; idx += kSoftmaxThreads - kN) {
            const int kc = idx / (pad * 8);
            const int rem = idx - kc * pad * 8;
            *reinterpret_cast<uint4*>(q_s + kc * kHalf * 128 + (rows_mine + rem / 8) * 128 + (rem % 8) * 16) =
                make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // the peer's barriers are initialised before any remote arrival
    tc_fence_after();
    cudaTriggerProgrammaticLaunchCompletion();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tmem_s = tmem;                 // S^T buffers: columns [0, 128) and [128, 256)
    const uint32_t tmem_o = tmem + 2 * kN;        // O^T chunk c: columns [256 + 128c, ..)
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;

    auto load16 = [&](uint32_t taddr, uint32_t (&r16)[16]) {
        tmem_ld16(taddr, r16);
        tmem_ld_wait();
        reg_fence16(r16);
    };
    // cluster address of a shared-memory location at the same offset in CTA `r`
    auto in_cta = [&](const void* ptr, uint32_t r) -> uint32_t { return mapa_shared(smem_u32(ptr), r); };

    if (warp >= kProducerWarp && warp < kProducerWarp + kNumProducers) {
        // ------------------------------------------------------------ TMA producers
        // The ring runs on across units: stage seq of the whole sequence goes to slot seq mod S,
        // and the first stage of each unit also carries the unit's Q.
        const uint32_t full0 = in_cta(full, 0);
        bool ok = true;
        uint32_t issued_parity[S];
#pragma unroll
        for (int s = 0; s < S; ++s) issued_parity[s] = 2;  // 2 = nothing outstanding
        const int box = Psz * 128;  // bytes of one page x 64 dims
        // K/V pages are read once: they leave L2 first, ahead of the split partials, which the
        // combine reads back after the kernel
        const uint64_t kv_policy = l2_policy_evict_first();
        int seq = 0;
        int last_k = -1;            // sequence number of the last K stage so far (reads Q)
#pragma unroll 1
        for (int k_item = 0, n_run = 0; ok; k_item += n_run) {
            const int unit = pair_run(p, x, pp, pair_id, k_item, n_run);
            if (unit < 0) break;
            const PairUnit U = pair_unit(p, x, pp, unit, n_run);
            if (U.ntiles == 0) continue;
            int wbase = 0;
            load_window(U, 0);
            const int seq0 = seq;
#pragma unroll 1
            for (int k = 0; k < 2 * U.ntiles && ok; ++k) {
                bool is_k;
                int tile;
                pair_ring_unit(k, U.ntiles, is_k, tile);
                const int n_st = is_k ? KC : 4 * VC2;
#pragma unroll 1
                for (int sq = 0; sq < n_st && ok; ++sq, ++seq) {
                    const int prev_k = last_k;
                    if (is_k) last_k = seq;
                    if (seq % kNumProducers != pw) continue;
                    // relative pages this stage reads: K: own 128 keys; V: quarter of 64 keys
                    const int rel0 = tile * pages_per_tile +
                                     (is_k ? (int)rank * (kOwnKeys / Psz) : (sq / VC2) * (64 / Psz));
                    const int npg = (is_k ? kOwnKeys : 64) / Psz;
                    if (rel0 < wbase || rel0 + npg > wbase + kMaxPids) {
                        wbase = rel0;
                        load_window(U, wbase);
                    }
                    const int slot = seq % S;
                    const uint32_t ph = (uint32_t)((seq / S) & 1);
                    // a polling wait with a short sleep between polls: producers spinning flat out
                    // beside the softmax warps slow it down, and a suspending wait wakes late
                    if (lane == 0) ok = backoff_wait(empty + slot, ph ^ 1u, abort_flag, p.err, p.wait_ns);
                    const bool with_q = (seq == seq0);
                    // The unit's Q replaces the previous unit's: the pair MMAs of that unit's last
                    // K stage must be done. The slot wait above covers stages up to seq - S.
                    if (lane == 0 && ok && with_q && prev_k >= 0 && prev_k > seq - S)
                        ok = backoff_wait(empty + prev_k % S, (uint32_t)((prev_k / S) & 1), abort_flag, p.err,
                                          p.wait_ns);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) break;
                    if (lane == 0) {
                        uint8_t* dst = ring + slot * kStageBytes;
                        // the even CTA expects both CTAs' bytes of the stage on its barrier
                        const uint32_t qbytes = with_q ? (uint32_t)(x.Gc * x.Tb * 128 * KC) : 0u;
                        if (leader) mbar_expect_tx(full + slot, 2u * (kStageBytes + qbytes));
                        const uint32_t fb = full0 + (uint32_t)(slot * 8);
                        if (with_q)
                            for (int kc = 0; kc < KC; ++kc)
                                tma_load_3d_pair(q_s + kc * kHalf * 128, &tm_q, fb, kc * 64, U.h0,
                                                 U.b * T + (int)rank * x.Tb);
                        // the stage's page ids go to registers before its copies are issued (each
                        // copy instruction is also a compiler memory barrier)
                        int32_t ids[8];
#pragma unroll
                        for (int pg = 0; pg < 8; ++pg) ids[pg] = pg < npg ? pid_w[rel0 + pg - wbase] : 0;
                        if (is_k) {
#pragma unroll
                            for (int pg = 0; pg < 8; ++pg)
                                if (pg < npg)
                                    tma_load_4d_pair_hint(dst + pg * box, &tm_k, fb, sq * 64, U.g, 0, ids[pg], kv_policy);
                        } else {
                            const int c = sq % VC2;
                            const int d0 = c * 256 + (int)rank * 128;
#pragma unroll
                            for (int pg = 0; pg < 4; ++pg)
                                if (pg < npg)
#pragma unroll
                                    for (int m = 0; m < 2; ++m)
                                        tma_load_4d_pair_hint(dst + m * 8192 + pg * box, &tm_v, fb, d0 + m * 64, U.g,
                                                              0, ids[pg], kv_policy);
                        }
                        issued_parity[slot] = ph;
                    }
                    __syncwarp();
                }
            }
        }
        if (lane == 0 && !ok) {
            // Copies of ours may still be landing. The even CTA waits for the stages it armed;
            // both CTAs then give copies in flight a grace period (a copy lands within
            // microseconds while the memory system works) before this CTA may leave.
            if (leader) {
#pragma unroll 1
                for (int s = 0; s < S; ++s) {
                    if (issued_parity[s] > 1) continue;
                    const unsigned long long t_start = globaltimer();
                    while (!mbar_try_wait(full + s, issued_parity[s]) && globaltimer() - t_start < p.wait_ns) {
                    }
                }
            }
            const unsigned long long t_start = globaltimer();
            while (globaltimer() - t_start < kCopyGraceNs) {
            }
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer (even CTA)
        // Tiles are numbered across the pair's units (gj): the S^T buffer, the P^T buffer and
        // the phases of s_full, p_full and p_free follow gj; the accumulate flags follow the
        // tile's place in its unit.
        if (leader) {
            constexpr uint32_t idesc_s = make_idesc(256, kN, 0, 0);  // S^T  = K . Q^T
            constexpr uint32_t idesc_o = make_idesc(256, kN, 1, 1);  // O^T += V^T . P^T
            const uint32_t q_addr = smem_u32(q_s);
            const uint32_t p_addr = smem_u32(smem + Lay::kPOff);
            const uint32_t ring_addr = smem_u32(ring);
            bool ok = true;
            int seq = 0;
            int G = 0;  // tiles of the earlier units
            auto wait_lane0 = [&](uint64_t* bar, uint32_t par) -> bool {
                bool got = true;
                if (lane == 0) got = ring_wait_cluster(bar, par, abort_flag, p.err, p.wait_ns);
                return __shfl_sync(0xffffffffu, got, 0);
            };
            // both CTAs' copies of the next stage have landed (one barrier counts both)
            auto next_stage = [&](uint32_t& addr, int& slot) -> bool {
                slot = seq % S;
                const uint32_t ph = (uint32_t)((seq / S) & 1);
                const bool got = wait_lane0(full + slot, ph);
                addr = ring_addr + slot * kStageBytes;
                return got;
            };
            auto release = [&](int slot) {
                if (lane == 0) tc_commit2_both(empty + slot);
                __syncwarp();
                ++seq;
            };
#pragma unroll 1
            for (int k_item = 0, n_run = 0; ok; k_item += n_run) {
                const int unit = pair_run(p, x, pp, pair_id, k_item, n_run);
                if (unit < 0) break;
                const PairUnit U = pair_unit(p, x, pp, unit, n_run);
                if (U.ntiles == 0) continue;
                // V rows past seq_len in the sequence's last, partial page are zeroed before PV in
                // both CTAs' copies of the stage (the zero probabilities there must not meet
                // non-finite garbage); the peer's copy through distributed shared memory
                auto zero_tail = [&](int tile, int q, uint32_t st_off) {
                    const int key0 = U.t0 + tile * kPairKeys + q * 64;
                    const int zlo = U.L - key0;
                    if (U.L % Psz != 0 && zlo > 0 && zlo < 64 && U.ch.ke == U.L) {
                        const int zhi = min(64, ((U.L + Psz - 1) / Psz) * Psz - key0);
                        const int rows = zhi - zlo;
                        const uint32_t peer_st = in_cta(smem + st_off, peer);
                        for (int idx = lane; idx < rows * 16; idx += 32) {
                            const int m = idx / (rows * 8);
                            const int rem = idx - m * rows * 8;
                            const uint32_t off = (uint32_t)(m * 8192 + (zlo + rem / 8) * 128 + (rem % 8) * 16);
                            *reinterpret_cast<uint4*>(smem + st_off + off) = make_uint4(0, 0, 0, 0);
                            st_cluster_v4(peer_st + off, make_uint4(0, 0, 0, 0));
                        }
                        fence_proxy_async_cluster();
                    }
                    __syncwarp();
                };
#pragma unroll 1
                for (int k = 0; k < 2 * U.ntiles && ok; ++k) {
                    bool is_k;
                    int j;
                    pair_ring_unit(k, U.ntiles, is_k, j);
                    const int gj = G + j;
                    if (is_k) {
                        // S^T(gj) into buffer gj mod 2: its previous tile gj - 2 has been read by
                        // both softmaxes (their P(gj-2) was waited for by the V(gj-2) unit, which
                        // comes earlier in the ring order, in this unit or the one before)
                        const uint32_t sb = tmem_s + (uint32_t)(gj & 1) * kN;
#pragma unroll 1
                        for (int kc = 0; kc < KC && ok; ++kc) {
                            uint32_t st;
                            int slot;
                            ok = next_stage(st, slot);
                            if (!ok) break;
                            tc_fence_after();
                            if (lane == 0) {
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk)
                                    tc_mma2(sb, sw128_desc(st + kk * 32, 16, 1024),
                                            sw128_desc(q_addr + kc * kHalf * 128 + kk * 32, 16, 1024), idesc_s,
                                            (kc > 0 || kk > 0) ? 1u : 0u);
                            }
                            release(slot);
                        }
                        if (!ok) break;
                        if (lane == 0) tc_commit2_both(s_full + (gj & 1));
                        __syncwarp();
                        continue;
                    }
                    ok = wait_lane0(p_full, (uint32_t)(gj & 1));
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t pb_addr = p_addr + (uint32_t)((gj % kPBufs) * Lay::kPBuf);
#pragma unroll 1
                    for (int q = 0; q < 4 && ok; ++q) {
#pragma unroll 1
                        for (int c = 0; c < VC2 && ok; ++c) {
                            uint32_t st;
                            int slot;
                            ok = next_stage(st, slot);
                            if (!ok) break;
                            zero_tail(j, q, st - smem_u32(smem));
                            tc_fence_after();
                            if (lane == 0) {
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk)
                                    tc_mma2(tmem_o + c * kN, sw128_desc(st + kk * 2048, 8192, 1024),
                                            sw32_desc(pb_addr + q * Lay::kPQuarter + kk * 512, 2048, 256), idesc_o,
                                            (j > 0 || q > 0 || kk > 0) ? 1u : 0u);
                            }
                            release(slot);
                        }
                    }
                    if (!ok) break;
                    if (lane == 0) tc_commit2_both(p_free + gj % kPBufs);
                    __syncwarp();
                }
                G += U.ntiles;
            }
            // drain our MMAs before either CTA frees TMEM or leaves (they read both CTAs' memory)
            if (lane == 0) {
                tc_commit2_local(drain);
                const unsigned long long t_start = globaltimer();
                while (!mbar_try_wait(drain, 0) && globaltimer() - t_start < p.wait_ns) {
                }
            }
            __syncwarp();
        }
        // (the odd CTA's MMA warp has no role: the even CTA issues the pair MMAs)
    } else {
        // ------------------------------------------------------------ softmax (warps 0-7)
        const float sl2 = p.scale * kLog2e;
        const bool plain = (p.causal == 0 && p.window == 0);
        const int kl = tid & 127;         // key lane of this CTA's 128 keys (TMEM lane)
        const int chh = tid >> 7;         // rows [64 chh, 64 chh + 64): the P^T buffer of CTA chh
        const int col0 = chh * kHalf;
        const int pk = (int)rank * kOwnKeys + kl;  // key index within the pair tile
        // P^T (MN-major, 32-byte swizzle): quarter of 64 keys, 16-row atoms of 2 KB, 8-key
        // groups of 256 B, 32 B per key with the 16-byte halves swapped for keys 4-7 of a group
        const int kig = pk & 7;
        const uint32_t prow_off = (uint32_t)(Lay::kPOff + (pk >> 6) * Lay::kPQuarter + ((pk & 63) >> 3) * 256 +
                                             kig * 32);
        const uint32_t pswz0 = (uint32_t)((0 ^ (kig >> 2)) << 4);
        const uint32_t pswz1 = (uint32_t)((1 ^ (kig >> 2)) << 4);
        const bool p_local = (chh == (int)rank);
        const uint32_t prow0 = (p_local ? smem_u32(smem) : mapa_shared(smem_u32(smem), (uint32_t)chh)) + prow_off;
        const uint32_t p_full_bar = in_cta(p_full, 0);
        bool ok = true;
        int nx = 0;     // maxima exchanges so far (they happen only on tiles that raise a row max)
        int G = 0;      // tiles of the earlier units: tile j of a unit is tile G + j of the pair
        int un = 0;     // units done (the row-sum exchange buffer of unit un is un mod 2)
        const int lcol = col0 + (lane & 15);
        auto group_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
            bool got = true;
            if (tid == 0) got = ring_wait_cluster(bar, parity, abort_flag, p.err, p.wait_ns);
            return !bar_or_256(!got);
        };
        // PV of tile t done (its P^T buffer is free and O^T holds every tile up to t)
        auto wait_pv = [&](int t) -> bool {
            return group_wait(p_free + t % kPBufs, (uint32_t)((t / kPBufs) & 1));
        };
#pragma unroll 1
        for (int k_item = 0, n_run = 0; ok; k_item += n_run) {
            const int unit = pair_run(p, x, pp, pair_id, k_item, n_run);
            if (unit < 0) break;
            const PairUnit U = pair_unit(p, x, pp, unit, n_run);
            if (tid == 0 && leader && !U.len_ok) raise_error(p.err, DFLASH_DEVERR_SEQ_LEN);
            // the unit's rows: column c of S^T / O^T is row c mod 64 of CTA c / 64's Q
            if (tid < kN) {
                const int hc = tid / kHalf, lr = tid % kHalf;
                const int i = hc * x.Tb + lr / x.Gc, hh = lr % x.Gc;
                int32_t lo = -(1 << 30), hi = (1 << 30);
                int64_t orow = -1;
                if (lr < rows_mine && i < T) {
                    const KeyRange kr = row_range(U.L, T, i, p.causal, p.window);
                    lo = kr.lo;
                    hi = kr.hi;
                    orow = (int64_t)(U.b * T + i) * p.Hq + (U.h0 + hh);
                }
                lo_s[tid] = lo;
                hi_s[tid] = hi;
                orow_s[tid] = orow;
                m_s[tid] = -INFINITY;
                a_s[tid] = 1.f;
                l_acc[tid] = 0.f;
            }
            bar_sync_256();
            // a key inside every row's range [max lo, min hi] needs no test per row
            int lo_all = -(1 << 30), hi_all = (1 << 30);
            if (!plain) {
                for (int r = 0; r < kN; ++r) {
                    lo_all = max(lo_all, lo_s[r]);
                    hi_all = min(hi_all, hi_s[r]);
                }
            }
            // row sums over this warp's 32 keys and the unit's tiles so far: lane l holds the sum
            // of row col0 + 16q + (l mod 16) in ls[q]
            float ls[4] = {0.f, 0.f, 0.f, 0.f};
            for (int j = 0; j < U.ntiles && ok; ++j) {
                const int gj = G + j;
                if (!group_wait(s_full + (gj & 1), (uint32_t)((gj >> 1) & 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sb = tmem_s + (uint32_t)(gj & 1) * kN + lane_base + (uint32_t)col0;
                const int key = U.t0 + j * kPairKeys + pk;
                const bool kvalid = key >= U.ch.kb && key < U.ch.ke;
                const bool allvis = plain || (key >= lo_all && key <= hi_all);
                auto score = [&](uint32_t raw, int col) -> float {
                    bool vis = kvalid;
                    if (!allvis) vis = vis && key >= lo_s[col] && key <= hi_s[col];
                    return vis ? u2f(raw) * sl2 : -INFINITY;
                };
                // Every column of this key lane visible (all but the chunk's edge keys and the
                // window's or the block's own few): no selects, and the scale folds into one FMA.
                // The running maxima are then finite, since pass 1 raises any -inf one.
                const bool open = kvalid && allvis;
                // pass 1: does any score of this CTA exceed its row's running max by more than the
                // threshold? Both CTAs exchange the answer (one word); only when either says yes
                // do they form and exchange the column maxima, so both take the same update.
                bool nd = false;
#pragma unroll 1
                for (int q = 0; q < 4; ++q) {
                    float mv[16];
                    load_row16(m_s + col0 + q * 16, mv);
                    uint32_t r16[16];
                    load16(sb + q * 16, r16);
                    if (open) {
#pragma unroll
                        for (int u = 0; u < 16; ++u) nd |= fmaf(u2f(r16[u]), sl2, -mv[u]) > kRescaleThresh;
                    } else {
#pragma unroll
                        for (int u = 0; u < 16; ++u) nd |= score(r16[u], col0 + q * 16 + u) > mv[u] + kRescaleThresh;
                    }
                }
                nd = bar_or_256(nd);
                if (tid == 0)
                    st_async_f32(in_cta(nflag + (gj & 1), peer), nd ? 1.f : 0.f, in_cta(nf_full + (gj & 1), peer));
                if (!group_wait(nf_full + (gj & 1), (uint32_t)((gj >> 1) & 1))) {
                    ok = false;
                    break;
                }
                const bool need = nd || nflag[gj & 1] != 0.f;
                // the flag of tile gj has been read: expect the peer's flag of tile gj + 2
                if (tid == 0) mbar_expect_tx(nf_full + (gj & 1), 4);
                if (need) {
                    // column maxima over this warp's 32 keys (transposing shuffle reduction), then
                    // over this CTA's 128 keys, then with the peer's
#pragma unroll 1
                    for (int q = 0; q < 4; ++q) {
                        uint32_t r16[16];
                        load16(sb + q * 16, r16);
                        float v[16];
#pragma unroll
                        for (int u = 0; u < 16; ++u) v[u] = score(r16[u], col0 + q * 16 + u);
                        const float mx = pair_transpose_max16(v, lane);
                        if (lane < 16) red[warp * 64 + q * 16 + lane] = mx;
                    }
                    bar_sync_256();
                    float mloc = -INFINITY;
                    if (tid < kN) {
                        const int hc = tid >> 6, cl = tid & 63;
                        mloc = fmaxf(fmaxf(red[(hc * 4 + 0) * 64 + cl], red[(hc * 4 + 1) * 64 + cl]),
                                     fmaxf(red[(hc * 4 + 2) * 64 + cl], red[(hc * 4 + 3) * 64 + cl]));
                        st_async_f32(in_cta(px + (nx & 1) * kN + tid, peer), mloc, in_cta(px_full + (nx & 1), peer));
                    }
                    if (!group_wait(px_full + (nx & 1), (uint32_t)((nx >> 1) & 1))) {
                        ok = false;
                        break;
                    }
                    if (tid < kN) {
                        const float mx = fmaxf(mloc, px[(nx & 1) * kN + tid]);
                        const float mo = m_s[tid];
                        if (mx > mo + kRescaleThresh) {
                            m_s[tid] = mx;
                            a_s[tid] = (mo == -INFINITY) ? 0.f : ex2(mo - mx);
                        } else {
                            a_s[tid] = 1.f;
                        }
                    }
                    bar_sync_256();
                    // px of this exchange has been read: expect the peer's maxima of exchange nx + 2
                    if (tid == 0) mbar_expect_tx(px_full + (nx & 1), kN * 4);
                    ++nx;
                    // the row sums so far follow the new maxima
#pragma unroll
                    for (int q = 0; q < 4; ++q) ls[q] *= a_s[lcol + q * 16];
                    if (j > 0) {
                        // O^T holds the unit's tiles < j once PV(gj-1) is done: rescale it in TMEM
                        if (!wait_pv(gj - 1)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        constexpr int nsplit = 2 / VC2;  // warps w and w+4: one chunk each, or half the columns
                        const int c = (warp >> 2) % VC2;
#pragma unroll 1
                        for (int q = (warp >> 2) / VC2; q < kN / 16; q += nsplit) {
                            uint32_t r16[16];
                            const uint32_t ta = tmem_o + c * kN + lane_base + q * 16;
                            load16(ta, r16);
                            float av[16];
                            load_row16(a_s + q * 16, av);
#pragma unroll
                            for (int u = 0; u < 16; ++u) r16[u] = f2u(u2f(r16[u]) * av[u]);
                            tmem_st16(ta, r16);
                        }
                        tmem_st_wait();
                    }
                }
                if (gj >= kPBufs) {
                    // the P^T buffer of tile gj: PV(gj - kPBufs) must have read it
                    if (!wait_pv(gj - kPBufs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                }
                // pass 2: P = exp2(s - m) as bf16 pairs into the P^T buffer of CTA chh, and the
                // rounded P (what the PV MMA reads) summed over the warp's keys into the row sums.
                // A rolled loop: the softmax's steady-state code stays small enough for the
                // instruction cache.
#pragma unroll 1
                for (int q = 0; q < 4; ++q) {
                    float mv[16];
                    load_row16(m_s + col0 + q * 16, mv);
                    uint32_t r16[16];
                    load16(sb + q * 16, r16);
                    float e[16];
                    if (open) {
#pragma unroll
                        for (int u = 0; u < 16; ++u) e[u] = ex2(fmaf(u2f(r16[u]), sl2, -mv[u]));
                    } else {
#pragma unroll
                        for (int u = 0; u < 16; ++u) {
                            const float sv = score(r16[u], col0 + q * 16 + u);
                            e[u] = (sv == -INFINITY) ? 0.f : ex2(sv - mv[u]);
                        }
                    }
                    uint32_t pk2[8];
                    float pr[16];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const __nv_bfloat162 h2 = __floats2bfloat162_rn(e[2 * u], e[2 * u + 1]);
                        pk2[u] = *reinterpret_cast<const uint32_t*>(&h2);
                        pr[2 * u] = __low2float(h2);
                        pr[2 * u + 1] = __high2float(h2);
                    }
                    const uint32_t dst = prow0 + (uint32_t)((gj % kPBufs) * Lay::kPBuf + q * 2048);
                    const uint4 lo4 = make_uint4(pk2[0], pk2[1], pk2[2], pk2[3]);
                    const uint4 hi4 = make_uint4(pk2[4], pk2[5], pk2[6], pk2[7]);
                    if (p_local) {
                        uint8_t* d8 = smem + (dst - smem_u32(smem));
                        *reinterpret_cast<uint4*>(d8 + pswz0) = lo4;
                        *reinterpret_cast<uint4*>(d8 + pswz1) = hi4;
                    } else {
                        st_cluster_v4(dst + pswz0, lo4);
                        st_cluster_v4(dst + pswz1, hi4);
                    }
                    const float sm = pair_transpose_sum16(pr, lane);
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq)
                        if (qq == q) ls[qq] += sm;
                }
                // every thread's P stores are made visible to the tensor cores (a warp writes
                // either only its own CTA's buffer, which needs the CTA-scope fence alone, or only
                // the peer's) and its TMEM reads are ordered before the next MMAs; one thread of
                // each CTA then tells the even CTA. (An arrive per warp measured slower: each
                // cluster-scope release costs about what the barrier saves.)
                if (p_local)
                    fence_proxy_async_smem();
                else
                    fence_proxy_async_cluster();
                tc_fence_before();
                bar_sync_256();
                if (tid == 0) mbar_arrive_cluster(p_full_bar);
            }
            // the row sums over this CTA's keys: across the 4 warps of each half of the rows
            if (ok && U.ntiles > 0 && lane < 16) {
#pragma unroll
                for (int q = 0; q < 4; ++q) red2[warp * 64 + q * 16 + lane] = ls[q];
            }
            bar_sync_256();
            if (ok && U.ntiles > 0 && tid < kN) {
                const int hc = tid >> 6, cl = tid & 63;
                l_acc[tid] = (red2[(hc * 4 + 0) * 64 + cl] + red2[(hc * 4 + 1) * 64 + cl]) +
                             (red2[(hc * 4 + 2) * 64 + cl] + red2[(hc * 4 + 3) * 64 + cl]);
            }
            // ------------------------------------------------------------ the unit's epilogue
            // The row sums and the lse need only the softmax's own results: they are exchanged
            // and written while the last PV of the unit is still running.
            const bool have_l = ok && U.ntiles > 0;
            // row sums: this CTA's keys' part to the peer, the peer's part from it (two buffers:
            // the peer may send the next unit's before this CTA has read this one's)
            const int lb = un & 1;
            if (tid < kN)
                st_async_f32(in_cta(lx + lb * kN + tid, peer), have_l ? l_acc[tid] : 0.f, in_cta(lx_full + lb, peer));
            {
                bool got = true;
                if (tid == 0) got = ring_wait_cluster(lx_full + lb, (uint32_t)((un >> 1) & 1), abort_flag, p.err, p.wait_ns);
                if (bar_or_256(!got)) ok = false;
            }
            const int64_t part_base = (int64_t)U.c_split * p.B * p.T * p.Hq;
            const bool final_out = (p.splits == 1);
            if (tid < kN) {
                const float tot = (have_l ? l_acc[tid] : 0.f) + lx[lb * kN + tid];
                a_s[tid] = tot > 0.f ? 1.f / tot : 0.f;
                // each CTA writes the lse of half of the rows
                if ((tid >> 6) == (int)rank && orow_s[tid] >= 0) {
                    const float lse_v = tot > 0.f ? (m_s[tid] + __log2f(tot)) * kLn2 : -INFINITY;
                    if (final_out) {
                        if (p.lse) p.lse[orow_s[tid]] = lse_v;
                    } else {
                        p.part_lse[part_base + orow_s[tid]] = lse_v;
                        // the slots of the run's later chunks hold nothing: an lse of -inf, whose
                        // partial rows the combine does not read
                        for (int c = 1; c < U.n_run; ++c)
                            p.part_lse[part_base + (int64_t)c * p.B * p.T * p.Hq + orow_s[tid]] = -INFINITY;
                    }
                }
            }
            bar_sync_256();
            // this unit's row sums have been read: expect the peer's of unit un + 2
            if (tid == 0) mbar_expect_tx(lx_full + lb, kN * 4);
            bool have_o = have_l;
            if (have_o) have_o = ok = wait_pv(G + U.ntiles - 1);
            tc_fence_after();
            // O^T: warp w reads TMEM lanes 32(w%4).. = dims of chunk c; each column is one output
            // row. A warp's 16 rows x 32 dims go through a 2 KB scratch in the idle P^T buffers
            // (the peer writes this CTA's P^T again only after this CTA's next raise flag), so
            // that each lane stores 4 consecutive dims of a row: 4 stores of 16 bytes per lane
            // per 16 rows in place of 16 of 4 bytes.
            {
                constexpr int nsplit = 2 / VC2;
                const int c = (warp >> 2) % VC2;
                const int dbase = c * 256 + (int)rank * 128 + (warp & 3) * 32;
                float* scr = reinterpret_cast<float*>(smem + Lay::kPOff) + warp * 512;  // [16 rows][32 dims]
                const int er = lane >> 3;        // row within a group of 4 this lane stores
                const int dq = (lane & 7) * 4;   // its 4 dims within the warp's 32
#pragma unroll 1
                for (int q = (warp >> 2) / VC2; q < kN / 16; q += nsplit) {
                    uint32_t r16[16];
                    if (have_o) {
                        load16(tmem_o + c * kN + lane_base + q * 16, r16);
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e) r16[e] = 0u;
                    }
                    float iv[16];
                    load_row16(a_s + q * 16, iv);
                    // the output indices of this lane's 4 rows go to registers before any global
                    // store (a store through a global pointer may alias shared memory for the
                    // compiler, which would keep each later shared load behind it)
                    int64_t orows[4];
#pragma unroll
                    for (int s4 = 0; s4 < 4; ++s4) orows[s4] = orow_s[q * 16 + 4 * s4 + er];
#pragma unroll
                    for (int e = 0; e < 16; ++e) scr[e * 32 + lane] = u2f(r16[e]) * iv[e];
                    __syncwarp();
                    float4 v4[4];
#pragma unroll
                    for (int s4 = 0; s4 < 4; ++s4)
                        v4[s4] = *reinterpret_cast<const float4*>(scr + (4 * s4 + er) * 32 + dq);
                    __syncwarp();
#pragma unroll
                    for (int s4 = 0; s4 < 4; ++s4) {
                        const int64_t orow = orows[s4];
                        if (orow < 0) continue;
                        if (final_out) {
                            const __nv_bfloat162 lo = __floats2bfloat162_rn(v4[s4].x, v4[s4].y);
                            const __nv_bfloat162 hi = __floats2bfloat162_rn(v4[s4].z, v4[s4].w);
                            uint2 pk;
                            pk.x = *reinterpret_cast<const uint32_t*>(&lo);
                            pk.y = *reinterpret_cast<const uint32_t*>(&hi);
                            *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + orow * D + dbase + dq) = pk;
                        } else {
                            *reinterpret_cast<float4*>(p.part_out + (part_base + orow) * D + dbase + dq) = v4[s4];
                        }
                    }
                }
            }
            // the read-out is done with O^T (the next unit's first PV overwrites it only after this
            // CTA's P of that unit's first tile) and with the tables the next unit rewrites
            tc_fence_before();
            bar_sync_256();
            G += U.ntiles;
            ++un;
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // no CTA leaves while the pair MMAs or the peer may still touch its memory
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc2(tmem, Lay::kTmemCols);
    }
}

// ----------------------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn pair_encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// CTA pairs of tc_pair_attn_kernel<D> that fit the device at once (cached per device).
template <int D>
cudaError_t pair_resident_pairs(int* pairs)
{
    using Lay = PairLayout<D>;
    static std::mutex mu;
    static int cached[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(mu);
    if (cached[dev] == 0) {
        auto kern = tc_pair_attn_kernel<D>;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kAlloc);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = Lay::kAlloc;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
        if (e != cudaSuccess) return e;
        cached[dev] = n > 0 ? n : 1;
    }
    *pairs = cached[dev];
    return cudaSuccess;
}

// A persistent grid: one CTA pair per cluster slot the device holds at once (or one per unit
// when there are fewer units), each pair looping over its units.
template <int D>
cudaError_t launch_pair_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p,
                          const PairExtra& x, cudaStream_t stream)
{
    using Lay = PairLayout<D>;
    auto kern = tc_pair_attn_kernel<D>;
    int pairs = 0;
    cudaError_t e = pair_resident_pairs<D>(&pairs);
    if (e != cudaSuccess) return e;
    pairs = std::min(pairs, x.units);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * pairs);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Lay::kAlloc;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, p, x);
}

}  // namespace

// Query heads per pair: the largest divisor of G whose rows fit 64 per CTA (ceil(T/2) block
// positions each), or 0.
int pair_choose_gc(int G, int T)
{
    const int tb = (T + 1) / 2;
    for (int gc = G; gc >= 1; --gc)
        if (G % gc == 0 && gc * tb <= kHalf) return gc;
    return 0;
}

bool tc_pair_supports(const AttnParams& p)
{
    if (p.dtype != DFLASH_BF16) return false;
    if (p.D != 256 && p.D != 512) return false;
    if (p.page_size != 16 && p.page_size != 32 && p.page_size != 64) return false;
    if (p.T < 2 || pair_choose_gc(p.G, p.T) == 0) return false;
    if (p.sh % 8 || p.ss % 8 || p.sp % 8) return false;
    return true;
}

int tc_pair_ctas_per_split(const AttnParams& p)
{
    const int gc = pair_choose_gc(p.G, p.T);
    return gc > 0 ? 2 * p.B * p.Hkv * (p.G / gc) : 0;
}

cudaError_t tc_pair_grid_ctas(const AttnParams& p, int64_t* ctas)
{
    const int gc = pair_choose_gc(p.G, p.T);
    if (gc <= 0) return cudaErrorNotSupported;
    const int64_t units = (int64_t)p.splits * p.Hkv * (p.G / gc) * p.B;
    int pairs = 0;
    cudaError_t e = (p.D == 512) ? pair_resident_pairs<512>(&pairs) : pair_resident_pairs<256>(&pairs);
    if (e != cudaSuccess) return e;
    *ctas = 2 * std::min<int64_t>(pairs, units);
    return cudaSuccess;
}

int tc_pair_row_groups(const AttnParams& p)
{
    const int gc = pair_choose_gc(p.G, p.T);
    return gc > 0 ? p.G / gc : 0;
}

cudaError_t launch_tc_pair_attn(const AttnParams& p, cudaStream_t stream)
{
    if (!tc_pair_supports(p) || p.balanced) return cudaErrorNotSupported;
    EncodeTiledFn enc = pair_encode_fn();
    if (!enc) return cudaErrorNotSupported;
    PairExtra x;
    x.Gc = pair_choose_gc(p.G, p.T);
    x.n_rg = p.G / x.Gc;
    x.Tb = (p.T + 1) / 2;
    const int64_t units = (int64_t)p.splits * p.Hkv * x.n_rg * p.B;
    if (units > (int64_t)INT32_MAX) return cudaErrorNotSupported;
    x.units = (int32_t)units;

    CUtensorMap tq, tk, tv;
    {
        const cuuint64_t dims[3] = {(cuuint64_t)p.D, (cuuint64_t)p.Hq, (cuuint64_t)p.B * p.T};
        const cuuint64_t strides[2] = {(cuuint64_t)p.D * 2, (cuuint64_t)p.Hq * p.D * 2};
        const cuuint32_t box[3] = {64, (cuuint32_t)x.Gc, (cuuint32_t)x.Tb};
        const cuuint32_t es[3] = {1, 1, 1};
        if (enc(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(p.q), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[4] = {(cuuint64_t)p.D, (cuuint64_t)p.Hkv, (cuuint64_t)p.page_size,
                                    (cuuint64_t)p.num_pages};
        const cuuint64_t strides[3] = {(cuuint64_t)p.sh * 2, (cuuint64_t)p.ss * 2, (cuuint64_t)p.sp * 2};
        const cuuint32_t box[4] = {64, 1, (cuuint32_t)p.page_size, 1};
        const cuuint32_t es[4] = {1, 1, 1, 1};
        if (enc(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(p.k), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        if (enc(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(p.v), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    cudaError_t e;
    switch (p.D) {
    case 256: e = launch_pair_d<256>(tq, tk, tv, p, x, stream); break;
    case 512: e = launch_pair_d<512>(tq, tk, tv, p, x, stream); break;
    default: e = cudaErrorNotSupported;
    }
    if (e != cudaSuccess || p.splits == 1) return e;
    return launch_combine(p.part_out, p.part_lse, p.splits, (int64_t)p.B * p.T * p.Hq, p.D, p.dtype, p.out, p.lse,
                          stream);
}

}  // namespace dflash
