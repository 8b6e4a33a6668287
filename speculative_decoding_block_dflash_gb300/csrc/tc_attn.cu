// Tensor-core block attention for bf16 on sm_103a: tcgen05.mma with TMEM
// accumulators, paged K/V staged by TMA into a shared-memory ring.
//
// Problem (DFlash block attention): per (request b, KV head g) the G query
// heads x T block queries that share g are packed into R = Gc*T rows of one
// tile ("num_query_per_req = 1 + num_speculative_tokens", kenforever1
// "dflash-gemma4-31b-notes"; GQA 8 x 9 = 72 rows at the Gemma-4-31B global
// layer shape). Every key byte is read once per CTA and feeds all R rows, so
// the packed tile is a dense contraction: QK^T and PV run on the tensor cores.
//
// Transposed formulation. head_dim reaches 512 ("head_size <= 512", same
// page), and an fp32 O accumulator of 128 x 512 would fill all 512 TMEM
// columns. So the kernel computes
//     S^T [128 keys x N rows]     = K_tile [128 x D] . Q^T [D x N]        (M = 128 keys)
//     O^T [D x N] (D/128 chunks) += V_tile^T [D x 128] . P^T [128 x N]  (M = 128 dims)
//     l^T [128 x 16]             += P [128 rows x 128] . ones [128 x 16] (lane r = row r's sum)
// with N = R rounded up to 16 (<= 80). The row-sum MMA reads P as a 128-row
// operand (rows >= N only feed unused lanes), so l takes 16 TMEM columns and
// S^T fits twice: TMEM holds two S^T buffers, O^T and l^T, 2N + (D/128) N + 16
// columns (496 at D = 512, N = 80).
//
// Pipeline. The ring is filled in the order the MMA warp consumes it, K(0) K(1)
// V(0) K(2) V(1) ... V(n-1): S(j+1) is computed into the other S^T buffer while
// the softmax of tile j runs, and the TMA copies only wait for a softmax when
// the ring is full of V(j) stages.
//
// Softmax (thread = one key lane of the tile, warps 0-7; warps w and w + 4 share
// the TMEM lanes of w mod 4 and take alternate 16-column groups): S^T is read from TMEM
// in 16-column groups in rolled loops; this code runs once or twice per SM per
// call, so it is kept small, and a dry run over fully masked scores executes it
// once while the first K tile is still in flight so that the first real tile
// does not stall on instruction fetches. Scores are masked by select
// (non-causal rows see every key up to L-1, causal rows keys up to their own
// position, a window W keeps the last W keys -- vLLM PR #43445 "Allow causal
// DFlash"). The running row max m is shared by the 256 softmax threads and only
// raised when a score exceeds it by more than 2^8 in the exp2 domain (a
// transposing shuffle reduction leaves each lane with one column's maximum over
// its warp, then the four warps meet in shared memory; O^T and l^T are then
// rescaled by exp2(m_old - m_new) in TMEM). P = exp2(s - m) is rounded to bf16
// pairs and written to shared memory as the operand of the PV and row-sum MMAs,
// MN-major with a 32-byte swizzle so that a key lane's 16 rows of a group are two
// 16-byte stores. P^T has two buffers: the softmax of tile j+1 writes while
// PV(j) still reads.
//
// Warp roles (384 threads): warps 0-7 softmax, then the epilogue; warps 8-10 TMA
// producers; warp 11 MMA issuer. Every role's loops are rolled: with unrolled stage
// loops the kernel was about 150 KB of code and its warps stalled on instruction fetch.
// One warp's tensor copies are processed in order, so a single producer warp caps a CTA
// near 26 GB/s with 2 KB boxes; the ring stages are dealt round-robin to the three
// producer warps (stage i of the sequence to warp i mod 3), each filling whole stages. Ring
// stages are 16 KB: a K stage is 128 keys x 64 dims (K-major, 128-byte
// swizzle), a V stage 64 keys x 128 dims (MN-major). One TMA box is one page's
// tokens of one KV head x 64 dims; the page id comes from the page table
// (validated; out-of-range ids and pages past the chunk are fetched at an
// out-of-bounds page coordinate, which the TMA unit fills with zeros without
// touching memory). V rows of the last, partial page past seq_len are zeroed in
// shared memory before the PV MMA so garbage there can never reach the output.
//
// Epilogue: the output tile is normalised by 1/l, assembled row-major in the
// freed Q / P / ring shared memory by eight warps and written with bulk
// asynchronous copies, one per block position (its Gc head rows are contiguous).
//
// Every mbarrier wait is bounded (p.wait_ns of %globaltimer, 2 s unless the
// caller sets dflash_opts.wait_limit_us); on expiry the kernel records
// DFLASH_DEVERR_TIMEOUT, drains its own TMA copies and MMAs (bounded), frees
// TMEM and returns.
#include <cuda.h>

#include <cmath>
#include <mutex>

#include "dflash_device.cuh"
#include "tc_ptx.cuh"

namespace dflash {
namespace {

using namespace ptx;

constexpr int kThreads = 384;
constexpr int kSoftmaxThreads = 256;  // warps 0..7
constexpr int kProducerWarp = 8;      // warps 8..10 issue TMA copies
constexpr int kNumProducers = 3;
constexpr int kMmaWarp = 11;
constexpr int kTileKeys = 128;
constexpr int kStageBytes = 16384;
constexpr int kMaxPids = 128;  // page ids held per producer warp (one window)
constexpr int kMaxRows = 80;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThresh = 8.0f;
constexpr int kOnesBytes = 4096;

struct TcExtra {
    int32_t Gc;     // query heads per CTA
    int32_t n_rg;   // row groups per KV head (G / Gc)
    int32_t R;      // packed rows per CTA (Gc * T)
    int32_t fused;  // 1: the split CTAs of a row group combine their partials in this kernel
};

__device__ __forceinline__ int32_t ld_acquire_gpu(const int32_t* ptr)
{
    int32_t v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
    return v;
}

constexpr int pow2ceil(int x)
{
    int p = 32;
    while (p < x) p <<= 1;
    return p;
}

template <int D, int N>
struct TcLayout {
    static constexpr int kPBytes = N * 128 * 2;                         // one P^T buffer: 2 key halves
    static constexpr int kFixed = N * D * 2 + 2 * kPBytes + 4096 + kOnesBytes;
    static constexpr int kStagesFit = (227 * 1024 - 1024 - kFixed) / kStageBytes;
    static constexpr int kStages = kStagesFit > 12 ? 12 : kStagesFit;
    static constexpr int kQOff = 0;                                     // [D/64][N rows][128 B]
    static constexpr int kPOff = kQOff + N * D * 2;                     // [2 buffers][2 key halves][N rows][128 B]
    static constexpr int kRingOff = kPOff + 2 * kPBytes;                // [stages][16 KB]
    static constexpr int kOnesOff = kRingOff + kStages * kStageBytes;   // bf16 ones [16 x 64] (row-sum MMA)
    static constexpr int kBarOff = kOnesOff + kOnesBytes;
    // Stages of the first K tile that do not fit the ring borrow the P^T buffers, which
    // are not written before the first softmax (it starts after those stages are consumed).
    static constexpr int kExtraWant = D / 64 - kStages;
    static constexpr int kExtra = (kPBytes < kStageBytes || kExtraWant <= 0) ? 0 : (kExtraWant > 2 ? 2 : kExtraWant);
    static constexpr int kNumBars = 2 * kStages + 6 + kExtra;
    static constexpr int kMiscOff = (kBarOff + kNumBars * 8 + 15) / 16 * 16;  // tmem base, abort flag
    static constexpr int kMOff = kMiscOff + 16;                         // float m_s[N]
    static constexpr int kAOff = kMOff + N * 4;                         // float alpha_s[N] (1/l at the end)
    static constexpr int kRedOff = kAOff + N * 4;                       // float red[4][N]
    static constexpr int kLoOff = kRedOff + 4 * N * 4;                  // int lo_s[N]
    static constexpr int kHiOff = kLoOff + N * 4;                       // int hi_s[N]
    static constexpr int kRowOff = kHiOff + N * 4;                      // int64 orow_s[N]
    static constexpr int kPidOff = kRowOff + N * 8;                     // int pid_s[kNumProducers][kMaxPids]
    static constexpr int kTotal = kPidOff + kNumProducers * kMaxPids * 4;
    static constexpr int kAlloc = kTotal + 1024;
    static constexpr int kTmemUsed = 2 * N + (D / 128) * N + 16;        // S^T x 2, O^T, l^T
    static constexpr int kTmemCols = pow2ceil(kTmemUsed);
    // each producer warp fills every kNumProducers-th stage; with fewer slots than producers
    // a warp could pass a slot two phases ahead (the parity wait cannot tell them apart)
    static_assert(kStages >= kNumProducers, "ring too shallow for the producer warps");
    static_assert(kOnesOff - kQOff >= N * D * 4, "output tile staging (Q, P and the ring)");
    static_assert(kPOff + kPBytes + N * 128 + 128 * 128 <= kOnesOff, "128-row P operand of the row-sum MMA");
    static_assert(kTmemUsed <= 512, "TMEM budget");
    static_assert((N * D * 2) % 1024 == 0 && (N * 128) % 1024 == 0, "1024-byte swizzle atoms");
    static_assert(kTotal + 1024 <= 227 * 1024, "shared memory budget");
};

// ----------------------------------------------------------------------------- kernel

// Column maxima over a warp: v holds 16 consecutive columns of this lane's row.
// Each step swaps half of the live columns with the partner lane and keeps the
// maximum of the half it owns; after four steps lane l holds the maximum over
// its 16-lane half of column l mod 16, and one exchange across the halves
// completes it: 16 shuffles for 16 columns instead of 80 (one butterfly each).
__device__ __forceinline__ float transpose_max16(float (&v)[16], int lane)
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

// The k-th unit (0 <= k < 2n) of the ring sequence K(0) K(1) V(0) K(2) V(1) ...
// K(n-1) V(n-2) V(n-1): whether it is a K tile, and which tile. K(j+1) is loaded
// ahead of V(j) so S(j+1) can be computed while the softmax of tile j runs.
__device__ __forceinline__ void ring_unit(int k, int n, bool& is_k, int& tile)
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

// Buffer and phase of the stage with sequence number seq: stages S .. S+E-1 (the tail of the
// first K tile) go to the E extra slots, used once; every other stage cycles through the
// S ring slots.
struct RingSlot {
    int idx;
    uint32_t phase;
    bool extra;
};

__device__ __forceinline__ RingSlot ring_slot(int seq, int S, int E)
{
    RingSlot r;
    if (seq >= S && seq < S + E) {
        r.idx = seq - S;
        r.phase = 0;
        r.extra = true;
    } else {
        const int q = seq < S ? seq : seq - E;
        r.idx = q % S;
        r.phase = (uint32_t)((q / S) & 1);
        r.extra = false;
    }
    return r;
}

// Length-balanced plan: the splits chunk slots of a row group are dealt to the B requests so
// that the longest chunk is as short as it can be. With t_b the 128-key tiles of request b's
// key span, C is the least tile count for which every request cut into ceil(t_b / C) chunks
// fits the slots; the spare slots go one each to requests 0, 1, ... in turn. Request b then
// has n_b chunks (split_chunk of n_b, none longer than C tiles), and slot `slot` is chunk c of
// n of request b, whose chunks start at slot `first`. (Slots dealt in proportion to the spans,
// rounded, left batch_sweep_b8's longest chunk at 33 tiles against 31 here, for a mean of 27.)
// Every warp computes it alike: its lanes take the requests in turn, and with at most 32
// requests the lanes test 32 candidate bounds at once, so that the common case costs one pass.
struct ReqChunk {
    int32_t b, c, n, first;
};

__device__ inline int64_t key_span(const AttnParams& p, int32_t b)
{
    int32_t L = __ldg(p.seq_lens + b);
    if (L < 0) L = 0;
    if (L > p.max_seq_len) L = p.max_seq_len;
    int32_t lo = 0;
    if (p.window > 0) {
        lo = L - p.T - p.window + 1;
        if (lo < 0) lo = 0;
    }
    const int64_t n = (int64_t)L - (lo / p.page_size) * p.page_size;
    return n > 0 ? n : 1;
}

// ceil(a / c) for 0 <= a < 2^24, c >= 1, through a float reciprocal and a one-step fix-up
__device__ __forceinline__ int32_t ceil_div_small(int32_t a, int32_t c)
{
    const int32_t num = a + c - 1;
    int32_t q = __float2int_rz(__fdividef((float)num, (float)c));
    if (q * c > num)
        --q;
    else if ((q + 1) * c <= num)
        ++q;
    return q;
}

// Slots the requests need when no chunk exceeds C tiles (t_lane: lane's request's tiles), summed
// over the warp. Out of line: it serves the rare search past 32 candidate bounds.
__device__ __noinline__ int32_t balanced_slots_for(const AttnParams& p, int32_t t_lane, int32_t C)
{
    const int lane = threadIdx.x & 31;
    int32_t n = ceil_div_small(t_lane, C);
#pragma unroll 1
    for (int32_t b = lane + 32; b < p.B; b += 32) n += ceil_div_small((int32_t)((key_span(p, b) + kTileKeys - 1) / kTileKeys), C);
    return __reduce_add_sync(0xffffffffu, n);
}

__device__ inline ReqChunk balanced_chunk(const AttnParams& p, int32_t slot)
{
    // requests b = lane + 32 k; loops stay rolled (this runs once per CTA, and unrolled it added
    // a quarter to the kernel's code)
    const int lane = threadIdx.x & 31;
    auto tiles_of = [&](int32_t b) -> int32_t { return (int32_t)((key_span(p, b) + kTileKeys - 1) / kTileKeys); };
    const int32_t t_lane = lane < p.B ? tiles_of(lane) : 0;  // all of them when B <= 32
    int32_t tmax = max(1, t_lane), ttot = t_lane;
#pragma unroll 1
    for (int32_t b = lane + 32; b < p.B; b += 32) {
        const int32_t t = tiles_of(b);
        tmax = max(tmax, t);
        ttot += t;
    }
    tmax = __reduce_max_sync(0xffffffffu, tmax);
    ttot = __reduce_add_sync(0xffffffffu, ttot);
    auto slots_for = [&](int32_t C) -> int32_t { return balanced_slots_for(p, t_lane, C); };
    // the least C that fits. Lane j tests lo + j when there are at most 32 requests (the answer
    // is usually within a few tiles of the mean); past that, or with more requests, gallop up
    // from the mean, then bisect.
    int32_t lo = max(1, (ttot + p.splits - 1) / p.splits);  // a C below lo cannot fit
    int32_t C = lo;
    int32_t used = -1;  // slots C takes, once known
    if (p.B <= 32) {
        const int32_t cj = lo + lane;
        int32_t need = 0;
#pragma unroll 1
        for (int32_t r = 0; r < p.B; ++r) need += ceil_div_small(__shfl_sync(0xffffffffu, t_lane, r), cj);
        const uint32_t fits = __ballot_sync(0xffffffffu, need <= p.splits);
        if (fits) {
            C = lo + __ffs(fits) - 1;
            used = __shfl_sync(0xffffffffu, need, __ffs(fits) - 1);
        } else {
            lo += 32;
            C = lo;
        }
    }
    if (used < 0 && slots_for(C) > p.splits) {
        int32_t step = 1, hi = tmax;  // C = tmax always fits: B <= splits
#pragma unroll 1
        for (;;) {
            const int32_t c2 = min(tmax, lo + step);
            if (slots_for(c2) <= p.splits) {
                hi = c2;
                break;
            }
            lo = c2 + 1;
            step <<= 1;
            if (c2 == tmax) break;  // not reached
        }
#pragma unroll 1
        while (lo < hi) {
            const int32_t mid = (lo + hi) >> 1;
            if (slots_for(mid) <= p.splits)
                hi = mid;
            else
                lo = mid + 1;
        }
        C = hi;
    }
    if (used < 0) used = slots_for(C);
    const int32_t left = p.splits - used;
    const int32_t every = left / p.B, some = left % p.B;
    // the request whose chunks hold `slot`: an inclusive scan of n_b over the lanes, 32 at a time
    int32_t base = 0;
#pragma unroll 1
    for (int32_t b0 = 0; b0 < p.B; b0 += 32) {
        const int32_t b = b0 + lane;
        const int32_t t = b0 == 0 ? t_lane : (b < p.B ? tiles_of(b) : 0);
        const int32_t n = b < p.B ? ceil_div_small(t, C) + every + (b < some ? 1 : 0) : 0;
        int32_t incl = n;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int32_t v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += v;
        }
        const uint32_t hit = __ballot_sync(0xffffffffu, b < p.B && slot < base + incl);
        if (hit) {
            const int src = __ffs(hit) - 1;
            const int32_t nb = __shfl_sync(0xffffffffu, n, src);
            const int32_t first = base + __shfl_sync(0xffffffffu, incl, src) - nb;
            return ReqChunk{b0 + src, slot - first, nb, first};
        }
        base += __shfl_sync(0xffffffffu, incl, 31);
    }
    return ReqChunk{p.B - 1, 0, 1, base};  // not reached: the n_b add up to the slots
}

template <int D, int N>
__global__ void __launch_bounds__(kThreads, 1)
    tc_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const AttnParams p, const TcExtra x)
{
    using Lay = TcLayout<D, N>;
    constexpr int S = Lay::kStages;
    constexpr int KC = D / 64;   // K stages per tile (64-dim chunks)
    constexpr int VC = D / 128;  // O^T chunks (128 dims); V stages per 64-key half
    constexpr int NQ = N / 16;   // 16-column groups of S^T / O^T

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* q_s = smem + Lay::kQOff;
    uint8_t* ring = smem + Lay::kRingOff;
    uint8_t* p_s = smem + Lay::kPOff;
    uint8_t* ones_s = smem + Lay::kOnesOff;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kBarOff);
    uint64_t* full = bars;
    uint64_t* empty = bars + S;
    uint64_t* s_full = bars + 2 * S;  // [2] MMA -> softmax: S^T of the tile is in TMEM buffer j mod 2
    uint64_t* p_full = s_full + 2;    // softmax -> MMA: P^T written and S^T buffer read
    uint64_t* p_free = s_full + 3;    // [2] MMA -> softmax: PV of the tile done (P^T buffer j mod 2 free)
    uint64_t* drain = s_full + 5;
    uint64_t* xfull = s_full + 6;     // [kExtra] TMA -> MMA: extra stage landed (used once)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lay::kMiscOff + 4);
    float* m_s = reinterpret_cast<float*>(smem + Lay::kMOff);
    float* a_s = reinterpret_cast<float*>(smem + Lay::kAOff);
    float* red = reinterpret_cast<float*>(smem + Lay::kRedOff);
    int32_t* lo_s = reinterpret_cast<int32_t*>(smem + Lay::kLoOff);
    int32_t* hi_s = reinterpret_cast<int32_t*>(smem + Lay::kHiOff);
    int64_t* orow_s = reinterpret_cast<int64_t*>(smem + Lay::kRowOff);
    int32_t* pid_s = reinterpret_cast<int32_t*>(smem + Lay::kPidOff);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    // (request, chunk of its n_split chunks); partial rows of chunk k sit at
    // (slot0 + k) * rstride + rbias + output row
    int b, c_split, n_split, slot0;
    int64_t rstride, rbias;
    if (p.balanced) {
        const ReqChunk rc = balanced_chunk(p, blockIdx.x);
        b = rc.b;
        c_split = rc.c;
        n_split = rc.n;
        slot0 = rc.first;
        rstride = (int64_t)p.T * p.Hq;
        rbias = -(int64_t)b * p.T * p.Hq;
    } else {
        b = blockIdx.z;
        c_split = blockIdx.x;
        n_split = p.splits;
        slot0 = 0;
        rstride = (int64_t)p.B * p.T * p.Hq;
        rbias = 0;
    }
    const int g = blockIdx.y / x.n_rg;
    const int rg = blockIdx.y % x.n_rg;
    const int T = p.T;
    const int Psz = p.page_size;
    const int R = x.R;
    const int h0 = g * p.G + rg * x.Gc;

    const int32_t L = __ldg(p.seq_lens + b);
    const bool len_ok = seq_len_ok(p, L);
    Chunk ch;
    ch.kb = 0;
    ch.ke = 0;
    if (len_ok) ch = split_chunk(L, T, p.window, Psz, n_split, c_split);
    const int t0 = (ch.kb / Psz) * Psz;
    const int ntiles = (ch.kb < ch.ke) ? (ch.ke - t0 + kTileKeys - 1) / kTileKeys : 0;
    const int pages_per_tile = kTileKeys / Psz;
    const int chunk_pages = ntiles * pages_per_tile;
    const int first_page = t0 / Psz;

    // Page ids of relative pages [base, base + kMaxPids) -> this producer warp's pid_w.
    // Pages past the chunk and invalid ids map to the out-of-bounds coordinate num_pages.
    const int pw = warp - kProducerWarp;
    int32_t* pid_w = pid_s + (pw >= 0 && pw < kNumProducers ? pw : 0) * kMaxPids;
    auto load_window = [&](int base) {
        for (int k = lane; k < kMaxPids; k += 32) {
            const int pr = base + k;
            int32_t id = p.num_pages;
            if (pr < chunk_pages && t0 + pr * Psz < ch.ke) {
                const int32_t v = __ldg(p.page_table + (int64_t)b * p.max_pages + first_page + pr);
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
        for (int i = 0; i < Lay::kNumBars; ++i) {
            uint64_t* bar = bars + i;
            mbar_init(bar, bar == p_full ? (uint32_t)kSoftmaxThreads : 1u);
        }
        *abort_flag = 0;
        if (!len_ok) raise_error(p.err, DFLASH_DEVERR_SEQ_LEN);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        // Q's copies go out now, counted on ring stage 0's barrier (whose producer arms it with
        // Q's bytes as well), so that Q lands while the producers still read the page table
        if (ntiles > 0)
            for (int kc = 0; kc < KC; ++kc) tma_load_3d(q_s + kc * N * 128, &tm_q, full, kc * 64, h0, b * T);
    }
    if (warp >= kProducerWarp && warp < kProducerWarp + kNumProducers) {
        if (ntiles > 0) load_window(0);
    } else if (warp == kMmaWarp) {
        for (int idx = lane; idx < kOnesBytes / 16; idx += 32)
            *reinterpret_cast<uint4*>(ones_s + idx * 16) =
                make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);  // bf16 1.0
        fence_proxy_async_smem();
        tmem_alloc(tmem_slot, Lay::kTmemCols);
        tmem_relinquish();
    } else {
        if (tid < N) {
            int32_t lo = -(1 << 30), hi = (1 << 30);
            int64_t orow = -1;
            if (tid < R) {
                const int i = tid / x.Gc;
                const int hh = tid - i * x.Gc;
                const KeyRange kr = row_range(L, T, i, p.causal, p.window);
                lo = kr.lo;
                hi = kr.hi;
                orow = (int64_t)(b * T + i) * p.Hq + (h0 + hh);
            }
            lo_s[tid] = lo;
            hi_s[tid] = hi;
            orow_s[tid] = orow;
            m_s[tid] = -INFINITY;
            a_s[tid] = 1.f;
        }
        // zero the padding rows [R, N) of Q (the TMA writes rows [0, R) of every 64-dim chunk)
        for (int idx = tid; idx < KC * (N - R) * 8; idx += kSoftmaxThreads) {
            const int kc = idx / ((N - R) * 8);
            const int rem = idx - kc * (N - R) * 8;
            *reinterpret_cast<uint4*>(q_s + kc * N * 128 + (R + rem / 8) * 128 + (rem % 8) * 16) =
                make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // let a dependent split-combine grid start launching; it waits for our completion
    cudaTriggerProgrammaticLaunchCompletion();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tmem_s = tmem;                   // S^T buffers: columns [0, N) and [N, 2N)
    const uint32_t tmem_o = tmem + 2 * N;           // O^T chunk c: columns [2N + cN, 2N + (c+1)N)
    const uint32_t tmem_l = tmem + 2 * N + VC * N;  // l^T: lane r holds row r's sum (16 equal columns)
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    bool role_ok = true;

    auto load16 = [&](uint32_t taddr, uint32_t (&r16)[16]) {
        tmem_ld16(taddr, r16);
        tmem_ld_wait();
        reg_fence16(r16);
    };

    if (warp >= kProducerWarp && warp < kProducerWarp + kNumProducers) {
        // ------------------------------------------------------------ TMA producers
        constexpr int E = Lay::kExtra;
        bool ok = true;
        int wbase = 0;
        uint32_t issued_parity[S];
        uint32_t issued_extra = 0;
#pragma unroll
        for (int s = 0; s < S; ++s) issued_parity[s] = 2;  // 2 = nothing outstanding
        if (ntiles > 0) {
            const int box = Psz * 128;  // bytes of one page x 64 dims
            // K/V pages are read once: they leave L2 first, ahead of the split partials
            const uint64_t kv_policy = l2_policy_evict_first();
            int seq = 0;                // index of the stage in the whole sequence; this warp fills seq = pw (mod kNumProducers)
            for (int k = 0; k < 2 * ntiles && ok; ++k) {
                bool is_k;
                int tile;
                ring_unit(k, ntiles, is_k, tile);
                const int rel0 = tile * pages_per_tile;
                const int n_st = is_k ? KC : 2 * VC;
                // K: KC stages of 128 keys x 64 dims; V: 2 x VC stages of 64 keys x 128 dims
                // (rolled, like every loop of the roles: unrolled, they made the kernel's code
                // too large for the instruction cache)
#pragma unroll 1
                for (int sq = 0; sq < n_st && ok; ++sq, ++seq) {
                    if (seq % kNumProducers == pw) {
                        if (rel0 < wbase || rel0 + pages_per_tile > wbase + kMaxPids) {
                            wbase = (tile > 0 ? tile - 1 : 0) * pages_per_tile;
                            load_window(wbase);
                        }
                        const RingSlot sl = ring_slot(seq, S, E);
                        uint64_t* fb = sl.extra ? xfull + sl.idx : full + sl.idx;
                        if (!sl.extra) {
                            if (lane == 0) ok = ring_wait(empty + sl.idx, sl.phase ^ 1u, abort_flag, p.err, p.wait_ns);
                            ok = __shfl_sync(0xffffffffu, ok, 0);
                            if (!ok) break;
                        }
                        if (lane == 0) {
                            uint8_t* dst = sl.extra ? p_s + sl.idx * Lay::kPBytes : ring + sl.idx * kStageBytes;
                            // The Q tile rides on the first stage's barrier (thread 0 issued its
                            // copies at set-up): the MMA warp's first wait covers it. (A separate
                            // barrier completed by the tensor-copy unit and waited on ahead of the
                            // ring made every later K/V copy of the CTA land about twice as late.)
                            const bool with_q = (seq == 0);
                            mbar_expect_tx(fb, kStageBytes + (with_q ? (uint32_t)(R * 128 * KC) : 0u));
                            // The stage's page ids go to registers before its copies are issued:
                            // each copy instruction is also a compiler memory barrier, so reading
                            // an id between two copies made every box wait for a shared-memory
                            // load, which halved the rate at which a warp issues copies.
                            if (is_k) {
                                int32_t ids[8];
#pragma unroll
                                for (int pg = 0; pg < 8; ++pg)
                                    ids[pg] = pg < pages_per_tile ? pid_w[rel0 + pg - wbase] : 0;
#pragma unroll
                                for (int pg = 0; pg < 8; ++pg)
                                    if (pg < pages_per_tile)
                                        tma_load_4d_hint(dst + pg * box, &tm_k, fb, sq * 64, g, 0, ids[pg], kv_policy);
                            } else {
                                const int h = sq / VC, c = sq % VC;
                                const int ppg = 64 / Psz;  // pages per 64-key half
                                int32_t ids[4];
#pragma unroll
                                for (int pg = 0; pg < 4; ++pg)
                                    ids[pg] = pg < ppg ? pid_w[rel0 + h * ppg + pg - wbase] : 0;
#pragma unroll
                                for (int pg = 0; pg < 4; ++pg)
                                    if (pg < ppg)
#pragma unroll
                                        for (int m = 0; m < 2; ++m)
                                            tma_load_4d_hint(dst + m * 8192 + pg * box, &tm_v, fb, c * 128 + m * 64,
                                                             g, 0, ids[pg], kv_policy);
                            }
                            if (sl.extra)
                                issued_extra |= 1u << sl.idx;
                            else
                                issued_parity[sl.idx] = sl.phase;
                        }
                        __syncwarp();
                    }
                }
            }
        }
        // Drain: no TMA copy of ours may still be landing when the ring is reused or the CTA exits.
        if (lane == 0 && !ok) {
#pragma unroll 1
            for (int s = 0; s < S; ++s) {
                if (issued_parity[s] > 1) continue;
                const unsigned long long t_start = globaltimer();
                while (!mbar_try_wait(full + s, issued_parity[s]) && globaltimer() - t_start < p.wait_ns) {
                }
            }
#pragma unroll 1
            for (int e = 0; e < E; ++e) {
                if (!(issued_extra & (1u << e))) continue;
                const unsigned long long t_start = globaltimer();
                while (!mbar_try_wait(xfull + e, 0) && globaltimer() - t_start < p.wait_ns) {
                }
            }
        }
        __syncwarp();
        role_ok = ok;
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t idesc_s = make_idesc(128, N, 0, 0);   // S^T  = K . Q^T   (A K-major, B K-major)
        constexpr uint32_t idesc_o = make_idesc(128, N, 1, 1);   // O^T += V^T . P^T (A MN-major, B MN-major)
        constexpr uint32_t idesc_l = make_idesc(128, 16, 1, 0);  // l^T += P . 1     (A MN-major, B K-major)
        const uint32_t q_addr = smem_u32(q_s);
        const uint32_t p_addr = smem_u32(p_s);
        const uint32_t ring_addr = smem_u32(ring);
        const uint32_t ones_addr = smem_u32(ones_s);
        constexpr int E = Lay::kExtra;
        int mseq = 0;  // sequence number of the next ring stage
        bool ok = true;
        auto wait_lane0 = [&](uint64_t* bar, uint32_t par) -> bool {
            bool got = true;
            if (lane == 0) got = ring_wait(bar, par, abort_flag, p.err, p.wait_ns);
            return __shfl_sync(0xffffffffu, got, 0);
        };
        // wait for the next stage; its shared address (and whether it is an extra slot)
        auto next_stage = [&](uint32_t& addr, RingSlot& sl) -> bool {
            sl = ring_slot(mseq, S, E);
            const bool got = wait_lane0(sl.extra ? xfull + sl.idx : full + sl.idx, sl.phase);
            addr = sl.extra ? p_addr + sl.idx * Lay::kPBytes : ring_addr + sl.idx * kStageBytes;
            return got;
        };
        auto release = [&](const RingSlot& sl) {
            if (lane == 0 && !sl.extra) tc_commit(empty + sl.idx);
            __syncwarp();
            ++mseq;
        };
        for (int k = 0; k < 2 * ntiles && ok; ++k) {
            bool is_k;
            int j;
            ring_unit(k, ntiles, is_k, j);
            if (is_k) {
                // S^T(j) = K(j) . Q^T into buffer j mod 2, whose previous tile j - 2 the
                // softmax has finished with (its p_full was waited for by the V(j-2) unit)
                const uint32_t sb = tmem_s + (uint32_t)(j & 1) * N;
#pragma unroll 1
                for (int kc = 0; kc < KC && ok; ++kc) {
                    uint32_t st;
                    RingSlot sl;
                    ok = next_stage(st, sl);
                    if (!ok) break;
                    tc_fence_after();
                    if (lane == 0) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            tc_mma(sb, sw128_desc(st + kk * 32, 16, 1024),
                                   sw128_desc(q_addr + kc * N * 128 + kk * 32, 16, 1024), idesc_s,
                                   (kc > 0 || kk > 0) ? 1u : 0u);
                    }
                    release(sl);
                }
                if (!ok) break;
                if (lane == 0) tc_commit(s_full + (j & 1));
                __syncwarp();
                continue;
            }
            // O^T += V(j)^T . P^T and l^T += P . 1 once the softmax has written P(j)
            ok = wait_lane0(p_full, (uint32_t)(j & 1));
            if (!ok) break;
            tc_fence_after();
            const int tile_key0 = t0 + j * kTileKeys;
            const uint32_t pb_addr = p_addr + (uint32_t)(j & 1) * Lay::kPBytes;
#pragma unroll 1
            for (int h = 0; h < 2 && ok; ++h) {
#pragma unroll 1
                for (int c = 0; c < VC && ok; ++c) {
                    uint32_t st_addr;
                    RingSlot sl;
                    ok = next_stage(st_addr, sl);
                    if (!ok) break;
                    tc_fence_after();
                    // V rows past seq_len in the sequence's last, partial page -> zero
                    const int key0 = tile_key0 + h * 64;
                    const int zlo = L - key0;
                    if (L % Psz != 0 && zlo > 0 && zlo < 64 && ch.ke == L) {
                        const int zhi = min(64, ((L + Psz - 1) / Psz) * Psz - key0);
                        uint8_t* st = smem + (st_addr - smem_u32(smem));
                        const int rows = zhi - zlo;
                        for (int idx = lane; idx < rows * 16; idx += 32) {
                            const int m = idx / (rows * 8);
                            const int rem = idx - m * rows * 8;
                            *reinterpret_cast<uint4*>(st + m * 8192 + (zlo + rem / 8) * 128 + (rem % 8) * 16) =
                                make_uint4(0, 0, 0, 0);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                    }
                    if (lane == 0) {
                        const uint32_t st = st_addr;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            tc_mma(tmem_o + c * N, sw128_desc(st + kk * 2048, 8192, 1024),
                                   sw32_desc(pb_addr + h * N * 128 + kk * 512, 2048, 256), idesc_o,
                                   (j > 0 || h > 0 || kk > 0) ? 1u : 0u);
                    }
                    release(sl);
                }
                // Row sums: P read as a 128-row A operand (rows >= N fall on the next shared
                // memory region and only produce unused TMEM lanes) times a 64 x 16 block of ones.
                if (lane == 0) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc_mma(tmem_l, sw32_desc(pb_addr + h * N * 128 + kk * 512, 2048, 256),
                               sw128_desc(ones_addr + kk * 32, 16, 1024), idesc_l,
                               (j > 0 || h > 0 || kk > 0) ? 1u : 0u);
                }
                __syncwarp();
            }
            if (!ok) break;
            if (lane == 0) tc_commit(p_free + (j & 1));
            __syncwarp();
        }
        // Drain our MMAs before TMEM is released.
        if (lane == 0) {
            tc_commit(drain);
            const unsigned long long t_start = globaltimer();
            while (!mbar_try_wait(drain, 0) && globaltimer() - t_start < p.wait_ns) {
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax warps 0-7
        // Thread = key lane kl of the tile; warps w and w + 4 share TMEM lanes 32 (w mod 4) ..
        // and take alternate 16-column groups of S^T (half 0: groups 0, 2, ..; half 1: 1, 3, ..).
        const float sl2 = p.scale * kLog2e;
        const int kl = tid & 127;
        const int half = tid >> 7;
        const bool plain = (p.causal == 0 && p.window == 0);
        // A key inside every row's range [max lo, min hi] needs no test per row: with a window
        // or the causal switch only a few keys (the window's first, the block's own) fall
        // outside it, and the per-row test (two shared-memory reads per score) made the
        // masked softmax several times slower than the plain one.
        int lo_all = -(1 << 30), hi_all = (1 << 30);
        if (!plain) {
            for (int r = 0; r < N; ++r) {
                lo_all = max(lo_all, lo_s[r]);
                hi_all = min(hi_all, hi_s[r]);
            }
        }
        // P^T is MN-major with a 32-byte swizzle: per key half, 16-row groups (atoms) of
        // 2048 B = 8 key groups x (8 keys x 32 B); this key lane owns one 32-byte row of
        // every atom, the two 16-byte halves swapped for keys 4-7 of a group.
        const int pr = kl & 7;
        uint8_t* prow0 = p_s + (kl >> 6) * (N * 128) + ((kl & 63) >> 3) * 256 + pr * 32;
        const int pswz0 = (0 ^ (pr >> 2)) << 4;
        const int pswz1 = (1 ^ (pr >> 2)) << 4;
        bool ok = true;
        // One thread waits on the mbarrier; the named barrier makes the outcome
        // uniform across the 256 softmax threads (so none is left at a barrier).
        auto group_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
            bool got = true;
            if (tid == 0) got = ring_wait(bar, parity, abort_flag, p.err, p.wait_ns);
            return !named_bar_or_256(!got);
        };

        // Iteration j = -1 is a dry run over fully masked scores while the first K tile is
        // in flight: it executes the instructions of a real tile, the row-max path
        // included, without touching a barrier or P^T (whose buffers may hold the first
        // tile's extra K stages), so the first real tile does not wait on instruction
        // fetches from a memory system busy with K/V traffic. It reads the O^T columns
        // (not written before p_full) and leaves m = -inf and alpha = 0.
        for (int j = (ntiles > 0 ? -1 : 0); j < ntiles && ok; ++j) {
            const bool dry = j < 0;
            const uint32_t sb = (dry ? tmem_o : tmem_s + (uint32_t)(j & 1) * N) + lane_base;
            if (!dry) {
                if (!group_wait(s_full + (j & 1), (uint32_t)((j >> 1) & 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
            const int key = t0 + j * kTileKeys + kl;
            const bool kvalid = !dry && key >= ch.kb && key < ch.ke;
            const bool allvis = plain || (key >= lo_all && key <= hi_all);
            // masked, log2-scaled score of column col from raw S^T bits
            auto score = [&](uint32_t raw, int col) -> float {
                bool vis = kvalid;
                if (!allvis) vis = vis && key >= lo_s[col] && key <= hi_s[col];
                return vis ? u2f(raw) * sl2 : -INFINITY;
            };
            // Every column of this key lane visible (all but the chunk's edge keys and the
            // window's or the block's own few): no selects, and the scale folds into one FMA.
            // The running maxima are then finite, since pass 1 raises any -inf one.
            // (the dry run sends half of the warps down each path, so both are fetched)
            const bool open = dry ? (half == 0) : (kvalid && allvis);
            // pass 1: does any score exceed the running max by more than the threshold? On
            // the first tile every running max is -inf, so the answer is yes without looking.
            bool need = false;
#pragma unroll 1
            for (int q = half; q < (j == 0 ? 0 : NQ); q += 2) {
                float mv[16];
                load_row16(m_s + q * 16, mv);
                uint32_t r16[16];
                load16(sb + q * 16, r16);
                if (open) {
#pragma unroll
                    for (int u = 0; u < 16; ++u) need |= fmaf(u2f(r16[u]), sl2, -mv[u]) > kRescaleThresh;
                } else {
#pragma unroll
                    for (int u = 0; u < 16; ++u) need |= score(r16[u], q * 16 + u) > mv[u] + kRescaleThresh;
                }
            }
            need = named_bar_or_256(need || dry || j == 0);
            if (need) {
                // new row maxima: each warp's column maxima (transposing shuffle reduction,
                // one column per lane), then the maximum over the 4 warps of the column's half
#pragma unroll 1
                for (int q = half; q < NQ; q += 2) {
                    uint32_t r16[16];
                    load16(sb + q * 16, r16);
                    float v[16];
#pragma unroll
                    for (int u = 0; u < 16; ++u) v[u] = score(r16[u], q * 16 + u);
                    const float mx = transpose_max16(v, lane);
                    if (lane < 16) red[(warp & 3) * N + q * 16 + lane] = mx;
                }
                named_bar_sync_256();
                if (tid < N) {
                    const float mo = m_s[tid];
                    const float mn =
                        fmaxf(fmaxf(mo, fmaxf(red[tid], red[N + tid])), fmaxf(red[2 * N + tid], red[3 * N + tid]));
                    m_s[tid] = mn;
                    a_s[tid] = (mo == -INFINITY) ? 0.f : ex2(mo - mn);
                }
                named_bar_sync_256();
            }
            // O^T and l^T hold tile j-1 once its PV has completed: only a rescale waits for it.
            // P^T buffer j mod 2 is free once PV(j-2) has completed. (p_free[b] completes once
            // per two tiles and every phase is waited for in order.)
            if (j > 0 && need) {
                if (!group_wait(p_free + ((j - 1) & 1), (uint32_t)(((j - 1) >> 1) & 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                {
#pragma unroll 1
                    for (int cq = half; cq < VC * NQ; cq += 2) {
                        const int c = cq / NQ, q = cq % NQ;
                        uint32_t r16[16];
                        const uint32_t ta = tmem_o + c * N + lane_base + q * 16;
                        load16(ta, r16);
                        float av[16];
                        load_row16(a_s + q * 16, av);
#pragma unroll
                        for (int u = 0; u < 16; ++u) r16[u] = f2u(u2f(r16[u]) * av[u]);
                        tmem_st16(ta, r16);
                    }
                    if (half == 0) {
                        // l^T: this thread's lane is row tid
                        uint32_t r16[16];
                        load16(tmem_l + lane_base, r16);
                        const float a = tid < N ? a_s[tid] : 1.f;
#pragma unroll
                        for (int u = 0; u < 16; ++u) r16[u] = f2u(u2f(r16[u]) * a);
                        tmem_st16(tmem_l + lane_base, r16);
                    }
                    tmem_st_wait();
                }
            }
            if (j > 1) {
                if (!group_wait(p_free + (j & 1), (uint32_t)(((j - 2) >> 1) & 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
            // pass 2: P = exp2(s - m), bf16 pairs, into P^T buffer j mod 2
            uint8_t* prow = prow0 + (j & 1) * Lay::kPBytes;
#pragma unroll 1
            for (int q = half; q < NQ; q += 2) {
                // row maxima into registers first: the P^T stores below must not be ordered
                // against these loads (both are shared-memory accesses the compiler cannot separate)
                float mv[16];
                load_row16(m_s + q * 16, mv);
                uint32_t r16[16];
                load16(sb + q * 16, r16);
                float e[16];
                if (open) {
#pragma unroll
                    for (int u = 0; u < 16; ++u) e[u] = ex2(fmaf(u2f(r16[u]), sl2, -mv[u]));
                } else {
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        const float sv = score(r16[u], q * 16 + u);
                        e[u] = (sv == -INFINITY) ? 0.f : ex2(sv - mv[u]);
                    }
                }
                uint32_t pk[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const __nv_bfloat162 h2 = __floats2bfloat162_rn(e[2 * u], e[2 * u + 1]);
                    pk[u] = *reinterpret_cast<const uint32_t*>(&h2);
                }
                if (!dry) {
                    uint8_t* dst = prow + q * 2048;
                    *reinterpret_cast<uint4*>(dst + pswz0) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    *reinterpret_cast<uint4*>(dst + pswz1) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                }
            }
            if (!dry) {
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(p_full);
            }
        }
        bool good = ok && ntiles > 0;
        if (good) good = group_wait(p_free + ((ntiles - 1) & 1), (uint32_t)(((ntiles - 1) >> 1) & 1));
        role_ok = good;
    }

    // ---------------------------------------------------------------- epilogue (warps 0-7)
    // The softmax warps 0-7 do the read-out: TMEM lanes 32 (w mod 4) .. +31 are open to
    // warp w, so warps w and w + 4 take alternate 128-dim chunks of O^T. The output tile (R rows x D, bf16 for the final output,
    // fp32 for a split's partial) is assembled row-major over Q, P and the ring (all
    // free once the last PV has completed) and written with bulk asynchronous copies:
    // for each block position i the Gc heads' rows are contiguous in global memory.
    // Every role's outcome, the producers' and the MMA warp's included: an aborted producer
    // may still drain copies into the ring, which the read-out below reuses.
    const bool any_failed = __syncthreads_or(!role_ok) != 0;
    if (warp < 8) {
        const bool have_o = !any_failed && ntiles > 0;
        tc_fence_after();
        const int64_t part_base = (slot0 + c_split) * rstride + rbias;
        const bool final_out = (p.splits == 1);
        if (warp < 4) {
            // row tid's sum sits in TMEM lane tid of l^T
            uint32_t l16[16];
            if (have_o) {
                load16(tmem_l + lane_base, l16);
            } else {
#pragma unroll
                for (int u = 0; u < 16; ++u) l16[u] = 0u;
            }
            const float tot = u2f(l16[0]);
            if (tid < N) a_s[tid] = tot > 0.f ? 1.f / tot : 0.f;
            if (tid < R) {
                const float lse_v = tot > 0.f ? (m_s[tid] + __log2f(tot)) * kLn2 : -INFINITY;
                if (final_out) {
                    if (p.lse) p.lse[orow_s[tid]] = lse_v;
                } else {
                    p.part_lse[part_base + orow_s[tid]] = lse_v;
                }
            }
        }
        named_bar_sync_256();
        uint8_t* tile_o = smem + Lay::kQOff;
        float* tile_f = reinterpret_cast<float*>(tile_o);
        __nv_bfloat16* tile_b = reinterpret_cast<__nv_bfloat16*>(tile_o);
        const int dl = (warp & 3) * 32 + lane;  // dim within a 128-dim chunk = TMEM lane
#pragma unroll 1
        for (int c = warp >> 2; c < VC; c += 2) {
#pragma unroll 1
            for (int q = 0; q < NQ; ++q) {
                float iv[16];
                load_row16(a_s + q * 16, iv);
                uint32_t r16[16];
                if (have_o) {
                    load16(tmem_o + c * N + lane_base + q * 16, r16);
                } else {
#pragma unroll
                    for (int u = 0; u < 16; ++u) r16[u] = 0u;
                }
                const int d = c * 128 + dl;
                if (final_out) {
#pragma unroll
                    for (int u = 0; u < 16; ++u)
                        if (q * 16 + u < R) tile_b[(q * 16 + u) * D + d] = __float2bfloat16_rn(u2f(r16[u]) * iv[u]);
                } else {
#pragma unroll
                    for (int u = 0; u < 16; ++u)
                        if (q * 16 + u < R) tile_f[(q * 16 + u) * D + d] = u2f(r16[u]) * iv[u];
                }
            }
        }
        fence_proxy_async_smem();
        named_bar_sync_256();
        if (tid == 0) {
            const uint32_t esz = final_out ? 2u : 4u;
            const uint32_t run = (uint32_t)x.Gc * D * esz;  // bytes of one block position's Gc rows
            for (int i = 0; i < T; ++i) {
                const int64_t row0 = (int64_t)(b * T + i) * p.Hq + h0;
                void* dst = final_out ? static_cast<void*>(static_cast<__nv_bfloat16*>(p.out) + row0 * D)
                                      : static_cast<void*>(p.part_out + (part_base + row0) * D);
                bulk_store_global(dst, tile_o + (size_t)i * run, run);
            }
            bulk_commit_group();
            if (x.fused)
                bulk_wait_all_0();   // the partial must be in global memory before the arrival below
            else
                bulk_wait_read_0();  // the tile must stay in shared memory until the copies have read it
        }
    }

    if (x.fused) {
        // ------------------------------------------------------------ split combine
        // The splits CTAs of this (request, row group) are co-resident (cooperative
        // launch). Each publishes its partial (the bulk copy above, the lse stores
        // before it), arrives on the group's counter and waits for all of them; then
        // all 12 warps of each combine a slice of the group's R x D outputs (one float4
        // column per thread: a global_verify slice of 288 float4s takes one round of loads):
        //   m = max_c lse_c, w_c = exp(lse_c - m), out = sum_c w_c o_c / sum_c w_c,
        //   lse = m + log(sum_c w_c)
        // The last CTA to finish resets the two counters to zero for the next call.
        __threadfence();
        __syncthreads();
        int32_t* cnt = p.counters + 2 * (b * gridDim.y + blockIdx.y);
        bool arrived = true;
        if (tid == 0) {
            asm volatile("fence.proxy.async.global;" ::: "memory");
            __threadfence();
            atomicAdd(cnt, 1);
            const unsigned long long t_start = globaltimer();
            while (ld_acquire_gpu(cnt) < n_split) {
                if (globaltimer() - t_start > p.wait_ns) {
                    raise_error(p.err, DFLASH_DEVERR_TIMEOUT);
                    arrived = false;
                    break;
                }
            }
        }
        arrived = __syncthreads_or(!arrived) == 0;
        if (arrived) {
            const int total = R * D;
            const int per = ((total + n_split - 1) / n_split + 3) & ~3;
            const int e0 = c_split * per;
            const int e1 = min(total, e0 + per);
            if (e0 < e1) {
                const int r0 = e0 / D;
                const int nr = (e1 - 1) / D - r0 + 1;
                float* w_sm = reinterpret_cast<float*>(smem + Lay::kQOff);  // [nr][splits] weights
                float* r_sm = w_sm + nr * n_split;                           // [nr][2]: 1/sum, lse
                for (int rr = warp; rr < nr; rr += kThreads / 32) {
                    const int64_t orow = orow_s[r0 + rr];
                    float m = -INFINITY;
                    const float* lse_row = p.part_lse + slot0 * rstride + rbias + orow;
                    for (int c = lane; c < n_split; c += 32) m = fmaxf(m, __ldcg(lse_row + c * rstride));
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
                    float tot = 0.f;
                    for (int c = lane; c < n_split; c += 32) {
                        const float l = __ldcg(lse_row + c * rstride);
                        const float w = (l == -INFINITY) ? 0.f : expf(l - m);
                        w_sm[rr * n_split + c] = w;
                        tot += w;
                    }
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
                    if (lane == 0) {
                        const bool empty_row = (m == -INFINITY) || !(tot > 0.f);
                        r_sm[2 * rr] = empty_row ? 0.f : 1.f / tot;
                        r_sm[2 * rr + 1] = empty_row ? -INFINITY : m + logf(tot);
                    }
                }
                __syncthreads();
                for (int e = e0 + tid * 4; e < e1; e += kThreads * 4) {
                    const int r = e / D, d = e - r * D, rr = r - r0;
                    const float inv = r_sm[2 * rr];
                    const int64_t orow = orow_s[r];
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (inv > 0.f) {
                        const float* base = p.part_out + (slot0 * rstride + rbias + orow) * D + d;
                        const int64_t cstride = rstride * D;
                        for (int c0 = 0; c0 < n_split; c0 += 16) {
                            float4 v[16];
#pragma unroll
                            for (int k = 0; k < 16; ++k)
                                v[k] = c0 + k < n_split
                                           ? __ldcg(reinterpret_cast<const float4*>(base + (c0 + k) * cstride))
                                           : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                            for (int k = 0; k < 16; ++k) {
                                const float w = c0 + k < n_split ? w_sm[rr * n_split + c0 + k] : 0.f;
                                acc.x = fmaf(w, v[k].x, acc.x);
                                acc.y = fmaf(w, v[k].y, acc.y);
                                acc.z = fmaf(w, v[k].z, acc.z);
                                acc.w = fmaf(w, v[k].w, acc.w);
                            }
                        }
                    }
                    const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
                    const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
                    uint2 pk;
                    pk.x = *reinterpret_cast<const uint32_t*>(&lo);
                    pk.y = *reinterpret_cast<const uint32_t*>(&hi);
                    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + orow * D + d) = pk;
                }
                // a row's lse is written by the CTA whose slice holds the row's first element
                for (int rr = tid; rr < nr; rr += kThreads)
                    if ((r0 + rr) * D >= e0 && p.lse) p.lse[orow_s[r0 + rr]] = r_sm[2 * rr + 1];
            }
        }
        __syncthreads();
        if (tid == 0) {
            // A CTA whose arrival wait ran out still counts itself here, so a group whose
            // counters held stale arrivals (every CTA times out) is reset like any other.
            __threadfence();
            if (atomicAdd(cnt + 1, 1) == n_split - 1) {
                // every CTA of the group has passed (or given up) the arrival wait and read its slice
                atomicExch(cnt, 0);
                atomicExch(cnt + 1, 0);
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, Lay::kTmemCols);
    }
}

// ----------------------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
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

// Query heads per CTA: the largest divisor of G whose packed rows fit kMaxRows.
int choose_gc(int G, int T)
{
    for (int gc = G; gc >= 1; --gc)
        if (G % gc == 0 && gc * T <= kMaxRows) return gc;
    return 0;
}

template <int D, int N>
cudaError_t launch_dn(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p,
                      const TcExtra& x, cudaStream_t stream, bool* combined)
{
    using Lay = TcLayout<D, N>;
    auto kern = tc_attn_kernel<D, N>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kAlloc);
    if (e != cudaSuccess) return e;
    dim3 grid(p.splits, p.Hkv * x.n_rg, p.balanced ? 1 : p.B);
    TcExtra xx = x;
    bool coop = false;
    if (p.balanced && !p.counters) return cudaErrorInvalidValue;  // the balanced plan combines in-kernel
    if (p.splits > 1 && p.counters) {
        // fused combine: every CTA of the grid must be resident at once
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, Lay::kAlloc) == cudaSuccess &&
            (int64_t)grid.x * grid.y * grid.z <= (int64_t)per_sm * device_sm_count() &&
            (int64_t)grid.y * grid.z <= DFLASH_MAX_COMBINE_GROUPS)
            coop = true;
    }
    if (p.balanced && !coop) return cudaErrorInvalidConfiguration;  // its partials need the in-kernel combine
    xx.fused = coop ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Lay::kAlloc;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = coop ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, p, xx);
    if (coop && e == cudaErrorCooperativeLaunchTooLarge && !p.balanced) {
        (void)cudaGetLastError();  // not resident after all: plain launch, separate combine
        coop = false;
        xx.fused = 0;
        cfg.numAttrs = 0;
        e = cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, p, xx);
    }
    *combined = (e == cudaSuccess) && coop;
    return e;
}

// Grid size and whether launch_dn would combine in-kernel (same rule, no launch).
template <int D, int N>
cudaError_t grid_info_dn(const AttnParams& p, const TcExtra& x, int64_t* ctas, bool* fused)
{
    using Lay = TcLayout<D, N>;
    auto kern = tc_attn_kernel<D, N>;
    const int64_t gx = p.splits, gy = (int64_t)p.Hkv * x.n_rg, gz = p.balanced ? 1 : p.B;
    *ctas = gx * gy * gz;
    *fused = false;
    if (p.splits > 1) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kAlloc);
        if (e != cudaSuccess) return e;
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, Lay::kAlloc);
        if (e != cudaSuccess) return e;
        *fused = *ctas <= (int64_t)per_sm * device_sm_count() && gy * gz <= DFLASH_MAX_COMBINE_GROUPS;
    }
    return cudaSuccess;
}

template <int D>
cudaError_t grid_info_d(int n, const AttnParams& p, const TcExtra& x, int64_t* ctas, bool* fused)
{
    switch (n) {
    case 16: return grid_info_dn<D, 16>(p, x, ctas, fused);
    case 32: return grid_info_dn<D, 32>(p, x, ctas, fused);
    case 48: return grid_info_dn<D, 48>(p, x, ctas, fused);
    case 64: return grid_info_dn<D, 64>(p, x, ctas, fused);
    case 80: return grid_info_dn<D, 80>(p, x, ctas, fused);
    }
    return cudaErrorNotSupported;
}

template <int D>
cudaError_t launch_d(int n, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p,
                     const TcExtra& x, cudaStream_t stream, bool* combined)
{
    switch (n) {
    case 16: return launch_dn<D, 16>(tq, tk, tv, p, x, stream, combined);
    case 32: return launch_dn<D, 32>(tq, tk, tv, p, x, stream, combined);
    case 48: return launch_dn<D, 48>(tq, tk, tv, p, x, stream, combined);
    case 64: return launch_dn<D, 64>(tq, tk, tv, p, x, stream, combined);
    case 80: return launch_dn<D, 80>(tq, tk, tv, p, x, stream, combined);
    }
    return cudaErrorNotSupported;
}

}  // namespace

bool tc_supports(const AttnParams& p)
{
    if (p.dtype != DFLASH_BF16) return false;
    if (p.D != 128 && p.D != 256 && p.D != 512) return false;
    if (p.page_size != 16 && p.page_size != 32 && p.page_size != 64) return false;
    if (choose_gc(p.G, p.T) == 0) return false;
    if (p.sh % 8 || p.ss % 8 || p.sp % 8) return false;
    return true;  // the tensor-map encoder is resolved from the driver at launch
}

int tc_row_groups(const AttnParams& p)
{
    const int gc = choose_gc(p.G, p.T);
    return gc > 0 ? p.G / gc : 0;
}

int tc_ctas_per_split(const AttnParams& p)
{
    const int gc = choose_gc(p.G, p.T);
    return gc > 0 ? p.B * p.Hkv * (p.G / gc) : 0;
}

cudaError_t tc_grid_info(const AttnParams& p, int64_t* ctas, bool* fused)
{
    if (!tc_supports(p)) return cudaErrorNotSupported;
    TcExtra x;
    x.fused = 0;
    x.Gc = choose_gc(p.G, p.T);
    x.n_rg = p.G / x.Gc;
    x.R = x.Gc * p.T;
    const int n = ((x.R + 15) / 16) * 16;
    switch (p.D) {
    case 128: return grid_info_d<128>(n, p, x, ctas, fused);
    case 256: return grid_info_d<256>(n, p, x, ctas, fused);
    case 512: return grid_info_d<512>(n, p, x, ctas, fused);
    }
    return cudaErrorNotSupported;
}

cudaError_t launch_tc_attn(const AttnParams& p, cudaStream_t stream)
{
    if (!tc_supports(p)) return cudaErrorNotSupported;
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    TcExtra x;
    x.fused = 0;
    x.Gc = choose_gc(p.G, p.T);
    x.n_rg = p.G / x.Gc;
    x.R = x.Gc * p.T;
    const int n = ((x.R + 15) / 16) * 16;

    CUtensorMap tq, tk, tv;
    {
        const cuuint64_t dims[3] = {(cuuint64_t)p.D, (cuuint64_t)p.Hq, (cuuint64_t)p.B * p.T};
        const cuuint64_t strides[2] = {(cuuint64_t)p.D * 2, (cuuint64_t)p.Hq * p.D * 2};
        const cuuint32_t box[3] = {64, (cuuint32_t)x.Gc, (cuuint32_t)p.T};
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
    bool combined = false;
    switch (p.D) {
    case 128: e = launch_d<128>(n, tq, tk, tv, p, x, stream, &combined); break;
    case 256: e = launch_d<256>(n, tq, tk, tv, p, x, stream, &combined); break;
    case 512: e = launch_d<512>(n, tq, tk, tv, p, x, stream, &combined); break;
    default: e = cudaErrorNotSupported;
    }
    if (e != cudaSuccess || p.splits == 1 || combined) return e;
    return launch_combine(p.part_out, p.part_lse, p.splits, (int64_t)p.B * p.T * p.Hq, p.D, p.dtype, p.out, p.lse,
                          stream);
}

}  // namespace dflash
