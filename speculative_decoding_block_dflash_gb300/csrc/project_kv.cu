// Context K/V projection for the draft pass, fused with the paged-cache write.
//
// The drafter's cross-attention reads context K/V computed from the target's hidden states
// (kenforever1 "dflash-gemma4-31b-notes", the code lines under "why non-causal attention";
// the vLLM DFlash review's risk list names this precompute as a bare linear layer). For
// every token t with cache slot s_t >= 0:
//   K[s_t, h, d] = bf16( sum_k hidden[t, k] * W_k[h*D + d, k] )   (fp32 accumulation)
//   V[s_t, h, d] = bf16( sum_k hidden[t, k] * W_v[h*D + d, k] )
// where slot s maps to page s / page_size, position s % page_size.
//
// The grid is persistent and made of CTA pairs (clusters of 2 sharing each tcgen05 MMA,
// cta_group::2), one pair per cluster slot the device holds at once. A pair walks output tiles
// of 256 tokens x 256 features (of K or of V), the tile index t = m * (2 * n_half) + nt
// (feature tiles fastest, so that the pairs running at once share their hidden rows and the
// whole weight set stays in L2). CTA r of a pair owns tokens [128 r, 128 r + 128) of the tile.
// Per 64-wide slice of the hidden dimension each CTA lands 16 KB of its hidden rows and 16 KB
// of weight rows (features [128 r, 128 r + 128) of the tile), and the even CTA issues one
// M=256 N=256 K=16 MMA per 16-wide step, taking the B operand's halves from both CTAs. Each
// CTA's TMEM receives its 128 token rows x 256 features, in one of two accumulators (256
// columns each) that alternate between tiles, so the epilogue of a tile runs while the MMAs
// of the next one do. (Against a single-CTA 256 x 256 tile in one 512-column accumulator, which
// lands the same bytes per flop: 244 -> 235 us on the 8192-token workload; a 256 x 512 pair
// tile, which lands a quarter fewer bytes per flop but fills TMEM with one accumulator: 239 us.)
// Warp roles per CTA:
//   warp 0     TMA producer: the CTA's two boxes of a stage into a 6-stage ring of 32 KB,
//              counted on the even CTA's barrier;
//   warp 1     MMA issuer (even CTA);
//   warps 2-9  epilogue: two warps per TMEM lane quarter (one per 128-feature half), thread =
//              token row, 16 columns at a time, bf16 pack and two 16-byte stores into the
//              token's cache slot.
//
// When the tiles leave a partial last round (tiles mod pairs = rem, 2 * rem <= pairs) and the
// caller gives a workspace, the last rem tiles are split in two along the hidden dimension,
// the halves running on 2 * rem pairs of the last round. For each CTA rank, the first half to
// reach its epilogue (an arrival counter) writes its fp32 accumulator rows to the workspace and
// raises a flag; the other waits for the flag (bounded), adds the partial to its own
// accumulator and writes the bf16 rows. Both halves of a tile are in the same round, so the
// waiter only waits for a CTA that is already writing. Rows past the token count, hidden
// columns past H and feature rows past N are zero-filled by the tensor copies. Every wait is
// bounded (DFLASH_DEVERR_TIMEOUT, the kernel returns), and both CTAs of a pair meet at a
// cluster barrier before TMEM is freed.
#include <algorithm>
#include <mutex>

#include "tc_ptx.cuh"

namespace dflash {
namespace {

using namespace ptx;

constexpr int kBM = 256;      // tokens per pair tile (128 per CTA)
constexpr int kRows = 128;    // tokens per CTA
constexpr int kBN = 256;      // features per pair tile (the MMA's N; 128 of the weight rows per CTA)
constexpr int kBK = 64;       // hidden elements per stage (128 bytes: one swizzle row)
constexpr int kStages = 6;
constexpr int kABytes = kRows * kBK * 2;        // this CTA's 128 hidden rows
constexpr int kBBytes = (kBN / 2) * kBK * 2;    // this CTA's half of the weight rows
constexpr int kStageBytes = kABytes + kBBytes;  // 32 KB
constexpr int kTmaWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 32 * (2 + kEpiWarps);
constexpr int kTmemCols = 2 * kBN;  // two accumulators: tile i in columns [256 (i mod 2), +256)
constexpr int kBarOff = kStages * kStageBytes;
constexpr int kNumBars = 2 * kStages + 5;  // full, empty, acc_full[2], acc_empty[2], drain
constexpr int kMiscOff = kBarOff + kNumBars * 8;
constexpr int kSmemUsed = kMiscOff + 16;
constexpr int kAlloc = kSmemUsed + 1024;  // the ring is aligned up to 1024 bytes (swizzle atoms)
static_assert(kAlloc <= 227 * 1024, "shared memory");
static_assert(kStageBytes % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
constexpr size_t kProjectSyncBytes = 8192;  // two int32 per (split tile, CTA rank), a fixed block
constexpr unsigned long long kCopyGraceNs = 200000ull;  // after an abort: time for copies in flight to land

struct ProjParams {
    const int32_t* slot_mapping;
    __nv_bfloat16* k_cache;
    __nv_bfloat16* v_cache;
    uint32_t* err;
    int32_t L, H, N, D, page_size;
    int32_t n_half;  // feature tiles of one projection: ceil(N / kBN)
    int32_t tiles;   // ceil(L / kBM) * 2 * n_half
    int32_t full_tiles;  // tiles computed whole; tiles [full_tiles, tiles) are split in two
    int32_t units;       // full_tiles + 2 * (tiles - full_tiles): the persistent loop's work units
    float* partial;      // [tiles - full_tiles][2 ranks][kRows][kBN] fp32: the first half's accumulator rows
    int32_t* sync;       // [tiles - full_tiles][2 ranks][2]: arrivals, partial-ready flag (zero between calls)
    int64_t total_slots;
    int64_t sp, ss, sh;
};

// Work unit u of the persistent loop: a whole tile, or one half (along the hidden dimension) of
// a split tile.
struct Unit {
    int tile, kb0, kb1, slot, half;  // slot < 0: a whole tile
};

__device__ __forceinline__ Unit unit_of(const ProjParams& p, int u, int KB)
{
    Unit w;
    if (u < p.full_tiles) {
        w.tile = u;
        w.kb0 = 0;
        w.kb1 = KB;
        w.slot = -1;
        w.half = 0;
    } else {
        const int v = u - p.full_tiles;
        w.slot = v >> 1;
        w.half = v & 1;
        w.tile = p.full_tiles + w.slot;
        w.kb0 = w.half ? KB / 2 : 0;
        w.kb1 = w.half ? KB : KB / 2;
    }
    return w;
}

__device__ __forceinline__ int ld_acquire_gpu(const int32_t* ptr)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
    return v;
}

// A pair's 2-D tensor copy into this CTA's shared memory, its bytes counted on the mbarrier at
// cluster address mbar_cluster (the even CTA's).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, uint32_t mbar_cluster, int c0,
                                                 int c1)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(mbar_cluster), "r"(c0), "r"(c1)
        : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo, uint32_t hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(lo), __uint_as_float(hi));
    return *reinterpret_cast<const uint32_t*>(&v);
}

// 16 fp32 accumulator columns -> 16 bf16 at dst (16-byte aligned).
__device__ __forceinline__ void store16(__nv_bfloat16* dst, const uint32_t (&r)[16])
{
    uint4 a, b;
    a.x = pack_bf16x2(r[0], r[1]);
    a.y = pack_bf16x2(r[2], r[3]);
    a.z = pack_bf16x2(r[4], r[5]);
    a.w = pack_bf16x2(r[6], r[7]);
    b.x = pack_bf16x2(r[8], r[9]);
    b.y = pack_bf16x2(r[10], r[11]);
    b.z = pack_bf16x2(r[12], r[13]);
    b.w = pack_bf16x2(r[14], r[15]);
    reinterpret_cast<uint4*>(dst)[0] = a;
    reinterpret_cast<uint4*>(dst)[1] = b;
}

__global__ void __launch_bounds__(kThreads, 1)
    project_kv_kernel(const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_wk,
                      const __grid_constant__ CUtensorMap tm_wv, const ProjParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ring = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);
    uint64_t* full = bars;                    // [kStages] TMA -> MMA: both CTAs' boxes of the stage landed (even CTA)
    uint64_t* empty = bars + kStages;         // [kStages] MMA -> TMA: stage consumed (both CTAs)
    uint64_t* acc_full = bars + 2 * kStages;  // [2] MMA -> epilogue: accumulator b holds a finished tile (both CTAs)
    uint64_t* acc_empty = acc_full + 2;       // [2] epilogues -> MMA: both CTAs have read accumulator b out (even CTA)
    uint64_t* drain = acc_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kMiscOff + 4);
    __shared__ int ticket_s;  // arrival order of this CTA's half of a split tile
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = (rank == 0);
    const int pair_id = blockIdx.x >> 1;
    const int npairs = gridDim.x >> 1;
    const int KB = (p.H + kBK - 1) / kBK;
    const int row_tiles = 2 * p.n_half;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(acc_full + b, 1);
            mbar_init(acc_empty + b, 2 * kEpiWarps);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kMmaWarp) {
        tmem_alloc2(tmem_slot, kTmemCols);
        tmem_relinquish2();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // the peer's barriers are initialised before any remote arrival
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kTmaWarp) {
        // ------------------------------------------------------------ TMA producer (both CTAs)
        const uint32_t full0 = mapa_shared(smem_u32(full), 0);
        bool ok = true;
        uint32_t issued_par[kStages];
#pragma unroll
        for (int s = 0; s < kStages; ++s) issued_par[s] = 2;  // 2 = nothing issued
        int seq = 0;
        for (int u = pair_id; u < p.units && ok; u += npairs) {
            const Unit w = unit_of(p, u, KB);
            const int m = w.tile / row_tiles;
            const int nt = w.tile - m * row_tiles;
            const bool is_v = nt >= p.n_half;
            const int col0 = (is_v ? nt - p.n_half : nt) * kBN;
            const CUtensorMap* tw = is_v ? &tm_wv : &tm_wk;
            for (int kb = w.kb0; kb < w.kb1; ++kb, ++seq) {
                const int s = seq % kStages;
                const uint32_t ph = (uint32_t)(seq / kStages) & 1u;
                // the even CTA's MMA commit frees the slot in both CTAs
                if (lane == 0) ok = ring_wait_cluster(empty + s, ph ^ 1u, abort_flag, p.err, kTimeoutNs);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                if (lane == 0) {
                    uint8_t* st = ring + s * kStageBytes;
                    // the even CTA's barrier counts both CTAs' bytes of the stage
                    if (leader) mbar_expect_tx(full + s, 2u * kStageBytes);
                    const uint32_t fb = full0 + (uint32_t)(s * 8);
                    tma_load_2d_pair(st, &tm_h, fb, kb * kBK, m * kBM + (int)rank * kRows);
                    tma_load_2d_pair(st + kABytes, tw, fb, kb * kBK, col0 + (int)rank * (kBN / 2));
                    issued_par[s] = ph;
                }
                __syncwarp();
            }
        }
        if (lane == 0 && !ok) {
            // Copies of ours may still be landing. The even CTA waits for the stages it armed;
            // both CTAs then give copies in flight a grace period (the odd CTA's copies count on
            // the even CTA's barriers, which it cannot wait for) before this CTA may leave.
            if (leader) {
                for (int s = 0; s < kStages; ++s) {
                    if (issued_par[s] > 1) continue;
                    const unsigned long long t_start = globaltimer();
                    while (!mbar_try_wait_cluster(full + s, issued_par[s]) && globaltimer() - t_start < kTimeoutNs) {
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
        if (leader) {
            constexpr uint32_t idesc = make_idesc(2 * kRows, kBN, 0, 0);  // M = 256 over the pair, K-major A and B
            const uint32_t ring_addr = smem_u32(ring);
            bool ok = true;
            int seq = 0;
            int i = 0;
            for (int u = pair_id; u < p.units && ok; u += npairs, ++i) {
                const Unit w = unit_of(p, u, KB);
                const int ab = i & 1;  // accumulator of this tile
                const uint32_t acc = tmem + (uint32_t)(ab * kBN);
                // both CTAs' epilogues have read out the tile two back (accumulator ab's last use)
                if (lane == 0)
                    ok = ring_wait_cluster(acc_empty + ab, ((uint32_t)(i >> 1) & 1u) ^ 1u, abort_flag, p.err,
                                           kTimeoutNs);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                tc_fence_after();
                for (int kb = w.kb0; kb < w.kb1; ++kb, ++seq) {
                    const int s = seq % kStages;
                    const uint32_t ph = (uint32_t)(seq / kStages) & 1u;
                    if (lane == 0) ok = ring_wait_cluster(full + s, ph, abort_flag, p.err, kTimeoutNs);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) break;
                    tc_fence_after();
                    if (lane == 0) {
                        const uint32_t sa = ring_addr + (uint32_t)(s * kStageBytes);
                        const uint32_t sb = sa + kABytes;
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk)
                            tc_mma2(acc, sw128_desc(sa + kk * 32, 16, 1024), sw128_desc(sb + kk * 32, 16, 1024), idesc,
                                    (kb > w.kb0 || kk > 0) ? 1u : 0u);
                        tc_commit2_both(empty + s);
                    }
                    __syncwarp();
                }
                if (!ok) break;
                if (lane == 0) tc_commit2_both(acc_full + ab);
                __syncwarp();
            }
            // our MMAs are complete before either CTA frees TMEM or leaves (they read both CTAs' memory)
            if (lane == 0) {
                tc_commit2_local(drain);
                const unsigned long long t_start = globaltimer();
                while (!mbar_try_wait(drain, 0) && globaltimer() - t_start < kTimeoutNs) {
                }
            }
            __syncwarp();
        }
        // (the odd CTA's MMA warp has no role: the even CTA issues the pair MMAs)
    } else {
        // ------------------------------------------------------------ epilogue (thread = token row)
        const int quarter = warp & 3;      // the TMEM lane quarter this warp may read
        constexpr int kCols = kBN / 2;     // columns per epilogue warp
        const int half = (warp - 2) >> 2;  // 0: features [0, 128) of the tile, 1: [128, 256)
        const int lrow = quarter * 32 + lane;  // row within this CTA's 128
        const uint32_t acc_empty0 = mapa_shared(smem_u32(acc_empty), 0);
        int i = 0;
        for (int u = pair_id; u < p.units; u += npairs, ++i) {
            const Unit w = unit_of(p, u, KB);
            const int m = w.tile / row_tiles;
            const int nt = w.tile - m * row_tiles;
            const bool is_v = nt >= p.n_half;
            const int col0 = (is_v ? nt - p.n_half : nt) * kBN + half * kCols;  // first feature of this half
            const int ncols = max(0, min(kCols, p.N - col0));                     // a multiple of 16
            const int ab = i & 1;
            const uint32_t acc = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(ab * kBN + half * kCols);
            const int row = m * kBM + (int)rank * kRows + lrow;
            __nv_bfloat16* dst = nullptr;  // this token's slot, or none
            if (row < p.L) {
                const int32_t slot = __ldg(p.slot_mapping + row);
                if (slot >= 0) {
                    if ((int64_t)slot < p.total_slots)
                        dst = (is_v ? p.v_cache : p.k_cache) + (int64_t)(slot / p.page_size) * p.sp +
                              (int64_t)(slot % p.page_size) * p.ss;
                    else
                        raise_error(p.err, DFLASH_DEVERR_PAGE_ID);
                }
            }
            // One thread spins on the accumulators (the other epilogue warps sleep at the named
            // barrier, leaving the issue slots to the producer and MMA warps); the barrier's OR
            // gives all 8 warps the wait's outcome, so that they leave together.
            bool got = true;
            if (threadIdx.x == 64)
                got = ring_wait_cluster(acc_full + ab, (uint32_t)(i >> 1) & 1u, abort_flag, p.err, kTimeoutNs);
            const bool ok = !named_bar_or_256(!got);
            if (!ok) break;
            tc_fence_after();
            // a split tile: per CTA rank, the first half to arrive publishes its partial rows,
            // the second adds them
            int role = 0;  // 0: whole tile, 1: publish the partial, 2: add the partial and store
            float* part = nullptr;
            if (w.slot >= 0) {
                int32_t* sync = p.sync + 2 * (2 * w.slot + (int)rank);
                if (threadIdx.x == 64) ticket_s = atomicAdd(sync, 1);
                named_bar_sync_256();  // the 8 epilogue warps
                role = ticket_s == 0 ? 1 : 2;
                part = p.partial + ((int64_t)(2 * w.slot + (int)rank) * kRows + lrow) * kBN + half * kCols;
                if (role == 2) {
                    // wait (bounded) until the first half's partial is visible
                    if (threadIdx.x == 64) {
                        const unsigned long long t_start = globaltimer();
                        int ready = ld_acquire_gpu(sync + 1);
                        while (!ready && globaltimer() - t_start < kTimeoutNs) ready = ld_acquire_gpu(sync + 1);
                        if (!ready) raise_error(p.err, DFLASH_DEVERR_TIMEOUT);
                    }
                    named_bar_sync_256();  // the 8 epilogue warps
                }
            }
            for (int c = 0; c < ncols; c += 32) {
                uint32_t r0[16], r1[16];
                tmem_ld16(acc + c, r0);
                tmem_ld16(acc + c + 16, r1);  // inside this half's 128 columns even when past ncols
                tmem_ld_wait();
                reg_fence16(r0);
                reg_fence16(r1);
                if (role == 1) {
                    float4* pp = reinterpret_cast<float4*>(part + c);
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        pp[v] = make_float4(__uint_as_float(r0[4 * v]), __uint_as_float(r0[4 * v + 1]),
                                            __uint_as_float(r0[4 * v + 2]), __uint_as_float(r0[4 * v + 3]));
                        pp[4 + v] = make_float4(__uint_as_float(r1[4 * v]), __uint_as_float(r1[4 * v + 1]),
                                                __uint_as_float(r1[4 * v + 2]), __uint_as_float(r1[4 * v + 3]));
                    }
                    continue;
                }
                if (role == 2) {
                    const float4* pp = reinterpret_cast<const float4*>(part + c);
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const float4 a = __ldcg(pp + v), b = __ldcg(pp + 4 + v);
                        r0[4 * v] = __float_as_uint(__uint_as_float(r0[4 * v]) + a.x);
                        r0[4 * v + 1] = __float_as_uint(__uint_as_float(r0[4 * v + 1]) + a.y);
                        r0[4 * v + 2] = __float_as_uint(__uint_as_float(r0[4 * v + 2]) + a.z);
                        r0[4 * v + 3] = __float_as_uint(__uint_as_float(r0[4 * v + 3]) + a.w);
                        r1[4 * v] = __float_as_uint(__uint_as_float(r1[4 * v]) + b.x);
                        r1[4 * v + 1] = __float_as_uint(__uint_as_float(r1[4 * v + 1]) + b.y);
                        r1[4 * v + 2] = __float_as_uint(__uint_as_float(r1[4 * v + 2]) + b.z);
                        r1[4 * v + 3] = __float_as_uint(__uint_as_float(r1[4 * v + 3]) + b.w);
                    }
                }
                if (dst) {
                    const int f0 = col0 + c;  // feature of column c: head f / D, dim f % D
                    store16(dst + (int64_t)(f0 / p.D) * p.sh + f0 % p.D, r0);
                    if (c + 16 < ncols) {
                        const int f1 = f0 + 16;
                        store16(dst + (int64_t)(f1 / p.D) * p.sh + f1 % p.D, r1);
                    }
                }
            }
            if (role == 1) {
                // publish: every thread's partial rows are written before the flag is raised
                __threadfence();
                named_bar_sync_256();  // the 8 epilogue warps
                if (threadIdx.x == 64) atomicExch(p.sync + 2 * (2 * w.slot + (int)rank) + 1, 1);
            } else if (role == 2) {
                named_bar_sync_256();  // the 8 epilogue warps
                if (threadIdx.x == 64) {  // both halves are done with this slot: reset it
                    p.sync[2 * (2 * w.slot + (int)rank)] = 0;
                    p.sync[2 * (2 * w.slot + (int)rank) + 1] = 0;
                }
            }
            // this CTA's read-out is done: one arrival per warp on the even CTA's barrier
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(acc_empty0 + (uint32_t)(ab * 8));
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // no CTA leaves while the pair MMAs or the peer may still touch its memory
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc2(tmem, kTmemCols);
    }
}

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

// 2D bf16 map of `rows` rows of `cols` elements (row stride `stride` elements), box 64 x box_rows,
// 128-byte swizzle; out-of-range elements read as zero.
bool encode_2d(EncodeTiledFn enc, CUtensorMap* map, const void* base, int64_t cols, int64_t rows, int64_t stride,
               int box_rows)
{
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)stride * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
    const cuuint32_t es[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Pairs of this kernel the current device holds at once (cached per device).
cudaError_t resident_pairs(int* pairs)
{
    static int cached[64] = {};
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(mu);
    if (cached[dev] == 0) {
        e = cudaFuncSetAttribute(project_kv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAlloc);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kAlloc;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, project_kv_kernel, &cfg);
        if (e != cudaSuccess) return e;
        cached[dev] = n > 0 ? n : 1;
    }
    *pairs = cached[dev];
    return cudaSuccess;
}

}  // namespace

int32_t project_kv_grid(int32_t L, int32_t N)
{
    const int64_t tiles = (int64_t)((L + kBM - 1) / kBM) * 2 * ((N + kBN - 1) / kBN);
    int pairs = 0;
    if (resident_pairs(&pairs) != cudaSuccess) return 0;
    return (int32_t)(2 * std::min<int64_t>(tiles, pairs));
}

size_t project_kv_workspace_bytes()
{
    // the sync block, then the fp32 rows of one split tile per two pairs (a split tile's halves
    // take two pairs of the last round)
    return kProjectSyncBytes + (size_t)(device_sm_count() / 4) * kBM * kBN * sizeof(float);
}

cudaError_t launch_project_kv(const void* hidden, int32_t L, int32_t H, int64_t hidden_stride, const void* w_k,
                              const void* w_v, const int32_t* slot_mapping, void* k_cache, void* v_cache,
                              int32_t Hkv, int32_t D, int32_t page_size, int32_t num_pages, int64_t sp, int64_t ss,
                              int64_t sh, uint32_t* err, void* workspace, size_t workspace_bytes, cudaStream_t stream)
{
    if (L == 0) return cudaSuccess;
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const int32_t N = Hkv * D;
    CUtensorMap th, twk, twv;
    if (!encode_2d(enc, &th, hidden, H, L, hidden_stride, kRows) || !encode_2d(enc, &twk, w_k, H, N, H, 128) ||
        !encode_2d(enc, &twv, w_v, H, N, H, 128))
        return cudaErrorInvalidValue;
    ProjParams p;
    p.slot_mapping = slot_mapping;
    p.k_cache = static_cast<__nv_bfloat16*>(k_cache);
    p.v_cache = static_cast<__nv_bfloat16*>(v_cache);
    p.err = err;
    p.L = L;
    p.H = H;
    p.N = N;
    p.D = D;
    p.page_size = page_size;
    p.n_half = (N + kBN - 1) / kBN;
    p.tiles = ((L + kBM - 1) / kBM) * 2 * p.n_half;
    p.total_slots = (int64_t)num_pages * page_size;
    p.sp = sp;
    p.ss = ss;
    p.sh = sh;
    int pairs = 0;
    cudaError_t e = resident_pairs(&pairs);
    if (e != cudaSuccess) return e;
    pairs = std::min(pairs, p.tiles);
    // split the tiles of a partial last round in two along the hidden dimension when the
    // halves fit in that round and the workspace holds their partials
    const int rem = p.tiles % pairs;
    const int KB = (H + kBK - 1) / kBK;
    const bool split = workspace && rem > 0 && 2 * rem <= pairs && KB >= 2 &&
                       2 * rem * 2 * 2 * (int64_t)sizeof(int32_t) <= (int64_t)kProjectSyncBytes &&
                       workspace_bytes >= kProjectSyncBytes + (size_t)rem * kBM * kBN * sizeof(float);
    p.full_tiles = split ? p.tiles - rem : p.tiles;
    p.units = split ? p.tiles + rem : p.tiles;
    p.sync = static_cast<int32_t*>(workspace);
    p.partial = workspace ? reinterpret_cast<float*>(static_cast<char*>(workspace) + kProjectSyncBytes) : nullptr;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * pairs);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kAlloc;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, project_kv_kernel, th, twk, twv, p);
}

}  // namespace dflash
