// Tensor-core block attention for bf16 on sm_103a, operand-split CTA pair.
//
// Same mathematics as tc_attn.cu (transposed S^T = K.Q^T, O^T += V^T.P^T,
// row sums l += 1.P^T on tcgen05 with TMEM accumulators; see that file). What
// differs is the schedule. With head_dim 512 a 128-key tile is 256 KB of K and
// V, more than the shared-memory ring of one CTA, and V(j) cannot be consumed
// before the softmax of tile j has produced P: a single CTA's ring then sits
// full of V(j) while the softmax runs, and HBM idles.
//
// Here a 2-CTA cluster shares one (request, KV head, row group, key chunk):
//   K-CTA (rank 0): streams only K, computes S^T into a double-buffered TMEM
//     region (QK of tile j+1 overlaps the softmax of tile j), runs the softmax
//     and ships each tile's P^T (bf16, in the MMA's shared-memory layout) with
//     the running row max and, when the max moved, the rescale factors, to the
//     V-CTA with one shared-to-shared bulk copy completing on the V-CTA's
//     mbarrier;
//   V-CTA (rank 1): streams only V through a deep ring (no Q to hold),
//     accumulates O^T and l, rescales them when told, and writes the output.
// Each SM streams one operand continuously. Flow control: the V-CTA's PV
// commit is multicast to the K-CTA's "message free" barrier of that buffer.
//
// Warps (288 threads) per CTA: 0-3 softmax (K-CTA) or rescale + epilogue
// (V-CTA), 4-7 TMA producers (ring stages dealt round-robin), 8 MMA issuer.
// Every wait is bounded (2 s of %globaltimer) and reports DFLASH_DEVERR_TIMEOUT.
#include <cuda.h>

#include <cmath>
#include <mutex>

#include "dflash_device.cuh"
#include "tc_ptx.cuh"

namespace dflash {
namespace {

using namespace ptx;

constexpr int kThreads = 288;
constexpr int kProducerWarp = 4;
constexpr int kNumProducers = 4;
constexpr int kMmaWarp = 8;
constexpr int kTileKeys = 128;
constexpr int kStageBytes = 16384;
constexpr int kMaxPids = 128;
constexpr int kMaxRows = 80;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThresh = 8.0f;
constexpr int kOnesBytes = 4096;
constexpr int kSmemCap = 227 * 1024;

struct PairExtra {
    int32_t Gc;    // query heads per pair
    int32_t n_rg;  // row groups per KV head
    int32_t R;     // packed rows (Gc * T)
};

constexpr int pow2ceil32(int x)
{
    int p = 32;
    while (p < x) p <<= 1;
    return p;
}

constexpr int round_up_c(int x, int a) { return (x + a - 1) / a * a; }

// Cluster-visible barriers sit at the same offsets in both CTAs: [0..1] msg_full
// (in the V-CTA: P^T of the buffer has landed), [2..3] msg_free (in the K-CTA:
// the V-CTA has finished with the buffer).
template <int D, int N>
struct PairLayout {
    // message: P^T [2 key halves][N rows][128 B], alpha[N], m[N], flag word
    static constexpr int kMsgBytes = N * 256 + 8 * N + 16;
    static constexpr int kMsgStride = round_up_c(kMsgBytes, 1024);
    static constexpr int kClusterBars = 0;   // 4 x uint64
    static constexpr int kBase = 1024;       // rank-specific layout starts here

    // ---- K-CTA
    static constexpr int kKQ = kBase;                                  // [D/64][N][128 B]
    static constexpr int kKStage = kKQ + N * D * 2;                    // 2 x message staging
    static constexpr int kKTable = kKStage + 2 * kMsgStride;           // m, alpha, red[4], lo, hi
    static constexpr int kKPid = kKTable + 8 * N * 4;                  // 4 x kMaxPids int
    static constexpr int kKBars = kKPid + 4 * kMaxPids * 4;            // local barriers
    static constexpr int kKMisc = kKBars + 64 * 8;                     // tmem slot, abort, flags
    static constexpr int kKRing = round_up_c(kKMisc + 64, 1024);
    static constexpr int kKStagesFit = (kSmemCap - 1024 - kKRing) / kStageBytes;
    static constexpr int kKStages = kKStagesFit > 12 ? 12 : kKStagesFit;
    static constexpr int kKTotal = kKRing + kKStages * kStageBytes;
    static constexpr int kKTmemCols = pow2ceil32(2 * N);

    // ---- V-CTA
    static constexpr int kVMsg = kBase;                                // 2 x message
    static constexpr int kVOnes = kVMsg + 2 * kMsgStride;
    static constexpr int kVRow = kVOnes + kOnesBytes;                  // int64 orow[N]
    static constexpr int kVPid = kVRow + N * 8;
    static constexpr int kVBars = kVPid + 4 * kMaxPids * 4;
    static constexpr int kVMisc = kVBars + 64 * 8;
    static constexpr int kVRing = round_up_c(kVMisc + 64, 1024);
    static constexpr int kVStagesFit = (kSmemCap - 1024 - kVRing) / kStageBytes;
    static constexpr int kVStages = kVStagesFit > 12 ? 12 : kVStagesFit;
    static constexpr int kVTotal = kVRing + kVStages * kStageBytes;
    static constexpr int kVTmemCols = pow2ceil32(N * (1 + D / 128));

    static constexpr int kAlloc = (kKTotal > kVTotal ? kKTotal : kVTotal) + 1024;
    static_assert(kKStages >= 3 && kVStages >= 3, "ring too shallow");
    static_assert(kAlloc <= kSmemCap, "shared memory budget");
    static_assert(N * (1 + D / 128) <= 512, "TMEM budget");
    static_assert(kMsgBytes % 16 == 0, "bulk copy size");
};

template <int D, int N>
__global__ void __launch_bounds__(kThreads, 1)
    tc_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const AttnParams p, const PairExtra x)
{
    using Lay = PairLayout<D, N>;
    constexpr int KC = D / 64;   // K stages per tile
    constexpr int VC = D / 128;  // O^T chunks; V stages per 64-key half
    constexpr int NQ = N / 16;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t rank = cluster_ctarank();
    const bool is_k = (rank == 0);
    uint64_t* cbars = reinterpret_cast<uint64_t*>(smem + Lay::kClusterBars);
    uint64_t* msg_full = cbars;      // [2], used in the V-CTA
    uint64_t* msg_free = cbars + 2;  // [2], used in the K-CTA

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int c_split = blockIdx.x >> 1;
    const int g = blockIdx.y / x.n_rg;
    const int rg = blockIdx.y % x.n_rg;
    const int b = blockIdx.z;
    const int T = p.T;
    const int Psz = p.page_size;
    const int R = x.R;
    const int h0 = g * p.G + rg * x.Gc;

    const int S = is_k ? Lay::kKStages : Lay::kVStages;
    uint8_t* ring = smem + (is_k ? Lay::kKRing : Lay::kVRing);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (is_k ? Lay::kKBars : Lay::kVBars));
    uint64_t* full = bars;            // [S]
    uint64_t* empty = bars + 12;      // [S]
    uint64_t* q_full = bars + 24;     // K-CTA
    uint64_t* s_full = bars + 25;     // [2] K-CTA
    uint64_t* s_free = bars + 27;     // [2] K-CTA (count 128)
    uint64_t* drain = bars + 29;
    uint64_t* rq = bars + 30;         // V-CTA: MMA -> rescale warps (count 1)
    uint64_t* rd = bars + 31;         // V-CTA: rescale warps -> MMA (count 128)
    uint8_t* misc = smem + (is_k ? Lay::kKMisc : Lay::kVMisc);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);
    volatile int* rq_cmd = reinterpret_cast<volatile int*>(misc + 8);  // V-CTA: buffer to rescale, -1 = finish
    int32_t* pid_s = reinterpret_cast<int32_t*>(smem + (is_k ? Lay::kKPid : Lay::kVPid));

    const int32_t L = __ldg(p.seq_lens + b);
    const bool len_ok = seq_len_ok(p, L);
    Chunk ch;
    ch.kb = 0;
    ch.ke = 0;
    if (len_ok) ch = split_chunk(L, T, p.window, Psz, p.splits, c_split);
    const int t0 = (ch.kb / Psz) * Psz;
    const int ntiles = (ch.kb < ch.ke) ? (ch.ke - t0 + kTileKeys - 1) / kTileKeys : 0;
    const int pages_per_tile = kTileKeys / Psz;
    const int chunk_pages = ntiles * pages_per_tile;
    const int first_page = t0 / Psz;

    const int pw = warp - kProducerWarp;
    int32_t* pid_w = pid_s + (pw & 3) * kMaxPids;
    auto load_window = [&](int base) {
        for (int k = lane; k < kMaxPids; k += 32) {
            const int pr = base + k;
            int32_t id = p.num_pages;
            if (pr < chunk_pages && t0 + pr * Psz < ch.ke) {
                const int32_t v = __ldg(p.page_table + (int64_t)b * p.max_pages + first_page + pr);
                if (v >= 0 && v < p.num_pages)
                    id = v;
                else if (is_k)
                    raise_error(p.err, DFLASH_DEVERR_PAGE_ID);
            }
            pid_w[k] = id;
        }
        __syncwarp();
    };

    // ---------------------------------------------------------------- set-up
    if (tid == 0) {
        for (int i = 0; i < 4; ++i) mbar_init(cbars + i, 1);
        for (int i = 0; i < 32; ++i) {
            uint64_t* bar = bars + i;
            mbar_init(bar, (bar == s_free || bar == s_free + 1 || bar == rd) ? 128u : 1u);
        }
        *abort_flag = 0;
        *rq_cmd = 0;
        if (!len_ok && is_k) raise_error(p.err, DFLASH_DEVERR_SEQ_LEN);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp >= kProducerWarp && warp < kProducerWarp + kNumProducers) {
        if (ntiles > 0) load_window(0);
    } else if (warp == kMmaWarp) {
        if (!is_k) {
            uint8_t* ones_s = smem + Lay::kVOnes;
            for (int idx = lane; idx < kOnesBytes / 16; idx += 32)
                *reinterpret_cast<uint4*>(ones_s + idx * 16) =
                    make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);  // bf16 1.0
            fence_proxy_async_smem();
        }
        tmem_alloc(tmem_slot, is_k ? Lay::kKTmemCols : Lay::kVTmemCols);
        tmem_relinquish();
    } else if (is_k) {
        float* m_s = reinterpret_cast<float*>(smem + Lay::kKTable);
        int32_t* lo_s = reinterpret_cast<int32_t*>(smem + Lay::kKTable + 6 * N * 4);
        int32_t* hi_s = reinterpret_cast<int32_t*>(smem + Lay::kKTable + 7 * N * 4);
        if (tid < N) {
            int32_t lo = -(1 << 30), hi = (1 << 30);
            if (tid < R) {
                const KeyRange kr = row_range(L, T, tid / x.Gc, p.causal, p.window);
                lo = kr.lo;
                hi = kr.hi;
            }
            lo_s[tid] = lo;
            hi_s[tid] = hi;
            m_s[tid] = -INFINITY;
        }
        uint8_t* q_s = smem + Lay::kKQ;
        for (int idx = tid; idx < KC * (N - R) * 8; idx += 128) {
            const int kc = idx / ((N - R) * 8);
            const int rem = idx - kc * (N - R) * 8;
            *reinterpret_cast<uint4*>(q_s + kc * N * 128 + (R + rem / 8) * 128 + (rem % 8) * 16) =
                make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
    } else {
        int64_t* orow_s = reinterpret_cast<int64_t*>(smem + Lay::kVRow);
        if (tid < N) {
            int64_t orow = -1;
            if (tid < R) {
                const int i = tid / x.Gc;
                orow = (int64_t)(b * T + i) * p.Hq + (h0 + tid - i * x.Gc);
            }
            orow_s[tid] = orow;
        }
    }
    tc_fence_before();
    // barriers of both CTAs initialised before any cross-CTA traffic
    cluster_sync_all();
    tc_fence_after();
    cudaTriggerProgrammaticLaunchCompletion();
    const uint32_t tmem = *tmem_slot;
    const uint32_t peer = rank ^ 1u;

    if (warp >= kProducerWarp && warp < kProducerWarp + kNumProducers) {
        // ------------------------------------------------------------ TMA producers (one operand each)
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        int wbase = 0;
        uint32_t issued_parity[12];
#pragma unroll
        for (int s = 0; s < 12; ++s) issued_parity[s] = 2;
        if (ntiles > 0) {
            if (is_k && pw == 0 && lane == 0) {
                uint8_t* q_s = smem + Lay::kKQ;
                mbar_expect_tx(q_full, (uint32_t)(R * 128 * KC));
                for (int kc = 0; kc < KC; ++kc) tma_load_3d(q_s + kc * N * 128, &tm_q, q_full, kc * 64, h0, b * T);
            }
            const int box = Psz * 128;
            const int per_tile = is_k ? KC : 2 * VC;
            int seq = 0;
            for (int j = 0; j < ntiles && ok; ++j) {
                const int rel0 = j * pages_per_tile;
                for (int st = 0; st < per_tile && ok; ++st, ++seq) {
                    if ((seq & 3) == pw) {
                        if (rel0 + pages_per_tile > wbase + kMaxPids) {
                            wbase = rel0;
                            load_window(wbase);
                        }
                        if (lane == 0) ok = wait_bounded(empty + stage, phase ^ 1u, abort_flag, p.err);
                        ok = __shfl_sync(0xffffffffu, ok, 0);
                        if (!ok) break;
                        if (lane == 0) {
                            uint8_t* dst = ring + stage * kStageBytes;
                            mbar_expect_tx(full + stage, kStageBytes);
                            if (is_k) {
                                for (int pg = 0; pg < pages_per_tile; ++pg)
                                    tma_load_4d(dst + pg * box, &tm_k, full + stage, st * 64, g, 0,
                                                pid_w[rel0 + pg - wbase]);
                            } else {
                                const int h = st / VC, c = st % VC;
                                const int ppg = 64 / Psz;
                                for (int pg = 0; pg < ppg; ++pg) {
                                    const int32_t page = pid_w[rel0 + h * ppg + pg - wbase];
                                    for (int m = 0; m < 2; ++m)
                                        tma_load_4d(dst + m * 8192 + pg * box, &tm_v, full + stage, c * 128 + m * 64,
                                                    g, 0, page);
                                }
                            }
                            issued_parity[stage] = phase;
                        }
                        __syncwarp();
                    }
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
        if (lane == 0 && !ok) {
            for (int s = 0; s < S; ++s) {
                if (issued_parity[s] > 1) continue;
                const unsigned long long t_start = globaltimer();
                while (!mbar_try_wait(full + s, issued_parity[s]) && globaltimer() - t_start < kTimeoutNs) {
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        const uint32_t ring_addr = smem_u32(ring);
        auto wait_lane0 = [&](uint64_t* bar, uint32_t par, bool cluster_scope) -> bool {
            bool got = true;
            if (lane == 0)
                got = cluster_scope ? wait_bounded_cluster(bar, par, abort_flag, p.err)
                                    : wait_bounded(bar, par, abort_flag, p.err);
            return __shfl_sync(0xffffffffu, got, 0);
        };
        auto advance = [&]() {
            if (++stage == S) {
                stage = 0;
                phase ^= 1u;
            }
        };
        if (is_k) {
            constexpr uint32_t idesc_s = make_idesc(128, N, 0, 0);
            const uint32_t q_addr = smem_u32(smem + Lay::kKQ);
            if (ntiles > 0) {
                ok = wait_lane0(q_full, 0, false);
                tc_fence_after();
            }
            for (int j = 0; j < ntiles && ok; ++j) {
                const int bf = j & 1;
                if (j >= 2) {
                    ok = wait_lane0(s_free + bf, (uint32_t)(((j >> 1) - 1) & 1), false);
                    if (!ok) break;
                    tc_fence_after();
                }
                const uint32_t tmem_s = tmem + bf * N;
                for (int kc = 0; kc < KC && ok; ++kc) {
                    ok = wait_lane0(full + stage, phase, false);
                    if (!ok) break;
                    tc_fence_after();
                    if (lane == 0) {
                        const uint32_t st = ring_addr + stage * kStageBytes;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            tc_mma(tmem_s, sw128_desc(st + kk * 32, 16, 1024),
                                   sw128_desc(q_addr + kc * N * 128 + kk * 32, 16, 1024), idesc_s,
                                   (kc > 0 || kk > 0) ? 1u : 0u);
                        tc_commit(empty + stage);
                    }
                    __syncwarp();
                    advance();
                }
                if (!ok) break;
                if (lane == 0) tc_commit(s_full + bf);
                __syncwarp();
            }
        } else {
            constexpr uint32_t idesc_o = make_idesc(128, N, 1, 0);
            constexpr uint32_t idesc_l = make_idesc(128, N, 0, 0);
            const uint32_t ones_addr = smem_u32(smem + Lay::kVOnes);
            const uint32_t tmem_o = tmem;
            const uint32_t tmem_l = tmem + VC * N;
            uint32_t rq_phase = 0;
            for (int j = 0; j < ntiles && ok; ++j) {
                const int bf = j & 1;
                uint8_t* msg = smem + Lay::kVMsg + bf * Lay::kMsgStride;
                if (lane == 0) mbar_expect_tx(msg_full + bf, (uint32_t)Lay::kMsgBytes);
                ok = wait_lane0(msg_full + bf, (uint32_t)((j >> 1) & 1), true);
                if (!ok) break;
                tc_fence_after();
                const int rescale = *reinterpret_cast<volatile int*>(msg + N * 256 + 8 * N);
                if (rescale) {
                    // O^T and l must be scaled by alpha before this tile's PV: wait for the
                    // previous PV, then hand the TMEM rescale to warps 0-3
                    if (lane == 0) {
                        tc_commit(drain);
                        const unsigned long long t_start = globaltimer();
                        while (!mbar_try_wait(drain, (uint32_t)(rq_phase & 1)) &&
                               globaltimer() - t_start < kTimeoutNs) {
                        }
                        *rq_cmd = bf;
                        mbar_arrive(rq);
                    }
                    ok = wait_lane0(rd, rq_phase & 1, false);
                    ++rq_phase;
                    if (!ok) break;
                    tc_fence_after();
                }
                const uint32_t p_addr = smem_u32(msg);
                const int tile_key0 = t0 + j * kTileKeys;
                for (int h = 0; h < 2 && ok; ++h) {
                    for (int c = 0; c < VC && ok; ++c) {
                        ok = wait_lane0(full + stage, phase, false);
                        if (!ok) break;
                        tc_fence_after();
                        const int key0 = tile_key0 + h * 64;
                        const int zlo = L - key0;
                        if (L % Psz != 0 && zlo > 0 && zlo < 64 && ch.ke == L) {
                            const int zhi = min(64, ((L + Psz - 1) / Psz) * Psz - key0);
                            uint8_t* st = ring + stage * kStageBytes;
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
                            const uint32_t st = ring_addr + stage * kStageBytes;
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                tc_mma(tmem_o + c * N, sw128_desc(st + kk * 2048, 8192, 1024),
                                       sw128_desc(p_addr + h * N * 128 + kk * 32, 16, 1024), idesc_o,
                                       (j > 0 || h > 0 || kk > 0) ? 1u : 0u);
                            tc_commit(empty + stage);
                        }
                        __syncwarp();
                        advance();
                    }
                    if (lane == 0) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            tc_mma(tmem_l, noswz_desc(ones_addr, 2048, 128),
                                   sw128_desc(p_addr + h * N * 128 + kk * 32, 16, 1024), idesc_l,
                                   (j > 0 || h > 0 || kk > 0) ? 1u : 0u);
                    }
                    __syncwarp();
                }
                if (!ok) break;
                // the K-CTA may refill this message buffer once these MMAs have read it
                if (lane == 0) tc_commit_multicast(msg_free + bf, (uint16_t)1u);
                __syncwarp();
            }
            // all PV done, then release the rescale/epilogue warps
            if (lane == 0) {
                tc_commit(drain);
                const unsigned long long t_start = globaltimer();
                while (!mbar_try_wait(drain, (uint32_t)(rq_phase & 1)) && globaltimer() - t_start < kTimeoutNs) {
                }
                *rq_cmd = -1;
                mbar_arrive(rq);
            }
            __syncwarp();
        }
        if (is_k && lane == 0) {
            tc_commit(drain);
            const unsigned long long t_start = globaltimer();
            while (!mbar_try_wait(drain, 0) && globaltimer() - t_start < kTimeoutNs) {
            }
        }
        __syncwarp();
    } else if (is_k) {
        // ------------------------------------------------------------ K-CTA softmax (thread = key lane)
        float* m_s = reinterpret_cast<float*>(smem + Lay::kKTable);
        float* a_s = m_s + N;
        float* red = m_s + 2 * N;
        int32_t* lo_s = reinterpret_cast<int32_t*>(smem + Lay::kKTable + 6 * N * 4);
        int32_t* hi_s = reinterpret_cast<int32_t*>(smem + Lay::kKTable + 7 * N * 4);
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const float sl2 = p.scale * kLog2e;
        const bool plain = (p.causal == 0 && p.window == 0);
        const int pchunk = (tid & 63) >> 3;
        const int pbyte = (tid & 7) * 2;
        bool ok = true;
        auto group_wait = [&](uint64_t* bar, uint32_t parity, bool cluster_scope) -> bool {
            bool got = true;
            if (tid == 0)
                got = cluster_scope ? wait_bounded_cluster(bar, parity, abort_flag, p.err)
                                    : wait_bounded(bar, parity, abort_flag, p.err);
            return !named_bar_or_128(!got);
        };
        auto load16 = [&](uint32_t taddr, uint32_t (&r16)[16]) {
            tmem_ld16(taddr, r16);
            tmem_ld_wait();
            reg_fence16(r16);
        };
        const uint32_t msg_peer0 = mapa_shared(smem_u32(smem + Lay::kVMsg), peer);
        const uint32_t full_peer0 = mapa_shared(smem_u32(msg_full), peer);
        int sent = 0;
        for (int j = 0; j < ntiles && ok; ++j) {
            const int bf = j & 1;
            const uint32_t tmem_s = tmem + bf * N;
            if (!group_wait(s_full + bf, (uint32_t)((j >> 1) & 1), false)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int key = t0 + j * kTileKeys + tid;
            const bool kvalid = key >= ch.kb && key < ch.ke;
            auto score = [&](uint32_t raw, int col) -> float {
                bool vis = kvalid;
                if (!plain) vis = vis && key >= lo_s[col] && key <= hi_s[col];
                return vis ? u2f(raw) * sl2 : -INFINITY;
            };
            bool need = false;
#pragma unroll 1
            for (int q = 0; q < NQ; ++q) {
                float mv[16];
                load_row16(m_s + q * 16, mv);
                uint32_t r16[16];
                load16(tmem_s + lane_base + q * 16, r16);
#pragma unroll
                for (int u = 0; u < 16; ++u) need |= score(r16[u], q * 16 + u) > mv[u] + kRescaleThresh;
            }
            need = named_bar_or_128(need);
            if (need) {
#pragma unroll 1
                for (int q = 0; q < NQ; ++q) {
                    uint32_t r16[16];
                    load16(tmem_s + lane_base + q * 16, r16);
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        float v = score(r16[u], q * 16 + u);
#pragma unroll
                        for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
                        if (((q * 16 + u) & 31) == lane) red[warp * N + q * 16 + u] = v;
                    }
                }
                named_bar_sync_128();
                if (tid < N) {
                    const float mo = m_s[tid];
                    const float mn =
                        fmaxf(fmaxf(mo, fmaxf(red[tid], red[N + tid])), fmaxf(red[2 * N + tid], red[3 * N + tid]));
                    m_s[tid] = mn;
                    a_s[tid] = (mo == -INFINITY) ? 0.f : ex2(mo - mn);
                }
                named_bar_sync_128();
            }
            // the staging buffer of this tile was last sent two tiles ago: that copy must have read it
            uint8_t* stg = smem + Lay::kKStage + bf * Lay::kMsgStride;
            if (j >= 2 && tid == 0) bulk_wait_read_1();
            named_bar_sync_128();
            uint8_t* pcol = stg + (tid >> 6) * (N * 128);
#pragma unroll 1
            for (int q = 0; q < NQ; ++q) {
                float mv[16];
                load_row16(m_s + q * 16, mv);
                uint32_t r16[16];
                load16(tmem_s + lane_base + q * 16, r16);
                __nv_bfloat16 pb[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const float sc = score(r16[u], q * 16 + u);
                    pb[u] = __float2bfloat16_rn((sc == -INFINITY) ? 0.f : ex2(sc - mv[u]));
                }
                uint8_t* prow = pcol + q * 16 * 128 + pbyte;
#pragma unroll
                for (int u = 0; u < 16; ++u)
                    *reinterpret_cast<__nv_bfloat16*>(prow + u * 128 + ((pchunk ^ (u & 7)) << 4)) = pb[u];
            }
            // S^T of this buffer is no longer needed: QK of tile j+2 may overwrite it
            tc_fence_before();
            mbar_arrive(s_free + bf);
            if (tid < N) {
                reinterpret_cast<float*>(stg + N * 256)[tid] = (need && j > 0) ? a_s[tid] : 1.f;
                reinterpret_cast<float*>(stg + N * 256 + 4 * N)[tid] = m_s[tid];
            }
            if (tid == 0) {
                int* fl = reinterpret_cast<int*>(stg + N * 256 + 8 * N);
                fl[0] = (need && j > 0) ? 1 : 0;
                fl[1] = 0;
                fl[2] = 0;
                fl[3] = 0;
            }
            fence_proxy_async_smem();
            named_bar_sync_128();
            bool go = true;
            if (tid == 0) {
                if (j >= 2) go = wait_bounded_cluster(msg_free + bf, (uint32_t)(((j >> 1) - 1) & 1), abort_flag, p.err);
                if (go) {
                    bulk_copy_to_peer(msg_peer0 + bf * Lay::kMsgStride, stg, (uint32_t)Lay::kMsgBytes,
                                      full_peer0 + bf * 8);
                    bulk_commit_group();
                }
            }
            ok = !named_bar_or_128(!go);
            if (ok) ++sent;
        }
        // every copy has left our shared memory, and the V-CTA has released every buffer
        if (tid == 0) {
            bulk_wait_read_0();
            for (int j = (sent >= 2 ? sent - 2 : 0); j < sent; ++j)
                if (!wait_bounded_cluster(msg_free + (j & 1), (uint32_t)((j >> 1) & 1), abort_flag, p.err)) break;
        }
    } else {
        // ------------------------------------------------------------ V-CTA rescale + epilogue
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const uint32_t tmem_o = tmem;
        const uint32_t tmem_l = tmem + VC * N;
        int64_t* orow_s = reinterpret_cast<int64_t*>(smem + Lay::kVRow);
        bool ok = true;
        auto load16 = [&](uint32_t taddr, uint32_t (&r16)[16]) {
            tmem_ld16(taddr, r16);
            tmem_ld_wait();
            reg_fence16(r16);
        };
        uint32_t rq_phase = 0;
        for (;;) {
            bool got = true;
            if (tid == 0) got = wait_bounded(rq, rq_phase & 1, abort_flag, p.err);
            ok = !named_bar_or_128(!got);
            ++rq_phase;
            if (!ok) break;
            const int cmd = *rq_cmd;
            if (cmd < 0) break;
            tc_fence_after();
            const float* alpha = reinterpret_cast<const float*>(smem + Lay::kVMsg + cmd * Lay::kMsgStride + N * 256);
#pragma unroll 1
            for (int cq = 0; cq < (VC + 1) * NQ; ++cq) {  // O^T chunks, then the row sums
                const int c = cq / NQ, q = cq % NQ;
                uint32_t r16[16];
                const uint32_t ta = tmem_o + c * N + lane_base + q * 16;
                load16(ta, r16);
                float av[16];
                load_row16(alpha + q * 16, av);
#pragma unroll
                for (int u = 0; u < 16; ++u) r16[u] = f2u(u2f(r16[u]) * av[u]);
                tmem_st16(ta, r16);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(rd);
        }
        tc_fence_after();
        // ---------------------------------------------------------------- epilogue
        const bool have_o = ok && ntiles > 0;
        const float* m_fin = reinterpret_cast<const float*>(smem + Lay::kVMsg + ((ntiles - 1) & 1) * Lay::kMsgStride +
                                                            N * 256 + 4 * N);
        const int64_t part_base = (int64_t)c_split * p.B * T * p.Hq;
        const bool final_out = (p.splits == 1);
        __nv_bfloat16* __restrict__ out_bf = reinterpret_cast<__nv_bfloat16*>(p.out);
        float* __restrict__ part_out = p.part_out;
#pragma unroll 1
        for (int q = 0; q < NQ; ++q) {
            int64_t orow[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) orow[u] = orow_s[q * 16 + u];
            uint32_t l16[16];
            if (have_o) {
                load16(tmem_l + lane_base + q * 16, l16);
            } else {
#pragma unroll
                for (int u = 0; u < 16; ++u) l16[u] = 0u;
            }
            float inv[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const float tot = u2f(l16[u]);
                inv[u] = tot > 0.f ? __frcp_rn(tot) : 0.f;
            }
            const int my = tid - q * 16;
            if (my >= 0 && my < 16 && tid < R) {
                float tot = 0.f;
#pragma unroll
                for (int u = 0; u < 16; ++u)
                    if (u == my) tot = u2f(l16[u]);
                const float lse_v = tot > 0.f ? (m_fin[tid] + __log2f(tot)) * kLn2 : -INFINITY;
                if (final_out) {
                    if (p.lse) p.lse[orow_s[tid]] = lse_v;
                } else {
                    p.part_lse[part_base + orow_s[tid]] = lse_v;
                }
            }
#pragma unroll 1
            for (int c = 0; c < VC; ++c) {
                const int d = c * 128 + tid;
                uint32_t r16[16];
                if (have_o) {
                    load16(tmem_o + c * N + lane_base + q * 16, r16);
                } else {
#pragma unroll
                    for (int u = 0; u < 16; ++u) r16[u] = 0u;
                }
                if (final_out) {
#pragma unroll
                    for (int u = 0; u < 16; ++u)
                        if (q * 16 + u < R) out_bf[orow[u] * D + d] = __float2bfloat16_rn(u2f(r16[u]) * inv[u]);
                } else {
#pragma unroll
                    for (int u = 0; u < 16; ++u)
                        if (q * 16 + u < R) part_out[(part_base + orow[u]) * D + d] = u2f(r16[u]) * inv[u];
                }
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, is_k ? Lay::kKTmemCols : Lay::kVTmemCols);
    }
    // no CTA of the pair leaves while its peer may still address its shared memory
    cluster_sync_all();
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

int choose_gc(int G, int T)
{
    for (int gc = G; gc >= 1; --gc)
        if (G % gc == 0 && gc * T <= kMaxRows) return gc;
    return 0;
}

template <int D, int N>
cudaError_t launch_dn(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p,
                      const PairExtra& x, cudaStream_t stream)
{
    using Lay = PairLayout<D, N>;
    auto kern = tc_pair_kernel<D, N>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kAlloc);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * p.splits, p.Hkv * x.n_rg, p.B);
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

template <int D>
cudaError_t launch_d(int n, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p,
                     const PairExtra& x, cudaStream_t stream)
{
    switch (n) {
    case 16: return launch_dn<D, 16>(tq, tk, tv, p, x, stream);
    case 32: return launch_dn<D, 32>(tq, tk, tv, p, x, stream);
    case 48: return launch_dn<D, 48>(tq, tk, tv, p, x, stream);
    case 64: return launch_dn<D, 64>(tq, tk, tv, p, x, stream);
    case 80: return launch_dn<D, 80>(tq, tk, tv, p, x, stream);
    }
    return cudaErrorNotSupported;
}

}  // namespace

bool tc_pair_supports(const AttnParams& p)
{
    if (p.dtype != DFLASH_BF16) return false;
    if (p.D != 128 && p.D != 256 && p.D != 512) return false;
    if (p.page_size != 16 && p.page_size != 32 && p.page_size != 64) return false;
    if (choose_gc(p.G, p.T) == 0) return false;
    if (p.sh % 8 || p.ss % 8 || p.sp % 8) return false;
    return true;
}

int tc_pair_ctas_per_split(const AttnParams& p)
{
    const int gc = choose_gc(p.G, p.T);
    return gc > 0 ? 2 * p.B * p.Hkv * (p.G / gc) : 0;
}

cudaError_t launch_tc_pair_attn(const AttnParams& p, cudaStream_t stream)
{
    if (!tc_pair_supports(p)) return cudaErrorNotSupported;
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    PairExtra x;
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
    switch (p.D) {
    case 128: e = launch_d<128>(n, tq, tk, tv, p, x, stream); break;
    case 256: e = launch_d<256>(n, tq, tk, tv, p, x, stream); break;
    case 512: e = launch_d<512>(n, tq, tk, tv, p, x, stream); break;
    default: e = cudaErrorNotSupported;
    }
    if (e != cudaSuccess || p.splits == 1) return e;
    return launch_combine(p.part_out, p.part_lse, p.splits, (int64_t)p.B * p.T * p.Hq, p.D, p.dtype, p.out, p.lse,
                          stream);
}

}  // namespace dflash
