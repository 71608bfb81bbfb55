// gemm2.cu -- CTA-pair (tcgen05 cta_group::2) variant of the block-scaled
// GEMM, for outputs whose width is a multiple of 256.
//
// Method: as gemm.cu ("Add an NVFP4 quantization converter", torchtitan PR
// #3914; "Hybrid quantization", TransformerEngine PR #2817): TN-form
// C = alpha * A B^T with NVFP4 or MXFP8 block-scaled operands.
//
// Two CTAs of a cluster form a pair that owns a 256 x 256 output tile: CTA c
// stages rows [128c, 128c+128) of the A tile and rows [128c, 128c+128) of the
// B tile; the leader (c = 0) issues 256x256 MMAs that read both CTAs' shared
// memory and write each CTA's half of the accumulator into its own TMEM
// (128 rows x 256 fp32 columns).  Per CTA a stage holds 32 KB of operands
// (against 48 KB for a 128x256 tile in one CTA) plus the A scales of its rows
// and the B scales of all 256 columns (the pair MMA reads the full B scale
// set from each CTA's TMEM), so each SM writes less into shared memory per
// MMA FLOP.  bf16 outputs leave through 4 KB per-warp staging buffers and
// TMA tensor stores (full 128-byte lines).  This kernel takes every GEMM whose
// output width is a multiple of 256 unless NVQ_GEMM_PAIR=0.
//
// Signalling (every wait bounded, as in gemm.cu):
//   full[s]      leader: A/B bytes of both CTAs (each CTA's TMA load signals the
//                leader's barrier, .cta_group::2) and the arrivals of the 8 scale
//                warps of both CTAs once their TMEM scales are written, so the MMA
//                issuer waits on one barrier per stage;
//   sf_full[s]   per CTA: this CTA's block-scale tiles;
//   empty[s]     per CTA: the leader's MMAs of stage s finished (multicast commit);
//   acc_full     per CTA: the tile's accumulator is complete (multicast commit);
//   acc_empty    leader: the 8 epilogue warps of both CTAs read the accumulator.
// A cluster barrier brackets the kernel so no CTA exits while its partner's
// MMAs, copies or arrivals may still reach it.
#include <cuda.h>

#include "gemm_epilogue.cuh"
#include "nvq_device.cuh"
#include "nvq_kernels.h"

namespace nvq {

namespace gemm2 {

constexpr int BM = 128;                  // rows per CTA (256 per pair)
constexpr int BN = 256;                  // MMA N = output columns per pair tile
constexpr int kHalfTileBytes = 128 * 128;
constexpr int kScaleWarps = 4;
constexpr int kEpiWarps = 8;
// Warp roles, by warpgroup: 0 = TMA producer (warp 0), MMA issuer (1),
// block-scale loader (2), idle (3); 1 = scale staging (warps 4-7, lane
// quadrant = warp & 3); 2-3 = epilogue (warps 8-15).
constexpr int kScaleLoadWarp = 2;
constexpr int kFirstScaleWarp = 4;
constexpr int kFirstEpiWarp = 8;
constexpr int kThreads = 32 * (kFirstEpiWarp + kEpiWarps);
// Register split (setmaxnreg): warpgroups 0-1 drop to kRegsLow so the
// epilogue warpgroups can hold a whole 128-column accumulator slice (128
// registers) and release the accumulator after one TMEM round trip.  The two
// shares add up to the launch allocation: 8 x 32 x 80 + 8 x 32 x 176 = 65536
// = kThreads x 128.
constexpr int kRegsLow = 80;
constexpr int kRegsHigh = 176;
static_assert(8 * 32 * kRegsLow + 8 * 32 * kRegsHigh == kThreads * 128, "register split");
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kAbortGraceNs = 1000000;  // 1 ms

// Each CTA's TMEM holds the B scales of all 256 columns (both halves of B):
// the pair MMA reads the full B scale set from each CTA's TMEM (holding only
// the half a CTA stages gives wrong products).
template <int FMT>
struct Cfg {
    static constexpr int kStageK = FMT == 1 ? 256 : 128;
    static constexpr int kMmaK = FMT == 1 ? 64 : 32;
    static constexpr int kAtomsK = FMT == 1 ? 4 : 1;
    static constexpr int kElemPerAtom = FMT == 1 ? 64 : 128;
    static constexpr int kSfbHalves = 2;
    static constexpr int kSfaBytes = kAtomsK * 512;
    static constexpr int kSfbBytes = kAtomsK * 512 * kSfbHalves;
    static constexpr int kStageBytes = 2 * kHalfTileBytes + kSfaBytes + kSfbBytes;
    static constexpr int kEpiBytes = kEpiWarps * 4096;  // TMA-store staging, 4 KB per epilogue warp
    static constexpr int kStagesFit = (232448 - 1024 - 1024 - kEpiBytes) / kStageBytes;
    static constexpr int kStages = kStagesFit < 6 ? kStagesFit : 6;
    static constexpr uint32_t kSfaCols = 4 * kAtomsK;
    static constexpr uint32_t kSfbCols = 4 * kAtomsK * kSfbHalves;
    static constexpr uint32_t kSfColsPerStage = kSfaCols + kSfbCols;
    static constexpr uint32_t kSfCol0 = BN;
    static_assert(kSfCol0 + kStages * kSfColsPerStage <= kTmemCols, "TMEM budget");
    static constexpr int kA = 0;
    static constexpr int kB = kA + kStages * kHalfTileBytes;
    static constexpr int kSfa = kB + kStages * kHalfTileBytes;
    static constexpr int kSfb = kSfa + kStages * kSfaBytes;
    static constexpr int kBar = kSfb + kStages * kSfbBytes;
    static constexpr int kNumBars = 3 * kStages + 3;  // full, empty, sf_full, acc_full, acc_empty, done
    static constexpr int kMisc = kBar + kNumBars * 8;
    static constexpr int kEpi = (kMisc + 16 + 1023) / 1024 * 1024;
    static constexpr int kAlloc = kEpi + kEpiBytes + 1024;
    static_assert(kAlloc <= 232448, "shared memory budget");
};

// Instruction descriptor: as gemm.cu with M = 256 (bits 24-28 = M >> 4).
template <int FMT>
__device__ __forceinline__ uint32_t make_idesc(uint32_t sf_id)
{
    uint32_t d = 0;
    if (FMT == 1) d |= (1u << 7) | (1u << 10);
    d |= (uint32_t)(BN >> 3) << 17;
    if (FMT == 2) d |= 1u << 23;
    d |= (uint32_t)(256 >> 4) << 24;
    d |= (sf_id & 3) << 4;
    d |= (sf_id & 3) << 29;
    return d;
}

struct PairTile {
    int g, mt_local, n_tile, a_row, b_row_pair, a_k0, b_k0, k_len, num_kb;
};

// Pair tile t: column tile fastest; rows of the pair = 128-row tiles
// 2 * mp and 2 * mp + 1 of the group; CTA `rank` takes the second index.
// A row tile past the group's end loads the group's last tile (in bounds)
// and stores nothing.
template <int STAGE_K>
__device__ __forceinline__ PairTile decode(const GemmArgs& a, int t, uint32_t rank)
{
    PairTile r;
    const int mp = t / a.n_tiles;
    r.n_tile = t - mp * a.n_tiles;
    int lo = 0;  // last group whose first pair tile <= mp (fixed-length branchless search)
#pragma unroll
    for (int step = kMaxGroups / 2; step >= 1; step >>= 1) {
        const int mid = lo + step;
        lo = (mid < a.G && a.groups[mid].pm_tile0 <= mp) ? mid : lo;
    }
    const GemmGroup& gr = a.groups[lo];
    r.g = lo;
    r.mt_local = 2 * (mp - gr.pm_tile0) + (int)rank;
    const int mt_load = r.mt_local < gr.m_tiles ? r.mt_local : gr.m_tiles - 1;
    r.a_row = gr.a_row0 + mt_load * BM;
    r.b_row_pair = gr.b_row0 + r.n_tile * BN;
    r.a_k0 = gr.a_k0;
    r.b_k0 = gr.b_k0;
    r.k_len = gr.k_len;
    r.num_kb = (gr.k_len + STAGE_K - 1) / STAGE_K;
    return r;
}

// Bounded wait that gives up when this CTA has aborted; a wait that runs out
// raises the abort flags of both CTAs of the pair.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, int* status, volatile int* abort_flag)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63) == 63) {
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
                record_error(status, kErrTimeout);
                *abort_flag = 1;
                set_partner_abort(abort_flag);
                return false;
            }
        }
    }
}

// Arrive on barrier `bar` of the leader CTA (local arrive in the leader).  Both
// uses (scales staged in TMEM, accumulator read out of TMEM) signal completed,
// fenced tcgen05 work, so the remote arrive is relaxed.
__device__ __forceinline__ void arrive_leader(uint64_t* bar, uint32_t rank)
{
    if (rank == 0) mbar_arrive(bar);
    else mbar_arrive_cluster_relaxed(map_to_rank(bar, 0));
}

template <int FMT>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap a_map, const __grid_constant__ CUtensorMap b_map,
                     const __grid_constant__ CUtensorMap c_map, const __grid_constant__ GemmArgs args)
{
    using C = Cfg<FMT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBar);
    uint64_t* empty = full + C::kStages;
    uint64_t* sf_full = empty + C::kStages;
    uint64_t* acc_full = sf_full + C::kStages;
    uint64_t* acc_empty = acc_full + 1;
    uint64_t* mma_done = acc_empty + 1;
    uint32_t* tmem_ptr = reinterpret_cast<uint32_t*>(smem + C::kMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMisc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int pair = (int)cluster_id_x(), n_pairs = (int)num_clusters_x();
    const int total = args.total_pm_tiles * args.n_tiles;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1 + 2 * kScaleWarps);  // producer (+ A/B bytes) and the scale warps
            mbar_init(&empty[s], 1);
            mbar_init(&sf_full[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 2 * kEpiWarps);
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
        if (args.any_k) {
            tma_prefetch_desc(&a_map);
            tma_prefetch_desc(&b_map);
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_ptr, kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();  // both CTAs' barriers initialised and TMEM allocated
    tc_fence_after();
    const uint32_t tmem_base = *tmem_ptr;

    // Each role's code sits inside its warpgroups' setmaxnreg branch, so the
    // compiler gives the epilogue the raised register budget.
    if (warp >= kFirstEpiWarp) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh));
        // ------------------------------------------------ epilogue (both CTAs)
        constexpr int kCols = BN / 2;
        const int quad = warp & 3;
        const int half = (warp - kFirstEpiWarp) >> 2;
        const int r = quad * 32 + lane;
        EpiAmax am = epi_amax_init(args, lane);
        uint32_t tl_i = 0;
        for (int t = pair; t < total; t += n_pairs, ++tl_i) {
            const PairTile tl = decode<C::kStageK>(args, t, rank);
            const GemmGroup& gr = args.groups[tl.g];
            int ok = 1;
            if (lane == 0) ok = wait_or_abort(acc_full, tl_i & 1, args.status, abort_flag);
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            const int out_row = tl.mt_local * BM + r;
            const bool row_ok = out_row < gr.rows_valid;
            float alpha = 1.0f;
            if (FMT == 1) {
                // row-scaled A: this lane's row's own outer scale (rows past the group's are not stored)
                const float aa = !args.a_row_scaled ? args.a_amax[gr.amax_idx]
                                 : row_ok ? args.a_amax[gr.a_row0 + out_row] : 0.0f;
                const float ga = __fdiv_rn(aa, 2688.0f);
                const float gb = __fdiv_rn(args.b_amax[gr.amax_idx], 2688.0f);
                alpha = __fmul_rn(ga, gb);
            }
            const int col0 = tl.n_tile * BN + half * kCols;
            const int64_t rowoff = gr.c_off + (int64_t)out_row * args.ldc + col0;
            const uint32_t taddr = tmem_base + (uint32_t)(half * kCols) + ((uint32_t)(quad * 32) << 16);
            auto release = [&] {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) arrive_leader(acc_empty, rank);
            };
            if (args.c_tma && tl.mt_local * BM + BM <= gr.rows_valid)
                epilogue_slice_tma<kCols>(args, &c_map, smem + C::kEpi + (warp - kFirstEpiWarp) * 4096, taddr,
                                          tl.num_kb > 0, alpha, col0, gr.c_row0 + tl.mt_local * BM + quad * 32, lane,
                                          am, release);
            else
                epilogue_slice<kCols>(args, taddr, tl.num_kb > 0, alpha, col0, rowoff, row_ok, am, release);
        }
        epi_amax_publish(args, am, lane);
        if (lane == 0) bulk_wait_group0();  // this warp's C stores completed before the CTA exits
    } else {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));
        if (warp == 0) {
            // ------------------------------------------------ TMA producer (both CTAs)
            // Straight-line issue as in gemm.cu: PTX-loop waits, copies guarded by
            // the CTA's live flag.
            if (lane == 0) {
                uint32_t it = 0, n_armed = 0;
                const uint32_t leader = rank == 0 ? 1u : 0u;
                for (int t = pair; t < total; t += n_pairs) {
                    const PairTile tl = decode<C::kStageK>(args, t, rank);
                    for (int kb = 0; kb < tl.num_kb; ++kb, ++it) {
                        const int s = it % C::kStages;
                        mbar_wait_flag_pair(&empty[s], ((it / C::kStages) & 1) ^ 1, abort_flag);
                        uint32_t live = live_flag(abort_flag);
                        // test hook: the leader arms the first stage, neither CTA loads into it
                        const uint32_t arm = live & leader;
                        live = (args.debug_drop_first_load && it == 0) ? 0u : live;
                        const int ka = tl.a_k0 + kb * C::kStageK, kbb = tl.b_k0 + kb * C::kStageK;
                        mbar_arrive_expect_tx_if(&full[s], 4u * kHalfTileBytes, arm);  // A + B of both CTAs
                        n_armed += arm;
                        const uint32_t bar = map_to_rank(&full[s], 0);
                        const int b_row = tl.b_row_pair + (int)rank * 128;
                        tma_load_2d_pair_if(smem + C::kA + s * kHalfTileBytes, &a_map, bar, FMT == 1 ? ka / 2 : ka, tl.a_row, live);
                        tma_load_2d_pair_if(smem + C::kB + s * kHalfTileBytes, &b_map, bar, FMT == 1 ? kbb / 2 : kbb, b_row, live);
                    }
                }
                // the leader drains the A/B copies of both CTAs (they complete on its full barriers)
                const uint32_t n = n_armed < (uint32_t)C::kStages ? n_armed : (uint32_t)C::kStages;
                for (uint32_t i = 0; i < n; ++i) {
                    const uint32_t k = n_armed - 1 - i;
                    if (rank == 0) mbar_wait(&full[k % C::kStages], (k / C::kStages) & 1, args.status);
                }
            }
        } else if (warp == 1) {
            // ------------------------------------------------ MMA issuer (leader CTA)
            if (lane == 0 && rank == 0) {
                constexpr int kMmas = C::kStageK / C::kMmaK;
                const uint64_t a_desc0 = smem_desc(smem_u32(smem + C::kA), 16, 1024, kSwizzle128B);
                const uint64_t b_desc0 = smem_desc(smem_u32(smem + C::kB), 16, 1024, kSwizzle128B);
                // ring position carried across tiles: slot s, phase parity par,
                // the slot's operand descriptors and its TMEM scale columns
                uint32_t s = 0, par = 0, tl_i = 0, live = 1u;
                uint64_t ad = a_desc0, bd = b_desc0;
                uint32_t sfa_col = tmem_base + C::kSfCol0;
                for (int t = pair; t < total; t += n_pairs, ++tl_i) {
                    const PairTile tl = decode<C::kStageK>(args, t, 0);
                    mbar_wait_flag_pair(acc_empty, (tl_i & 1) ^ 1, abort_flag);
                    tc_fence_after();
                    for (int kb = 0; kb < tl.num_kb; ++kb) {
                        live = mbar_wait_live_pair(&full[s], par, abort_flag);  // A/B bytes and scales
                        tc_fence_after();
                        const int n_mma = min(C::kStageK, tl.k_len - kb * C::kStageK) / C::kMmaK;
                        const uint32_t sfb_col = sfa_col + C::kSfaCols;
#pragma unroll
                        for (int j = 0; j < kMmas; ++j) {
                            const uint32_t on = (j < n_mma) ? live : 0u;
                            const uint32_t acc = (kb > 0 || j > 0) ? 1u : 0u;
                            if constexpr (FMT == 1)
                                tc_mma_nvf4_pair_if(tmem_base, ad + 2 * j, bd + 2 * j, make_idesc<1>(0), sfa_col + 4 * j,
                                                    sfb_col + 4 * C::kSfbHalves * j, acc, on);
                            else
                                tc_mma_mxf8_pair_if(tmem_base, ad + 2 * j, bd + 2 * j, make_idesc<2>((uint32_t)j), sfa_col,
                                                    sfb_col, acc, on);
                        }
                        tc_commit_pair_if(&empty[s], 0x3, live);
                        const bool wrap = s == (uint32_t)C::kStages - 1;
                        s = wrap ? 0u : s + 1;
                        par ^= wrap ? 1u : 0u;
                        ad = wrap ? a_desc0 : ad + (uint64_t)(kHalfTileBytes >> 4);
                        bd = wrap ? b_desc0 : bd + (uint64_t)(kHalfTileBytes >> 4);
                        sfa_col = wrap ? tmem_base + C::kSfCol0 : sfa_col + C::kSfColsPerStage;
                    }
                    tc_commit_pair_if(acc_full, 0x3, live);
                }
                tc_commit_pair(mma_done, 0x1);
                mbar_wait(mma_done, 0, args.status);
                if (*abort_flag) record_error(args.status, kErrTimeout);
            }
        } else if (warp >= kFirstScaleWarp) {
            // ------------------------------------------------ scale staging (both CTAs)
            const int q = warp & 3;
            uint32_t it = 0;
            bool ok = true;
            for (int t = pair; t < total && ok; t += n_pairs) {
                const PairTile tl = decode<C::kStageK>(args, t, rank);
                for (int kb = 0; kb < tl.num_kb; ++kb, ++it) {
                    const int s = it % C::kStages;
                    int good = 1;
                    if (lane == 0)
                        good = wait_or_abort(&sf_full[s], (it / C::kStages) & 1, args.status, abort_flag);
                    good = __shfl_sync(0xFFFFFFFFu, good, 0);
                    if (!good) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sfa_col = tmem_base + C::kSfCol0 + (uint32_t)s * C::kSfColsPerStage;
                    const uint32_t sfb_col = sfa_col + C::kSfaCols;
                    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
                    const uint8_t* sfa = smem + C::kSfa + s * C::kSfaBytes + lane * 16;
                    const uint8_t* sfb = smem + C::kSfb + s * C::kSfbBytes + lane * 16;
                    stage_block_scales<C::kAtomsK, C::kSfbHalves>(sfa_col, sfb_col, lane_base, q, sfa, sfb);
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) arrive_leader(&full[s], rank);
                }
            }
        } else if (warp == kScaleLoadWarp) {
            // ------------------------------------------------ block-scale loader (both CTAs)
            // This CTA's A scale tiles and the B scale tiles of all 256 columns,
            // on its own thread (every copy costs its issuing thread ~100 cycles).
            if (lane == 0) {
                uint32_t it = 0, n_armed = 0;
                for (int t = pair; t < total; t += n_pairs) {
                    const PairTile tl = decode<C::kStageK>(args, t, rank);
                    for (int kb = 0; kb < tl.num_kb; ++kb, ++it) {
                        const int s = it % C::kStages;
                        mbar_wait_flag_pair(&empty[s], ((it / C::kStages) & 1) ^ 1, abort_flag);
                        const uint32_t live = live_flag(abort_flag);
                        const int ka = tl.a_k0 + kb * C::kStageK, kbb = tl.b_k0 + kb * C::kStageK;
                        const int left = tl.k_len - kb * C::kStageK;
                        const int atoms = min(C::kAtomsK, (left + C::kElemPerAtom - 1) / C::kElemPerAtom);
                        const uint32_t sf_bytes = (uint32_t)atoms * 512u;
                        mbar_arrive_expect_tx_if(&sf_full[s], sf_bytes * (1 + C::kSfbHalves), live);
                        n_armed += live;
                        bulk_load_if(smem + C::kSfa + s * C::kSfaBytes,
                                     args.a_scale + ((int64_t)(tl.a_row / 128) * args.a_scale_ctiles + ka / C::kElemPerAtom) * 512,
                                     sf_bytes, &sf_full[s], live);
#pragma unroll
                        for (int h = 0; h < C::kSfbHalves; ++h) {
                            const int brow = tl.b_row_pair + h * 128;
                            bulk_load_if(smem + C::kSfb + s * C::kSfbBytes + h * C::kAtomsK * 512,
                                         args.b_scale + ((int64_t)(brow / 128) * args.b_scale_ctiles + kbb / C::kElemPerAtom) * 512,
                                         sf_bytes, &sf_full[s], live);
                        }
                    }
                }
                const uint32_t n = n_armed < (uint32_t)C::kStages ? n_armed : (uint32_t)C::kStages;
                for (uint32_t i = 0; i < n; ++i) {
                    const uint32_t k = n_armed - 1 - i;
                    mbar_wait(&sf_full[k % C::kStages], (k / C::kStages) & 1, args.status);
                }
            }
        }
    }  // warpgroups 0-1

    // After an abort, copies this CTA issued into stages the leader never
    // armed complete on no barrier anyone waits for: give them a bounded
    // grace period (a copy lands within microseconds) before the CTA can exit.
    if (threadIdx.x == 0 && *abort_flag) grace_wait_ns(kAbortGraceNs);
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the partner no longer issues MMAs, copies or arrivals that reach this CTA
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

template <int FMT>
cudaError_t set_smem()
{
    using C = Cfg<FMT>;
    return cudaFuncSetAttribute(gemm_pair_kernel<FMT>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, C::kAlloc);
}

}  // namespace gemm2

cudaError_t init_gemm_pair_attributes(bool* usable)
{
    *usable = false;
    cudaError_t e = gemm2::set_smem<1>();
    if (e == cudaSuccess) e = gemm2::set_smem<2>();
    // The register split assumes the launch allocation is 128 registers per
    // thread (kThreads x 128 = 65536).  With any other count, setmaxnreg.inc
    // could wait for registers that never come free, so the pair kernel is
    // then not used (the single-CTA kernel takes its GEMMs).
    cudaFuncAttributes a1{}, a2{};
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&a1, gemm2::gemm_pair_kernel<1>);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&a2, gemm2::gemm_pair_kernel<2>);
    if (e == cudaSuccess) *usable = a1.numRegs == 128 && a2.numRegs == 128;
    return e;
}

cudaError_t launch_gemm_pair(const void* a_map, const void* b_map, const void* c_map, const GemmArgs& g, int num_sms,
                             cudaStream_t s)
{
    const int tiles = g.total_pm_tiles * g.n_tiles;
    if (tiles == 0) return cudaSuccess;
    const int pairs = tiles < num_sms / 2 ? tiles : num_sms / 2;
    const CUtensorMap& am = *reinterpret_cast<const CUtensorMap*>(a_map);
    const CUtensorMap& bm = *reinterpret_cast<const CUtensorMap*>(b_map);
    const CUtensorMap& cm = *reinterpret_cast<const CUtensorMap*>(c_map);
    if (g.fmt == 1)
        gemm2::gemm_pair_kernel<1><<<2 * pairs, gemm2::kThreads, gemm2::Cfg<1>::kAlloc, s>>>(am, bm, cm, g);
    else
        gemm2::gemm_pair_kernel<2><<<2 * pairs, gemm2::kThreads, gemm2::Cfg<2>::kAlloc, s>>>(am, bm, cm, g);
    return cudaGetLastError();
}

}  // namespace nvq
