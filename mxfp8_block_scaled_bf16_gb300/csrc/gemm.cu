// gemm.cu -- block-scaled GEMMs on the 5th-generation tensor cores (tcgen05)
// for the three GEMMs of a linear layer (forward, dgrad, wgrad) and their
// grouped (MoE) forms, in TN form: C[r][c] = alpha * sum_k A[r][k] B[c][k].
//
// Method: "Add an NVFP4 quantization converter" (torchtitan PR #3914): the
// NVFP4 GEMM with E4M3 1x16 block scales and an FP32 tensor scale folded into
// alpha; "Hybrid quantization" (TransformerEngine PR #2817, Flowchart): the
// MXFP8 GEMM (E8M0 1x32 block scales) on direction-specific sub-storages,
// and the grouped GEMM over experts.
//
// Structure: a persistent kernel, one CTA per SM, each CTA walking output
// tiles of 128 x BN (BN = 256 when the output width allows, else 128) in a
// static round-robin order (column tiles fastest, so the CTAs in flight share
// A rows and sweep B from L2).  15 warps:
//   warp 0      TMA producer: A (128 rows x 128 bytes) and B (BN rows x 128
//               bytes) tiles with cp.async.bulk.tensor (128B swizzle) into a
//               ring of smem stages (full/empty mbarriers);
//   warp 1      TMEM owner and MMA issuer: 4 block-scaled MMAs per stage
//               (NVFP4: kind::mxf4nvf4 scale_vec::4X, K = 64; MXFP8:
//               kind::mxf8f6f4 scale_vec::1X, K = 32, the scale byte chosen by
//               the scale-factor id) into one of the TMEM accumulator stages;
//   warps 2..5  scale staging into TMEM with tcgen05.st, warp w writing lane
//               quadrant q = w % 4 (the smem->TMEM tcgen05.cp path runs in the
//               MMA's in-order pipe, where it cost more than the MMAs
//               themselves).  A 128x4 scale tile is 32 rows of 16 bytes, row l
//               holding tile rows l, l+32, l+64, l+96.  The MMA reads the A
//               scales of rows 32q..32q+31 from quadrant q, column base + q, so
//               warp q writes only word q of each row there; every quadrant
//               reads the B scales of all N columns, so each gets the whole
//               16-byte rows (4 columns per tile) -- both found by testing
//               layouts against the exact results;
//   warps 6..13 epilogue: warp w reads TMEM lane quadrant w % 4, half
//               (w - 6) / 4 of the columns; after its last load it releases the
//               accumulator to the MMA warp, then stores the scaled (+ bias)
//               bf16 / fp32 rows while the next tile's MMAs run;
//   warp 14     block-scale loader: the stage's A and B scale tiles with
//               cp.async.bulk (a separate thread from the A/B producer, since
//               every copy costs its issuing thread ~100 cycles).
// Every mbarrier wait is bounded; a wait that runs out records
// NVQ_ERR_TIMEOUT and raises a CTA-wide abort flag so all roles leave their
// loops; the producer then waits (bounded) for its copies in flight and the
// MMA warp for its tensor-core work before TMEM is freed.
#include <cuda.h>

#include "gemm_epilogue.cuh"
#include "nvq_device.cuh"
#include "nvq_kernels.h"

namespace nvq {

namespace gemm {

constexpr int BM = 128;
constexpr int kTileBytesA = 128 * 128;
constexpr int kScaleWarps = 4;
constexpr int kEpiWarps = 8;
constexpr int kFirstEpiWarp = 2 + kScaleWarps;
constexpr int kScaleLoadWarp = kFirstEpiWarp + kEpiWarps;  // block-scale copies
constexpr int kThreads = 32 * (kScaleLoadWarp + 1);
constexpr uint32_t kTmemCols = 512;

template <int FMT, int BN>
struct Cfg {
    static constexpr int kStageK = FMT == 1 ? 256 : 128;        // elements per stage (128 bytes)
    static constexpr int kMmaK = FMT == 1 ? 64 : 32;
    static constexpr int kAtomsK = FMT == 1 ? 4 : 1;            // 128x4 scale tiles along K per stage
    static constexpr int kElemPerAtom = FMT == 1 ? 64 : 128;
    static constexpr int kBHalves = BN / 128;
    static constexpr int kStages = BN == 256 ? 4 : 6;
    static constexpr int kAccStages = BN == 256 ? 1 : 2;
    static constexpr int kTileBytesB = BN * 128;
    static constexpr int kSfaBytes = kAtomsK * 512;
    static constexpr int kSfbBytes = kAtomsK * 512 * kBHalves;
    static constexpr uint32_t kSfaCols = 4 * kAtomsK;
    static constexpr uint32_t kSfbCols = 4 * kAtomsK * kBHalves;
    static constexpr uint32_t kSfCol0 = BN * kAccStages;
    static constexpr uint32_t kSfColsPerStage = kSfaCols + kSfbCols;
    static_assert(kSfCol0 + kStages * kSfColsPerStage <= kTmemCols, "TMEM budget");
    // shared memory layout (offsets from a 1024-aligned base)
    static constexpr int kA = 0;
    static constexpr int kB = kA + kStages * kTileBytesA;
    static constexpr int kSfa = kB + kStages * kTileBytesB;
    static constexpr int kSfb = kSfa + kStages * kSfaBytes;
    static constexpr int kBar = kSfb + kStages * kSfbBytes;
    static constexpr int kNumBars = 4 * kStages + 2 * kAccStages + 1;  // full, empty, sf_ready, sf_full, acc x2, done
    static constexpr int kMisc = kBar + kNumBars * 8;  // tmem address, abort flag
    static constexpr int kAlloc = kMisc + 16 + 1024;
    static_assert(kAlloc <= 232448, "shared memory budget");
};

// Instruction descriptor (kind::mxf4nvf4 / kind::mxf8f6f4 block-scaled):
// bits 4-5 B scale id, 7-9 A type, 10-12 B type, 15/16 K-major (0),
// 17-22 N >> 3, 23 scale type (0 UE4M3, 1 UE8M0), 24-28 M >> 4, 29-30 A scale id.
template <int FMT, int BN>
__device__ __forceinline__ uint32_t make_idesc(uint32_t sf_id)
{
    uint32_t d = 0;
    if (FMT == 1) d |= (1u << 7) | (1u << 10);  // E2M1 x E2M1 (E4M3 = 0 for MXFP8)
    d |= (uint32_t)(BN >> 3) << 17;
    if (FMT == 2) d |= 1u << 23;
    d |= (uint32_t)(BM >> 4) << 24;
    d |= (sf_id & 3) << 4;
    d |= (sf_id & 3) << 29;
    return d;
}

struct Tile {
    int g, mt_local, n_tile, a_row, b_row, a_k0, b_k0, k_len, num_kb;
};

template <int BN, int STAGE_K>
__device__ __forceinline__ Tile decode(const GemmArgs& a, int t)
{
    Tile r;
    const int m_tile = t / a.n_tiles;
    r.n_tile = t - m_tile * a.n_tiles;
    // last group whose first tile <= m_tile (empty groups own no tile):
    // fixed-length branchless search over at most kMaxGroups groups
    int lo = 0;
#pragma unroll
    for (int step = kMaxGroups / 2; step >= 1; step >>= 1) {
        const int mid = lo + step;
        lo = (mid < a.G && a.groups[mid].m_tile0 <= m_tile) ? mid : lo;
    }
    const GemmGroup& gr = a.groups[lo];
    r.g = lo;
    r.mt_local = m_tile - gr.m_tile0;
    r.a_row = gr.a_row0 + r.mt_local * BM;
    r.b_row = gr.b_row0 + r.n_tile * BN;
    r.a_k0 = gr.a_k0;
    r.b_k0 = gr.b_k0;
    r.k_len = gr.k_len;
    r.num_kb = (gr.k_len + STAGE_K - 1) / STAGE_K;
    return r;
}

// Bounded wait that also gives up when another role has aborted the CTA.
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
                return false;
            }
        }
    }
}

template <int FMT, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap a_map, const __grid_constant__ CUtensorMap b_map,
                const __grid_constant__ GemmArgs args)
{
    using C = Cfg<FMT, BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBar);
    uint64_t* empty = full + C::kStages;
    uint64_t* sf_ready = empty + C::kStages;
    uint64_t* acc_full = sf_ready + C::kStages;
    uint64_t* acc_empty = acc_full + C::kAccStages;
    uint64_t* mma_done = acc_empty + C::kAccStages;
    uint64_t* sf_full = mma_done + 1;
    uint32_t* tmem_ptr = reinterpret_cast<uint32_t*>(smem + C::kMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMisc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int total = args.total_m_tiles * args.n_tiles;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&sf_ready[s], kScaleWarps);
            mbar_init(&sf_full[s], 1);
        }
        for (int s = 0; s < C::kAccStages; ++s) {
            mbar_init(&acc_full[s], 1);
            mbar_init(&acc_empty[s], kEpiWarps);
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
        if (args.any_k) {
            tma_prefetch_desc(&a_map);
            tma_prefetch_desc(&b_map);
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_ptr, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_ptr;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (A and B tiles)
        // Straight-line issue: waits are PTX loops (mbar_wait_flag) and every
        // copy is guarded by the CTA's live flag instead of a branch.  Each
        // copy costs its issuing thread on the order of 100 cycles, so the
        // block-scale copies have their own thread (the scale loader warp).
        if (lane == 0) {
            uint32_t it = 0, n_armed = 0;
            for (int t = blockIdx.x; t < total; t += gridDim.x) {
                const Tile tl = decode<BN, C::kStageK>(args, t);
                for (int kb = 0; kb < tl.num_kb; ++kb, ++it) {
                    const int s = it % C::kStages;
                    mbar_wait_flag(&empty[s], ((it / C::kStages) & 1) ^ 1, abort_flag);
                    uint32_t live = live_flag(abort_flag);
                    // test hook: live = 2 arms the stage but loads nothing
                    live = (args.debug_drop_first_load && it == 0) ? 2u * live : live;
                    const int ka = tl.a_k0 + kb * C::kStageK, kbb = tl.b_k0 + kb * C::kStageK;
                    mbar_arrive_expect_tx_if(&full[s], (uint32_t)(kTileBytesA + C::kTileBytesB), live);
                    n_armed += live != 0 ? 1u : 0u;
                    live = live == 1 ? 1u : 0u;
                    tma_load_2d_if(smem + C::kA + s * kTileBytesA, &a_map, &full[s], FMT == 1 ? ka / 2 : ka, tl.a_row, live);
                    tma_load_2d_if(smem + C::kB + s * C::kTileBytesB, &b_map, &full[s], FMT == 1 ? kbb / 2 : kbb, tl.b_row,
                                   live);
                }
            }
            // drain: the armed stages are a prefix of the iterations (abort is
            // sticky); the last copy issued into each stage has landed before exit
            const uint32_t n = n_armed < (uint32_t)C::kStages ? n_armed : (uint32_t)C::kStages;
            for (uint32_t i = 0; i < n; ++i) {
                const uint32_t k = n_armed - 1 - i;
                mbar_wait(&full[k % C::kStages], (k / C::kStages) & 1, args.status);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        // Straight-line issue as in the producer: the per-stage MMAs are
        // unrolled (the short last stage of a ragged K predicates the rest
        // off), descriptors advance by adding to the start-address field
        // (smem addresses < 256 KB keep it within its 14 bits).
        if (lane == 0) {
            constexpr int kMmas = C::kStageK / C::kMmaK;
            const uint64_t a_desc0 = smem_desc(smem_u32(smem + C::kA), 16, 1024, kSwizzle128B);
            const uint64_t b_desc0 = smem_desc(smem_u32(smem + C::kB), 16, 1024, kSwizzle128B);
            uint32_t it = 0, tl_i = 0;
            for (int t = blockIdx.x; t < total; t += gridDim.x, ++tl_i) {
                const Tile tl = decode<BN, C::kStageK>(args, t);
                const int as = tl_i % C::kAccStages;
                mbar_wait_flag(&acc_empty[as], ((tl_i / C::kAccStages) & 1) ^ 1, abort_flag);
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(as * BN);
                for (int kb = 0; kb < tl.num_kb; ++kb, ++it) {
                    const int s = it % C::kStages;
                    const uint32_t par = (it / C::kStages) & 1;
                    mbar_wait_flag(&full[s], par, abort_flag);
                    mbar_wait_flag(&sf_ready[s], par, abort_flag);
                    tc_fence_after();
                    const uint32_t live = live_flag(abort_flag);
                    const int n_mma = min(C::kStageK, tl.k_len - kb * C::kStageK) / C::kMmaK;
                    const uint32_t sfa_col = tmem_base + C::kSfCol0 + (uint32_t)s * C::kSfColsPerStage;
                    const uint32_t sfb_col = sfa_col + C::kSfaCols;
                    const uint64_t ad = a_desc0 + (uint64_t)((s * kTileBytesA) >> 4);
                    const uint64_t bd = b_desc0 + (uint64_t)((s * C::kTileBytesB) >> 4);
#pragma unroll
                    for (int j = 0; j < kMmas; ++j) {
                        const uint32_t on = (j < n_mma) ? live : 0u;
                        const uint32_t acc = (kb > 0 || j > 0) ? 1u : 0u;
                        if constexpr (FMT == 1)
                            tc_mma_nvf4_if(d_tmem, ad + 2 * j, bd + 2 * j, make_idesc<1, BN>(0), sfa_col + 4 * j,
                                           sfb_col + 4 * C::kBHalves * j, acc, on);
                        else
                            tc_mma_mxf8_if(d_tmem, ad + 2 * j, bd + 2 * j, make_idesc<2, BN>((uint32_t)j), sfa_col,
                                           sfb_col, acc, on);
                    }
                    tc_commit_if(&empty[s], live);
                }
                tc_commit_if(&acc_full[as], live_flag(abort_flag));
            }
            // all of this thread's tensor-core work has finished before TMEM is freed
            tc_commit(mma_done);
            mbar_wait(mma_done, 0, args.status);
            if (*abort_flag) record_error(args.status, kErrTimeout);
        }
    } else if (warp < kFirstEpiWarp) {
        // ------------------------------------------------ scale staging (warps 2..5)
        // A 512-byte 128x4 scale tile is 32 rows of 16 bytes; row l holds tile
        // rows l, l+32, l+64, l+96 (one 32-bit word each: the scales of the
        // tile's four 16- or 32-element k-blocks).  A scales: the MMA of lane
        // quadrant q reads word q of row l from TMEM lane 32 q + l, column
        // base + q.  B scales: every quadrant reads all of them, so warp q
        // writes the whole 16-byte row l into lane l of its quadrant (4
        // columns), the layout a replicating smem->TMEM copy produces.
        const int q = warp & 3;
        uint32_t it = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
            const Tile tl = decode<BN, C::kStageK>(args, t);
            for (int kb = 0; kb < tl.num_kb; ++kb, ++it) {
                const int s = it % C::kStages;
                int good = 1;
                if (lane == 0) good = wait_or_abort(&sf_full[s], (it / C::kStages) & 1, args.status, abort_flag);
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
                stage_block_scales<C::kAtomsK, C::kBHalves>(sfa_col, sfb_col, lane_base, q, sfa, sfb);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sf_ready[s]);
            }
        }
    } else if (warp == kScaleLoadWarp) {
        // ------------------------------------------------ block-scale loader
        // The 512-byte 128x4 scale tiles of A and B for each stage, into the
        // stage's scale slots, completing on sf_full (same ring and empty
        // barriers as the A/B tiles).
        if (lane == 0) {
            uint32_t it = 0, n_armed = 0;
            for (int t = blockIdx.x; t < total; t += gridDim.x) {
                const Tile tl = decode<BN, C::kStageK>(args, t);
                for (int kb = 0; kb < tl.num_kb; ++kb, ++it) {
                    const int s = it % C::kStages;
                    mbar_wait_flag(&empty[s], ((it / C::kStages) & 1) ^ 1, abort_flag);
                    const uint32_t live = live_flag(abort_flag);
                    const int ka = tl.a_k0 + kb * C::kStageK, kbb = tl.b_k0 + kb * C::kStageK;
                    const int left = tl.k_len - kb * C::kStageK;
                    const int atoms = min(C::kAtomsK, (left + C::kElemPerAtom - 1) / C::kElemPerAtom);
                    const uint32_t sf_bytes = (uint32_t)atoms * 512u;
                    mbar_arrive_expect_tx_if(&sf_full[s], sf_bytes * (1 + C::kBHalves), live);
                    n_armed += live;
                    bulk_load_if(smem + C::kSfa + s * C::kSfaBytes,
                                 args.a_scale + ((int64_t)(tl.a_row / 128) * args.a_scale_ctiles + ka / C::kElemPerAtom) * 512,
                                 sf_bytes, &sf_full[s], live);
#pragma unroll
                    for (int h = 0; h < C::kBHalves; ++h)
                        bulk_load_if(smem + C::kSfb + s * C::kSfbBytes + h * C::kAtomsK * 512,
                                     args.b_scale +
                                         ((int64_t)(tl.b_row / 128 + h) * args.b_scale_ctiles + kbb / C::kElemPerAtom) * 512,
                                     sf_bytes, &sf_full[s], live);
                }
            }
            const uint32_t n = n_armed < (uint32_t)C::kStages ? n_armed : (uint32_t)C::kStages;
            for (uint32_t i = 0; i < n; ++i) {
                const uint32_t k = n_armed - 1 - i;
                mbar_wait(&sf_full[k % C::kStages], (k / C::kStages) & 1, args.status);
            }
        }
    } else {
        // ------------------------------------------------ epilogue (warps 6..13)
        constexpr int kCols = BN / 2;       // columns per warp
        const int quad = warp & 3;
        const int half = (warp - kFirstEpiWarp) >> 2;
        const int r = quad * 32 + lane;     // tile row = TMEM lane
        EpiAmax am = epi_amax_init(args, lane);
        uint32_t tl_i = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++tl_i) {
            const Tile tl = decode<BN, C::kStageK>(args, t);
            const GemmGroup& gr = args.groups[tl.g];
            const int as = tl_i % C::kAccStages;
            // one lane polls, the warp reconverges before the .sync.aligned TMEM loads
            int ok = 1;
            if (lane == 0) ok = wait_or_abort(&acc_full[as], (tl_i / C::kAccStages) & 1, args.status, abort_flag);
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
            const uint32_t taddr = tmem_base + (uint32_t)(as * BN + half * kCols) + ((uint32_t)(quad * 32) << 16);
            epilogue_slice<kCols>(args, taddr, tl.num_kb > 0, alpha, col0, rowoff, row_ok, am, [&] {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[as]);
            });
        }
        epi_amax_publish(args, am, lane);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

template <int FMT, int BN>
cudaError_t set_smem()
{
    return cudaFuncSetAttribute(gemm_kernel<FMT, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<FMT, BN>::kAlloc);
}

template <int FMT, int BN>
void launch(const CUtensorMap& am, const CUtensorMap& bm, const GemmArgs& g, int grid, cudaStream_t s)
{
    gemm_kernel<FMT, BN><<<grid, kThreads, Cfg<FMT, BN>::kAlloc, s>>>(am, bm, g);
}

}  // namespace gemm

cudaError_t init_gemm_attributes()
{
    cudaError_t e = gemm::set_smem<1, 128>();
    if (e == cudaSuccess) e = gemm::set_smem<1, 256>();
    if (e == cudaSuccess) e = gemm::set_smem<2, 128>();
    if (e == cudaSuccess) e = gemm::set_smem<2, 256>();
    return e;
}

int gemm_block_n(int64_t n_out) { return n_out % 256 == 0 ? 256 : 128; }

cudaError_t launch_gemm(const void* a_map, const void* b_map, const GemmArgs& g, int num_sms, cudaStream_t s)
{
    const int tiles = g.total_m_tiles * g.n_tiles;
    if (tiles == 0) return cudaSuccess;
    const int grid = tiles < num_sms ? tiles : num_sms;
    const CUtensorMap& am = *reinterpret_cast<const CUtensorMap*>(a_map);
    const CUtensorMap& bm = *reinterpret_cast<const CUtensorMap*>(b_map);
    if (g.fmt == 1) {
        if (g.block_n == 256) gemm::launch<1, 256>(am, bm, g, grid, s);
        else gemm::launch<1, 128>(am, bm, g, grid, s);
    } else {
        if (g.block_n == 256) gemm::launch<2, 256>(am, bm, g, grid, s);
        else gemm::launch<2, 128>(am, bm, g, grid, s);
    }
    return cudaGetLastError();
}

}  // namespace nvq
