// nvq_device.cuh -- device helpers shared by the libnvq kernels (sm_103a).
//
// Inline PTX wrappers for mbarriers, TMA (cp.async.bulk[.tensor] loads and
// stores) and the 5th-generation tensor core (tcgen05: TMEM alloc, block-scaled
// MMA, TMEM loads and stores), plus the element-format conversions and the
// Philox4x32-10 generator used by stochastic rounding.
//
// Every wait here is bounded: a wait that runs past its time limit records
// NVQ_ERR_TIMEOUT in the device status word (or raises the CTA's abort flag,
// for the PTX-loop wait) and gives up, so a broken pipeline ends the kernel
// instead of spinning forever.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace nvq {

// Device-side errors go to the library's status word (first error wins),
// passed to every kernel as a pointer; read and cleared by
// nvq_get_device_status().
__device__ __forceinline__ void record_error(int* status, int code)
{
    if (status) atomicCAS(status, 0, code);
}

constexpr int kErrTimeout = 7;
constexpr int kErrBounds = 8;

// Time limit of one bounded wait (ns).  Far above any legitimate stall of
// these kernels (a full pipeline stage is microseconds).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbarrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* status)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63) == 63 && globaltimer_ns() - t0 > kWaitLimitNs) {
            record_error(status, kErrTimeout);
            return false;
        }
    }
}

// Bounded wait whose whole polling loop is PTX, so no value flows back into
// the caller's control flow: the issuing loops of the GEMM's producer and MMA
// threads stay free of data-dependent branches, which on this part slowed
// tensor-core and TMA issue (a loop around tcgen05.mma issue measured ~1.5x
// slower than straight-line issue).  Returns when the phase completes, when
// *abort_flag is already set, or after kWaitLimitNs, in which case it sets
// *abort_flag itself; callers read the flag afterwards (a "live" predicate)
// and guard their async work with it.
__device__ __forceinline__ void mbar_wait_flag(uint64_t* bar, uint32_t parity, volatile int* abort_flag)
{
    asm volatile(
        "{\n\t.reg .pred P1;\n\t.reg .b64 t0, t1;\n\t.reg .b32 ab;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 P1, [%0], %1;\n\t"
        "@P1 bra.uni DONE;\n\t"
        "mov.u64 t0, %%globaltimer;\n\t"
        "LOOP:\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 P1, [%0], %1;\n\t"
        "@P1 bra.uni DONE;\n\t"
        "ld.volatile.shared.u32 ab, [%2];\n\t"
        "setp.ne.u32 P1, ab, 0;\n\t"
        "@P1 bra.uni DONE;\n\t"
        "mov.u64 t1, %%globaltimer;\n\t"
        "sub.u64 t1, t1, t0;\n\t"
        "setp.lt.u64 P1, t1, %3;\n\t"
        "@P1 bra.uni LOOP;\n\t"
        "st.volatile.shared.u32 [%2], 1;\n\t"
        "DONE:\n\t}" ::"r"(smem_u32(bar)),
        "r"(parity), "r"(smem_u32(const_cast<int*>(abort_flag))), "l"(kWaitLimitNs)
        : "memory");
}

// mbar_wait_flag that also yields the live predicate: 1 when the phase
// completed, 0 when the wait gave up (abort flag set by another thread, or
// the time limit, in which case it sets the flag).
__device__ __forceinline__ uint32_t mbar_wait_live(uint64_t* bar, uint32_t parity, volatile int* abort_flag)
{
    uint32_t live;
    asm volatile(
        "{\n\t.reg .pred P1;\n\t.reg .b64 t0, t1;\n\t.reg .b32 ab;\n\t"
        "mov.u32 %0, 1;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 P1, [%1], %2;\n\t"
        "@P1 bra.uni DONE;\n\t"
        "mov.u64 t0, %%globaltimer;\n\t"
        "LOOP:\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 P1, [%1], %2;\n\t"
        "@P1 bra.uni DONE;\n\t"
        "ld.volatile.shared.u32 ab, [%3];\n\t"
        "setp.ne.u32 P1, ab, 0;\n\t"
        "@P1 bra.uni GAVEUP;\n\t"
        "mov.u64 t1, %%globaltimer;\n\t"
        "sub.u64 t1, t1, t0;\n\t"
        "setp.lt.u64 P1, t1, %4;\n\t"
        "@P1 bra.uni LOOP;\n\t"
        "st.volatile.shared.u32 [%3], 1;\n\t"
        "GAVEUP:\n\t"
        "mov.u32 %0, 0;\n\t"
        "DONE:\n\t}"
        : "=r"(live)
        : "r"(smem_u32(bar)), "r"(parity), "r"(smem_u32(const_cast<int*>(abort_flag))), "l"(kWaitLimitNs)
        : "memory");
    return live;
}

// CTA-pair forms of the two waits above: a wait that runs out also raises the
// partner CTA's abort flag (the same shared-memory offset in CTA rank ^ 1 of
// the cluster, mapped only on that path so it costs no register), so both
// CTAs of the pair stop issuing copies and tensor-core work together instead
// of the partner finding out only when its own waits run out.
__device__ __forceinline__ void mbar_wait_flag_pair(uint64_t* bar, uint32_t parity, volatile int* abort_flag)
{
    asm volatile(
        "{\n\t.reg .pred P1;\n\t.reg .b64 t0, t1;\n\t.reg .b32 ab, pr, pa;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 P1, [%0], %1;\n\t"
        "@P1 bra.uni DONE;\n\t"
        "mov.u64 t0, %%globaltimer;\n\t"
        "LOOP:\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 P1, [%0], %1;\n\t"
        "@P1 bra.uni DONE;\n\t"
        "ld.volatile.shared.u32 ab, [%2];\n\t"
        "setp.ne.u32 P1, ab, 0;\n\t"
        "@P1 bra.uni DONE;\n\t"
        "mov.u64 t1, %%globaltimer;\n\t"
        "sub.u64 t1, t1, t0;\n\t"
        "setp.lt.u64 P1, t1, %3;\n\t"
        "@P1 bra.uni LOOP;\n\t"
        "st.volatile.shared.u32 [%2], 1;\n\t"
        "mov.u32 pr, %%cluster_ctarank;\n\t"
        "xor.b32 pr, pr, 1;\n\t"
        "mapa.shared::cluster.u32 pa, %2, pr;\n\t"
        "st.relaxed.cluster.shared::cluster.u32 [pa], 1;\n\t"
        "DONE:\n\t}" ::"r"(smem_u32(bar)),
        "r"(parity), "r"(smem_u32(const_cast<int*>(abort_flag))), "l"(kWaitLimitNs)
        : "memory");
}

__device__ __forceinline__ uint32_t mbar_wait_live_pair(uint64_t* bar, uint32_t parity, volatile int* abort_flag)
{
    uint32_t live;
    asm volatile(
        "{\n\t.reg .pred P1;\n\t.reg .b64 t0, t1;\n\t.reg .b32 ab, pr, pa;\n\t"
        "mov.u32 %0, 1;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 P1, [%1], %2;\n\t"
        "@P1 bra.uni DONE;\n\t"
        "mov.u64 t0, %%globaltimer;\n\t"
        "LOOP:\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 P1, [%1], %2;\n\t"
        "@P1 bra.uni DONE;\n\t"
        "ld.volatile.shared.u32 ab, [%3];\n\t"
        "setp.ne.u32 P1, ab, 0;\n\t"
        "@P1 bra.uni GAVEUP;\n\t"
        "mov.u64 t1, %%globaltimer;\n\t"
        "sub.u64 t1, t1, t0;\n\t"
        "setp.lt.u64 P1, t1, %4;\n\t"
        "@P1 bra.uni LOOP;\n\t"
        "st.volatile.shared.u32 [%3], 1;\n\t"
        "mov.u32 pr, %%cluster_ctarank;\n\t"
        "xor.b32 pr, pr, 1;\n\t"
        "mapa.shared::cluster.u32 pa, %3, pr;\n\t"
        "st.relaxed.cluster.shared::cluster.u32 [pa], 1;\n\t"
        "GAVEUP:\n\t"
        "mov.u32 %0, 0;\n\t"
        "DONE:\n\t}"
        : "=r"(live)
        : "r"(smem_u32(bar)), "r"(parity), "r"(smem_u32(const_cast<int*>(abort_flag))), "l"(kWaitLimitNs)
        : "memory");
    return live;
}

// Raises the partner CTA's abort flag (the flag at the same offset in CTA
// rank ^ 1 of the cluster).
__device__ __forceinline__ void set_partner_abort(volatile int* abort_flag)
{
    asm volatile(
        "{\n\t.reg .b32 pr, pa;\n\t"
        "mov.u32 pr, %%cluster_ctarank;\n\t"
        "xor.b32 pr, pr, 1;\n\t"
        "mapa.shared::cluster.u32 pa, %0, pr;\n\t"
        "st.relaxed.cluster.shared::cluster.u32 [pa], 1;\n\t}" ::"r"(smem_u32(const_cast<int*>(abort_flag)))
        : "memory");
}

// Spins for `ns` nanoseconds of %globaltimer (bounded by construction).
__device__ __forceinline__ void grace_wait_ns(uint64_t ns)
{
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < ns) {
    }
}

// 1 while the CTA has not aborted (read after a mbar_wait_flag).
__device__ __forceinline__ uint32_t live_flag(volatile int* abort_flag) { return *abort_flag == 0 ? 1u : 0u; }

// Arrive with an expected transaction byte count, when live != 0.
__device__ __forceinline__ void mbar_arrive_expect_tx_if(uint64_t* bar, uint32_t bytes, uint32_t live)
{
    asm volatile(
        "{\n\t.reg .pred g;\n\tsetp.ne.b32 g, %2, 0;\n\t"
        "@g mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
        "r"(bytes), "r"(live)
        : "memory");
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_prefetch_desc(const void* desc)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(desc) : "memory");
}

// 2-D tiled load of box (x = inner, y = outer) into smem, completing on bar,
// issued only when live != 0.
__device__ __forceinline__ void tma_load_2d_if(void* dst, const void* desc, uint64_t* bar, int32_t x, int32_t y,
                                               uint32_t live)
{
    asm volatile(
        "{\n\t.reg .pred g;\n\tsetp.ne.b32 g, %5, 0;\n\t"
        "@g cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];\n\t}" ::"r"(smem_u32(dst)),
        "l"(desc), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(live)
        : "memory");
}

// Untiled bulk copy global -> smem (16-byte aligned, size % 16 == 0), completing
// on bar, issued only when live != 0.
__device__ __forceinline__ void bulk_load_if(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint32_t live)
{
    asm volatile(
        "{\n\t.reg .pred g;\n\tsetp.ne.b32 g, %4, 0;\n\t"
        "@g cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n\t}" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "r"(live)
        : "memory");
}

// 2-D tiled store smem -> global (bulk-group completion); x (inner) must be a
// multiple of 16 bytes, and neither coordinate negative.
__device__ __forceinline__ void tma_store_2d(const void* desc, const void* src, int32_t x, int32_t y)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(desc),
                 "r"(smem_u32(src)), "r"(x), "r"(y)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// This thread's bulk stores have finished reading their smem sources.
__device__ __forceinline__ void bulk_wait_group_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// This thread's bulk stores have completed.
__device__ __forceinline__ void bulk_wait_group0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Generic-proxy smem writes become visible to the async proxy (TMA).
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Arrive on an mbarrier once all prior tcgen05 async ops of this thread finish.
__device__ __forceinline__ void tc_commit(uint64_t* bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_commit_if(uint64_t* bar, uint32_t live)
{
    asm volatile(
        "{\n\t.reg .pred g;\n\tsetp.ne.b32 g, %1, 0;\n\t"
        "@g tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar)),
        "r"(live)
        : "memory");
}

// Shared-memory matrix descriptor (tcgen05): start, leading/stride byte
// offsets (>> 4), fixed version bits 46..48 = 0b001, swizzle mode in 61..63.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swz)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)(swz & 7) << 61;
    return d;
}

constexpr uint32_t kSwizzleNone = 0;
constexpr uint32_t kSwizzle128B = 2;

// D(tmem) (+)= A(smem) x B(smem)^T with per-16-block E4M3 scales (NVFP4),
// issued only when live != 0; `accumulate` = 0 overwrites D.
__device__ __forceinline__ void tc_mma_nvf4_if(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                               uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate,
                                               uint32_t live)
{
    asm volatile(
        "{\n\t.reg .pred p, g;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "setp.ne.b32 g, %7, 0;\n\t"
        "@g tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X"
        " [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate), "r"(live)
        : "memory");
}

// Same with E4M3 elements and per-32-block E8M0 scales (MXFP8), the scale byte
// of each k-step chosen by the scale-factor id in the instruction descriptor.
__device__ __forceinline__ void tc_mma_mxf8_if(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                               uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate,
                                               uint32_t live)
{
    asm volatile(
        "{\n\t.reg .pred p, g;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "setp.ne.b32 g, %7, 0;\n\t"
        "@g tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X"
        " [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate), "r"(live)
        : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns -> 32 registers per thread.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32"
        " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15,"
        " %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Issued after tmem_ld_wait(): the loaded registers pass through this empty
// statement, so no computation on them can be scheduled before the wait.
__device__ __forceinline__ void tmem_regs_ready(uint32_t (&r)[32])
{
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31]));
}

// 32 lanes x 1 column: lane i of the warp's lane quadrant gets v.
__device__ __forceinline__ void tmem_st_32x32b_x1(uint32_t taddr, uint32_t v)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}

// 32 lanes x 4 consecutive columns.
__device__ __forceinline__ void tmem_st_32x32b_x4(uint32_t taddr, const uint4& v)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// 32 lanes x N consecutive columns (N = 8, 16 or 32).
template <int N>
__device__ __forceinline__ void tmem_st_32x32b_xn(uint32_t taddr, const uint32_t (&r)[N])
{
    static_assert(N == 8 || N == 16 || N == 32, "store width");
    if constexpr (N == 8) {
        asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                     "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                     : "memory");
    } else if constexpr (N == 16) {
        asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
                     "%12, %13, %14, %15, %16};" ::"r"(taddr),
                     "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
                     "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
                     : "memory");
    } else {
        asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
                     "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, "
                     "%31, %32};" ::"r"(taddr),
                     "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
                     "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
                     "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
                     "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
                     : "memory");
    }
}

// One pipeline stage's block scales, shared memory -> TMEM, by the warp of
// lane quadrant q (TMEM lanes 32q..32q+31; `lane_base` = their address bits).
// The stage holds kAtomsK 128x4 scale tiles of A at `sfa` and kAtomsK x
// kBHalves tiles of B at `sfb` (512 bytes each, this lane's 16-byte row
// already added), laid out as the block-scaled MMA reads them:
//   A: the word of atom j for the row of this lane goes to column
//      sfa_col + 4j + q (the MMA reads column 4j + q in quadrant q);
//   B: the whole 16-byte tile row of atom j, half h, goes to columns
//      sfb_col + 4 (kBHalves j + h) .. + 3 in every quadrant.
// Each operand leaves in one wide store: the A word is written to all four
// columns of its atom (the three the MMA does not read in this quadrant get
// copies), because one wide store per operand ran faster than one narrow
// store per atom (forward GEMM 354 -> 334 us, dgrad 324 -> 295 us).  Atoms
// past a ragged stage end are written too (stale shared memory, in bounds);
// their MMAs are predicated off.
template <int kAtomsK, int kBHalves>
__device__ __forceinline__ void stage_block_scales(uint32_t sfa_col, uint32_t sfb_col, uint32_t lane_base, int q,
                                                   const uint8_t* sfa, const uint8_t* sfb)
{
    if constexpr (kAtomsK == 1) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(sfa + 4 * q);
        tmem_st_32x32b_x4(sfa_col + lane_base, make_uint4(w, w, w, w));
    } else {
        uint32_t ra[4 * kAtomsK];
#pragma unroll
        for (int j = 0; j < kAtomsK; ++j) {
            const uint32_t w = *reinterpret_cast<const uint32_t*>(sfa + 512 * j + 4 * q);
            ra[4 * j] = ra[4 * j + 1] = ra[4 * j + 2] = ra[4 * j + 3] = w;
        }
        tmem_st_32x32b_xn<4 * kAtomsK>(sfa_col + lane_base, ra);
    }
    constexpr int kNb = 4 * kAtomsK * kBHalves;
    if constexpr (kNb == 4) {
        tmem_st_32x32b_x4(sfb_col + lane_base, *reinterpret_cast<const uint4*>(sfb));
    } else {
        uint32_t rb[kNb];
#pragma unroll
        for (int j = 0; j < kAtomsK; ++j)
#pragma unroll
            for (int h = 0; h < kBHalves; ++h) {
                const uint4 u = *reinterpret_cast<const uint4*>(sfb + 512 * (h * kAtomsK + j));
                const int c = 4 * (kBHalves * j + h);
                rb[c] = u.x;
                rb[c + 1] = u.y;
                rb[c + 2] = u.z;
                rb[c + 3] = u.w;
            }
        tmem_st_32x32b_xn<kNb>(sfb_col + lane_base, rb);
    }
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ------------------------------------------------------------------ CTA pairs (clusters of 2)
__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_id_x()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t num_clusters_x()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// shared::cluster address of the same smem offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(const void* p, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}

// Relaxed cluster-scope arrive, for a signal that only orders tcgen05 work:
// the arriving thread has already waited for its TMEM stores / loads to
// complete (tcgen05.wait::st / ::ld) and fenced them with
// tcgen05.fence::before_thread_sync; the waiter issues
// tcgen05.fence::after_thread_sync before its MMAs.  On the CTA-pair GEMM the
// release form cost ~0.4 ms per forward GEMM (the MMA waited ~875 cycles per
// stage on it); the relaxed form gives the same, exact, results.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// tma_load_2d_pair issued only when live != 0.
__device__ __forceinline__ void tma_load_2d_pair_if(void* dst, const void* desc, uint32_t bar_cluster_addr, int32_t x,
                                                    int32_t y, uint32_t live)
{
    asm volatile(
        "{\n\t.reg .pred g;\n\tsetp.ne.b32 g, %5, 0;\n\t"
        "@g cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];\n\t}" ::"r"(smem_u32(dst)),
        "l"(desc), "r"(bar_cluster_addr), "r"(x), "r"(y), "r"(live)
        : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Arrive on the mbarrier at the same smem offset in every CTA of `mask` once
// all prior tcgen05 async ops of this thread (pair MMAs) have finished.
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar, uint16_t mask)
{
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(mask)
        : "memory");
}

// tc_commit_pair issued only when live != 0.
__device__ __forceinline__ void tc_commit_pair_if(uint64_t* bar, uint16_t mask, uint32_t live)
{
    asm volatile(
        "{\n\t.reg .pred g;\n\tsetp.ne.b32 g, %2, 0;\n\t"
        "@g tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}" ::"r"(
            smem_u32(bar)),
        "h"(mask), "r"(live)
        : "memory");
}

// Pair MMAs issued only when live != 0.
__device__ __forceinline__ void tc_mma_nvf4_pair_if(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                    uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate,
                                                    uint32_t live)
{
    asm volatile(
        "{\n\t.reg .pred p, g;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "setp.ne.b32 g, %7, 0;\n\t"
        "@g tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X"
        " [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate), "r"(live)
        : "memory");
}

__device__ __forceinline__ void tc_mma_mxf8_pair_if(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                    uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate,
                                                    uint32_t live)
{
    asm volatile(
        "{\n\t.reg .pred p, g;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "setp.ne.b32 g, %7, 0;\n\t"
        "@g tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X"
        " [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate), "r"(live)
        : "memory");
}

// 32-byte global store (256-bit vector; the address must be 32-byte aligned).
__device__ __forceinline__ void st_global_v8(void* dst, const uint32_t* w)
{
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

// ------------------------------------------------------------------ formats
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// E4M3 round-to-nearest-even with saturation to +-448.
__device__ __forceinline__ uint32_t e4m3_rn(float v)
{
    uint16_t r;  // both halves converted from v, so either byte is the code
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(v), "f"(v));
    return r & 0xFFu;
}

// Exact decode of an E4M3 code to fp32 (via f16, which holds every E4M3 value).
__device__ __forceinline__ float e4m3_to_f32(uint32_t code)
{
    uint32_t h2;
    uint16_t in = (uint16_t)(code | (code << 8));  // same code in both bytes
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
    return __half2float(__ushort_as_half((uint16_t)(h2 & 0xFFFF)));
}

// Four E4M3 codes (RN, satfinite) packed into 32 bits, element 0 in the low byte.
__device__ __forceinline__ uint32_t e4m3x4_rn(float a0, float a1, float a2, float a3)
{
    uint16_t lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(a1), "f"(a0));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(a3), "f"(a2));
    return (uint32_t)lo | ((uint32_t)hi << 16);
}

// Eight E2M1 codes (RN, satfinite) packed into 32 bits, element 0 in the low nibble.
__device__ __forceinline__ uint32_t e2m1x8_rn(const float (&v)[8])
{
    uint32_t out;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(out)
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
    return out;
}

// ------------------------------------------------------------------ packed fp32 pairs
// Two fp32 values in one 64-bit register pair (element 0 in the low word); the
// f32x2 instructions apply one IEEE operation, with the stated rounding, to
// each half -- the same result as two scalar operations in one issue slot.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi)
{
    return ((uint64_t)__float_as_uint(hi) << 32) | (uint64_t)__float_as_uint(lo);
}
__device__ __forceinline__ float f2_lo(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float f2_hi(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }

__device__ __forceinline__ uint64_t f2_add_rn(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_sub_rn(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_add_rp(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("add.rp.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul_rn(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_fma_rn(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_fma_rp(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rp.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ float fmin3(float a, float b, float c)
{
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// ------------------------------------------------------------------ stochastic rounding to E2M1
// Stochastic rounding of a pair of values onto the E2M1 grid with 16 random
// bits r each, as E2M1 codes: a magnitude between neighbours lo <= |v| < hi
// rounds up iff r < ceil(2^16 (|v| - lo) / (hi - lo)); 6 and above saturate;
// the sign is kept.  Computed in the index domain, where the grid
// {0, .5, 1, 1.5, 2, 3, 4, 6} becomes the integers 0..7:
// idx(x) = min(2x, x + 2, x/2 + 4) is the concave piecewise-linear map that
// sends each grid interval linearly onto [k, k + 1], so frac is the
// fractional part of idx and the code is ceil(idx - r/2^16).
//  - x = min(|v|, 6): values at or above 6 give idx = 7, code 7.
//  - The three lines are formed with 128 added, one round-up fma / add each:
//    on [128, 256) the fp32 ulp is 2^-16, the grid of r, and rounding frac up
//    onto that grid moves no ceiling, so the minimum of the rounded lines
//    gives the same decision (the sign of idx - r/2^16 when |v| < 0.5).
//  - d = (128 + idx) - (128 + r/2^16) is exact; fl_ru(d + 1.5 * 2^23, + 8 for
//    a negative v) holds ceil(d) (+ 8) in its low mantissa bits: the code
//    nibble, sign included.
// A CPU sweep checks this against the rounding rule on every finite bf16
// value and 2.9e8 (value, r) pairs (tests/test_sr_formulation.py).
//   v2:    the two values (v_lo, v_hi);
//   negr2: the two values -(128 + r / 2^16), from sr_neg_r;
//   z_lo, z_hi: bit patterns whose low nibbles are the two codes.
__device__ __forceinline__ void e2m1_sr_pair(uint64_t v2, uint64_t negr2, uint32_t& z_lo, uint32_t& z_hi)
{
    const uint64_t kTwo = 0x4000000040000000ull, kHalf = 0x3F0000003F000000ull;
    const uint64_t k128 = 0x4300000043000000ull, k130 = 0x4302000043020000ull, k132 = 0x4304000043040000ull;
    const uint64_t kNegOne = 0xBF800000BF800000ull, kMagic4 = 0x4B4000044B400004ull;  // 1.5 * 2^23 + 4
    const float vl = f2_lo(v2), vh = f2_hi(v2);
    const uint64_t x = f2_pack(fminf(fabsf(vl), 6.0f), fminf(fabsf(vh), 6.0f));
    const uint64_t a = f2_fma_rp(x, kTwo, k128);
    const uint64_t b = f2_add_rp(x, k130);
    const uint64_t c = f2_fma_rp(x, kHalf, k132);
    const uint64_t m = f2_pack(fmin3(f2_lo(a), f2_lo(b), f2_lo(c)), fmin3(f2_hi(a), f2_hi(b), f2_hi(c)));
    const uint64_t d = f2_add_rn(m, negr2);
    const uint64_t sgn4 = f2_pack(copysignf(4.0f, vl), copysignf(4.0f, vh));
    const uint64_t z = f2_add_rp(d, f2_fma_rn(sgn4, kNegOne, kMagic4));  // + 1.5 * 2^23 (+ 8 for a negative v)
    z_lo = (uint32_t)z;
    z_hi = (uint32_t)(z >> 32);
}

// -(128 + r / 2^16) for the 16-bit field `half` (0 low, 1 high) of a Philox word.
__device__ __forceinline__ float sr_neg_r(uint32_t w, int half)
{
    return __uint_as_float(__byte_perm(w, 0xC3000000u, half ? 0x7432u : 0x7410u));
}

// Horner packing of 8 code nibbles from e2m1_sr_pair's bit patterns (each
// 0x4B4000cc): sum_j bits_j * 16^j mod 2^32 carries the constant
// 0x4B400000 * 0x11111111 on top of the packed codes.
constexpr uint32_t kSrPackBias = 0x4B400000u * 0x11111111u;

// ------------------------------------------------------------------ Philox4x32-10
struct Philox4 {
    uint32_t x, y, z, w;
};

// Philox4x32-10 (Salmon et al., SC'11) of counter (c0, c1, c2, c3) with the
// key schedule precomputed on the host: rk[2r], rk[2r+1] are the key words of
// round r (the key plus r Weyl increments).
__device__ __forceinline__ Philox4 philox4x32_10_rk(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                                    const uint32_t (&rk)[20])
{
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
        const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
        const uint32_t n0 = hi1 ^ c1 ^ rk[2 * round], n2 = hi0 ^ c3 ^ rk[2 * round + 1];
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
    }
    return {c0, c1, c2, c3};
}

// Word i (0..3) of a Philox block: it holds the 16-bit random fields 2i (low
// half) and 2i + 1 (high half).
__device__ __forceinline__ uint32_t philox_word(const Philox4& p, int i)
{
    return i == 0 ? p.x : i == 1 ? p.y : i == 2 ? p.z : p.w;
}

}  // namespace nvq
