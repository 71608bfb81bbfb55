// gemm_epilogue.cuh -- the accumulator epilogue shared by the single-CTA and
// CTA-pair GEMM kernels: one warp turns its TMEM slice (32 accumulator rows,
// kCols fp32 columns) into C = alpha * acc (+ bias) rows.
#pragma once

#include <cuda.h>

#include "nvq_device.cuh"
#include "nvq_kernels.h"

namespace nvq {

// Optional amaxes of the stored output, for the quantizer of the next
// operation (so it can skip its own amax pass).  Each epilogue warp keeps
// running maxima across its tiles and publishes them once, at the end of the
// kernel (one atomic per warp instead of one per tile).
//   plain: max |C| over the stored values (after rounding to the output type);
//   rht:   max |H16 (s .* u)| over the 16-row column blocks u of C, before the
//          1/4 of the transform (applied once to the maximum: rounding is
//          monotonic).  A lane holds one row, so the 16 rows of a block are 16
//          consecutive lanes and the fp32 butterfly runs across them: stage h
//          pairs lanes i and i ^ h, the lane with bit h clear keeps a + b and
//          the other a - b, in the order the columnwise quantizer applies
//          (spans 1, 2, 4, 8).
struct EpiAmax {
    float plain;
    float rht;
    uint32_t flip;       // sign bit to apply to this lane's row (sign[lane & 15] == -1)
    uint32_t neg[4];     // sign bit of the own value in stage h = 1, 2, 4, 8
    bool on_plain, on_rht;
};

__device__ __forceinline__ EpiAmax epi_amax_init(const GemmArgs& args, int lane)
{
    EpiAmax am;
    am.plain = 0.0f;
    am.rht = 0.0f;
    am.flip = ((args.rht_sign_mask >> (lane & 15)) & 1u) << 31;
#pragma unroll
    for (int b = 0; b < 4; ++b) am.neg[b] = (lane & (1 << b)) ? 0x80000000u : 0u;
    am.on_plain = args.c_amax != nullptr;
    am.on_rht = args.c_amax_rht != nullptr;
    return am;
}

__device__ __forceinline__ void epi_amax_add(EpiAmax& am, float v)
{
    am.plain = fmaxf(am.plain, fabsf(v));
    if (am.on_rht) {  // warp-uniform
        float u = __uint_as_float(__float_as_uint(v) ^ am.flip);
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const float p = __shfl_xor_sync(0xFFFFFFFFu, u, 1 << b);
            u = __fadd_rn(p, __uint_as_float(__float_as_uint(u) ^ am.neg[b]));
        }
        am.rht = fmaxf(am.rht, fabsf(u));
    }
}

// n packed bf16 pairs (the stored values)
template <int n>
__device__ __forceinline__ void epi_amax_add_bf16(EpiAmax& am, const uint32_t* w)
{
    if (!am.on_plain && !am.on_rht) return;
#pragma unroll
    for (int i = 0; i < n; ++i) {
        epi_amax_add(am, __uint_as_float(w[i] << 16));
        epi_amax_add(am, __uint_as_float(w[i] & 0xFFFF0000u));
    }
}

// Both amaxes of a 32-row x 64-column bf16 block staged in shared memory for a
// TMA store (row r at r * 128 bytes, 16-byte chunks XOR-swizzled by r & 7), read
// back by columns: lane l takes columns 2l and 2l + 1 (one 4-byte word per row;
// the 32 lanes read a row's 128 bytes, one word per bank) and runs the
// Hadamard butterfly of each 16-row block in registers on packed fp32 pairs.
// Replaces the lane-shuffle form on this path (four shuffles per value made
// the epilogue, not the tensor core, set the tile rate).
__device__ __forceinline__ void epi_amax_add_staged(EpiAmax& am, const GemmArgs& args, const uint8_t* stage, int lane)
{
    if (!am.on_plain && !am.on_rht) return;
    const int chunk = lane >> 2, within = (lane & 3) * 4;
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
        uint64_t v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int r = 16 * blk + i;
            uint32_t w = *reinterpret_cast<const uint32_t*>(stage + r * 128 + ((chunk ^ (r & 7)) << 4) + within);
            am.plain = fmaxf(am.plain, fmaxf(fabsf(__uint_as_float(w << 16)), fabsf(__uint_as_float(w & 0xFFFF0000u))));
            if (am.on_rht && ((args.rht_sign_mask >> i) & 1u)) w ^= 0x80008000u;  // s .* u (row i of the block)
            v[i] = ((uint64_t)(w & 0xFFFF0000u) << 32) | (uint64_t)(w << 16);
        }
        if (am.on_rht) {
#pragma unroll
            for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    if ((i & h) == 0) {
                        const uint64_t a = v[i], b = v[i + h];
                        v[i] = f2_add_rn(a, b);
                        v[i + h] = f2_sub_rn(a, b);
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < 16; ++i)
                am.rht = fmaxf(am.rht, fmaxf(fabsf(__uint_as_float((uint32_t)v[i])),
                                             fabsf(__uint_as_float((uint32_t)(v[i] >> 32)))));
        }
    }
}

__device__ __forceinline__ float epi_warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// Publishes the warp's maxima (non-negative floats order like their bits).
__device__ __forceinline__ void epi_amax_publish(const GemmArgs& args, EpiAmax& am, int lane)
{
    if (am.on_plain) {
        const float m = epi_warp_max(am.plain);
        if (lane == 0) atomicMax(reinterpret_cast<unsigned int*>(args.c_amax), __float_as_uint(m));
    }
    if (am.on_rht) {
        const float m = __fmul_rn(epi_warp_max(am.rht), 0.25f);
        if (lane == 0) atomicMax(reinterpret_cast<unsigned int*>(args.c_amax_rht), __float_as_uint(m));
    }
}

// 32 accumulator columns (fp32 bits) -> alpha * acc (+ bias) as 16 bf16 pairs
// (column 2i in the low half of out[i]); bcol: C column of v[0].
__device__ __forceinline__ void pack32_bf16(const GemmArgs& args, const uint32_t (&v)[32], float alpha, int bcol,
                                            uint32_t* out)
{
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        float y0 = __fmul_rn(alpha, __uint_as_float(v[2 * i]));
        float y1 = __fmul_rn(alpha, __uint_as_float(v[2 * i + 1]));
        if (args.bias) {
            y0 = __fadd_rn(y0, __uint_as_float((uint32_t)args.bias[bcol + 2 * i] << 16));
            y1 = __fadd_rn(y1, __uint_as_float((uint32_t)args.bias[bcol + 2 * i + 1] << 16));
        }
        __nv_bfloat162 b2 = __floats2bfloat162_rn(y0, y1);
        out[i] = *reinterpret_cast<uint32_t*>(&b2);
    }
}

// 32 accumulator columns from TMEM (zero for an empty contraction).
__device__ __forceinline__ void load32(uint32_t taddr, bool have_k, uint32_t (&v)[32])
{
    if (have_k) {
        tmem_ld_32x32b_x32(taddr, v);
        tmem_ld_wait();
        tmem_regs_ready(v);
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0u;
    }
}

// Reads the warp's slice in 32-column chunks, scales, adds the bias and packs
// to bf16 pairs.  taddr: TMEM address of the slice (its lane quadrant, first
// column); have_k: false for an empty contraction (the slice is zero).
template <int kCols>
__device__ __forceinline__ void pack_slice_bf16(const GemmArgs& args, uint32_t taddr, bool have_k, float alpha,
                                                int col0, uint32_t (&packed)[kCols / 2])
{
#pragma unroll
    for (int c = 0; c < kCols / 32; ++c) {
        uint32_t v[32];
        load32(taddr + (uint32_t)(c * 32), have_k, v);
        pack32_bf16(args, v, alpha, col0 + c * 32, &packed[c * 16]);
    }
}

// rowoff: element offset of the row's first column in C; release(): hands the
// accumulator back to the MMA issuer once every TMEM load of the slice has
// completed.
template <int kCols, typename Release>
__device__ __forceinline__ void epilogue_slice(const GemmArgs& args, uint32_t taddr, bool have_k, float alpha,
                                               int col0, int64_t rowoff, bool row_ok, EpiAmax& am, Release release)
{
    static_assert(kCols % 64 == 0, "64-column granularity");
    if (!args.c_fp32) {
        // bf16: pack the whole slice in registers, release the accumulator,
        // then store -- the next tile's MMAs overlap the global stores.
        uint32_t packed[kCols / 2];
        pack_slice_bf16<kCols>(args, taddr, have_k, alpha, col0, packed);
        release();
        epi_amax_add_bf16<kCols / 2>(am, packed);
        if (!row_ok) return;
        if (args.c_st32) {  // 32-byte stores, one full L2 sector each
            uint16_t* dst = reinterpret_cast<uint16_t*>(args.C) + rowoff;
#pragma unroll
            for (int i = 0; i < kCols / 16; ++i) st_global_v8(dst + 16 * i, &packed[8 * i]);
        } else {
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(args.C) + rowoff);
#pragma unroll
            for (int i = 0; i < kCols / 8; ++i)
                dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
        }
        return;
    }
    // fp32: 64-column passes, the accumulator released after the last load
#pragma unroll 1
    for (int p = 0; p < kCols / 64; ++p) {
        uint32_t v[64];
        if (have_k) {
            tmem_ld_32x32b_x32(taddr + (uint32_t)(p * 64), *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
            tmem_ld_32x32b_x32(taddr + (uint32_t)(p * 64 + 32), *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
            tmem_ld_wait();
            tmem_regs_ready(*reinterpret_cast<uint32_t(*)[32]>(&v[0]));
            tmem_regs_ready(*reinterpret_cast<uint32_t(*)[32]>(&v[32]));
        } else {
#pragma unroll
            for (int i = 0; i < 64; ++i) v[i] = 0u;
        }
        if (p == kCols / 64 - 1) release();
        if (!row_ok && !am.on_plain && !am.on_rht) continue;
        float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(args.C) + rowoff + p * 64);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float f[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float y = __fmul_rn(alpha, __uint_as_float(v[4 * i + e]));
                if (args.bias) y = __fadd_rn(y, __uint_as_float((uint32_t)args.bias[col0 + p * 64 + 4 * i + e] << 16));
                f[e] = y;
                if (am.on_plain || am.on_rht) epi_amax_add(am, y);
            }
            if (row_ok) dst[i] = make_float4(f[0], f[1], f[2], f[3]);
        }
    }
}

// bf16 slice whose 32 rows are all valid, stored through the TMA.  The
// whole 128-column slice comes out of TMEM in one round trip (four x32 loads,
// 128 registers: the caller runs with a raised register budget), the
// accumulator is released, and only then are the values scaled, packed and
// stored.  Each 64-column half is written into the warp's 4 KB staging buffer
// (32 rows x 128 bytes, 128B-swizzled as the store's tensor map expects) and
// leaves through one bulk tensor store, so every global write is a full
// 128-byte line (register stores write one 32-byte sector per row and
// instruction, and their L1 traffic slowed the tensor pipe).  stage:
// 1024-byte aligned, 4 KB, owned by this warp; c_row0: C row of the slice's
// first row.  The lane that issues the stores waits for their completion
// before the CTA exits.
template <int kCols, typename Release>
__device__ __forceinline__ void epilogue_slice_tma(const GemmArgs& args, const CUtensorMap* c_map, uint8_t* stage,
                                                   uint32_t taddr, bool have_k, float alpha, int col0, int c_row0,
                                                   int lane, EpiAmax& am, Release release)
{
    static_assert(kCols == 128, "four 32-column chunks");
    uint8_t* row = stage + lane * 128;
    uint32_t v[4][32];
    if (have_k) {
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(taddr + (uint32_t)(32 * c), v[c]);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_regs_ready(v[c]);
    } else {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i) v[c][i] = 0u;
    }
    release();  // every TMEM load of the slice has completed
#pragma unroll
    for (int b = 0; b < 2; ++b) {
        uint32_t packed[32];
        pack32_bf16(args, v[2 * b], alpha, col0 + 64 * b, &packed[0]);
        pack32_bf16(args, v[2 * b + 1], alpha, col0 + 64 * b + 32, &packed[16]);
        if (lane == 0) bulk_wait_group_read0();  // the previous store has read the buffer
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(row + ((c ^ (lane & 7)) << 4)) =
                make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(c_map, stage, col0 + 64 * b, c_row0);
            bulk_commit_group();
        }
        // the output amaxes from the staged block (read while the store reads it;
        // the next half's writes wait for every lane at the __syncwarp above)
        epi_amax_add_staged(am, args, stage, lane);
    }
}

}  // namespace nvq
