// quantize_kernel.cuh -- the fused rowwise + columnwise block quantizer of
// bf16 tensors into NVFP4 (E2M1 + E4M3 1x16 scales + FP32 tensor scale),
// MXFP8 (E4M3 + E8M0 1x32 scales) or the identity (bf16 kept), with the
// optional 16-point random Hadamard transform on the columnwise blocks,
// Philox stochastic rounding, and the columnwise direction built from the
// dequantized rowwise value ("rowwise_dequantized" source).  Included by
// quantize.cu (amax pass and the original-source variants) and
// quantize_hybrid.cu (identity and rowwise-dequantized variants), which
// compile in parallel.
//
// Method: "Add an NVFP4 quantization converter" (torchtitan PR #3914, "What
// changed"; review thread on "rowwise") and "Hybrid quantization"
// (TransformerEngine PR #2817, "Description", mxfp8 storage review, "Enable
// columnwise_source and hybrid recipes", IdentityQuantizer).
//
// Work decomposition (both kernels): a CTA owns a tile of 128 (padded) rows x
// 256 columns; warp w covers rows 32*(w&3).. and columns 128*(w>>2)..; lane l
// owns 16 consecutive rows (half (l>>4) of the warp's 32) x 8 consecutive
// columns (group l&15).  One 16-byte load per row brings a thread's 8 bf16
// values, so every element is read from HBM once per pass and held in
// registers: a columnwise 16-block lives entirely in one thread (Hadamard
// butterflies in registers), a rowwise 16-block spans a lane pair (one
// shuffle), a 32-block spans 4 lanes (rows) or a lane and lane^16 (columns).
// Outputs that are not contiguous per thread (transposed codes, swizzled
// scales) are staged in shared memory and written out with vector stores.
//
// Grouped tensors: rows are addressed in a padded space where each group
// starts at a multiple of 128, so no tile straddles two groups; rows of the
// padded space with no source row read as zero.
#pragma once

#include "nvq_kernels.h"
#include "nvq_device.cuh"

namespace nvq {

constexpr int kTileRows = 128;
constexpr int kTileCols = 256;
constexpr int kThreads = 256;

struct ThreadTile {
    uint4 w[16];  // 16 rows x 8 bf16
};

__device__ __forceinline__ int find_group(const QuantGroups& g, int64_t tile_row)
{
    int lo = 0, hi = g.G - 1;
    while (lo < hi) {  // last group whose first tile <= tile_row
        const int mid = (lo + hi + 1) >> 1;
        if (g.tile0[mid] <= tile_row) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// Loads the thread's 16 x 8 block; rows with no source row (padding) and
// columns >= K read as zero.
__device__ __forceinline__ void load_tile(const QuantArgs& a, int g, int64_t prow0, int64_t k0,
                                          ThreadTile& t)
{
    const int64_t gp0 = (int64_t)a.groups.tile0[g] * kTileRows;  // padded start of group
    const int64_t m = a.groups.rows[g];
    const int64_t src0 = a.groups.src_row0[g];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int64_t local = prow0 + i - gp0;
        if (local < m && k0 < a.K) {
            const uint4* p = reinterpret_cast<const uint4*>(a.x + (src0 + local) * a.ld + k0);
            t.w[i] = __ldg(p);
        } else {
            t.w[i] = make_uint4(0, 0, 0, 0);
        }
    }
}

__device__ __forceinline__ void unpack8(const uint4& w, float (&v)[8])
{
    v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x);
    v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
    v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z);
    v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
}

// Column j (0..7) of the thread's tile as 16 fp32 values.
__device__ __forceinline__ void column16(const ThreadTile& t, int j, float (&u)[16])
{
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t word = (j >> 1) == 0 ? t.w[i].x : (j >> 1) == 1 ? t.w[i].y : (j >> 1) == 2 ? t.w[i].z : t.w[i].w;
        u[i] = (j & 1) ? bf16_hi(word) : bf16_lo(word);
    }
}

// s .* u for the thread's 16 rows: row i of the tile is negated (sign bits of
// both bf16 halves of every word flipped) where sign[i] == -1.
__device__ __forceinline__ void flip_rows(ThreadTile& t, uint32_t sign_mask)
{
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t m = ((sign_mask >> i) & 1u) ? 0x80008000u : 0u;
        t.w[i].x ^= m;
        t.w[i].y ^= m;
        t.w[i].z ^= m;
        t.w[i].w ^= m;
    }
}

// H16 u for an already sign-flipped u: butterflies with spans 1, 2, 4, 8
// ((a, b) -> (a + b, a - b)), without the 1/4.
__device__ __forceinline__ void butterfly16(float (&u)[16])
{
#pragma unroll
    for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if ((i & h) == 0) {
                const float a = u[i], b = u[i + h];
                u[i] = __fadd_rn(a, b);
                u[i + h] = __fsub_rn(a, b);
            }
        }
    }
}

// T(u) = 1/4 H16 u for an already sign-flipped u: butterflies with spans
// 1, 2, 4, 8 ((a, b) -> (a + b, a - b)), then the exact 1/4.
__device__ __forceinline__ void hadamard16(float (&u)[16])
{
#pragma unroll
    for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if ((i & h) == 0) {
                const float a = u[i], b = u[i + h];
                u[i] = __fadd_rn(a, b);
                u[i + h] = __fsub_rn(a, b);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) u[i] = __fmul_rn(u[i], 0.25f);
}

// The same transform on two columns at once (packed pairs): u2[i] holds row i
// of both columns; butterflies with spans 1, 2, 4, 8, then the exact 1/4 when
// quarter.
template <bool kQuarter>
__device__ __forceinline__ void hadamard16x2(uint64_t (&u2)[16])
{
#pragma unroll
    for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if ((i & h) == 0) {
                const uint64_t a = u2[i], b = u2[i + h];
                u2[i] = f2_add_rn(a, b);
                u2[i + h] = f2_sub_rn(a, b);
            }
        }
    }
    if constexpr (kQuarter) {
#pragma unroll
        for (int i = 0; i < 16; ++i) u2[i] = f2_mul_rn(u2[i], 0x3E8000003E800000ull);  // * 0.25, exact
    }
}

// Columns 2m and 2m + 1 of the thread's tile (the two halves of word m) as 16
// packed pairs, row 0 first.
__device__ __forceinline__ void column_pair16(const ThreadTile& t, int m, uint64_t (&u2)[16])
{
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t w = m == 0 ? t.w[i].x : m == 1 ? t.w[i].y : m == 2 ? t.w[i].z : t.w[i].w;
        u2[i] = ((uint64_t)(w & 0xFFFF0000u) << 32) | (uint64_t)(w << 16);
    }
}

__device__ __forceinline__ void atomic_max_nonneg(float* addr, float v)
{
    atomicMax(reinterpret_cast<unsigned int*>(addr), __float_as_uint(v));
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}


// Plain and Hadamard-domain maxima of the thread's 16 x 8 tile: max |x|, and
// max |H16 (s .* u)| over its 8 columnwise 16-blocks u (before the 1/4 of the
// transform, applied once to the maximum by the caller: rounding is
// monotonic).  Flips t's sign bits when rht.
__device__ __forceinline__ void tile_amax(ThreadTile& t, bool rht, uint32_t sign_mask, float& m_plain, float& m_rht)
{
    m_plain = 0.0f;
    m_rht = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        float v[8];
        unpack8(t.w[i], v);
#pragma unroll
        for (int j = 0; j < 8; ++j) m_plain = fmaxf(m_plain, fabsf(v[j]));
    }
    if (rht) {
        flip_rows(t, sign_mask);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float u[16];
            column16(t, j, u);
            butterfly16(u);
#pragma unroll
            for (int i = 0; i < 16; ++i) m_rht = fmaxf(m_rht, fabsf(u[i]));
        }
    }
}

// CTA-wide maxima published with one atomic each (all threads call it).
__device__ __forceinline__ void cta_amax_publish(float m_plain, float m_rht, float* out_plain, float* out_plain2,
                                                 float* out_rht)
{
    __shared__ float red[2][kThreads / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    m_plain = warp_max(m_plain);
    m_rht = warp_max(m_rht);
    if (lane == 0) {
        red[0][warp] = m_plain;
        red[1][warp] = m_rht;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float p = 0.0f, r = 0.0f;
        for (int w = 0; w < kThreads / 32; ++w) {
            p = fmaxf(p, red[0][w]);
            r = fmaxf(r, red[1][w]);
        }
        // max |fl(u/4)| = fl(max |u| / 4): the 1/4 of the transform, once
        r = __fmul_rn(r, 0.25f);
        if (out_plain) atomic_max_nonneg(out_plain, p);
        if (out_plain2) atomic_max_nonneg(out_plain2, p);
        if (out_rht) atomic_max_nonneg(out_rht, r);
    }
}

// ------------------------------------------------------------------ NVFP4 block encode
struct Nvfp4Scale {
    float r448;   // 448 / A
    float s_enc;  // 2688 / A  (A = 0 -> 1, overflow -> FLT_MAX)
    bool zero;    // A == 0
};

__device__ __forceinline__ Nvfp4Scale nvfp4_tensor_scale(float A)
{
    Nvfp4Scale s;
    s.zero = (A == 0.0f);
    s.r448 = __fdiv_rn(448.0f, A);
    float se = __fdiv_rn(2688.0f, A);
    if (s.zero) se = 1.0f;
    if (isinf(se)) se = 3.402823466e38f;
    s.s_enc = se;
    return s;
}

// Block scale code S and element encode factor e = fl(s_enc / E4M3(S)) for
// block amax b, without a division per block: every finite E4M3 value is
// n * 2^j with n in 1..15 (normal codes: n = 8 + mantissa, j = exponent - 10;
// subnormal codes: n = mantissa, j = -9), so e = fl(s_enc / n) * 2^-j.  The
// power-of-two scaling is exact because s_enc / n and e stay normal for every
// finite tensor amax (e >= (2688 / FLT_MAX) / 448 > FLT_MIN), and it
// overflows exactly when the quotient does.  q_tab[n] = fl(s_enc / n).
__device__ __forceinline__ uint32_t nvfp4_block_scale(const Nvfp4Scale& ts, const float* q_tab, float b, float& e)
{
    uint32_t S = 0;
    if (b != 0.0f && !ts.zero) S = e4m3_rn(__fmul_rn(b, ts.r448));
    e = 0.0f;
    if (S != 0) {
        const uint32_t ex = S >> 3, mant = S & 7u;
        const uint32_t n = ex ? 8u + mant : mant;
        const uint32_t ex1 = ex ? ex : 1u;
        const float q = __fmul_rn(q_tab[n], __uint_as_float((137u - ex1) << 23));  // * 2^(10 - ex1)
        e = isinf(q) ? 3.402823466e38f : q;
    }
    return S;
}

// The same by division (kept for the NVFP4-row + MXFP8-column variant, where
// the table version makes the compiler spill registers and runs no faster:
// that variant is bound by memory, not by this division).
__device__ __forceinline__ uint32_t nvfp4_block_scale_div(const Nvfp4Scale& ts, float b, float& e)
{
    uint32_t S = 0;
    if (b != 0.0f && !ts.zero) S = e4m3_rn(__fmul_rn(b, ts.r448));
    e = 0.0f;
    if (S != 0) {
        const float q = __fdiv_rn(ts.s_enc, e4m3_to_f32(S));
        e = isinf(q) ? 3.402823466e38f : q;
    }
    return S;
}

// q_tab[dir][n] = fl(s_enc / n), n = 1..15, of the row (dir 0) and column
// (dir 1) NVFP4 tensor scales of group g; threads 0..31 fill it, the caller
// synchronizes before use.
template <int ROW_FMT, int COL_FMT>
__device__ __noinline__ void nvfp4_fill_q_tab(const QuantArgs& a, int g, float (&q_tab)[2][16])
{
    if (threadIdx.x < 32) {
        const int dir = threadIdx.x >> 4, n = threadIdx.x & 15;
        float A = 0.0f;
        if (dir == 0 && ROW_FMT == 1) A = a.row_amax[g];
        if (dir == 1 && (COL_FMT == 1 || COL_FMT == 5)) A = a.col_amax[g];
        const Nvfp4Scale ts = nvfp4_tensor_scale(A);
        q_tab[dir][n] = n ? __fdiv_rn(ts.s_enc, (float)n) : 0.0f;
    }
}

// 8 consecutive elements of one direction's output starting at linear index L0
// (L0 % 8 == 0): E2M1 codes, element 0 in the low nibble.
template <bool SR>
__device__ __forceinline__ uint32_t nvfp4_encode8(const float (&v)[8], float e, uint64_t L0, int dir,
                                                  const QuantArgs& a)
{
    if constexpr (SR) {
        const uint64_t e2 = f2_pack(e, e);
        uint64_t s2[4];  // v * e, elements (2h, 2h + 1) in pair h
#pragma unroll
        for (int h = 0; h < 4; ++h) s2[h] = f2_mul_rn(f2_pack(v[2 * h], v[2 * h + 1]), e2);
        const uint64_t blk = L0 >> 3;
        const Philox4 p = philox4x32_10_rk((uint32_t)blk, (uint32_t)(blk >> 32), (uint32_t)dir, a.sr_offset,
                                           a.sr_round_key);
        uint32_t packed = 0;  // Horner over the elements, element 0 last (lowest nibble)
#pragma unroll
        for (int h = 3; h >= 0; --h) {
            const uint32_t w = philox_word(p, h);  // fields 2h (low half) and 2h + 1 (high half)
            uint32_t zl, zh;
            e2m1_sr_pair(s2[h], f2_pack(sr_neg_r(w, 0), sr_neg_r(w, 1)), zl, zh);
            packed = packed * 16u + zh;
            packed = packed * 16u + zl;
        }
        return packed - kSrPackBias;
    } else {
        float s[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) s[j] = __fmul_rn(v[j], e);
        return e2m1x8_rn(s);
    }
}

// Two columns at once: v2[i] = (column A, column B) at row i of an 8-row
// group, e2 = (e_A, e_B), LA0 / LB0 the linear indices of row 0 of each
// column's group.  Codes of column A and column B, element 0 in the low nibble.
template <bool SR>
__device__ __forceinline__ void nvfp4_encode8x2(const uint64_t* v2, uint64_t e2, uint64_t LA0, uint64_t LB0, int dir,
                                                const QuantArgs& a, uint32_t& codes_a, uint32_t& codes_b)
{
    uint64_t s2[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) s2[i] = f2_mul_rn(v2[i], e2);
    if constexpr (SR) {
        const uint64_t ba = LA0 >> 3, bb = LB0 >> 3;
        const Philox4 pa = philox4x32_10_rk((uint32_t)ba, (uint32_t)(ba >> 32), (uint32_t)dir, a.sr_offset,
                                            a.sr_round_key);
        const Philox4 pb = philox4x32_10_rk((uint32_t)bb, (uint32_t)(bb >> 32), (uint32_t)dir, a.sr_offset,
                                            a.sr_round_key);
        uint32_t qa = 0, qb = 0;
#pragma unroll
        for (int i = 7; i >= 0; --i) {
            const uint64_t nr = f2_pack(sr_neg_r(philox_word(pa, i >> 1), i & 1), sr_neg_r(philox_word(pb, i >> 1), i & 1));
            uint32_t za, zb;
            e2m1_sr_pair(s2[i], nr, za, zb);
            qa = qa * 16u + za;
            qb = qb * 16u + zb;
        }
        codes_a = qa - kSrPackBias;
        codes_b = qb - kSrPackBias;
    } else {
        float sa[8], sb[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            sa[i] = f2_lo(s2[i]);
            sb[i] = f2_hi(s2[i]);
        }
        codes_a = e2m1x8_rn(sa);
        codes_b = e2m1x8_rn(sb);
    }
}

// ------------------------------------------------------------------ MXFP8 block encode
__device__ __forceinline__ int mx_exponent(float b)
{
    if (b == 0.0f) return -127;
    const uint32_t bits = __float_as_uint(b);
    const int ef = (int)((bits >> 23) & 0xFF);
    int lg;  // floor(log2 b), exact for normals and subnormals
    if (ef != 0) lg = ef - 127;
    else lg = -118 - __clz(bits & 0x7FFFFF);  // m * 2^-149 -> (31 - clz(m)) - 149
    int e = lg - 8;
    return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// 2^-e as fp32 for e in [-127, 127] (2^127 is finite; 2^-127 is subnormal).
__device__ __forceinline__ float exp2_neg(int e)
{
    const int p = -e;
    if (p >= -126) return __uint_as_float((uint32_t)(p + 127) << 23);
    return __uint_as_float(1u << (p + 149));
}

// ------------------------------------------------------------------ dequantized rowwise values
// The rowwise-dequantized source: each quantized value back in bf16, formed in
// fp32 -- NVFP4: the exact product E2M1(q) * E4M3(S), times g = A / 2688 with
// one rounding; MXFP8: E4M3(q) * 2^e, exact -- and rounded once to nearest
// even.  8 codes (element 0 in the low nibble) -> 8 bf16 (element 0 in the
// low half of word 0).
__device__ __forceinline__ uint4 nvfp4_dequant8(uint32_t codes, float sval, float g, const float* e2m1_tab)
{
    uint32_t w[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        const float v0 = __fmul_rn(__fmul_rn(e2m1_tab[(codes >> (8 * h)) & 15u], sval), g);
        const float v1 = __fmul_rn(__fmul_rn(e2m1_tab[(codes >> (8 * h + 4)) & 15u], sval), g);
        __nv_bfloat162 b2 = __floats2bfloat162_rn(v0, v1);
        w[h] = *reinterpret_cast<uint32_t*>(&b2);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// 4 E4M3 codes (element 0 in the low byte) times 2^e -> 2 bf16 pairs.
__device__ __forceinline__ uint2 mxfp8_dequant4(uint32_t codes, float p2e)
{
    uint32_t w[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const float v0 = __fmul_rn(e4m3_to_f32((codes >> (16 * h)) & 0xFFu), p2e);
        const float v1 = __fmul_rn(e4m3_to_f32((codes >> (16 * h + 8)) & 0xFFu), p2e);
        __nv_bfloat162 b2 = __floats2bfloat162_rn(v0, v1);
        w[h] = *reinterpret_cast<uint32_t*>(&b2);
    }
    return make_uint2(w[0], w[1]);
}

// Column j (0..7) of the thread's 16 rows as 16 bf16 (row 0 first) in 8 words.
__device__ __forceinline__ void column16_bf16(const ThreadTile& t, int j, uint32_t (&out)[8])
{
    const uint32_t sel = (j & 1) ? 0x7632u : 0x5410u;  // high or low halves
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        const uint4& a = t.w[2 * m];
        const uint4& c = t.w[2 * m + 1];
        const uint32_t wa = (j >> 1) == 0 ? a.x : (j >> 1) == 1 ? a.y : (j >> 1) == 2 ? a.z : a.w;
        const uint32_t wc = (j >> 1) == 0 ? c.x : (j >> 1) == 1 ? c.y : (j >> 1) == 2 ? c.z : c.w;
        out[m] = __byte_perm(wa, wc, sel);
    }
}

// ------------------------------------------------------------------ fused quantize
// Shared staging: transposed codes and both scale tiles.  Output row kk of
// the transposed codes holds 64 (NVFP4) or 128 (MXFP8) bytes; its 8- or
// 16-byte chunks are XOR-swizzled by (kk >> 3) & 7 so the lanes of a warp
// (8 output rows apart) hit different banks.
struct QuantSmem {
    uint8_t col_codes[kTileCols * kTileRows];
    uint8_t row_scales[2048];                      // 128 rows x up to 16 scale cols
    uint8_t col_scales[2][1024];                   // 2 x (128 k-rows x up to 8 scale cols)
};

__device__ __forceinline__ int col_chunk_nv(int kk, int ch8) { return kk * 64 + ((ch8 ^ ((kk >> 3) & 7)) << 3); }
__device__ __forceinline__ int col_chunk_mx(int kk, int ch16) { return kk * 128 + ((ch16 ^ ((kk >> 3) & 7)) << 4); }

// Formats: 0 none, 1 NVFP4, 2 MXFP8, 3 identity (bf16), 4 row-scaled NVFP4
// (rowwise only: row p's FP32 outer scale from its own amax row_amax[p]), 5
// NVFP4 with one scale per 16 x 16 tile (columnwise only: the tile's amax,
// the thread's 16 x 8 half and its lane partner's, sets the scale of all its
// 1 x 16 columnwise blocks).  DQ: the columnwise
// direction quantizes the dequantized rowwise values (the tile is replaced by
// them after the rowwise pass).  Run-time modes (CTA-uniform): row_data ==
// NULL skips the rowwise stores; col_data == NULL skips the columnwise pass;
// dq_amax != NULL writes the amax of the columnwise source (plain, or of its
// Hadamard transform when RHT) -- the first pass of a rowwise-dequantized
// NVFP4 columnwise direction, whose scale needs it before any block is
// quantized.
template <int ROW_FMT, int COL_FMT, bool RHT, bool SR, bool DQ>
__global__ void __launch_bounds__(kThreads, 2) quantize_kernel(QuantArgs a)
{
    static_assert(!DQ || ROW_FMT == 1 || ROW_FMT == 2, "the rowwise-dequantized source needs a quantized rowwise direction");
    __shared__ __align__(16) QuantSmem sm;
    const int64_t tile_row = blockIdx.y, tile_col = blockIdx.x;
    const int g = find_group(a.groups, tile_row);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r_loc = (warp & 3) * 32 + (lane >> 4) * 16;  // first of the thread's 16 rows in tile
    const int c_loc = (warp >> 2) * 128 + (lane & 15) * 8; // first of the thread's 8 cols in tile
    const int64_t prow0 = tile_row * kTileRows + r_loc;
    const int64_t k0 = tile_col * kTileCols + c_loc;
    const bool kvalid = k0 < a.K;
    const bool row_out = a.row_data != nullptr;
    const bool col_pass = COL_FMT != 0 && a.col_data != nullptr;

    for (int i = threadIdx.x; i < 2048 / 16; i += kThreads) {
        reinterpret_cast<uint4*>(sm.row_scales)[i] = make_uint4(0, 0, 0, 0);
        reinterpret_cast<uint4*>(&sm.col_scales[0][0])[i] = make_uint4(0, 0, 0, 0);
    }

    constexpr bool kRowTab = !(ROW_FMT == 1 && COL_FMT == 2);
    __shared__ float q_tab[2][16];
    if constexpr ((ROW_FMT == 1 && kRowTab) || COL_FMT == 1 || COL_FMT == 5) nvfp4_fill_q_tab<ROW_FMT, COL_FMT>(a, g, q_tab);
    __shared__ float e2m1_tab[16];  // signed E2M1 values by code (rowwise-dequantized NVFP4)
    if constexpr (DQ && ROW_FMT == 1) {
        if (threadIdx.x < 16) {
            const uint32_t m = threadIdx.x & 7u;
            const float mag = m < 2 ? 0.5f * (float)m : __uint_as_float((m + 252u) << 22);
            e2m1_tab[threadIdx.x] = (threadIdx.x & 8u) ? -mag : mag;
        }
    }

    ThreadTile t;
    load_tile(a, g, prow0, k0, t);
    __syncthreads();  // staging cleared, q_tab filled

    // ---------------- rowwise direction
    if constexpr (ROW_FMT == 1 || ROW_FMT == 4) {  // NVFP4, 16-blocks = lane pair
        constexpr bool kRowScaled = ROW_FMT == 4;
        const Nvfp4Scale ts_tensor = nvfp4_tensor_scale(kRowScaled ? 0.0f : a.row_amax[g]);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float v[8];
            unpack8(t.w[i], v);
            float b = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j) b = fmaxf(b, fabsf(v[j]));
            b = fmaxf(b, __shfl_xor_sync(0xFFFFFFFFu, b, 1));
            float e;
            uint32_t S;
            if constexpr (kRowScaled) {
                // the row's own amax (padded row index; rows past the stored ones read 0)
                const int64_t pr = prow0 + i;
                const float A_r = pr < a.row_rows_store ? a.row_amax[pr] : 0.0f;
                S = nvfp4_block_scale_div(nvfp4_tensor_scale(A_r), b, e);
            } else if constexpr (kRowTab) {
                S = nvfp4_block_scale(ts_tensor, q_tab[0], b, e);
            } else {
                S = nvfp4_block_scale_div(ts_tensor, b, e);
            }
            const int64_t p = prow0 + i;
            const uint64_t L0 = (uint64_t)p * (uint64_t)a.K + (uint64_t)k0;
            const uint32_t codes = nvfp4_encode8<SR>(v, e, L0, 0, a);
            if (row_out && kvalid && p < a.row_rows_store)
                *reinterpret_cast<uint32_t*>(a.row_data + p * (a.K / 2) + k0 / 2) = codes;
            if constexpr (DQ) t.w[i] = nvfp4_dequant8(codes, e4m3_to_f32(S), __fdiv_rn(a.row_amax[g], 2688.0f), e2m1_tab);
            if ((lane & 1) == 0) {
                const int r = r_loc + i, c = c_loc / 16;  // scale column within the CTA (0..15)
                sm.row_scales[(c >> 2) * 512 + (r & 31) * 16 + (r >> 5) * 4 + (c & 3)] = (uint8_t)(kvalid ? S : 0);
            }
        }
    } else if constexpr (ROW_FMT == 2) {  // MXFP8, 32-blocks = 4 lanes
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float v[8];
            unpack8(t.w[i], v);
            float b = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j) b = fmaxf(b, fabsf(v[j]));
            b = fmaxf(b, __shfl_xor_sync(0xFFFFFFFFu, b, 1));
            b = fmaxf(b, __shfl_xor_sync(0xFFFFFFFFu, b, 2));
            const int e = mx_exponent(b);
            const float sc = exp2_neg(e);
            const uint32_t lo = e4m3x4_rn(__fmul_rn(v[0], sc), __fmul_rn(v[1], sc), __fmul_rn(v[2], sc), __fmul_rn(v[3], sc));
            const uint32_t hi = e4m3x4_rn(__fmul_rn(v[4], sc), __fmul_rn(v[5], sc), __fmul_rn(v[6], sc), __fmul_rn(v[7], sc));
            const int64_t p = prow0 + i;
            if (row_out && kvalid && p < a.row_rows_store)
                *reinterpret_cast<uint2*>(a.row_data + p * a.K + k0) = make_uint2(lo, hi);
            if constexpr (DQ) {
                const float p2e = exp2_neg(-e);
                const uint2 d0 = mxfp8_dequant4(lo, p2e), d1 = mxfp8_dequant4(hi, p2e);
                t.w[i] = make_uint4(d0.x, d0.y, d1.x, d1.y);
            }
            if ((lane & 3) == 0) {
                const int r = r_loc + i, c = c_loc / 32;  // 0..7
                sm.row_scales[(c >> 2) * 512 + (r & 31) * 16 + (r >> 5) * 4 + (c & 3)] = (uint8_t)(kvalid ? (e + 127) : 0);
            }
        }
    } else if constexpr (ROW_FMT == 3) {  // identity: the bf16 rows themselves
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int64_t p = prow0 + i;
            if (row_out && kvalid && p < a.row_rows_store)
                *reinterpret_cast<uint4*>(a.row_data + (p * a.K + k0) * 2) = t.w[i];
        }
    }

    // The rowwise pass is done with t: pin its registers here so the compiler
    // does not start the columnwise extraction inside the rowwise pass (that
    // overlap spilled registers in the variants without the Hadamard transform).
#pragma unroll
    for (int i = 0; i < 16; ++i)
        asm volatile("" : "+r"(t.w[i].x), "+r"(t.w[i].y), "+r"(t.w[i].z), "+r"(t.w[i].w));

    // ---------------- amax of the rowwise-dequantized columnwise source
    if constexpr (DQ) {
        if (a.dq_amax) {
            float m_plain, m_rht;
            tile_amax(t, RHT, a.rht_sign_mask, m_plain, m_rht);
            cta_amax_publish(m_plain, m_rht, RHT ? nullptr : a.dq_amax + g, nullptr, RHT ? a.dq_amax + g : nullptr);
        }
    }

    // ---------------- columnwise direction (output row = column k, contraction = padded row p)
    if (!col_pass) {
    } else if constexpr (COL_FMT == 1 || COL_FMT == 5) {  // NVFP4: the thread's 16 rows form one block per column
        const Nvfp4Scale ts = nvfp4_tensor_scale(a.col_amax[g]);
        if constexpr (RHT) flip_rows(t, a.rht_sign_mask);  // the rowwise pass is done with t
        float tile_b = 0.0f;  // 2D: amax of the 16 x 16 tile (this lane's 16 x 8 and lane ^ 1's)
        if constexpr (COL_FMT == 5) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float v[8];
                unpack8(t.w[i], v);
#pragma unroll
                for (int j = 0; j < 8; ++j) tile_b = fmaxf(tile_b, fabsf(v[j]));
            }
            tile_b = fmaxf(tile_b, __shfl_xor_sync(0xFFFFFFFFu, tile_b, 1));
        }
        if constexpr (RHT || SR) {
        // columns 2m and 2m + 1 together, as packed pairs
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            uint64_t u2[16];
            column_pair16(t, m, u2);
            if constexpr (RHT) hadamard16x2<true>(u2);
            float b0 = 0.0f, b1 = 0.0f;
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
                b0 = fmax3(b0, fabsf(f2_lo(u2[i])), fabsf(f2_lo(u2[i + 1])));
                b1 = fmax3(b1, fabsf(f2_hi(u2[i])), fabsf(f2_hi(u2[i + 1])));
            }
            if constexpr (COL_FMT == 5) b0 = b1 = tile_b;
            float e0, e1;
            const uint32_t S0 = nvfp4_block_scale(ts, q_tab[1], b0, e0);
            const uint32_t S1 = nvfp4_block_scale(ts, q_tab[1], b1, e1);
            const uint64_t L0 = (uint64_t)(k0 + 2 * m) * (uint64_t)a.col_cols_store + (uint64_t)prow0;
            const uint64_t L1 = L0 + (uint64_t)a.col_cols_store;
            const uint64_t e2 = f2_pack(e0, e1);
            uint32_t ca0, cb0, ca1, cb1;
            nvfp4_encode8x2<SR>(&u2[0], e2, L0, L1, 1, a, ca0, cb0);
            nvfp4_encode8x2<SR>(&u2[8], e2, L0 + 8, L1 + 8, 1, a, ca1, cb1);
            const int kk = c_loc + 2 * m;  // output rows within the CTA (0..255): kk, kk + 1
            const int c = r_loc / 16;      // scale column within the CTA (0..7)
            *reinterpret_cast<uint2*>(&sm.col_codes[col_chunk_nv(kk, c)]) = make_uint2(ca0, ca1);
            *reinterpret_cast<uint2*>(&sm.col_codes[col_chunk_nv(kk + 1, c)]) = make_uint2(cb0, cb1);
            sm.col_scales[kk >> 7][(c >> 2) * 512 + (kk & 31) * 16 + ((kk >> 5) & 3) * 4 + (c & 3)] =
                (uint8_t)(kvalid ? S0 : 0);
            sm.col_scales[(kk + 1) >> 7][(c >> 2) * 512 + ((kk + 1) & 31) * 16 + (((kk + 1) >> 5) & 3) * 4 + (c & 3)] =
                (uint8_t)(kvalid ? S1 : 0);
        }
        } else {
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
            float u[16];
            column16(t, jj, u);
            float b = 0.0f;
#pragma unroll
            for (int i = 0; i < 16; ++i) b = fmaxf(b, fabsf(u[i]));
            if constexpr (COL_FMT == 5) b = tile_b;
            float e;
            const uint32_t S = nvfp4_block_scale(ts, q_tab[1], b, e);
            const uint64_t Lbase = (uint64_t)(k0 + jj) * (uint64_t)a.col_cols_store + (uint64_t)prow0;
            float h0[8], h1[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) { h0[i] = u[i]; h1[i] = u[i + 8]; }
            const uint32_t c0 = nvfp4_encode8<SR>(h0, e, Lbase, 1, a);
            const uint32_t c1 = nvfp4_encode8<SR>(h1, e, Lbase + 8, 1, a);
            *reinterpret_cast<uint2*>(&sm.col_codes[col_chunk_nv(c_loc + jj, r_loc / 16)]) = make_uint2(c0, c1);
            const int kk = c_loc + jj;
            const int c = r_loc / 16;
            sm.col_scales[kk >> 7][(c >> 2) * 512 + (kk & 31) * 16 + ((kk >> 5) & 3) * 4 + (c & 3)] =
                (uint8_t)(kvalid ? S : 0);
        }
        }
    } else if constexpr (COL_FMT == 2) {  // MXFP8: 32-blocks = this thread's 16 rows + lane^16's
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float u[16];
            column16(t, j, u);
            float b = 0.0f;
#pragma unroll
            for (int i = 0; i < 16; ++i) b = fmaxf(b, fabsf(u[i]));
            b = fmaxf(b, __shfl_xor_sync(0xFFFFFFFFu, b, 16));
            const int e = mx_exponent(b);
            const float sc = exp2_neg(e);
            uint4 q;
            q.x = e4m3x4_rn(__fmul_rn(u[0], sc), __fmul_rn(u[1], sc), __fmul_rn(u[2], sc), __fmul_rn(u[3], sc));
            q.y = e4m3x4_rn(__fmul_rn(u[4], sc), __fmul_rn(u[5], sc), __fmul_rn(u[6], sc), __fmul_rn(u[7], sc));
            q.z = e4m3x4_rn(__fmul_rn(u[8], sc), __fmul_rn(u[9], sc), __fmul_rn(u[10], sc), __fmul_rn(u[11], sc));
            q.w = e4m3x4_rn(__fmul_rn(u[12], sc), __fmul_rn(u[13], sc), __fmul_rn(u[14], sc), __fmul_rn(u[15], sc));
            *reinterpret_cast<uint4*>(&sm.col_codes[col_chunk_mx(c_loc + j, r_loc / 16)]) = q;
            if ((lane >> 4) == 0) {
                const int kk = c_loc + j;
                const int c = r_loc / 32;  // 0..3
                sm.col_scales[kk >> 7][(kk & 31) * 16 + ((kk >> 5) & 3) * 4 + (c & 3)] =
                    (uint8_t)(kvalid ? (e + 127) : 0);
            }
        }
    } else if constexpr (COL_FMT == 3) {  // identity: the bf16 columns, transposed (32 contiguous bytes per block)
        if (kvalid && prow0 < a.col_cols_store) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                uint32_t w[8];
                column16_bf16(t, j, w);
                uint4* dst = reinterpret_cast<uint4*>(a.col_data + ((k0 + j) * a.col_cols_store + prow0) * 2);
                dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
            }
        }
    }
    __syncthreads();

    // ---------------- write-out of staged outputs
    const int64_t p_tile0 = tile_row * kTileRows;
    if (!row_out) {
    } else if constexpr (ROW_FMT == 1 || ROW_FMT == 2 || ROW_FMT == 4) {
        // this CTA's scale columns: NVFP4 16 (4 tiles), MXFP8 8 (2 tiles), all in tile-row tile_row
        constexpr int ntiles = ROW_FMT == 2 ? 2 : 4;
        const int64_t ct0 = tile_col * ntiles;
        for (int i = threadIdx.x; i < ntiles * 32; i += kThreads) {
            const int tt = i >> 5;
            if (ct0 + tt < a.row_scale_ctiles) {
                uint8_t* dst = a.row_scale + ((tile_row * a.row_scale_ctiles + ct0 + tt) * 512) + (i & 31) * 16;
                *reinterpret_cast<uint4*>(dst) = reinterpret_cast<const uint4*>(sm.row_scales)[i];
            }
        }
    }
    if (!col_pass) {
    } else if constexpr (COL_FMT == 1 || COL_FMT == 2 || COL_FMT == 5) {
        constexpr bool kNv = COL_FMT != 2;
        const int64_t row_bytes = kNv ? a.col_cols_store / 2 : a.col_cols_store;
        const int64_t byte0 = kNv ? p_tile0 / 2 : p_tile0;
        for (int i = threadIdx.x; i < kTileCols * 8; i += kThreads) {
            const int kk = i >> 3, ch = i & 7;  // 8 chunks per output row
            const int64_t k = tile_col * kTileCols + kk;
            if (kNv) {
                const int64_t off = byte0 + ch * 8;
                if (k < a.K && off < row_bytes)
                    *reinterpret_cast<uint2*>(a.col_data + k * row_bytes + off) =
                        *reinterpret_cast<const uint2*>(&sm.col_codes[col_chunk_nv(kk, ch)]);
            } else {
                const int64_t off = byte0 + ch * 16;
                if (k < a.K && off < row_bytes)
                    *reinterpret_cast<uint4*>(a.col_data + k * row_bytes + off) =
                        *reinterpret_cast<const uint4*>(&sm.col_codes[col_chunk_mx(kk, ch)]);
            }
        }
        // scales: output rows k (two 128-row tile-rows), scale columns p/16 (NVFP4, 2 tiles) or p/32 (1 tile)
        constexpr int nct = kNv ? 2 : 1;
        const int64_t ct0 = kNv ? (p_tile0 / 16) / 4 : (p_tile0 / 32) / 4;
        for (int i = threadIdx.x; i < 2 * nct * 32; i += kThreads) {
            const int kt = i / (nct * 32), rem = i % (nct * 32), tt = rem >> 5, chunk = rem & 31;
            const int64_t ktile = tile_col * 2 + kt;  // 128-row tile of the output rows
            if (ktile * 128 < a.col_scale_rows_pad && ct0 + tt < a.col_scale_ctiles) {
                uint8_t* dst = a.col_scale + (ktile * a.col_scale_ctiles + ct0 + tt) * 512 + chunk * 16;
                *reinterpret_cast<uint4*>(dst) =
                    *reinterpret_cast<const uint4*>(&sm.col_scales[kt][tt * 512 + chunk * 16]);
            }
        }
    }
}


// One launch of a quantize_kernel variant.
template <int R, int C, bool RHT, bool SR, bool DQ>
inline void launch_quantize_variant(const QuantArgs& a, dim3 grid, cudaStream_t s)
{
    quantize_kernel<R, C, RHT, SR, DQ><<<grid, kThreads, 0, s>>>(a);
}

inline dim3 quantize_grid(const QuantArgs& a, int64_t row_tiles)
{
    return dim3((unsigned)((a.K + kTileCols - 1) / kTileCols), (unsigned)row_tiles);
}

}  // namespace nvq
