/*
 * oracle.c -- plain, slow CPU reference for the block-scaled quantize + GEMM
 * path.  TEST INFRASTRUCTURE ONLY: it is loaded by the tests, by the smoke
 * check and by the benchmark's CPU-baseline leg, never by the library.  It
 * shares no code, header, table or helper with the CUDA library.
 *
 * Sources (pages read for what the method computes):
 *   [TT]  "Add an NVFP4 quantization converter" (torchtitan PR #3914),
 *         section "What changed": NVFP4Linear with a per-rank Philox
 *         stochastic-rounding key (_sr_seed) and a 16-point random Hadamard
 *         sign vector (_rht_sign_vector) shared by both GEMM operands;
 *         review thread on "rowwise": NVFP4 = outer (tensor) scale plus an
 *         inner 1x16 block scale.
 *   [TE]  "Hybrid quantization" (TransformerEngine PR #2817), section
 *         "Description": rowwise / columnwise directions each with their own
 *         format; greptile review of mxfp8_tensor_storage: MXFP8 blocks of
 *         MXFP8_BLOCK_SCALING_SIZE = 32 rows, ceil(M/32) columnwise scales.
 *
 * The pages name the formats but never print their bit layouts, scale
 * formulas, the Hadamard construction or the Philox counter layout.  Every
 * such step below is a stated reading (marked READING) of the plainest kind
 * that agrees with the pages.
 *
 * Floating point: every operation that decides a code is done in IEEE fp32
 * with round-to-nearest-even and no contraction (built with
 * -ffp-contract=off); the dequantized GEMM accumulates in fp64.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------ */
/* bf16 / fp32 bit helpers                                             */
/* ------------------------------------------------------------------ */

static float bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

ORC_API float orc_bf16_to_f32(uint16_t h) { return bf16_to_f32(h); }

/* ------------------------------------------------------------------ */
/* Element and scale formats (READING: OCP "fn" formats)               */
/*   E2M1: sign | 2-bit exponent (bias 1) | 1-bit mantissa, no inf/NaN */
/*   E4M3: sign | 4-bit exponent (bias 7) | 3-bit mantissa, S.1111.111 */
/*         is NaN, no inf, max finite 448                               */
/*   E8M0: unsigned exponent, value 2^(e-127), 255 is NaN               */
/* ------------------------------------------------------------------ */

ORC_API double orc_e2m1_decode(uint8_t code)
{
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double mag = (e == 0) ? ldexp((double)m, -1)            /* subnormal: m/2 * 2^(1-1) */
                          : ldexp(1.0 + m / 2.0, e - 1);     /* normal: (1+m/2) 2^(e-1) */
    return s ? -mag : mag;
}

ORC_API double orc_e4m3_decode(uint8_t code)
{
    int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7) return NAN;
    double mag = (e == 0) ? ldexp((double)m, -9)             /* m/8 * 2^(1-7) */
                          : ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

ORC_API double orc_e8m0_decode(uint8_t code)
{
    if (code == 255) return NAN;
    return ldexp(1.0, (int)code - 127);
}

/* Round a >= 0 to the nearest multiple of q (a power of two), ties to an
 * even multiple.  a / q is exact, so this is an exact integer rounding. */
static double rne_multiple(double a, double q)
{
    double n = a / q;
    double fl = floor(n);
    double fr = n - fl;
    double k = fl;
    if (fr > 0.5 || (fr == 0.5 && fmod(fl, 2.0) != 0.0)) k = fl + 1.0;
    return k * q;
}

/* Exact grid value -> E2M1 magnitude bits (e<<1 | m). */
static uint8_t e2m1_mag_bits(double mag)
{
    if (mag == 0.0) return 0;
    int ex = ilogb(mag);                 /* floor(log2 mag) */
    if (ex < 0) return 1;                /* 0.5: subnormal, mantissa 1 */
    int m = (int)((mag / ldexp(1.0, ex) - 1.0) * 2.0);
    return (uint8_t)(((ex + 1) << 1) | m);
}

/* E2M1 round-to-nearest-even with saturation to +-6; the sign of v is
 * kept, so a negative value that rounds to zero gives code 0x8. */
ORC_API uint8_t orc_e2m1_encode_rn(float v)
{
    uint8_t s = signbit(v) ? 8 : 0;
    double a = fabs((double)v);
    if (a >= 6.0) return s | 7;
    double q = (a < 2.0) ? 0.5 : (a < 4.0 ? 1.0 : 2.0);   /* grid spacing in the binade */
    return s | e2m1_mag_bits(rne_multiple(a, q));
}

/* Exact grid value -> E4M3 magnitude bits. */
static uint8_t e4m3_mag_bits(double mag)
{
    if (mag == 0.0) return 0;
    int ex = ilogb(mag);
    if (ex < -6) return (uint8_t)(mag / ldexp(1.0, -9));  /* subnormal mantissa */
    int m = (int)((mag / ldexp(1.0, ex) - 1.0) * 8.0);
    return (uint8_t)(((ex + 7) << 3) | m);
}

/* E4M3 round-to-nearest-even, saturating to +-448 (satfinite). */
ORC_API uint8_t orc_e4m3_encode_rn(float v)
{
    uint8_t s = signbit(v) ? 0x80 : 0;
    double a = fabs((double)v);
    if (a >= 448.0) return s | 0x7E;
    double q;
    if (a < ldexp(1.0, -6)) q = ldexp(1.0, -9);           /* subnormal spacing */
    else q = ldexp(1.0, ilogb(a) - 3);                    /* 3 mantissa bits */
    return s | e4m3_mag_bits(rne_multiple(a, q));
}

/* ------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: */
/* as easy as 1, 2, 3", SC'11): 10 rounds of the 4x32 S-box keyed by a */
/* 64-bit key that is bumped by the Weyl constants between rounds.      */
/* ------------------------------------------------------------------ */

ORC_API void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) { k0 += W0; k1 += W1; }
        uint64_t p0 = (uint64_t)M0 * c0;
        uint64_t p1 = (uint64_t)M1 * c2;
        uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        uint32_t n1 = (uint32_t)p1;
        uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        uint32_t n3 = (uint32_t)p0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* READING (the pages say only "a Philox key", [TT] "What changed"): the
 * 16 random bits for the element at linear index L of a direction's output
 * (row: i*K + k; col: k*M_padded + i).  Key = the int64 seed as two 32-bit
 * words (low first).  One Philox call covers the 8 elements L>>3; its four
 * words hold two 16-bit fields each, low half first. */
ORC_API uint32_t orc_sr_bits(int64_t seed, uint32_t offset, int direction, uint64_t L)
{
    uint64_t useed = (uint64_t)seed, blk = L >> 3;
    uint32_t key[2] = {(uint32_t)useed, (uint32_t)(useed >> 32)};
    uint32_t ctr[4] = {(uint32_t)blk, (uint32_t)(blk >> 32), (uint32_t)direction, offset};
    uint32_t w[4];
    orc_philox4x32_10(ctr, key, w);
    return (w[(L & 7) >> 1] >> (16 * (L & 1))) & 0xFFFFu;
}

/* E2M1 stochastic rounding ([TT] "What changed": SR is unbiased).  With
 * lo <= |v| < hi the two neighbouring grid values, the magnitude rounds up
 * iff r < ceil(frac * 2^16), frac = (|v| - lo) / (hi - lo); both the
 * subtraction and the division by the power-of-two spacing are exact.  At
 * or above 6 the result saturates.  The sign of v is kept. */
ORC_API uint8_t orc_e2m1_encode_sr(float v, uint32_t r16)
{
    uint8_t s = signbit(v) ? 8 : 0;
    double a = fabs((double)v);
    if (a >= 6.0) return s | 7;
    double q = (a < 2.0) ? 0.5 : (a < 4.0 ? 1.0 : 2.0);
    double lo = floor(a / q) * q, hi = lo + q;
    double frac = (a - lo) / q;
    double thresh = ceil(frac * 65536.0);
    double mag = ((double)r16 < thresh) ? hi : lo;
    return s | e2m1_mag_bits(mag);
}

/* ------------------------------------------------------------------ */
/* 16-point random Hadamard transform ([TT] "What changed": the basis  */
/* only cancels when both GEMM operands share the sign vector).         */
/* READING: T(u) = (1/4) H16 (s . u), H16 the Sylvester Hadamard matrix */
/* H[i][j] = (-1)^popcount(i&j), applied by the in-place fast           */
/* Walsh-Hadamard butterfly in fp32 with spans 1, 2, 4, 8, each pair    */
/* (a, b) -> (a + b, a - b); the sign flip and the final 1/4 are exact. */
/* ------------------------------------------------------------------ */

ORC_API void orc_rht16(float u[16], const int8_t sign[16])
{
    for (int i = 0; i < 16; ++i)
        if (sign[i] < 0) u[i] = -u[i];
    for (int h = 1; h < 16; h <<= 1)
        for (int i = 0; i < 16; ++i)
            if ((i & h) == 0) {
                float a = u[i], b = u[i + h];
                u[i] = a + b;
                u[i + h] = a - b;
            }
    for (int i = 0; i < 16; ++i) u[i] = u[i] * 0.25f;
}

/* ------------------------------------------------------------------ */
/* Tensor amax (the FP32 per-tensor scale's input)                      */
/* ------------------------------------------------------------------ */

ORC_API float orc_amax(const uint16_t* x, int64_t M, int64_t K, int64_t ld)
{
    float amax = 0.0f;
    for (int64_t i = 0; i < M; ++i)
        for (int64_t k = 0; k < K; ++k) {
            float a = fabsf(bf16_to_f32(x[i * ld + k]));
            if (a > amax) amax = a;
        }
    return amax;
}

/* Column 16-block j of column k, rows beyond M read as zero. */
static void load_col_block(const uint16_t* x, int64_t M, int64_t ld, int64_t k, int64_t j, float u[16])
{
    for (int t = 0; t < 16; ++t) {
        int64_t i = 16 * j + t;
        u[t] = (i < M) ? bf16_to_f32(x[i * ld + k]) : 0.0f;
    }
}

/* amax of the Hadamard-transformed columnwise blocks. */
ORC_API float orc_amax_rht_col(const uint16_t* x, int64_t M, int64_t K, int64_t ld, const int8_t sign[16])
{
    float amax = 0.0f;
    int64_t nb = (M + 15) / 16;
    for (int64_t k = 0; k < K; ++k)
        for (int64_t j = 0; j < nb; ++j) {
            float u[16];
            load_col_block(x, M, ld, k, j, u);
            orc_rht16(u, sign);
            for (int t = 0; t < 16; ++t)
                if (fabsf(u[t]) > amax) amax = fabsf(u[t]);
        }
    return amax;
}

/* ------------------------------------------------------------------ */
/* NVFP4 block quantization (READING of "E4M3 block scale + FP32 tensor */
/* scale", [TT] review of "rowwise"):                                   */
/*   s_enc = 2688 / A   (2688 = 6 * 448; A = 0 -> 1; overflow -> FLT_MAX) */
/*   S     = E4M3_rn_sat(b * (448 / A))  (b = block amax; b = 0 -> S = 0) */
/*   e     = s_enc / E4M3(S)  (S = 0 -> 0; overflow -> FLT_MAX)          */
/*   q_i   = E2M1_round(x_i * e)                                        */
/* decoded value: E2M1(q) * E4M3(S) * g with g = A / 2688.              */
/* ------------------------------------------------------------------ */

ORC_API float orc_nvfp4_s_enc(float A)
{
    if (A == 0.0f) return 1.0f;
    float s = 2688.0f / A;
    return isinf(s) ? FLT_MAX : s;
}

ORC_API float orc_nvfp4_g(float A) { return A / 2688.0f; }

typedef struct {
    int on;
    int64_t seed;
    uint32_t offset;
} orc_sr;

/* Quantize one 16-block u (values already in the quantized domain). */
static void nvfp4_block(const float u[16], float A, const orc_sr* sr, int direction,
                        uint64_t L0, uint8_t codes[16], uint8_t* scale)
{
    float b = 0.0f;
    for (int t = 0; t < 16; ++t)
        if (fabsf(u[t]) > b) b = fabsf(u[t]);
    uint8_t S = 0;
    if (b != 0.0f && A != 0.0f) {
        float r448 = 448.0f / A;
        S = orc_e4m3_encode_rn(b * r448);
    }
    float e = 0.0f;
    if (S != 0) {
        e = orc_nvfp4_s_enc(A) / (float)orc_e4m3_decode(S);
        if (isinf(e)) e = FLT_MAX;
    }
    for (int t = 0; t < 16; ++t) {
        float v = u[t] * e;
        if (sr->on)
            codes[t] = orc_e2m1_encode_sr(v, orc_sr_bits(sr->seed, sr->offset, direction, L0 + (uint64_t)t));
        else
            codes[t] = orc_e2m1_encode_rn(v);
    }
    *scale = S;
}

/* Rowwise NVFP4 of the M rows x[0..M) that are rows row0.. of a larger
 * tensor with A its amax: 16-blocks along K, element (i, k) drawing its
 * stochastic-rounding bits at linear index (row0 + i) * K + k.  Outputs
 * codes[M][K/2] (low nibble = even k) and compact scales[M][K/16]. */
ORC_API void orc_nvfp4_quantize_rows_at(const uint16_t* x, int64_t M, int64_t K, int64_t ld, float A,
                                        int sr_on, int64_t seed, uint32_t offset, int64_t row0,
                                        uint8_t* codes, uint8_t* scales)
{
    orc_sr sr = {sr_on, seed, offset};
    int64_t nb = K / 16;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < nb; ++j) {
            float u[16];
            uint8_t q[16];
            for (int t = 0; t < 16; ++t) u[t] = bf16_to_f32(x[i * ld + 16 * j + t]);
            nvfp4_block(u, A, &sr, 0, (uint64_t)((row0 + i) * K + 16 * j), q, &scales[i * nb + j]);
            for (int t = 0; t < 8; ++t)
                codes[i * (K / 2) + 8 * j + t] = (uint8_t)(q[2 * t] | (q[2 * t + 1] << 4));
        }
}

/* Rowwise NVFP4: 16-blocks along K.  Outputs codes[M][K/2] (low nibble =
 * even k) and compact scales[M][K/16].  K % 16 == 0. */
ORC_API void orc_nvfp4_quantize_rows(const uint16_t* x, int64_t M, int64_t K, int64_t ld, float A,
                                     int sr_on, int64_t seed, uint32_t offset,
                                     uint8_t* codes, uint8_t* scales)
{
    orc_nvfp4_quantize_rows_at(x, M, K, ld, A, sr_on, seed, offset, 0, codes, scales);
}

/* Columnwise NVFP4 of the M rows x[0..M) that are rows row0.. (row0 % 16
 * == 0) of a larger tensor whose columnwise storage has Mp_total columns and
 * whose (transformed) amax is A: 16-blocks along the rows, stored transposed
 * as codes[K][Mp/2] and compact scales[K][Mp/16], Mp = M rounded up to 16
 * (rows beyond M are zero); element (k, i) draws its stochastic-rounding bits
 * at linear index k * Mp_total + row0 + i.  rht_sign != NULL applies T to
 * every block before quantizing. */
ORC_API void orc_nvfp4_quantize_cols_at(const uint16_t* x, int64_t M, int64_t K, int64_t ld, float A,
                                        const int8_t* rht_sign, int sr_on, int64_t seed, uint32_t offset,
                                        int64_t row0, int64_t Mp_total, uint8_t* codes, uint8_t* scales)
{
    orc_sr sr = {sr_on, seed, offset};
    int64_t nb = (M + 15) / 16, Mp = nb * 16;
#pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < K; ++k)
        for (int64_t j = 0; j < nb; ++j) {
            float u[16];
            uint8_t q[16];
            load_col_block(x, M, ld, k, j, u);
            if (rht_sign) orc_rht16(u, rht_sign);
            nvfp4_block(u, A, &sr, 1, (uint64_t)(k * Mp_total + row0 + 16 * j), q, &scales[k * nb + j]);
            for (int t = 0; t < 8; ++t)
                codes[k * (Mp / 2) + 8 * j + t] = (uint8_t)(q[2 * t] | (q[2 * t + 1] << 4));
        }
}

/* Columnwise NVFP4: 16-blocks along M, stored transposed: codes[K][Mp/2],
 * compact scales[K][Mp/16], Mp = M rounded up to 16 (rows beyond M are
 * zero).  rht_sign != NULL applies T to every block before quantizing; A is
 * then the amax of the transformed tensor. */
ORC_API void orc_nvfp4_quantize_cols(const uint16_t* x, int64_t M, int64_t K, int64_t ld, float A,
                                     const int8_t* rht_sign, int sr_on, int64_t seed, uint32_t offset,
                                     uint8_t* codes, uint8_t* scales)
{
    int64_t Mp = (M + 15) / 16 * 16;
    orc_nvfp4_quantize_cols_at(x, M, K, ld, A, rht_sign, sr_on, seed, offset, 0, Mp, codes, scales);
}

/* ------------------------------------------------------------------ */
/* NVFP4 2D block scaling, columnwise ([TE] "Hybrid quantization",        */
/* timeline: "[Common] Enable NVFP4 2D block scaling in columnwise only").  */
/* READING: the columnwise direction of x[M][K] takes one E4M3 scale per   */
/* 16 x 16 tile (rows 16j.., columns 16c..) from the tile's amax, with the */
/* per-tensor recipe otherwise unchanged (s_enc, the block scale from the  */
/* amax, the element factor, RTN); each of the tile's 16 columnwise        */
/* 1 x 16 blocks is stored with that scale.  The rowwise direction keeps   */
/* 1 x 16 blocks.  Rows past M read as zero; K % 16 == 0.                  */
/* ------------------------------------------------------------------ */

ORC_API void orc_nvfp4_quantize_cols_2d(const uint16_t* x, int64_t M, int64_t K, int64_t ld, float A,
                                        uint8_t* codes, uint8_t* scales)
{
    int64_t nb = (M + 15) / 16, Mp = nb * 16;
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < nb; ++j)
        for (int64_t c = 0; c < K / 16; ++c) {
            float tile[16][16];  /* [column in tile][row in block] */
            float b = 0.0f;
            for (int kk = 0; kk < 16; ++kk) {
                load_col_block(x, M, ld, 16 * c + kk, j, tile[kk]);
                for (int t = 0; t < 16; ++t)
                    if (fabsf(tile[kk][t]) > b) b = fabsf(tile[kk][t]);
            }
            uint8_t S = 0;
            if (b != 0.0f && A != 0.0f) S = orc_e4m3_encode_rn(b * (448.0f / A));
            float e = 0.0f;
            if (S != 0) {
                e = orc_nvfp4_s_enc(A) / (float)orc_e4m3_decode(S);
                if (isinf(e)) e = FLT_MAX;
            }
            for (int kk = 0; kk < 16; ++kk) {
                int64_t k = 16 * c + kk;
                uint8_t q[16];
                for (int t = 0; t < 16; ++t) q[t] = orc_e2m1_encode_rn(tile[kk][t] * e);
                for (int t = 0; t < 8; ++t)
                    codes[k * (Mp / 2) + 8 * j + t] = (uint8_t)(q[2 * t] | (q[2 * t + 1] << 4));
                scales[k * nb + j] = S;
            }
        }
}

/* ------------------------------------------------------------------ */
/* Row-scaled NVFP4 ([TE] "Hybrid quantization", Description: the grouped */
/* GEMM recipe's input quantizer NVFP4Quantizer(row_scaled_nvfp4=True)).  */
/* READING: the FP32 outer scale is per row instead of per tensor: row r   */
/* has its own amax A_r = max_k |x[r][k]|, which takes the place of the    */
/* tensor amax in every step above (s_enc, the block scale, the element    */
/* factor), and decodes with g_r = A_r / 2688.  Rowwise only.              */
/* ------------------------------------------------------------------ */

ORC_API void orc_nvfp4_dequant(const uint8_t* codes, const uint8_t* scales, int64_t R, int64_t C,
                               float g, double* out);

ORC_API void orc_nvfp4_quantize_rows_rowscaled(const uint16_t* x, int64_t M, int64_t K, int64_t ld,
                                               uint8_t* codes, uint8_t* scales, float* amax_rows)
{
    orc_sr rtn = {0, 0, 0};
    int64_t nb = K / 16;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i) {
        float A = orc_amax(x + i * ld, 1, K, ld);
        amax_rows[i] = A;
        for (int64_t j = 0; j < nb; ++j) {
            float u[16];
            uint8_t q[16];
            for (int t = 0; t < 16; ++t) u[t] = bf16_to_f32(x[i * ld + 16 * j + t]);
            nvfp4_block(u, A, &rtn, 0, (uint64_t)(i * K + 16 * j), q, &scales[i * nb + j]);
            for (int t = 0; t < 8; ++t)
                codes[i * (K / 2) + 8 * j + t] = (uint8_t)(q[2 * t] | (q[2 * t + 1] << 4));
        }
    }
}

ORC_API void orc_nvfp4_dequant_rowscaled(const uint8_t* codes, const uint8_t* scales, int64_t R, int64_t C,
                                         const float* amax_rows, double* out)
{
    for (int64_t r = 0; r < R; ++r)
        orc_nvfp4_dequant(codes + r * (C / 2), scales + r * (C / 16), 1, C, orc_nvfp4_g(amax_rows[r]), out + r * C);
}

/* ------------------------------------------------------------------ */
/* MXFP8 ([TE] mxfp8 storage review: 32-element blocks, E8M0 scale,     */
/* ceil(M/32) columnwise scale rows).  READING (OCP MX): with b the     */
/* block amax, e = clamp(floor(log2 b) - 8, -127, 127) (8 = emax of     */
/* E4M3; b = 0 gives -127), scale code e + 127, elements                */
/* E4M3_rn_sat(x * 2^-e).                                               */
/* ------------------------------------------------------------------ */

static int mx_exponent(float b)
{
    if (b == 0.0f) return -127;
    int e = ilogb((double)b) - 8;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

static void mxfp8_block(const float u[32], uint8_t codes[32], uint8_t* scale)
{
    float b = 0.0f;
    for (int t = 0; t < 32; ++t)
        if (fabsf(u[t]) > b) b = fabsf(u[t]);
    int e = mx_exponent(b);
    for (int t = 0; t < 32; ++t) codes[t] = orc_e4m3_encode_rn((float)ldexp((double)u[t], -e));
    *scale = (uint8_t)(e + 127);
}

/* Rowwise MXFP8: codes[M][K], compact scales[M][K/32].  K % 32 == 0. */
ORC_API void orc_mxfp8_quantize_rows(const uint16_t* x, int64_t M, int64_t K, int64_t ld,
                                     uint8_t* codes, uint8_t* scales)
{
    int64_t nb = K / 32;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < nb; ++j) {
            float u[32];
            for (int t = 0; t < 32; ++t) u[t] = bf16_to_f32(x[i * ld + 32 * j + t]);
            mxfp8_block(u, &codes[i * K + 32 * j], &scales[i * nb + j]);
        }
}

/* Columnwise MXFP8: codes[K][Mp], compact scales[K][Mp/32], Mp = M rounded
 * up to 32, the partial last block zero-padded (ceil, not floor). */
ORC_API void orc_mxfp8_quantize_cols(const uint16_t* x, int64_t M, int64_t K, int64_t ld,
                                     uint8_t* codes, uint8_t* scales)
{
    int64_t nb = (M + 31) / 32, Mp = nb * 32;
#pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < K; ++k)
        for (int64_t j = 0; j < nb; ++j) {
            float u[32];
            for (int t = 0; t < 32; ++t) {
                int64_t i = 32 * j + t;
                u[t] = (i < M) ? bf16_to_f32(x[i * ld + k]) : 0.0f;
            }
            mxfp8_block(u, &codes[k * Mp + 32 * j], &scales[k * nb + j]);
        }
}

/* ------------------------------------------------------------------ */
/* Scale layout for block-scaled GEMMs (READING: the public cuBLAS /     */
/* PTX block-scaling layout): scales[R][C] live in 128 x 4 tiles of      */
/* 512 bytes, tile (r/128)*ceil(C/4) + c/4, inside the tile at           */
/* (r%32)*16 + ((r%128)/32)*4 + c%4; pads are zero.                      */
/* ------------------------------------------------------------------ */

ORC_API int64_t orc_swizzled_size(int64_t R, int64_t C)
{
    return ((R + 127) / 128) * 128 * ((C + 3) / 4) * 4;
}

static int64_t swz_offset(int64_t r, int64_t c, int64_t C)
{
    int64_t ctiles = (C + 3) / 4;
    return ((r / 128) * ctiles + c / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + c % 4;
}

ORC_API void orc_scale_swizzle(const uint8_t* compact, int64_t R, int64_t C, uint8_t* out)
{
    memset(out, 0, (size_t)orc_swizzled_size(R, C));
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c) out[swz_offset(r, c, C)] = compact[r * C + c];
}

ORC_API void orc_scale_unswizzle(const uint8_t* swz, int64_t R, int64_t C, uint8_t* compact)
{
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c) compact[r * C + c] = swz[swz_offset(r, c, C)];
}

/* ------------------------------------------------------------------ */
/* Dequantization to fp64                                               */
/* ------------------------------------------------------------------ */

ORC_API void orc_nvfp4_dequant(const uint8_t* codes, const uint8_t* scales, int64_t R, int64_t C,
                               float g, double* out)
{
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c) {
            uint8_t byte = codes[r * (C / 2) + c / 2];
            uint8_t q = (c & 1) ? (byte >> 4) : (byte & 15);
            out[r * C + c] = orc_e2m1_decode(q) * orc_e4m3_decode(scales[r * (C / 16) + c / 16]) * (double)g;
        }
}

ORC_API void orc_mxfp8_dequant(const uint8_t* codes, const uint8_t* scales, int64_t R, int64_t C, double* out)
{
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c)
            out[r * C + c] = orc_e4m3_decode(codes[r * C + c]) * orc_e8m0_decode(scales[r * (C / 32) + c / 32]);
}

/* ------------------------------------------------------------------ */
/* Rowwise-dequantized source and the identity direction ([TE]          */
/* "Hybrid quantization", "Enable columnwise_source and hybrid recipes": */
/* with columnwise_source = "rowwise_dequantized" the columnwise operand  */
/* is built from dequantize(rowwise-quantized x) -- double quantization  */
/* when the columnwise quantizer is not the identity; IdentityQuantizer  */
/* passes the high-precision value through).                            */
/* READING: the dequantized value is formed in fp32 -- NVFP4: the exact  */
/* product E2M1(q) * E4M3(S), times g = A / 2688 with one rounding;      */
/* MXFP8: E4M3(q) * 2^e, exact -- and stored in the training dtype,      */
/* bf16, with one round to nearest even.                                 */
/* ------------------------------------------------------------------ */

ORC_API void orc_f64_to_bf16_rne(const double* v, int64_t n, uint16_t* out);

/* fp32 -> bf16 bits, round to nearest even (finite inputs). */
static uint16_t f32_to_bf16_rne(float f)
{
    uint16_t out;
    double d = (double)f;
    orc_f64_to_bf16_rne(&d, 1, &out);
    return out;
}

/* bf16 bits of the dequantized NVFP4 operand codes[R][C/2] with compact
 * scales[R][C/16] and tensor amax A. */
ORC_API void orc_nvfp4_dequant_bf16(const uint8_t* codes, const uint8_t* scales, int64_t R, int64_t C, float A,
                                    uint16_t* out)
{
    float g = orc_nvfp4_g(A);
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c) {
            uint8_t byte = codes[r * (C / 2) + c / 2];
            uint8_t q = (c & 1) ? (byte >> 4) : (byte & 15);
            float cs = (float)(orc_e2m1_decode(q) * orc_e4m3_decode(scales[r * (C / 16) + c / 16]));  /* exact */
            float v = cs * g;
            out[r * C + c] = f32_to_bf16_rne(v);
        }
}

/* bf16 bits of the dequantized MXFP8 operand codes[R][C], scales[R][C/32]. */
ORC_API void orc_mxfp8_dequant_bf16(const uint8_t* codes, const uint8_t* scales, int64_t R, int64_t C, uint16_t* out)
{
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c) {
            float v = (float)(orc_e4m3_decode(codes[r * C + c]) * orc_e8m0_decode(scales[r * (C / 32) + c / 32]));
            out[r * C + c] = f32_to_bf16_rne(v);
        }
}

/* Identity direction: the bf16 values themselves.  Rowwise: a copy of
 * x[M][K]; columnwise: the transpose, out[K][Mp] with Mp = M rounded up to
 * 16 and the columns past M zero. */
ORC_API void orc_identity_rows(const uint16_t* x, int64_t M, int64_t K, int64_t ld, uint16_t* out)
{
    for (int64_t i = 0; i < M; ++i)
        for (int64_t k = 0; k < K; ++k) out[i * K + k] = x[i * ld + k];
}

ORC_API void orc_identity_cols(const uint16_t* x, int64_t M, int64_t K, int64_t ld, uint16_t* out)
{
    int64_t Mp = (M + 15) / 16 * 16;
    for (int64_t k = 0; k < K; ++k)
        for (int64_t i = 0; i < Mp; ++i) out[k * Mp + i] = (i < M) ? x[i * ld + k] : 0;
}

/* ------------------------------------------------------------------ */
/* GEMM in TN form: out[r][c] = alpha * sum_k A[r][k] * B[c][k] + bias[c] */
/* (fp64 accumulation of the dequantized operands).                      */
/* ------------------------------------------------------------------ */

ORC_API void orc_gemm_tn_f64(const double* A, const double* B, int64_t R, int64_t Cn, int64_t K,
                             double alpha, const double* bias, double* out)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < Cn; ++c) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) acc += A[r * K + k] * B[c * K + k];
            out[r * Cn + c] = alpha * acc + (bias ? bias[c] : 0.0);
        }
}

/* Selected outputs of the same product straight from quantized operands
 * (for sizes whose fp64 operands would not fit): fmt 1 = NVFP4 (codes
 * packed two per byte, compact 1x16 E4M3 scales, tensor decode factor g),
 * fmt 2 = MXFP8 (E4M3 codes, compact 1x32 E8M0 scales). */
static double deq_elem(int fmt, const uint8_t* codes, const uint8_t* scales, int64_t r, int64_t k,
                       int64_t K, float g)
{
    if (fmt == 1) {
        uint8_t byte = codes[r * (K / 2) + k / 2];
        uint8_t q = (k & 1) ? (byte >> 4) : (byte & 15);
        return orc_e2m1_decode(q) * orc_e4m3_decode(scales[r * (K / 16) + k / 16]) * (double)g;
    }
    return orc_e4m3_decode(codes[r * K + k]) * orc_e8m0_decode(scales[r * (K / 32) + k / 32]);
}

ORC_API void orc_gemm_tn_sampled(int fmt, const uint8_t* a_codes, const uint8_t* a_scales, float g_a,
                                 const uint8_t* b_codes, const uint8_t* b_scales, float g_b, int64_t K,
                                 const double* bias, int64_t n_samples, const int64_t* rows,
                                 const int64_t* cols, double* out)
{
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t s = 0; s < n_samples; ++s) {
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k)
            acc += deq_elem(fmt, a_codes, a_scales, rows[s], k, K, g_a) *
                   deq_elem(fmt, b_codes, b_scales, cols[s], k, K, g_b);
        out[s] = acc + (bias ? bias[cols[s]] : 0.0);
    }
}

/* orc_gemm_tn_sampled for a row-scaled NVFP4 A (decode factor g_a_rows[r]
 * for row r) and an NVFP4 B with decode factor g_b. */
ORC_API void orc_gemm_tn_sampled_rowscaled(const uint8_t* a_codes, const uint8_t* a_scales, const float* g_a_rows,
                                           const uint8_t* b_codes, const uint8_t* b_scales, float g_b, int64_t K,
                                           int64_t n_samples, const int64_t* rows, const int64_t* cols, double* out)
{
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t s = 0; s < n_samples; ++s) {
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k)
            acc += deq_elem(1, a_codes, a_scales, rows[s], k, K, g_a_rows[rows[s]]) *
                   deq_elem(1, b_codes, b_scales, cols[s], k, K, g_b);
        out[s] = acc;
    }
}

/* fp64 -> bf16 with one round to nearest even (output rounding of the
 * bf16-output GEMM check); overflow goes to infinity like an IEEE cast. */
ORC_API void orc_f64_to_bf16_rne(const double* v, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i) {
        double x = v[i];
        uint16_t sign = signbit(x) ? 0x8000 : 0;
        double a = fabs(x);
        if (isnan(x)) { out[i] = 0x7FC0; continue; }
        if (a == 0.0) { out[i] = sign; continue; }
        int e = ilogb(a);
        if (e < -126) e = -126;                 /* subnormal spacing 2^-133 */
        double mag = rne_multiple(a, ldexp(1.0, e - 7));
        if (mag >= ldexp(1.0, 128)) { out[i] = sign | 0x7F80; continue; }
        float f = (float)mag;                   /* exact: 8 significant bits */
        uint32_t u;
        memcpy(&u, &f, sizeof u);
        out[i] = sign | (uint16_t)(u >> 16);
    }
}
