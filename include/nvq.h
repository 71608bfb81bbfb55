/*
 * nvq.h -- C ABI of libnvq: block-scaled NVFP4 / MXFP8 quantization and
 * block-scaled GEMMs of a training linear layer, for GB300 (sm_103a).
 *
 * What the calls compute follows two pages:
 *   [TT] "Add an NVFP4 quantization converter" (torchtitan PR #3914):
 *        NVFP4Linear -- E2M1 codes with an E4M3 scale per 1x16 block and an
 *        FP32 per-tensor scale ("outer scale rowwise, inner scale 1x16",
 *        review thread on "rowwise"); a 16-point random Hadamard transform
 *        whose sign vector both wgrad operands share, and stochastic rounding
 *        keyed by a Philox seed (_sr_seed, _rht_sign_vector, "What changed");
 *        every local GEMM dimension a multiple of 128 (review of
 *        parallelize()); quantized activations saved for backward
 *        (Table 1 takeaway).
 *   [TE] "Hybrid quantization" (TransformerEngine PR #2817): rowwise and
 *        columnwise directions quantized to different formats from the
 *        original tensor (Description, columnwise_source="original"); usage
 *        flags skip unneeded directions (review of quantize()); MXFP8 with
 *        32-element blocks and E8M0 scales, ceil(M/32) columnwise scales
 *        (mxfp8_tensor_storage review); grouped split-quantize and grouped
 *        GEMM for MoE experts (Flowchart, _hybrid_split_quantize).
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Every GEMM is "TN": C[r][c] = alpha * sum_k A[r][k] * B[c][k] (+ bias[c]),
 *    both operands stored K-major (the contraction index is contiguous).
 *    A rowwise quantization of x[M][K] is the K-major operand for y = x W^T;
 *    a columnwise quantization of x[M][K] is stored transposed, [K][M'], so
 *    it is the K-major operand of a contraction over M (wgrad).
 *  - Input tensors are bf16, row-major with a leading dimension `ld` in
 *    elements (ld >= K, ld % 8 == 0, base 16-byte aligned).
 *  - All device pointers are caller-owned.  The library allocates no device
 *    memory, keeps no per-tensor state, never frees caller memory and never
 *    synchronizes the stream: every call enqueues kernels on `stream` and
 *    returns.  Argument checks run on the host before anything is enqueued.
 *  - Errors: a non-NVQ_OK status means nothing was enqueued (NVQ_ERR_CUDA:
 *    a launch failed; later work on the stream may be affected).  Conditions
 *    detected on the device (a bounded wait that ran out, a checked-build
 *    bounds violation) are recorded in a device status word read by
 *    nvq_get_device_status(); no kernel traps or spins without a limit.
 */
#ifndef NVQ_H_
#define NVQ_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define NVQ_API __attribute__((visibility("default")))
#else
#define NVQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* nvq_stream; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
    NVQ_OK = 0,
    NVQ_ERR_NULL = 1,        /* a required pointer is NULL */
    NVQ_ERR_SHAPE = 2,       /* a size is negative, not a multiple the call needs, or mismatched */
    NVQ_ERR_ALIGN = 3,       /* a pointer or leading dimension is not 16-byte aligned */
    NVQ_ERR_WORKSPACE = 4,   /* reserved: no call here takes a workspace */
    NVQ_ERR_UNSUPPORTED = 5, /* a valid option this build does not implement */
    NVQ_ERR_CUDA = 6,        /* a CUDA runtime/driver call failed */
    NVQ_ERR_TIMEOUT = 7,     /* device: a bounded pipeline wait ran out */
    NVQ_ERR_BOUNDS = 8       /* device: a checked-build index check failed */
} nvq_status;

/* NVQ_FMT_IDENTITY: the high-precision value passed through ([TE]
 * IdentityQuantizer): bf16 data, no scales, no amax; a quantize direction
 * only (no GEMM takes it).
 * NVQ_FMT_NVFP4_ROWSCALED: NVFP4 with an FP32 outer scale per row instead of
 * per tensor ([TE] Description, the grouped GEMM recipe's input quantizer
 * NVFP4Quantizer(row_scaled_nvfp4=True)): row r's amax A_r takes the tensor
 * amax's place in every step of the NVFP4 recipe and it decodes as
 * E2M1 * E4M3 * (A_r / 2688).  A rowwise direction only; a GEMM takes it as A
 * with an NVFP4 B (alpha per output row). */
typedef enum {
    NVQ_FMT_NONE = 0,
    NVQ_FMT_NVFP4 = 1,
    NVQ_FMT_MXFP8 = 2,
    NVQ_FMT_IDENTITY = 3,
    NVQ_FMT_NVFP4_ROWSCALED = 4
} nvq_format;

/* Source of the columnwise direction of nvq_hybrid_quantize ([TE]
 * columnwise_source): the original tensor, or the dequantized rowwise value. */
enum { NVQ_COL_SOURCE_ORIGINAL = 0, NVQ_COL_SOURCE_ROWWISE_DEQUANTIZED = 1 };

enum { NVQ_DIR_ROW = 1, NVQ_DIR_COL = 2 };

/* Stochastic-rounding key ([TT] _sr_seed: an int64 drawn per rank).  The 16
 * random bits of the element at linear index L of a direction's stored output
 * are field (L & 7) of Philox4x32-10 with key (lo32(seed), hi32(seed)) and
 * counter (lo32(L >> 3), hi32(L >> 3), direction (0 row, 1 col), offset);
 * field f is bits [16*(f&1), 16*(f&1)+16) of word f >> 1.  A magnitude with
 * neighbours lo <= |v| < hi rounds up iff bits < ceil(2^16 (|v|-lo)/(hi-lo)).
 * Scales are always rounded to nearest. */
typedef struct {
    int64_t seed;
    uint32_t offset;
} nvq_sr;

/* Random Hadamard transform ([TT] _rht_sign_vector): 16 values of +1/-1.
 * Each 16-block u along the contraction dimension becomes
 * T(u) = 1/4 * H16 * (s .* u), H16 the Sylvester Hadamard matrix applied as
 * the fp32 butterfly with spans 1, 2, 4, 8 ((a, b) -> (a + b, a - b)). */
typedef struct {
    int8_t sign[16];
} nvq_rht;

/* One quantized operand, K-major: `rows` rows of `cols` contraction elements.
 *   NVFP4: data = E2M1 codes, rows x cols/2 bytes, two per byte, the even
 *          element in the low nibble; scale = E4M3 per 1x16 block; amax =
 *          device float[n] holding the FP32 tensor amax A (n = 1, or one per
 *          group for grouped calls); decoded value E2M1 * E4M3 * A / 2688.
 *   MXFP8: data = E4M3 codes, rows x cols bytes; scale = E8M0 per 1x32
 *          block; amax unused (may be NULL).
 *   IDENTITY: data = bf16 values, rows x cols x 2 bytes; scale and amax
 *          unused (may be NULL).
 *   NVFP4_ROWSCALED: as NVFP4, with amax = device float[rows], row r's amax
 *          (grouped storage: one per padded row, 0 for pad rows).
 * Scales are stored in the block-scaled GEMM layout: the scale matrix
 * [rows][nb] (nb = cols / block) is padded to [ceil(rows/128)*128]
 * [ceil(nb/4)*4] and cut into 128x4 tiles of 512 bytes; tile
 * (r/128)*ceil(nb/4) + c/4 sits at byte 512*tile, and inside it entry
 * (r, c) at (r%32)*16 + ((r%128)/32)*4 + c%4.  Pads are written as zero.
 * data and scale must be 16-byte aligned (data 128-byte aligned for GEMMs). */
typedef struct {
    nvq_format fmt;
    void* data;
    void* scale;
    float* amax;
    int64_t rows;
    int64_t cols;
} nvq_qtensor;

/* Bytes of data and scale storage for a [rows][cols] operand of `fmt`
 * (cols a multiple of the block: 16 for NVFP4 and IDENTITY, 32 for MXFP8;
 * IDENTITY has no scale storage). */
NVQ_API nvq_status nvq_query_sizes(nvq_format fmt, int64_t rows, int64_t cols, size_t* data_bytes,
                           size_t* scale_bytes);

/* Columns of the columnwise (transposed) operand made from M rows: M rounded
 * up to the block (ceil, [TE] mxfp8 storage review: ceil(M/32) scales; 16
 * for NVFP4 and IDENTITY). */
NVQ_API int64_t nvq_colwise_cols(nvq_format fmt, int64_t M);

/* Amax pass ([TT] FP32 per-tensor scale).  amax_out[0] = max |x| over
 * x[M][K]; if rht != NULL, amax_rht_out[0] = max |T(u)| over all columnwise
 * 16-blocks u (rows beyond M read as zero).  Either output may be NULL.
 * Outputs are overwritten (no prior zeroing needed). */
NVQ_API nvq_status nvq_amax(const void* x, int64_t M, int64_t K, int64_t ld, const nvq_rht* rht,
                    float* amax_out, float* amax_rht_out, nvq_stream stream);

/* NVFP4 quantization of bf16 x[M][K] ([TT]).  dirs = NVQ_DIR_ROW and/or
 * NVQ_DIR_COL.  row: rows = M, cols = K (K % 16 == 0).  col: rows = K,
 * cols = nvq_colwise_cols(NVFP4, M); rows past M are zero.  rht_col applies
 * the Hadamard transform to the columnwise blocks (its amax is then taken
 * over T(x)); sr (NULL = round to nearest) applies to both directions.
 * Runs the amax pass then one fused pass that reads x once for both
 * directions; writes row->amax[0] and col->amax[0].
 * Domain: x finite.  The transform adds up to 16 magnitudes in fp32, so with
 * rht_col every |x| <= FLT_MAX / 16 keeps it finite.  Where the transform of
 * some columnwise block overflows, the call still completes with no device
 * error and writes every output byte: col->amax[0] is +inf and the
 * columnwise codes and scales are unspecified; the rowwise direction does not
 * use the transform and is unaffected. */
NVQ_API nvq_status nvq_nvfp4_quantize(const void* x, int64_t M, int64_t K, int64_t ld, int dirs,
                              const nvq_rht* rht_col, const nvq_sr* sr, nvq_qtensor* row,
                              nvq_qtensor* col, nvq_stream stream);

/* Flags of the _ex entry points. */
enum {
    /* The NVFP4 tensor amax is given instead of measured: row->amax[0] holds
     * max |x| and col->amax[0] holds max |x| (or, with rht_col, the
     * Hadamard-domain max |T(u)| over the columnwise 16-blocks) before the
     * call, as the producer of x wrote them (nvq_gemm_tn_amax); the amax pass
     * is skipped and x is read once.  The codes equal those of the measured
     * call when the given amaxes equal the measured ones. */
    NVQ_AMAX_GIVEN = 1,
    /* The NVFP4 columnwise direction takes one E4M3 scale per 16 x 16 tile of
     * x (rows 16j.., columns 16c..) from the tile's amax instead of one per
     * 1 x 16 block ([TE] timeline: "[Common] Enable NVFP4 2D block scaling in
     * columnwise only"); the scale is stored for each of the tile's sixteen
     * columnwise blocks, so the GEMM reads it as usual.  Round to nearest, no
     * Hadamard transform (the weights' recipe); the rowwise direction keeps
     * 1 x 16 blocks. */
    NVQ_COL_2D = 4
};

/* nvq_nvfp4_quantize with flags (NVQ_AMAX_GIVEN or 0). */
NVQ_API nvq_status nvq_nvfp4_quantize_ex(const void* x, int64_t M, int64_t K, int64_t ld, int dirs,
                                         const nvq_rht* rht_col, const nvq_sr* sr, int flags, nvq_qtensor* row,
                                         nvq_qtensor* col, nvq_stream stream);

/* MXFP8 quantization of bf16 x[M][K] ([TE]): E8M0 scale 2^e per 32-block,
 * e = floor(log2 amax_block) - 8 clamped to [-127, 127], elements
 * E4M3_rn_satfinite(x * 2^-e).  row: [M][K] (K % 32 == 0); col: [K][ceil32(M)]. */
NVQ_API nvq_status nvq_mxfp8_quantize(const void* x, int64_t M, int64_t K, int64_t ld, int dirs,
                              nvq_qtensor* row, nvq_qtensor* col, nvq_stream stream);

/* Hybrid quantization ([TE] HybridQuantizer): rowwise in row_fmt and
 * columnwise in col_fmt, each NVFP4, MXFP8 or IDENTITY.  A direction whose
 * format is NVQ_FMT_NONE is skipped (usage flag).  rht_col / sr apply to
 * NVFP4 directions only.  hybrid(F, F) is bitwise equal to the single-format
 * call.  An IDENTITY direction stores the bf16 values: rowwise a copy
 * [M][K], columnwise the transpose [K][nvq_colwise_cols(IDENTITY, M)].
 *   col_source = NVQ_COL_SOURCE_ORIGINAL: both directions from the original
 *     x, from one read of it.
 *   col_source = NVQ_COL_SOURCE_ROWWISE_DEQUANTIZED ([TE] "Enable
 *     columnwise_source and hybrid recipes": the backward operand is built
 *     from dequantize(rowwise-quantized x), double quantization unless the
 *     columnwise quantizer is the identity): row_fmt must be NVFP4 or MXFP8;
 *     the columnwise direction quantizes (or, IDENTITY, stores) the
 *     dequantized rowwise value x^ = bf16_rn(fp32 (E2M1 * E4M3) * (A / 2688))
 *     (NVFP4, A the rowwise amax) or bf16_rn(E4M3 * 2^e) (MXFP8, exact).  An
 *     NVFP4 columnwise direction then takes its amax over x^ (or T(x^)), which
 *     costs a second pass over x.  Not available for grouped tensors. */
NVQ_API nvq_status nvq_hybrid_quantize(const void* x, int64_t M, int64_t K, int64_t ld,
                               nvq_format row_fmt, nvq_format col_fmt, int col_source,
                               const nvq_rht* rht_col, const nvq_sr* sr, nvq_qtensor* row,
                               nvq_qtensor* col, nvq_stream stream);

/* nvq_hybrid_quantize with flags (NVQ_AMAX_GIVEN, NVQ_COL_2D). */
NVQ_API nvq_status nvq_hybrid_quantize_ex(const void* x, int64_t M, int64_t K, int64_t ld, nvq_format row_fmt,
                                          nvq_format col_fmt, int col_source, const nvq_rht* rht_col,
                                          const nvq_sr* sr, int flags, nvq_qtensor* row, nvq_qtensor* col,
                                          nvq_stream stream);

/* Block-scaled GEMM, TN form: C[r][c] = alpha * sum_k A[r][k] B[c][k] + bias[c].
 * A, B: same format, or a row-scaled NVFP4 A with an NVFP4 B (alpha_r =
 * (A.amax[r]/2688) * (B.amax[0]/2688)); A.cols == B.cols = K; A.rows = Mr and B.rows = Nc
 * multiples of 128 ([TT] every GEMM dim a multiple of 128); K a multiple of
 * 128.  alpha = (A.amax[0]/2688) * (B.amax[0]/2688) for NVFP4, 1 for MXFP8,
 * read on the device.  C: row-major [Mr][ldc], bf16 (c_fp32 = 0) or fp32
 * (c_fp32 = 1), 16-byte aligned, ldc % 8 == 0.  bias: bf16[Nc] or NULL.
 * fp32 tensor-core accumulation; the bf16 output is rounded once. */
NVQ_API nvq_status nvq_gemm_tn(const nvq_qtensor* A, const nvq_qtensor* B, const void* bias, void* C,
                       int64_t ldc, int c_fp32, nvq_stream stream);

/* nvq_gemm_tn that also writes the amaxes of its stored output C (the values
 * after rounding to C's type), for the quantizer of the operation that reads
 * C next, which can then skip its amax pass (NVQ_AMAX_GIVEN; [TT] "What
 * changed": every NVFP4 input needs its FP32 per-tensor scale):
 *   c_amax[0]     = max |C|                                  (NULL: not computed);
 *   c_amax_rht[0] = max |T(u)| over the 16-row column blocks u of C, T the
 *                   Hadamard transform of nvq_rht with the sign vector rht
 *                   (the amax the columnwise NVFP4 quantization of C with
 *                   that sign vector needs; NULL: not computed).
 * Both are overwritten (zeroed on the stream first).  C's rows are a
 * multiple of 128, so every 16-row block is whole. */
NVQ_API nvq_status nvq_gemm_tn_amax(const nvq_qtensor* A, const nvq_qtensor* B, const void* bias, void* C,
                                    int64_t ldc, int c_fp32, const nvq_rht* rht, float* c_amax, float* c_amax_rht,
                                    nvq_stream stream);

/* NVFP4 linear forward ([TT] NVFP4Linear): quantizes x[M][K] rowwise (RTN)
 * into x_row and columnwise with the Hadamard transform into saved_x_col
 * (the wgrad operand, kept for backward); quantizes W[N][K] rowwise into
 * w_row and columnwise into saved_w_col (the dgrad operand); then
 * y[M][N] = x W^T (+ bias), bf16.  saved_* may have data == NULL to skip
 * that direction.  M, N, K multiples of 128. */
NVQ_API nvq_status nvq_nvfp4_linear_fwd(const void* x, const void* w, const void* bias, int64_t M,
                                int64_t N, int64_t K, const nvq_rht* rht, void* y,
                                nvq_qtensor* x_row, nvq_qtensor* w_row, nvq_qtensor* saved_x_col,
                                nvq_qtensor* saved_w_col, nvq_stream stream);

/* nvq_nvfp4_linear_fwd for a layer inside a stack: flags = NVQ_AMAX_GIVEN
 * takes x's amaxes from x_row->amax[0] and saved_x_col->amax[0] (written by
 * the previous layer's GEMM) instead of measuring them; y_amax / y_amax_rht
 * (NULL to skip) receive y's amaxes as nvq_gemm_tn_amax defines them, for the
 * next layer's quantization of y. */
NVQ_API nvq_status nvq_nvfp4_linear_fwd_ex(const void* x, const void* w, const void* bias, int64_t M, int64_t N,
                                           int64_t K, const nvq_rht* rht, int flags, void* y, float* y_amax,
                                           float* y_amax_rht, nvq_qtensor* x_row, nvq_qtensor* w_row,
                                           nvq_qtensor* saved_x_col, nvq_qtensor* saved_w_col, nvq_stream stream);

/* Backward quantization of dy[M][N]: rowwise (for dgrad) and columnwise with
 * the Hadamard transform (for wgrad), both with stochastic rounding. */
NVQ_API nvq_status nvq_nvfp4_linear_bwd_quantize(const void* dy, int64_t M, int64_t N,
                                         const nvq_rht* rht, const nvq_sr* sr,
                                         nvq_qtensor* dy_row, nvq_qtensor* dy_col,
                                         nvq_stream stream);

/* nvq_nvfp4_linear_bwd_quantize with flags (NVQ_AMAX_GIVEN: dy's amaxes were
 * written into dy_row->amax[0] / dy_col->amax[0] by the GEMM that produced dy). */
NVQ_API nvq_status nvq_nvfp4_linear_bwd_quantize_ex(const void* dy, int64_t M, int64_t N, const nvq_rht* rht,
                                                    const nvq_sr* sr, int flags, nvq_qtensor* dy_row,
                                                    nvq_qtensor* dy_col, nvq_stream stream);

/* dgrad: dx[M][K] = dy W = TN(dy_row [M][N], saved_w_col [K][N]), bf16. */
NVQ_API nvq_status nvq_nvfp4_linear_dgrad(const nvq_qtensor* dy_row, const nvq_qtensor* saved_w_col,
                                  void* dx, nvq_stream stream);

/* dgrad that also writes dx's amaxes (nvq_gemm_tn_amax; NULL to skip), for the
 * quantization of dx as the output gradient of the layer below. */
NVQ_API nvq_status nvq_nvfp4_linear_dgrad_ex(const nvq_qtensor* dy_row, const nvq_qtensor* saved_w_col,
                                             const nvq_rht* rht, void* dx, float* dx_amax, float* dx_amax_rht,
                                             nvq_stream stream);

/* wgrad: dW[N][K] = dy^T x = TN(dy_col [N][M], saved_x_col [K][M]), bf16;
 * the Hadamard transforms cancel because both operands share one sign vector. */
NVQ_API nvq_status nvq_nvfp4_linear_wgrad(const nvq_qtensor* dy_col, const nvq_qtensor* saved_x_col,
                                  void* dw, nvq_stream stream);

/* ------------------------------------------------------------------ */
/* Linear layer with per-direction formats ([TE] Description: "MXFP8 fwd */
/* and NVFP4 bwd (or vice versa)").  fwd_fmt, bwd_fmt: NVFP4 or MXFP8.    */
/* The forward GEMM takes x and W rowwise in fwd_fmt; dgrad and wgrad take */
/* the columnwise copies of W and x and both directions of dy in bwd_fmt, */
/* all quantized from the original bf16.  An NVFP4 backward follows the   */
/* NVFP4 recipe ([TT] "What changed"): the Hadamard transform on x's and  */
/* dy's columnwise copies (the wgrad operands) and stochastic rounding on */
/* dy.  M, N, K multiples of 128.                                         */
/* ------------------------------------------------------------------ */
enum {
    /* W's NVFP4 columnwise copy (the dgrad operand) takes 16 x 16 2D
     * scaling (NVQ_COL_2D). */
    NVQ_W_COL_2D = 4
};

/* y[M][N] = x W^T (+ bias) in fwd_fmt; writes x_row, w_row ([M][K], [N][K]
 * in fwd_fmt) and, when their data is non-NULL, saved_x_col ([K][M]) and
 * saved_w_col ([K][N]) in bwd_fmt.  flags: NVQ_W_COL_2D or 0. */
NVQ_API nvq_status nvq_hybrid_linear_fwd(const void* x, const void* w, const void* bias, int64_t M, int64_t N,
                                         int64_t K, nvq_format fwd_fmt, nvq_format bwd_fmt, const nvq_rht* rht,
                                         int flags, void* y, nvq_qtensor* x_row, nvq_qtensor* w_row,
                                         nvq_qtensor* saved_x_col, nvq_qtensor* saved_w_col, nvq_stream stream);

/* dy[M][N] -> dy_row [M][N] and dy_col [N][M] in bwd_fmt (NVFP4: sr on both,
 * rht on dy_col; MXFP8: both ignored). */
NVQ_API nvq_status nvq_hybrid_linear_bwd_quantize(const void* dy, int64_t M, int64_t N, nvq_format bwd_fmt,
                                                  const nvq_rht* rht, const nvq_sr* sr, nvq_qtensor* dy_row,
                                                  nvq_qtensor* dy_col, nvq_stream stream);

/* dgrad dx[M][K] = TN(dy_row, saved_w_col) and wgrad dW[N][K] =
 * TN(dy_col, saved_x_col) in whichever format the operands carry (both
 * NVFP4 or both MXFP8), bf16. */
NVQ_API nvq_status nvq_linear_dgrad(const nvq_qtensor* dy_row, const nvq_qtensor* saved_w_col, void* dx,
                                    nvq_stream stream);
NVQ_API nvq_status nvq_linear_wgrad(const nvq_qtensor* dy_col, const nvq_qtensor* saved_x_col, void* dw,
                                    nvq_stream stream);

/* ------------------------------------------------------------------ */
/* Grouped (MoE) calls ([TE] GroupedLinear, _hybrid_split_quantize).    */
/* Group g holds group_rows[g] >= 0 consecutive rows of the input        */
/* (host array, G <= NVQ_MAX_GROUPS).  Quantized storage is padded per   */
/* group to a multiple of 128 rows: with P_g = sum_{h<g} ceil128(m_h),   */
/* group g's rowwise operand occupies rows [P_g, P_g + ceil128(m_g)) of  */
/* a [P_G][K] operand, and its columnwise operand occupies contraction   */
/* columns [P_g, ...) of a [K][P_G] operand; pad rows are zero.  NVFP4   */
/* directions take a per-group amax (amax[g]).                           */
/* ------------------------------------------------------------------ */
#define NVQ_MAX_GROUPS 256

/* Rows of the padded grouped storage: sum over g of ceil128(group_rows[g]). */
NVQ_API int64_t nvq_grouped_padded_rows(const int64_t* group_rows, int G);

/* Grouped hybrid quantization of bf16 x[sum m_g][K] (row-major, ld):
 * row -> [P_G][K] in row_fmt, col -> [K][P_G] in col_fmt, per-group amax.
 * rht_col and sr act as in nvq_hybrid_quantize (RHT on an NVFP4 columnwise
 * direction, SR on NVFP4 directions; each may be NULL), for a grouped NVFP4
 * backward ([TE] Description: "MXFP8 fwd and NVFP4 bwd (or vice versa)";
 * [TT] "What changed": SR on the gradient, RHT on the wgrad operands):
 *  - the 16-row Hadamard blocks of the columnwise direction never straddle
 *    two groups (each group starts at a multiple of 128 padded rows), and the
 *    transformed amax is taken per group;
 *  - each group's columnwise operand quantizes its rows padded with zero rows
 *    to a multiple of 128, every 16-row block included: with RHT a block of
 *    pad rows transforms to signed zeros, whose codes keep the sign (0x8);
 *  - an element's stochastic-rounding index is its position in the padded
 *    output: P * K + k for rowwise element (padded row P, column k), and
 *    k * P_G + P for columnwise element (k, P). */
NVQ_API nvq_status nvq_grouped_hybrid_quantize(const void* x, int64_t K, int64_t ld,
                                       const int64_t* group_rows, int G, nvq_format row_fmt,
                                       nvq_format col_fmt, nvq_qtensor* row, nvq_qtensor* col,
                                       const nvq_rht* rht_col, const nvq_sr* sr,
                                       nvq_stream stream);

/* Grouped forward / dgrad (groups along the GEMM rows): for each g,
 * C[O_g + r][c] = alpha_g sum_k A[P_g + r][k] B[b_row0_g + c][k] (r < m_g),
 * O_g = sum_{h<g} m_h (unpadded output rows), b_row0_g = g * n_per_group
 * when b_col_groups == 0 (B rows grouped: forward, W_row = [G*N][K]), or
 * B = columns [g * b_cols_per_group, ...) of a [n][G*b_cols_per_group]
 * operand when b_col_groups == 1 (dgrad, W_col = [K][G*N]).  C is bf16
 * [sum m_g][ldc].  alpha_g uses A.amax[g] and B.amax[g] for NVFP4. */
NVQ_API nvq_status nvq_grouped_gemm_rows(const nvq_qtensor* A, const nvq_qtensor* B,
                                 const int64_t* group_rows, int G, int64_t n_per_group,
                                 int b_col_groups, void* C, int64_t ldc, nvq_stream stream);

/* Grouped wgrad (groups along the contraction): for each g,
 * C_g[r][c] = sum over k in [P_g, P_g + ceil128(m_g)) of A[r][k] B[c][k],
 * C_g = C + g * A.rows * ldc (bf16 [G][A.rows][ldc]); m_g = 0 gives zeros. */
NVQ_API nvq_status nvq_grouped_gemm_wgrad(const nvq_qtensor* A, const nvq_qtensor* B,
                                  const int64_t* group_rows, int G, void* C, int64_t ldc,
                                  nvq_stream stream);

/* Grouped linear layer in the recipe of the [TE] hybrid MoE example
 * ("Hybrid quantization", Description): forward in NVFP4 (rowwise x and W),
 * backward in MXFP8 (columnwise x and W quantized from the original bf16,
 * dy rowwise and columnwise).  T = sum m_g tokens, G experts of N outputs
 * and K inputs.  Compositions of the grouped calls above, on `stream`.
 *
 * fwd: x bf16 [T][K], w bf16 [G*N][K] (expert g = rows g*N..), y bf16
 * [T][N].  x_row NVFP4 [P_G][K] and w_row NVFP4 [G*N][K] (G amax each) are
 * written; saved_x_col MXFP8 [K][P_G] and saved_w_col MXFP8 [K][G*N] are
 * written when their data is non-NULL (needed by dgrad / wgrad). */
NVQ_API nvq_status nvq_grouped_linear_fwd(const void* x, const void* w, const int64_t* group_rows, int G,
                                          int64_t N, int64_t K, void* y, nvq_qtensor* x_row,
                                          nvq_qtensor* w_row, nvq_qtensor* saved_x_col,
                                          nvq_qtensor* saved_w_col, nvq_stream stream);

/* Flags of nvq_grouped_linear_fwd_ex. */
enum {
    /* The input's rowwise (forward) direction is row-scaled NVFP4 ([TE]
     * Description: "row-scaled NVFP4 fwd + MXFP8 bwd"): x_row has format
     * NVQ_FMT_NVFP4_ROWSCALED and P_G amaxes, one per padded row. */
    NVQ_X_ROW_SCALED = 2
};

/* nvq_grouped_linear_fwd with flags (NVQ_X_ROW_SCALED or 0). */
NVQ_API nvq_status nvq_grouped_linear_fwd_ex(const void* x, const void* w, const int64_t* group_rows, int G,
                                             int64_t N, int64_t K, int flags, void* y, nvq_qtensor* x_row,
                                             nvq_qtensor* w_row, nvq_qtensor* saved_x_col, nvq_qtensor* saved_w_col,
                                             nvq_stream stream);

/* dy bf16 [T][N] -> MXFP8 dy_row [P_G][N] and dy_col [N][P_G]. */
NVQ_API nvq_status nvq_grouped_linear_bwd_quantize(const void* dy, const int64_t* group_rows, int G, int64_t N,
                                                   nvq_qtensor* dy_row, nvq_qtensor* dy_col, nvq_stream stream);

/* dx bf16 [T][K]: dx_g = dy_g W_g for every group. */
NVQ_API nvq_status nvq_grouped_linear_dgrad(const nvq_qtensor* dy_row, const nvq_qtensor* saved_w_col,
                                            const int64_t* group_rows, int G, void* dx, nvq_stream stream);

/* dW bf16 [G][N][K]: dW_g = dy_g^T x_g (zero for an empty group). */
NVQ_API nvq_status nvq_grouped_linear_wgrad(const nvq_qtensor* dy_col, const nvq_qtensor* saved_x_col,
                                            const int64_t* group_rows, int G, void* dw, nvq_stream stream);

/* ------------------------------------------------------------------ */
/* Status                                                               */
/* ------------------------------------------------------------------ */
NVQ_API const char* nvq_status_string(nvq_status s);

/* Synchronizes `stream`, returns the device status word (NVQ_OK or the
 * first device-side error recorded since the last call) in *code and
 * clears it. */
NVQ_API nvq_status nvq_get_device_status(nvq_stream stream, int32_t* code);

/* Which GEMM kernel takes the GEMMs whose output width is a multiple of 256
 * on the current device: 1 = the CTA-pair kernel (tcgen05 cta_group::2),
 * 0 = the single-CTA kernel (the pair kernel is disabled by NVQ_GEMM_PAIR=0,
 * or its compiled register allocation is not the one its register split
 * needs), -1 = the device could not be set up.  Widths that are not a
 * multiple of 256 always take the single-CTA kernel.  Performs the library's
 * one-time per-device set-up if it has not run yet. */
NVQ_API int nvq_gemm_pair_available(void);

/* Library version string. */
NVQ_API const char* nvq_version(void);

#ifdef __cplusplus
}
#endif
#endif /* NVQ_H_ */
