// nvq_kernels.h -- argument blocks and launchers shared between the C-ABI
// layer (api.cu) and the kernels (quantize.cu, gemm.cu).  Internal.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace nvq {

constexpr int kMaxGroups = 256;

// Row groups of a (possibly grouped) input in a padded row space where each
// group starts at a multiple of 128 rows.  tile0[g] = first 128-row tile of
// group g; rows[g] = source rows of the group; src_row0[g] = its first row
// in the unpadded input.
struct QuantGroups {
    int G;
    int32_t tile0[kMaxGroups];
    int64_t rows[kMaxGroups];
    int64_t src_row0[kMaxGroups];
};

struct QuantArgs {
    const uint16_t* x;  // bf16 input
    int64_t ld;         // elements
    int64_t K;          // columns of x (contraction of the rowwise operand)
    QuantGroups groups;
    // rowwise output
    uint8_t* row_data;
    uint8_t* row_scale;
    const float* row_amax;     // per group (NVFP4)
    int64_t row_rows_store;    // rows of row_data written (rows >= it skipped)
    int64_t row_scale_ctiles;  // 128x4 scale tiles per 128 rows
    // columnwise output ([K][col_cols_store])
    uint8_t* col_data;
    uint8_t* col_scale;
    const float* col_amax;     // per group (NVFP4)
    int64_t col_cols_store;
    int64_t col_scale_ctiles;
    int64_t col_scale_rows_pad;  // ceil128(K)
    // amax pass outputs (per group), any may be NULL
    float* amax_out[2];
    float* amax_rht_out;
    // rowwise-dequantized source: the pass that measures the columnwise
    // source's amax (plain, or Hadamard-domain with RHT) writes it here
    float* dq_amax;
    // RHT and SR
    uint32_t rht_sign_mask;  // bit i set: sign[i] == -1
    uint32_t sr_offset;
    uint32_t sr_round_key[20];  // Philox key schedule: (k0 + r*W0, k1 + r*W1), r = 0..9
    int* status;  // device status word
};

cudaError_t launch_amax(const QuantArgs& a, int64_t row_tiles, cudaStream_t s);
cudaError_t launch_quantize(const QuantArgs& a, int row_fmt, int col_fmt, bool rht, bool sr,
                            int64_t row_tiles, cudaStream_t s);
// Variants with an identity direction (format 3) or the rowwise-dequantized
// columnwise source (dq): quantize_hybrid.cu.
cudaError_t launch_quantize_hybrid(const QuantArgs& a, int row_fmt, int col_fmt, bool rht, bool sr, bool dq,
                                   int64_t row_tiles, cudaStream_t s);
// Per-row amax of the padded row space (row-scaled NVFP4): amax_rows[n_rows].
cudaError_t launch_row_amax(const QuantArgs& a, int64_t n_rows, float* amax_rows, cudaStream_t s);

// ------------------------------------------------------------------ GEMM
// One GEMM problem (or one group of a grouped GEMM) in TN form.
struct GemmGroup {
    int32_t m_tile0;    // first 128-row output tile of this group (prefix over groups)
    int32_t pm_tile0;   // first 256-row pair tile of this group (CTA-pair kernel)
    int32_t m_tiles;    // 128-row tiles of this group
    int32_t a_row0;     // first row of A (padded space)
    int32_t b_row0;     // first row of B
    int32_t a_k0;       // first contraction element of A (multiple of 128)
    int32_t b_k0;       // first contraction element of B (multiple of 128)
    int32_t k_len;      // contraction length (multiple of 128; 0 allowed)
    int32_t rows_valid; // output rows written (<= m_tiles * 128)
    int32_t amax_idx;   // index into the amax arrays (NVFP4 alpha)
    int64_t c_off;      // element offset of the group's C[0][0]
    int32_t c_row0;     // C row of the group's first row (c_off / ldc)
};

struct GemmArgs {
    int fmt;               // 1 NVFP4, 2 MXFP8
    int block_n;           // output tile width BN (128 or 256)
    int use_pair;          // run the CTA-pair kernel (block_n == 256)
    int total_pm_tiles;    // sum over groups of ceil(m_tiles / 2)
    int any_k;             // some group has a nonzero contraction (tensor maps valid)
    int n_tiles;           // output column tiles (N / BN)
    int total_m_tiles;     // sum of m_tiles
    int G;
    const uint8_t* a_scale;
    const uint8_t* b_scale;
    int64_t a_scale_ctiles;  // 128x4 scale tiles per 128 rows of A
    int64_t b_scale_ctiles;
    const float* a_amax;
    const float* b_amax;
    int a_row_scaled;  // A is row-scaled NVFP4: a_amax holds one amax per (padded) row of A
    const uint16_t* bias;  // bf16 [N] or NULL
    void* C;
    int64_t ldc;
    int c_fp32;
    int c_st32;  // bf16 C, base and row pitch 32-byte aligned: 32-byte stores
    int c_tma;   // bf16 C stored through the C tensor map (CTA-pair kernel)
    int* status;           // device status word
    int debug_drop_first_load;  // test hook: arm stage 0's barrier but issue no copy
    // optional amax of the stored output (single-problem GEMMs): max |C|, and
    // max |T(u)| over 16-row column blocks u of C (T: 16-point Hadamard
    // transform with the sign vector below); zeroed by the caller
    float* c_amax;
    float* c_amax_rht;
    uint32_t rht_sign_mask;  // bit i set: sign[i] == -1
    GemmGroup groups[kMaxGroups];
};

// Output tile width for an output of n_out columns (a multiple of 128).
int gemm_block_n(int64_t n_out);

// A_map / B_map: CUtensorMap (boxes 128 x 128 bytes for A, block_n x 128 for B).
// Persistent launch: min(tiles, num_sms) CTAs.
cudaError_t launch_gemm(const void* a_map, const void* b_map, const GemmArgs& g, int num_sms, cudaStream_t s);

cudaError_t init_gemm_attributes();

// CTA-pair (cta_group::2) kernel for block_n == 256: 2 * min(tiles, num_sms / 2) CTAs.
cudaError_t launch_gemm_pair(const void* a_map, const void* b_map, const void* c_map, const GemmArgs& g, int num_sms,
                             cudaStream_t s);
cudaError_t init_gemm_pair_attributes(bool* usable);  // usable: the pair kernel may run

}  // namespace nvq
