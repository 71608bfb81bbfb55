// quantize_hybrid.cu -- the fused quantizer's variants with an identity
// direction (the bf16 value passed through, IdentityQuantizer) or with the
// columnwise direction built from the dequantized rowwise value
// (columnwise_source = "rowwise_dequantized"), for "Hybrid quantization"
// (TransformerEngine PR #2817, "Enable columnwise_source and hybrid recipes").
// The kernels are in quantize_kernel.cuh; this unit compiles beside
// quantize.cu.
#include "quantize_kernel.cuh"

namespace nvq {

// ------------------------------------------------------------------ per-row amax
// amax_rows[p] = max_k |x[src(p)][k]| for every row p of the padded row space
// (0 for pad rows): one warp per row, 16-byte loads, 8 rows per CTA.
__global__ void __launch_bounds__(kThreads) row_amax_kernel(QuantArgs a, int64_t n_rows, float* amax_rows)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t p = (int64_t)blockIdx.x * (kThreads / 32) + warp;
    if (p >= n_rows) return;
    const int g = find_group(a.groups, p / kTileRows);
    const int64_t local = p - (int64_t)a.groups.tile0[g] * kTileRows;
    float m = 0.0f;
    if (local < a.groups.rows[g]) {
        const uint16_t* row = a.x + (a.groups.src_row0[g] + local) * a.ld;
        for (int64_t k = (int64_t)lane * 8; k < a.K; k += 256) {
            float v[8];
            unpack8(__ldg(reinterpret_cast<const uint4*>(row + k)), v);
#pragma unroll
            for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(v[j]));
        }
    }
    m = warp_max(m);
    if (lane == 0) amax_rows[p] = m;
}

template <int R, int C, bool DQ>
static cudaError_t launch_h4(const QuantArgs& a, dim3 grid, cudaStream_t s, bool rht, bool sr)
{
    if (rht && sr) launch_quantize_variant<R, C, true, true, DQ>(a, grid, s);
    else if (rht) launch_quantize_variant<R, C, true, false, DQ>(a, grid, s);
    else if (sr) launch_quantize_variant<R, C, false, true, DQ>(a, grid, s);
    else launch_quantize_variant<R, C, false, false, DQ>(a, grid, s);
    return cudaGetLastError();
}

template <int R, int C, bool DQ>
static cudaError_t launch_h2(const QuantArgs& a, dim3 grid, cudaStream_t s, bool sr)
{
    if (sr) launch_quantize_variant<R, C, false, true, DQ>(a, grid, s);
    else launch_quantize_variant<R, C, false, false, DQ>(a, grid, s);
    return cudaGetLastError();
}

template <int R, int C, bool DQ>
static cudaError_t launch_h1(const QuantArgs& a, dim3 grid, cudaStream_t s)
{
    launch_quantize_variant<R, C, false, false, DQ>(a, grid, s);
    return cudaGetLastError();
}

cudaError_t launch_quantize_hybrid(const QuantArgs& a, int row_fmt, int col_fmt, bool rht, bool sr, bool dq,
                                   int64_t row_tiles, cudaStream_t s)
{
    const dim3 grid = quantize_grid(a, row_tiles);
    // RHT only reaches an NVFP4 columnwise direction; SR only NVFP4 directions.
    const bool nv = row_fmt == 1 || col_fmt == 1;
    rht = rht && col_fmt == 1;
    sr = sr && nv;
    if (col_fmt == 5) {
        switch (row_fmt * 4 + 1) {
            case 1: return launch_h1<0, 5, false>(a, grid, s);
            case 5: return launch_h1<1, 5, false>(a, grid, s);
            case 9: return launch_h1<2, 5, false>(a, grid, s);
            default: return cudaErrorInvalidValue;
        }
    }
    if (dq) {
        switch (row_fmt * 4 + col_fmt) {
            case 5: return launch_h4<1, 1, true>(a, grid, s, rht, sr);
            case 6: return launch_h2<1, 2, true>(a, grid, s, sr);
            case 7: return launch_h2<1, 3, true>(a, grid, s, sr);
            case 9: return launch_h4<2, 1, true>(a, grid, s, rht, sr);
            case 10: return launch_h1<2, 2, true>(a, grid, s);
            case 11: return launch_h1<2, 3, true>(a, grid, s);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (row_fmt * 4 + col_fmt) {
        case 3: return launch_h1<0, 3, false>(a, grid, s);
        case 7: return launch_h2<1, 3, false>(a, grid, s, sr);
        case 11: return launch_h1<2, 3, false>(a, grid, s);
        case 12: return launch_h1<3, 0, false>(a, grid, s);
        case 13: return launch_h4<3, 1, false>(a, grid, s, rht, sr);
        case 14: return launch_h1<3, 2, false>(a, grid, s);
        case 15: return launch_h1<3, 3, false>(a, grid, s);
        case 16: return launch_h2<4, 0, false>(a, grid, s, sr);
        case 18: return launch_h2<4, 2, false>(a, grid, s, sr);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_row_amax(const QuantArgs& a, int64_t n_rows, float* amax_rows, cudaStream_t s)
{
    if (n_rows == 0) return cudaSuccess;
    const int64_t per = kThreads / 32;
    row_amax_kernel<<<(unsigned)((n_rows + per - 1) / per), kThreads, 0, s>>>(a, n_rows, amax_rows);
    return cudaGetLastError();
}

}  // namespace nvq
