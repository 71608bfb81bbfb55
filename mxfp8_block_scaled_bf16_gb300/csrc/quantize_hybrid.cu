// quantize_hybrid.cu -- the fused quantizer's variants with an identity
// direction (the bf16 value passed through, IdentityQuantizer) or with the
// columnwise direction built from the dequantized rowwise value
// (columnwise_source = "rowwise_dequantized"), for "Hybrid quantization"
// (TransformerEngine PR #2817, "Enable columnwise_source and hybrid recipes").
// The kernels are in quantize_kernel.cuh; this unit compiles beside
// quantize.cu.
#include "quantize_kernel.cuh"

namespace nvq {

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
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace nvq
