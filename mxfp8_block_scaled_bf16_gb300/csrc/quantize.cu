// quantize.cu -- the amax pass and the fused quantizer's variants whose
// columnwise direction reads the original tensor (NVFP4 / MXFP8 in either
// direction), for "Add an NVFP4 quantization converter" (torchtitan PR #3914)
// and "Hybrid quantization" (TransformerEngine PR #2817).  The kernels are in
// quantize_kernel.cuh.
#include "quantize_kernel.cuh"

namespace nvq {

// ------------------------------------------------------------------ amax pass
__global__ void __launch_bounds__(kThreads, 2) amax_kernel(QuantArgs a)
{
    const int64_t tile_row = blockIdx.y;
    const int g = find_group(a.groups, tile_row);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t prow0 = tile_row * kTileRows + (warp & 3) * 32 + (lane >> 4) * 16;
    const int64_t k0 = (int64_t)blockIdx.x * kTileCols + (warp >> 2) * 128 + (lane & 15) * 8;

    ThreadTile t;
    load_tile(a, g, prow0, k0, t);
    float m_plain, m_rht;
    tile_amax(t, a.amax_rht_out != nullptr, a.rht_sign_mask, m_plain, m_rht);
    cta_amax_publish(m_plain, m_rht, a.amax_out[0] ? a.amax_out[0] + g : nullptr,
                     a.amax_out[1] ? a.amax_out[1] + g : nullptr, a.amax_rht_out ? a.amax_rht_out + g : nullptr);
}

// ------------------------------------------------------------------ launchers
cudaError_t launch_amax(const QuantArgs& a, int64_t row_tiles, cudaStream_t s)
{
    dim3 grid((unsigned)((a.K + kTileCols - 1) / kTileCols), (unsigned)row_tiles);
    amax_kernel<<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

template <int R, int C>
static cudaError_t launch_q3(const QuantArgs& a, dim3 grid, cudaStream_t s, bool rht, bool sr)
{
    if (rht && sr) launch_quantize_variant<R, C, true, true, false>(a, grid, s);
    else if (rht) launch_quantize_variant<R, C, true, false, false>(a, grid, s);
    else if (sr) launch_quantize_variant<R, C, false, true, false>(a, grid, s);
    else launch_quantize_variant<R, C, false, false, false>(a, grid, s);
    return cudaGetLastError();
}

cudaError_t launch_quantize(const QuantArgs& a, int row_fmt, int col_fmt, bool rht, bool sr,
                            int64_t row_tiles, cudaStream_t s)
{
    const dim3 grid = quantize_grid(a, row_tiles);
    // RHT only reaches an NVFP4 columnwise direction; SR only NVFP4 directions.
    const bool nv = row_fmt == 1 || col_fmt == 1;
    rht = rht && col_fmt == 1;
    sr = sr && nv;
    switch (row_fmt * 3 + col_fmt) {
        case 1: return launch_q3<0, 1>(a, grid, s, rht, sr);
        case 2: return launch_q3<0, 2>(a, grid, s, false, false);
        case 3: return launch_q3<1, 0>(a, grid, s, false, sr);
        case 4: return launch_q3<1, 1>(a, grid, s, rht, sr);
        case 5: return launch_q3<1, 2>(a, grid, s, false, sr);
        case 6: return launch_q3<2, 0>(a, grid, s, false, false);
        case 7: return launch_q3<2, 1>(a, grid, s, rht, sr);
        case 8: return launch_q3<2, 2>(a, grid, s, false, false);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace nvq
