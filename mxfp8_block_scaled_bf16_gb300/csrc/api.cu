// api.cu -- the extern "C" surface of libnvq (declared in include/nvq.h):
// argument validation on the host, TMA tensor-map encoding, group tables and
// kernel dispatch.  No call allocates device memory or synchronizes a stream
// (except nvq_get_device_status, which exists to do that).
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/nvq.h"
#include "nvq_kernels.h"

namespace nvq {

// Device status word; every kernel gets its address.
__device__ int g_status_word = 0;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInit {
    std::once_flag once;
    int* status = nullptr;
    int num_sms = 0;
    bool pair_ok = false;  // the CTA-pair kernel's register allocation is the one it was written for
    cudaError_t err = cudaSuccess;
};

// The CTA-pair kernel runs the GEMMs whose output width is a multiple of 256
// unless NVQ_GEMM_PAIR=0 (the single-CTA kernel then takes them too).
bool pair_gemm_enabled()
{
    static const bool on = [] {
        const char* e = std::getenv("NVQ_GEMM_PAIR");
        return !(e && e[0] == '0');
    }();
    return on;
}
DeviceInit g_dev[kMaxDevices];

// Per-device one-time setup: the status word's address and the GEMM
// kernels' shared-memory limit.
cudaError_t device_setup(int** status, int* num_sms = nullptr)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    DeviceInit& d = g_dev[dev];
    std::call_once(d.once, [&d, dev]() {
        d.err = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), g_status_word);
        if (d.err == cudaSuccess) d.err = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (d.err == cudaSuccess) d.err = init_gemm_attributes();
        if (d.err == cudaSuccess) d.err = init_gemm_pair_attributes(&d.pair_ok);
    });
    *status = d.status;
    if (num_sms) *num_sms = d.num_sms;
    return d.err;
}

// The current device's pair-kernel check (device_setup must have succeeded).
bool device_pair_ok()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    return g_dev[dev].pair_ok;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, []() {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D uint8 tensor map over [rows][row_bytes] with a box_rows x 128-byte box
// and the 128-byte swizzle the MMA descriptors expect.
nvq_status make_operand_map(CUtensorMap* map, const void* data, int64_t rows, int64_t row_bytes, uint32_t box_rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return NVQ_ERR_CUDA;
    cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {128, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(data), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? NVQ_OK : NVQ_ERR_CUDA;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }
// block of the format's scales; the identity (bf16) direction pads its
// columnwise storage to 16 like NVFP4 and has no scales
inline int block_of(nvq_format f) { return f == NVQ_FMT_MXFP8 ? 32 : 16; }
inline bool valid_fmt(nvq_format f) { return f == NVQ_FMT_NVFP4 || f == NVQ_FMT_MXFP8; }
inline bool valid_qfmt(nvq_format f) { return valid_fmt(f) || f == NVQ_FMT_IDENTITY || f == NVQ_FMT_NVFP4_ROWSCALED; }
inline bool is_nvfp4(nvq_format f) { return f == NVQ_FMT_NVFP4 || f == NVQ_FMT_NVFP4_ROWSCALED; }

int64_t data_bytes(nvq_format f, int64_t rows, int64_t cols)
{
    return is_nvfp4(f) ? rows * (cols / 2) : f == NVQ_FMT_IDENTITY ? rows * cols * 2 : rows * cols;
}

int64_t scale_ctiles(nvq_format f, int64_t cols) { return ceil_div(cols / block_of(f), 4); }

nvq_status check_qtensor(const nvq_qtensor* t, nvq_format fmt, int64_t rows, int64_t cols)
{
    if (!t || !t->data || (!t->scale && fmt != NVQ_FMT_IDENTITY)) return NVQ_ERR_NULL;
    if (t->fmt != fmt) return NVQ_ERR_UNSUPPORTED;
    if (is_nvfp4(fmt) && !t->amax) return NVQ_ERR_NULL;
    if (t->rows != rows || t->cols != cols) return NVQ_ERR_SHAPE;
    if (!aligned16(t->data) || (fmt != NVQ_FMT_IDENTITY && !aligned16(t->scale)) ||
        (is_nvfp4(fmt) && (reinterpret_cast<uintptr_t>(t->amax) & 3)))
        return NVQ_ERR_ALIGN;
    return NVQ_OK;
}

nvq_status cuda_status(cudaError_t e) { return e == cudaSuccess ? NVQ_OK : NVQ_ERR_CUDA; }

uint32_t sign_mask(const nvq_rht* rht, bool* ok)
{
    uint32_t m = 0;
    *ok = true;
    for (int i = 0; i < 16; ++i) {
        if (rht->sign[i] == -1) m |= 1u << i;
        else if (rht->sign[i] != 1) *ok = false;
    }
    return m;
}

// Shared body of every quantize entry point.  group_rows == NULL: one tensor
// of M rows (outputs unpadded: row rows = M, col cols = colwise_cols(M)).
nvq_status quantize_impl(const void* x, int64_t M, int64_t K, int64_t ld, const int64_t* group_rows, int G,
                         nvq_format row_fmt, nvq_format col_fmt, const nvq_rht* rht_col, const nvq_sr* sr,
                         nvq_qtensor* row, nvq_qtensor* col, cudaStream_t stream, bool amax_given = false,
                         int col_source = NVQ_COL_SOURCE_ORIGINAL, bool col_2d = false)
{
    if (row_fmt != NVQ_FMT_NONE && !valid_qfmt(row_fmt)) return NVQ_ERR_UNSUPPORTED;
    if (col_fmt != NVQ_FMT_NONE && !valid_qfmt(col_fmt)) return NVQ_ERR_UNSUPPORTED;
    const bool dq = col_source == NVQ_COL_SOURCE_ROWWISE_DEQUANTIZED;
    if (col_source != NVQ_COL_SOURCE_ORIGINAL && !dq) return NVQ_ERR_UNSUPPORTED;
    // the rowwise-dequantized source needs a quantized rowwise direction
    if (dq && (!valid_fmt(row_fmt) || col_fmt == NVQ_FMT_NONE)) return NVQ_ERR_UNSUPPORTED;
    // row-scaled NVFP4 is a rowwise format, with an MXFP8 columnwise direction or none
    if (col_fmt == NVQ_FMT_NVFP4_ROWSCALED) return NVQ_ERR_UNSUPPORTED;
    const bool row_scaled = row_fmt == NVQ_FMT_NVFP4_ROWSCALED;
    if (row_scaled && (dq || (col_fmt != NVQ_FMT_NONE && col_fmt != NVQ_FMT_MXFP8))) return NVQ_ERR_UNSUPPORTED;
    // 16 x 16 (2D) scaling of an NVFP4 columnwise direction, round to nearest
    // (the weights' recipe: no Hadamard transform, no stochastic rounding)
    if (col_2d && (col_fmt != NVQ_FMT_NVFP4 || rht_col || sr || dq || row_scaled || row_fmt == NVQ_FMT_IDENTITY))
        return NVQ_ERR_UNSUPPORTED;
    const bool hybrid_kernel =
        dq || row_scaled || col_2d || row_fmt == NVQ_FMT_IDENTITY || col_fmt == NVQ_FMT_IDENTITY;
    if (hybrid_kernel && !row_scaled && group_rows) return NVQ_ERR_UNSUPPORTED;
    if (K < 0 || ld < K || (ld % 8) != 0) return NVQ_ERR_SHAPE;
    if (!aligned16(x)) return NVQ_ERR_ALIGN;
    if ((row_fmt != NVQ_FMT_NONE && K % block_of(row_fmt)) || K % 16) return NVQ_ERR_SHAPE;
    if (K > INT32_MAX / 2) return NVQ_ERR_SHAPE;

    QuantArgs a;
    std::memset(&a, 0, sizeof a);
    a.x = static_cast<const uint16_t*>(x);
    a.ld = ld;
    a.K = K;
    int64_t padded = 0;
    if (group_rows) {
        if (G < 1 || G > kMaxGroups) return NVQ_ERR_SHAPE;
        a.groups.G = G;
        int64_t src = 0;
        for (int g = 0; g < G; ++g) {
            if (group_rows[g] < 0) return NVQ_ERR_SHAPE;
            a.groups.tile0[g] = (int32_t)(padded / 128);
            a.groups.rows[g] = group_rows[g];
            a.groups.src_row0[g] = src;
            src += group_rows[g];
            padded += round_up(group_rows[g], 128);
        }
        M = src;
    } else {
        if (M < 0) return NVQ_ERR_SHAPE;
        a.groups.G = 1;
        a.groups.tile0[0] = 0;
        a.groups.rows[0] = M;
        a.groups.src_row0[0] = 0;
        padded = round_up(M, 128);
    }
    if (padded / 128 > INT32_MAX || padded > INT32_MAX) return NVQ_ERR_SHAPE;
    if (!x && padded > 0 && K > 0) return NVQ_ERR_NULL;  // an empty input may have no storage

    const bool do_row = row_fmt != NVQ_FMT_NONE, do_col = col_fmt != NVQ_FMT_NONE;
    const int64_t row_rows = group_rows ? padded : M;
    const int64_t col_cols = group_rows ? padded : (do_col ? round_up(M, block_of(col_fmt)) : 0);
    if (do_row) {
        nvq_status s = check_qtensor(row, row_fmt, row_rows, K);
        if (s != NVQ_OK) return s;
    }
    if (do_col) {
        nvq_status s = check_qtensor(col, col_fmt, K, col_cols);
        if (s != NVQ_OK) return s;
    }
    const bool rht = rht_col != nullptr && col_fmt == NVQ_FMT_NVFP4;
    if (rht) {
        bool ok;
        a.rht_sign_mask = sign_mask(rht_col, &ok);
        if (!ok) return NVQ_ERR_SHAPE;
    }
    const bool any_nv = row_fmt == NVQ_FMT_NVFP4 || col_fmt == NVQ_FMT_NVFP4;
    if (sr && any_nv) {
        const uint64_t s = (uint64_t)sr->seed;
        uint32_t k0 = (uint32_t)s, k1 = (uint32_t)(s >> 32);
        for (int r = 0; r < 10; ++r) {  // Philox4x32-10 key schedule (Weyl increments)
            a.sr_round_key[2 * r] = k0;
            a.sr_round_key[2 * r + 1] = k1;
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        a.sr_offset = sr->offset;
    }
    if (!do_row && !do_col) return NVQ_OK;

    int* status = nullptr;
    if (cudaError_t e = device_setup(&status); e != cudaSuccess) return NVQ_ERR_CUDA;
    a.status = status;
    if (do_row) {
        a.row_data = static_cast<uint8_t*>(row->data);
        a.row_scale = static_cast<uint8_t*>(row->scale);
        a.row_amax = row->amax;
        a.row_rows_store = row_rows;
        a.row_scale_ctiles = scale_ctiles(row_fmt, K);
    }
    if (do_col) {
        a.col_data = static_cast<uint8_t*>(col->data);
        a.col_scale = static_cast<uint8_t*>(col->scale);
        a.col_amax = col->amax;
        a.col_cols_store = col_cols;
        a.col_scale_ctiles = scale_ctiles(col_fmt, col_cols);
        a.col_scale_rows_pad = round_up(K, 128);
    }
    const int64_t row_tiles = padded / 128;
    const int nG = a.groups.G;
    if (K == 0 || row_tiles == 0) {
        // nothing to read: zero the outputs that exist (scales / amax)
        cudaError_t e = cudaSuccess;
        if (do_row && row_fmt == NVQ_FMT_NVFP4) e = cudaMemsetAsync(row->amax, 0, sizeof(float) * nG, stream);
        if (e == cudaSuccess && do_row && row_scaled && row_rows > 0)
            e = cudaMemsetAsync(row->amax, 0, sizeof(float) * row_rows, stream);
        if (e == cudaSuccess && do_col && col_fmt == NVQ_FMT_NVFP4)
            e = cudaMemsetAsync(col->amax, 0, sizeof(float) * nG, stream);
        if (e == cudaSuccess && do_col && K > 0) {
            size_t db = (size_t)data_bytes(col_fmt, K, col_cols);
            if (db) e = cudaMemsetAsync(col->data, 0, db, stream);
            size_t sb = col_fmt == NVQ_FMT_IDENTITY ? 0 : (size_t)(round_up(K, 128) * round_up(col_cols / block_of(col_fmt), 4));
            if (e == cudaSuccess && sb) e = cudaMemsetAsync(col->scale, 0, sb, stream);
        }
        return cuda_status(e);
    }
    if (any_nv && !amax_given) {
        // amax pass: plain amax for NVFP4 rowwise (and NVFP4 columnwise without
        // RHT), Hadamard-domain amax for NVFP4 columnwise with RHT; a
        // rowwise-dequantized columnwise direction measures its own below
        float* plain_row = row_fmt == NVQ_FMT_NVFP4 ? row->amax : nullptr;
        float* plain_col = (col_fmt == NVQ_FMT_NVFP4 && !rht && !dq) ? col->amax : nullptr;
        float* rht_out = (col_fmt == NVQ_FMT_NVFP4 && rht && !dq) ? col->amax : nullptr;
        cudaError_t e = cudaSuccess;
        if (plain_row) e = cudaMemsetAsync(plain_row, 0, sizeof(float) * nG, stream);
        if (e == cudaSuccess && plain_col) e = cudaMemsetAsync(plain_col, 0, sizeof(float) * nG, stream);
        if (e == cudaSuccess && rht_out) e = cudaMemsetAsync(rht_out, 0, sizeof(float) * nG, stream);
        if (e != cudaSuccess) return NVQ_ERR_CUDA;
        a.amax_out[0] = plain_row ? plain_row : plain_col;
        a.amax_out[1] = plain_row ? plain_col : nullptr;
        a.amax_rht_out = rht_out;
        if ((plain_row || plain_col || rht_out) && launch_amax(a, row_tiles, stream) != cudaSuccess)
            return NVQ_ERR_CUDA;
        a.amax_out[0] = a.amax_out[1] = a.amax_rht_out = nullptr;
    }
    if (!hybrid_kernel)
        return cuda_status(launch_quantize(a, (int)row_fmt, (int)col_fmt, rht, sr != nullptr, row_tiles, stream));
    if (row_scaled && !amax_given && launch_row_amax(a, row_rows, row->amax, stream) != cudaSuccess)
        return NVQ_ERR_CUDA;
    if (dq && col_fmt == NVQ_FMT_NVFP4) {
        // The columnwise scale needs the amax of the dequantized values before
        // any block is quantized: a first pass writes the rowwise operand and
        // that amax, a second recomputes the dequantized values (the same
        // rowwise arithmetic) and quantizes them columnwise.
        if (cudaMemsetAsync(col->amax, 0, sizeof(float), stream) != cudaSuccess) return NVQ_ERR_CUDA;
        QuantArgs a1 = a;
        a1.col_data = nullptr;
        a1.dq_amax = col->amax;
        if (launch_quantize_hybrid(a1, (int)row_fmt, (int)col_fmt, rht, sr != nullptr, true, row_tiles, stream) !=
            cudaSuccess)
            return NVQ_ERR_CUDA;
        a.row_data = nullptr;
    }
    const int col_code = col_2d ? 5 : (int)col_fmt;  // 5: the kernel's tile-scaled NVFP4 columnwise format
    return cuda_status(launch_quantize_hybrid(a, (int)row_fmt, col_code, rht, sr != nullptr, dq, row_tiles, stream));
}

// Test hook for the bounded waits: with NVQ_DEBUG_DROP_TMA=1 in the
// environment (read once per process), the first GEMM the process launches
// arms its first pipeline stage but issues no copy into it, so every wait on
// that stage runs out, the kernel records NVQ_ERR_TIMEOUT and returns (the
// CTA-pair kernel stops both CTAs of a pair); later launches are normal.
// Nothing faults or hangs.
bool debug_drop_this_launch()
{
    static const bool on = [] {
        const char* e = std::getenv("NVQ_DEBUG_DROP_TMA");
        return e && e[0] == '1';
    }();
    static std::atomic<bool> used{false};
    return on && !used.exchange(true);
}

// Operand formats a GEMM takes: both NVFP4, both MXFP8, or a row-scaled NVFP4
// A with an NVFP4 B (the per-row outer scale of A goes into the epilogue's
// alpha).
bool gemm_formats_ok(const nvq_qtensor* A, const nvq_qtensor* B)
{
    if (A->fmt == NVQ_FMT_NVFP4_ROWSCALED) return B->fmt == NVQ_FMT_NVFP4;
    return A->fmt == B->fmt && valid_fmt(A->fmt);
}

nvq_status gemm_prepare(const nvq_qtensor* A, const nvq_qtensor* B, int64_t n_out, CUtensorMap* am, CUtensorMap* bm,
                        GemmArgs* g)
{
    if (!A || !B || !A->data || !B->data || !A->scale || !B->scale) return NVQ_ERR_NULL;
    if (!gemm_formats_ok(A, B)) return NVQ_ERR_UNSUPPORTED;
    const nvq_format f = B->fmt;  // the tensor-core format (a row-scaled A is NVFP4 on the tensor core)
    if (f == NVQ_FMT_NVFP4 && (!A->amax || !B->amax)) return NVQ_ERR_NULL;
    if (A->rows < 0 || B->rows < 0 || A->cols < 0 || A->rows % 128 || B->rows % 128) return NVQ_ERR_SHAPE;
    if (A->cols % 128 || B->cols % 128) return NVQ_ERR_SHAPE;
    if (A->rows > INT32_MAX || B->rows > INT32_MAX || A->cols > INT32_MAX / 2 || B->cols > INT32_MAX / 2)
        return NVQ_ERR_SHAPE;
    if (!aligned16(A->data) || !aligned16(B->data) || !aligned16(A->scale) || !aligned16(B->scale))
        return NVQ_ERR_ALIGN;
    std::memset(g, 0, sizeof *g);
    std::memset(am, 0, sizeof *am);
    std::memset(bm, 0, sizeof *bm);
    g->fmt = (int)f;
    g->a_scale = static_cast<const uint8_t*>(A->scale);
    g->b_scale = static_cast<const uint8_t*>(B->scale);
    g->a_scale_ctiles = scale_ctiles(f, A->cols);
    g->b_scale_ctiles = scale_ctiles(f, B->cols);
    g->a_amax = A->amax;
    g->b_amax = B->amax;
    g->a_row_scaled = A->fmt == NVQ_FMT_NVFP4_ROWSCALED ? 1 : 0;
    if (n_out % 128) return NVQ_ERR_SHAPE;
    g->block_n = gemm_block_n(n_out);
    int* status = nullptr;
    if (device_setup(&status) != cudaSuccess) return NVQ_ERR_CUDA;
    g->use_pair = (g->block_n == 256 && pair_gemm_enabled() && device_pair_ok()) ? 1 : 0;
    g->any_k = (A->rows > 0 && A->cols > 0 && B->rows > 0 && B->cols > 0) ? 1 : 0;
    const int64_t eb = f == NVQ_FMT_NVFP4 ? 2 : 1;  // elements per byte
    // the pair kernel loads 128 rows of B per CTA; the single-CTA one block_n rows
    const uint32_t b_box = g->use_pair ? 128u : (uint32_t)g->block_n;
    nvq_status s = NVQ_OK;
    if (g->any_k) s = make_operand_map(am, A->data, A->rows, A->cols / eb, 128);
    if (s == NVQ_OK && g->any_k) s = make_operand_map(bm, B->data, B->rows, B->cols / eb, b_box);
    return s;
}

// bf16 C viewed as [rows][ncols] with row pitch ldc, stored in boxes of 32
// rows x 64 columns (128 bytes, 128B swizzle) by the CTA-pair epilogue.
nvq_status make_c_map(CUtensorMap* map, void* C, int64_t rows, int64_t ncols, int64_t ldc)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return NVQ_ERR_CUDA;
    cuuint64_t dims[2] = {(cuuint64_t)ncols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(ldc * 2)};
    cuuint32_t box[2] = {64, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, C, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? NVQ_OK : NVQ_ERR_CUDA;
}

nvq_status check_c(const void* C, int64_t ldc, int64_t ncols, int c_fp32)
{
    if (!C) return NVQ_ERR_NULL;
    if (!aligned16(C) || ldc % 8) return NVQ_ERR_ALIGN;
    if (ldc < ncols) return NVQ_ERR_SHAPE;
    (void)c_fp32;
    return NVQ_OK;
}

nvq_status gemm_launch(const CUtensorMap& am, const CUtensorMap& bm, GemmArgs& g, int64_t n_out, cudaStream_t stream)
{
    int* status = nullptr;
    int num_sms = 0;
    if (device_setup(&status, &num_sms) != cudaSuccess) return NVQ_ERR_CUDA;
    g.status = status;
    g.debug_drop_first_load = debug_drop_this_launch() ? 1 : 0;
    // pair tiles: each group's 128-row tiles taken two at a time
    int pm = 0;
    for (int i = 0; i < g.G; ++i) {
        g.groups[i].pm_tile0 = pm;
        pm += (g.groups[i].m_tiles + 1) / 2;
    }
    g.total_pm_tiles = pm;
    // 32-byte epilogue stores need every row start 32-byte aligned
    bool st32 = !g.c_fp32 && (reinterpret_cast<uintptr_t>(g.C) & 31) == 0 && g.ldc % 16 == 0;
    for (int i = 0; i < g.G && st32; ++i) st32 = g.groups[i].c_off % 16 == 0;
    g.c_st32 = st32 ? 1 : 0;
    // C rows written by this call, and the C row of each group's first row
    int64_t rows_end = 0;
    for (int i = 0; i < g.G; ++i) {
        const int64_t r0 = g.ldc > 0 ? g.groups[i].c_off / g.ldc : 0;
        g.groups[i].c_row0 = (int32_t)r0;
        if (g.groups[i].rows_valid > 0 && r0 + g.groups[i].rows_valid > rows_end) rows_end = r0 + g.groups[i].rows_valid;
    }
    CUtensorMap cm;
    std::memset(&cm, 0, sizeof cm);
    g.c_tma = 0;
    if (g.use_pair && !g.c_fp32 && rows_end > 0 && rows_end <= INT32_MAX &&
        make_c_map(&cm, g.C, rows_end, n_out, g.ldc) == NVQ_OK)
        g.c_tma = 1;
    if (g.use_pair) return cuda_status(launch_gemm_pair(&am, &bm, &cm, g, num_sms, stream));
    return cuda_status(launch_gemm(&am, &bm, g, num_sms, stream));
}

// nvq_gemm_tn with the optional output amaxes.
nvq_status gemm_tn_impl(const nvq_qtensor* A, const nvq_qtensor* B, const void* bias, void* C, int64_t ldc,
                        int c_fp32, const nvq_rht* rht, float* c_amax, float* c_amax_rht, cudaStream_t stream)
{
    if (!A || !B) return NVQ_ERR_NULL;
    if (gemm_formats_ok(A, B) && A->cols != B->cols) return NVQ_ERR_SHAPE;
    if ((c_amax && (reinterpret_cast<uintptr_t>(c_amax) & 3)) || (c_amax_rht && (reinterpret_cast<uintptr_t>(c_amax_rht) & 3)))
        return NVQ_ERR_ALIGN;
    uint32_t mask = 0;
    if (c_amax_rht) {
        bool ok;
        mask = sign_mask(rht, &ok);
        if (!ok) return NVQ_ERR_SHAPE;
    }
    CUtensorMap am, bm;
    GemmArgs* g = new (std::nothrow) GemmArgs;
    if (!g) return NVQ_ERR_CUDA;
    nvq_status s = gemm_prepare(A, B, B->rows, &am, &bm, g);
    if (s == NVQ_OK) s = check_c(C, ldc, B->rows, c_fp32);
    if (s == NVQ_OK && bias && !aligned16(bias)) s = NVQ_ERR_ALIGN;
    if (s == NVQ_OK && c_amax && cudaMemsetAsync(c_amax, 0, sizeof(float), stream) != cudaSuccess) s = NVQ_ERR_CUDA;
    if (s == NVQ_OK && c_amax_rht && cudaMemsetAsync(c_amax_rht, 0, sizeof(float), stream) != cudaSuccess)
        s = NVQ_ERR_CUDA;
    if (s == NVQ_OK) {
        g->c_amax = c_amax;
        g->c_amax_rht = c_amax_rht;
        g->rht_sign_mask = mask;
        g->n_tiles = (int)(B->rows / g->block_n);
        g->total_m_tiles = (int)(A->rows / 128);
        g->G = 1;
        g->bias = static_cast<const uint16_t*>(bias);
        g->C = C;
        g->ldc = ldc;
        g->c_fp32 = c_fp32 ? 1 : 0;
        GemmGroup& gr = g->groups[0];
        gr.m_tile0 = 0;
        gr.m_tiles = g->total_m_tiles;
        gr.k_len = (int32_t)A->cols;
        gr.rows_valid = (int32_t)A->rows;
        s = gemm_launch(am, bm, *g, B->rows, stream);
    }
    delete g;
    return s;
}

}  // namespace
}  // namespace nvq

using namespace nvq;

extern "C" {

nvq_status nvq_query_sizes(nvq_format fmt, int64_t rows, int64_t cols, size_t* db, size_t* sb)
{
    if (!db || !sb) return NVQ_ERR_NULL;
    if (!valid_qfmt(fmt)) return NVQ_ERR_UNSUPPORTED;
    if (rows < 0 || cols < 0 || cols % block_of(fmt)) return NVQ_ERR_SHAPE;
    *db = (size_t)data_bytes(fmt, rows, cols);
    *sb = fmt == NVQ_FMT_IDENTITY ? 0 : (size_t)(round_up(rows, 128) * round_up(cols / block_of(fmt), 4));
    return NVQ_OK;
}

int64_t nvq_colwise_cols(nvq_format fmt, int64_t M)
{
    if (!valid_qfmt(fmt) || M < 0) return -1;
    return round_up(M, block_of(fmt));
}

nvq_status nvq_amax(const void* x, int64_t M, int64_t K, int64_t ld, const nvq_rht* rht, float* amax_out,
                    float* amax_rht_out, nvq_stream stream)
{
    if (!x) return NVQ_ERR_NULL;
    if (M < 0 || K < 0 || ld < K || ld % 8 || K % 8) return NVQ_ERR_SHAPE;
    if (!aligned16(x)) return NVQ_ERR_ALIGN;
    if (rht == nullptr) amax_rht_out = nullptr;
    QuantArgs a;
    std::memset(&a, 0, sizeof a);
    a.x = static_cast<const uint16_t*>(x);
    a.ld = ld;
    a.K = K;
    a.groups.G = 1;
    a.groups.rows[0] = M;
    if (rht) {
        bool ok;
        a.rht_sign_mask = sign_mask(rht, &ok);
        if (!ok) return NVQ_ERR_SHAPE;
    }
    int* status = nullptr;
    if (device_setup(&status) != cudaSuccess) return NVQ_ERR_CUDA;
    a.status = status;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (amax_out) e = cudaMemsetAsync(amax_out, 0, sizeof(float), s);
    if (e == cudaSuccess && amax_rht_out) e = cudaMemsetAsync(amax_rht_out, 0, sizeof(float), s);
    if (e != cudaSuccess) return NVQ_ERR_CUDA;
    if (M == 0 || K == 0 || (!amax_out && !amax_rht_out)) return NVQ_OK;
    a.amax_out[0] = amax_out;
    a.amax_rht_out = amax_rht_out;
    return cuda_status(launch_amax(a, ceil_div(M, 128), s));
}

nvq_status nvq_nvfp4_quantize(const void* x, int64_t M, int64_t K, int64_t ld, int dirs, const nvq_rht* rht_col,
                              const nvq_sr* sr, nvq_qtensor* row, nvq_qtensor* col, nvq_stream stream)
{
    if (dirs & ~(NVQ_DIR_ROW | NVQ_DIR_COL)) return NVQ_ERR_UNSUPPORTED;
    return quantize_impl(x, M, K, ld, nullptr, 1, (dirs & NVQ_DIR_ROW) ? NVQ_FMT_NVFP4 : NVQ_FMT_NONE,
                         (dirs & NVQ_DIR_COL) ? NVQ_FMT_NVFP4 : NVQ_FMT_NONE, rht_col, sr, row, col,
                         reinterpret_cast<cudaStream_t>(stream));
}

nvq_status nvq_mxfp8_quantize(const void* x, int64_t M, int64_t K, int64_t ld, int dirs, nvq_qtensor* row,
                              nvq_qtensor* col, nvq_stream stream)
{
    if (dirs & ~(NVQ_DIR_ROW | NVQ_DIR_COL)) return NVQ_ERR_UNSUPPORTED;
    return quantize_impl(x, M, K, ld, nullptr, 1, (dirs & NVQ_DIR_ROW) ? NVQ_FMT_MXFP8 : NVQ_FMT_NONE,
                         (dirs & NVQ_DIR_COL) ? NVQ_FMT_MXFP8 : NVQ_FMT_NONE, nullptr, nullptr, row, col,
                         reinterpret_cast<cudaStream_t>(stream));
}

nvq_status nvq_hybrid_quantize(const void* x, int64_t M, int64_t K, int64_t ld, nvq_format row_fmt,
                               nvq_format col_fmt, int col_source, const nvq_rht* rht_col, const nvq_sr* sr,
                               nvq_qtensor* row, nvq_qtensor* col, nvq_stream stream)
{
    return quantize_impl(x, M, K, ld, nullptr, 1, row_fmt, col_fmt, rht_col, sr, row, col,
                         reinterpret_cast<cudaStream_t>(stream), false, col_source);
}

nvq_status nvq_hybrid_quantize_ex(const void* x, int64_t M, int64_t K, int64_t ld, nvq_format row_fmt,
                                  nvq_format col_fmt, int col_source, const nvq_rht* rht_col, const nvq_sr* sr,
                                  int flags, nvq_qtensor* row, nvq_qtensor* col, nvq_stream stream)
{
    if (flags & ~(NVQ_AMAX_GIVEN | NVQ_COL_2D)) return NVQ_ERR_UNSUPPORTED;
    return quantize_impl(x, M, K, ld, nullptr, 1, row_fmt, col_fmt, rht_col, sr, row, col,
                         reinterpret_cast<cudaStream_t>(stream), (flags & NVQ_AMAX_GIVEN) != 0, col_source,
                         (flags & NVQ_COL_2D) != 0);
}

nvq_status nvq_hybrid_linear_fwd(const void* x, const void* w, const void* bias, int64_t M, int64_t N, int64_t K,
                                 nvq_format fwd_fmt, nvq_format bwd_fmt, const nvq_rht* rht, int flags, void* y,
                                 nvq_qtensor* x_row, nvq_qtensor* w_row, nvq_qtensor* saved_x_col,
                                 nvq_qtensor* saved_w_col, nvq_stream stream)
{
    if (!x || !w || !y || !x_row || !w_row) return NVQ_ERR_NULL;
    if (M % 128 || N % 128 || K % 128 || M <= 0 || N <= 0 || K <= 0) return NVQ_ERR_SHAPE;
    if (!valid_fmt(fwd_fmt) || !valid_fmt(bwd_fmt)) return NVQ_ERR_UNSUPPORTED;
    if (flags & ~NVQ_W_COL_2D) return NVQ_ERR_UNSUPPORTED;
    const bool nv_bwd = bwd_fmt == NVQ_FMT_NVFP4;
    if ((flags & NVQ_W_COL_2D) && !nv_bwd) return NVQ_ERR_UNSUPPORTED;
    const bool xc = saved_x_col && saved_x_col->data, wc = saved_w_col && saved_w_col->data;
    nvq_status s = nvq_hybrid_quantize_ex(x, M, K, K, fwd_fmt, xc ? bwd_fmt : NVQ_FMT_NONE, NVQ_COL_SOURCE_ORIGINAL,
                                          nv_bwd ? rht : nullptr, nullptr, 0, x_row, xc ? saved_x_col : nullptr, stream);
    if (s != NVQ_OK) return s;
    s = nvq_hybrid_quantize_ex(w, N, K, K, fwd_fmt, wc ? bwd_fmt : NVQ_FMT_NONE, NVQ_COL_SOURCE_ORIGINAL, nullptr,
                               nullptr, (wc && (flags & NVQ_W_COL_2D)) ? NVQ_COL_2D : 0, w_row,
                               wc ? saved_w_col : nullptr, stream);
    if (s != NVQ_OK) return s;
    return nvq_gemm_tn(x_row, w_row, bias, y, N, 0, stream);
}

nvq_status nvq_hybrid_linear_bwd_quantize(const void* dy, int64_t M, int64_t N, nvq_format bwd_fmt,
                                          const nvq_rht* rht, const nvq_sr* sr, nvq_qtensor* dy_row,
                                          nvq_qtensor* dy_col, nvq_stream stream)
{
    if (M % 128 || N % 128) return NVQ_ERR_SHAPE;
    if (!valid_fmt(bwd_fmt)) return NVQ_ERR_UNSUPPORTED;
    const bool nv = bwd_fmt == NVQ_FMT_NVFP4;
    return nvq_hybrid_quantize(dy, M, N, N, bwd_fmt, bwd_fmt, NVQ_COL_SOURCE_ORIGINAL, nv ? rht : nullptr,
                               nv ? sr : nullptr, dy_row, dy_col, stream);
}

nvq_status nvq_linear_dgrad(const nvq_qtensor* dy_row, const nvq_qtensor* saved_w_col, void* dx, nvq_stream stream)
{
    if (!dy_row || !saved_w_col) return NVQ_ERR_NULL;
    return nvq_gemm_tn(dy_row, saved_w_col, nullptr, dx, saved_w_col->rows, 0, stream);
}

nvq_status nvq_linear_wgrad(const nvq_qtensor* dy_col, const nvq_qtensor* saved_x_col, void* dw, nvq_stream stream)
{
    if (!dy_col || !saved_x_col) return NVQ_ERR_NULL;
    return nvq_gemm_tn(dy_col, saved_x_col, nullptr, dw, saved_x_col->rows, 0, stream);
}

nvq_status nvq_gemm_tn(const nvq_qtensor* A, const nvq_qtensor* B, const void* bias, void* C, int64_t ldc,
                       int c_fp32, nvq_stream stream)
{
    return gemm_tn_impl(A, B, bias, C, ldc, c_fp32, nullptr, nullptr, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

nvq_status nvq_gemm_tn_amax(const nvq_qtensor* A, const nvq_qtensor* B, const void* bias, void* C, int64_t ldc,
                            int c_fp32, const nvq_rht* rht, float* c_amax, float* c_amax_rht, nvq_stream stream)
{
    if (c_amax_rht && !rht) return NVQ_ERR_NULL;
    return gemm_tn_impl(A, B, bias, C, ldc, c_fp32, rht, c_amax, c_amax_rht, reinterpret_cast<cudaStream_t>(stream));
}

nvq_status nvq_nvfp4_quantize_ex(const void* x, int64_t M, int64_t K, int64_t ld, int dirs, const nvq_rht* rht_col,
                                 const nvq_sr* sr, int flags, nvq_qtensor* row, nvq_qtensor* col, nvq_stream stream)
{
    if (dirs & ~(NVQ_DIR_ROW | NVQ_DIR_COL)) return NVQ_ERR_UNSUPPORTED;
    if (flags & ~(NVQ_AMAX_GIVEN | NVQ_COL_2D)) return NVQ_ERR_UNSUPPORTED;
    return quantize_impl(x, M, K, ld, nullptr, 1, (dirs & NVQ_DIR_ROW) ? NVQ_FMT_NVFP4 : NVQ_FMT_NONE,
                         (dirs & NVQ_DIR_COL) ? NVQ_FMT_NVFP4 : NVQ_FMT_NONE, rht_col, sr, row, col,
                         reinterpret_cast<cudaStream_t>(stream), (flags & NVQ_AMAX_GIVEN) != 0,
                         NVQ_COL_SOURCE_ORIGINAL, (flags & NVQ_COL_2D) != 0);
}
nvq_status nvq_nvfp4_linear_fwd_ex(const void* x, const void* w, const void* bias, int64_t M, int64_t N, int64_t K,
                                   const nvq_rht* rht, int flags, void* y, float* y_amax, float* y_amax_rht,
                                   nvq_qtensor* x_row, nvq_qtensor* w_row, nvq_qtensor* saved_x_col,
                                   nvq_qtensor* saved_w_col, nvq_stream stream)
{
    if (!x || !w || !y || !x_row || !w_row) return NVQ_ERR_NULL;
    if (M % 128 || N % 128 || K % 128 || M <= 0 || N <= 0 || K <= 0) return NVQ_ERR_SHAPE;
    if (flags & ~NVQ_AMAX_GIVEN) return NVQ_ERR_UNSUPPORTED;
    if (y_amax_rht && !rht) return NVQ_ERR_NULL;
    const bool xc = saved_x_col && saved_x_col->data, wc = saved_w_col && saved_w_col->data;
    nvq_status s = nvq_nvfp4_quantize_ex(x, M, K, K, NVQ_DIR_ROW | (xc ? NVQ_DIR_COL : 0), rht, nullptr, flags, x_row,
                                         xc ? saved_x_col : nullptr, stream);
    if (s != NVQ_OK) return s;
    s = nvq_nvfp4_quantize(w, N, K, K, NVQ_DIR_ROW | (wc ? NVQ_DIR_COL : 0), nullptr, nullptr, w_row,
                           wc ? saved_w_col : nullptr, stream);
    if (s != NVQ_OK) return s;
    return nvq_gemm_tn_amax(x_row, w_row, bias, y, N, 0, rht, y_amax, y_amax_rht, stream);
}

nvq_status nvq_nvfp4_linear_fwd(const void* x, const void* w, const void* bias, int64_t M, int64_t N, int64_t K,
                                const nvq_rht* rht, void* y, nvq_qtensor* x_row, nvq_qtensor* w_row,
                                nvq_qtensor* saved_x_col, nvq_qtensor* saved_w_col, nvq_stream stream)
{
    return nvq_nvfp4_linear_fwd_ex(x, w, bias, M, N, K, rht, 0, y, nullptr, nullptr, x_row, w_row, saved_x_col,
                                   saved_w_col, stream);
}

nvq_status nvq_nvfp4_linear_bwd_quantize_ex(const void* dy, int64_t M, int64_t N, const nvq_rht* rht,
                                            const nvq_sr* sr, int flags, nvq_qtensor* dy_row, nvq_qtensor* dy_col,
                                            nvq_stream stream)
{
    if (M % 128 || N % 128) return NVQ_ERR_SHAPE;
    return nvq_nvfp4_quantize_ex(dy, M, N, N, NVQ_DIR_ROW | NVQ_DIR_COL, rht, sr, flags, dy_row, dy_col, stream);
}

nvq_status nvq_nvfp4_linear_bwd_quantize(const void* dy, int64_t M, int64_t N, const nvq_rht* rht,
                                         const nvq_sr* sr, nvq_qtensor* dy_row, nvq_qtensor* dy_col,
                                         nvq_stream stream)
{
    return nvq_nvfp4_linear_bwd_quantize_ex(dy, M, N, rht, sr, 0, dy_row, dy_col, stream);
}

nvq_status nvq_nvfp4_linear_dgrad_ex(const nvq_qtensor* dy_row, const nvq_qtensor* saved_w_col, const nvq_rht* rht,
                                     void* dx, float* dx_amax, float* dx_amax_rht, nvq_stream stream)
{
    if (!dy_row || !saved_w_col) return NVQ_ERR_NULL;
    if (dy_row->fmt != NVQ_FMT_NVFP4 || saved_w_col->fmt != NVQ_FMT_NVFP4) return NVQ_ERR_UNSUPPORTED;
    return nvq_gemm_tn_amax(dy_row, saved_w_col, nullptr, dx, saved_w_col->rows, 0, rht, dx_amax, dx_amax_rht, stream);
}

nvq_status nvq_nvfp4_linear_dgrad(const nvq_qtensor* dy_row, const nvq_qtensor* saved_w_col, void* dx,
                                  nvq_stream stream)
{
    return nvq_nvfp4_linear_dgrad_ex(dy_row, saved_w_col, nullptr, dx, nullptr, nullptr, stream);
}

nvq_status nvq_nvfp4_linear_wgrad(const nvq_qtensor* dy_col, const nvq_qtensor* saved_x_col, void* dw,
                                  nvq_stream stream)
{
    if (!dy_col || !saved_x_col) return NVQ_ERR_NULL;
    if (dy_col->fmt != NVQ_FMT_NVFP4 || saved_x_col->fmt != NVQ_FMT_NVFP4) return NVQ_ERR_UNSUPPORTED;
    return nvq_gemm_tn(dy_col, saved_x_col, nullptr, dw, saved_x_col->rows, 0, stream);
}

int64_t nvq_grouped_padded_rows(const int64_t* group_rows, int G)
{
    if (!group_rows || G < 0) return -1;
    int64_t p = 0;
    for (int g = 0; g < G; ++g) {
        if (group_rows[g] < 0) return -1;
        p += round_up(group_rows[g], 128);
    }
    return p;
}

nvq_status nvq_grouped_hybrid_quantize(const void* x, int64_t K, int64_t ld, const int64_t* group_rows, int G,
                                       nvq_format row_fmt, nvq_format col_fmt, nvq_qtensor* row, nvq_qtensor* col,
                                       const nvq_rht* rht_col, const nvq_sr* sr, nvq_stream stream)
{
    if (!group_rows) return NVQ_ERR_NULL;
    return quantize_impl(x, 0, K, ld, group_rows, G, row_fmt, col_fmt, rht_col, sr, row, col,
                         reinterpret_cast<cudaStream_t>(stream));
}

nvq_status nvq_grouped_gemm_rows(const nvq_qtensor* A, const nvq_qtensor* B, const int64_t* group_rows, int G,
                                 int64_t n_per_group, int b_col_groups, void* C, int64_t ldc, nvq_stream stream)
{
    if (!group_rows) return NVQ_ERR_NULL;
    if (G < 1 || G > kMaxGroups) return NVQ_ERR_SHAPE;
    CUtensorMap am, bm;
    GemmArgs* g = new (std::nothrow) GemmArgs;
    if (!g) return NVQ_ERR_CUDA;
    if (!A || !B) {
        delete g;
        return NVQ_ERR_NULL;
    }
    const int64_t n_out_guess = b_col_groups ? B->rows : n_per_group;
    nvq_status s = (b_col_groups && A->fmt == NVQ_FMT_NVFP4_ROWSCALED) ? NVQ_ERR_UNSUPPORTED
                                                                      : gemm_prepare(A, B, n_out_guess, &am, &bm, g);
    int64_t n_out = 0, klen = 0;
    if (s == NVQ_OK) {
        if (n_per_group <= 0 || n_per_group % 128) s = NVQ_ERR_SHAPE;
        else if (b_col_groups == 0) {  // B = [G * n][K]
            n_out = n_per_group;
            klen = A->cols;
            if (B->rows != (int64_t)G * n_per_group || B->cols != A->cols) s = NVQ_ERR_SHAPE;
        } else {  // B = [n][G * cpg], contraction slice per group
            n_out = B->rows;
            klen = n_per_group;
            if (B->cols != (int64_t)G * n_per_group || A->cols != n_per_group) s = NVQ_ERR_SHAPE;
        }
    }
    if (s == NVQ_OK && nvq_grouped_padded_rows(group_rows, G) != A->rows) s = NVQ_ERR_SHAPE;
    if (s == NVQ_OK) s = check_c(C, ldc, n_out, 0);
    if (s == NVQ_OK) {
        g->n_tiles = (int)(n_out / g->block_n);
        g->G = G;
        g->C = C;
        g->ldc = ldc;
        int64_t tiles = 0, prow = 0, orow = 0;
        for (int i = 0; i < G; ++i) {
            GemmGroup& gr = g->groups[i];
            const int64_t mt = round_up(group_rows[i], 128) / 128;
            gr.m_tile0 = (int32_t)tiles;
            gr.m_tiles = (int32_t)mt;
            gr.a_row0 = (int32_t)prow;
            gr.b_row0 = b_col_groups ? 0 : (int32_t)(i * n_per_group);
            gr.a_k0 = 0;
            gr.b_k0 = b_col_groups ? (int32_t)(i * n_per_group) : 0;
            gr.k_len = (int32_t)klen;
            gr.rows_valid = (int32_t)group_rows[i];
            gr.amax_idx = i;
            gr.c_off = orow * ldc;
            tiles += mt;
            prow += mt * 128;
            orow += group_rows[i];
        }
        g->total_m_tiles = (int)tiles;
        s = gemm_launch(am, bm, *g, n_out, reinterpret_cast<cudaStream_t>(stream));
    }
    delete g;
    return s;
}

nvq_status nvq_grouped_gemm_wgrad(const nvq_qtensor* A, const nvq_qtensor* B, const int64_t* group_rows, int G,
                                  void* C, int64_t ldc, nvq_stream stream)
{
    if (!group_rows) return NVQ_ERR_NULL;
    if (G < 1 || G > kMaxGroups) return NVQ_ERR_SHAPE;
    CUtensorMap am, bm;
    GemmArgs* g = new (std::nothrow) GemmArgs;
    if (!g) return NVQ_ERR_CUDA;
    if (!A || !B) {
        delete g;
        return NVQ_ERR_NULL;
    }
    nvq_status s = A->fmt == NVQ_FMT_NVFP4_ROWSCALED ? NVQ_ERR_UNSUPPORTED : gemm_prepare(A, B, B->rows, &am, &bm, g);
    if (s == NVQ_OK && (A->cols != B->cols || nvq_grouped_padded_rows(group_rows, G) != A->cols)) s = NVQ_ERR_SHAPE;
    if (s == NVQ_OK) s = check_c(C, ldc, B->rows, 0);
    if (s == NVQ_OK) {
        g->n_tiles = (int)(B->rows / g->block_n);
        g->G = G;
        g->C = C;
        g->ldc = ldc;
        const int64_t mt = A->rows / 128;
        int64_t pk = 0;
        for (int i = 0; i < G; ++i) {
            GemmGroup& gr = g->groups[i];
            const int64_t kl = round_up(group_rows[i], 128);
            gr.m_tile0 = (int32_t)(i * mt);
            gr.m_tiles = (int32_t)mt;
            gr.a_row0 = 0;
            gr.b_row0 = 0;
            gr.a_k0 = (int32_t)pk;
            gr.b_k0 = (int32_t)pk;
            gr.k_len = (int32_t)kl;
            gr.rows_valid = (int32_t)A->rows;
            gr.amax_idx = i;
            gr.c_off = (int64_t)i * A->rows * ldc;
            pk += kl;
        }
        g->total_m_tiles = (int)(G * mt);
        s = gemm_launch(am, bm, *g, B->rows, reinterpret_cast<cudaStream_t>(stream));
    }
    delete g;
    return s;
}

nvq_status nvq_grouped_linear_fwd(const void* x, const void* w, const int64_t* group_rows, int G, int64_t N,
                                  int64_t K, void* y, nvq_qtensor* x_row, nvq_qtensor* w_row,
                                  nvq_qtensor* saved_x_col, nvq_qtensor* saved_w_col, nvq_stream stream)
{
    return nvq_grouped_linear_fwd_ex(x, w, group_rows, G, N, K, 0, y, x_row, w_row, saved_x_col, saved_w_col, stream);
}

nvq_status nvq_grouped_linear_fwd_ex(const void* x, const void* w, const int64_t* group_rows, int G, int64_t N,
                                     int64_t K, int flags, void* y, nvq_qtensor* x_row, nvq_qtensor* w_row,
                                     nvq_qtensor* saved_x_col, nvq_qtensor* saved_w_col, nvq_stream stream)
{
    if (!group_rows || !x_row || !w_row || !y) return NVQ_ERR_NULL;
    if (G < 1 || G > kMaxGroups || N <= 0 || K <= 0) return NVQ_ERR_SHAPE;
    if (flags & ~NVQ_X_ROW_SCALED) return NVQ_ERR_UNSUPPORTED;
    const bool xc = saved_x_col && saved_x_col->data, wc = saved_w_col && saved_w_col->data;
    const nvq_format xf = (flags & NVQ_X_ROW_SCALED) ? NVQ_FMT_NVFP4_ROWSCALED : NVQ_FMT_NVFP4;
    nvq_status s = nvq_grouped_hybrid_quantize(x, K, K, group_rows, G, xf,
                                               xc ? NVQ_FMT_MXFP8 : NVQ_FMT_NONE, x_row, xc ? saved_x_col : nullptr,
                                               nullptr, nullptr, stream);
    if (s != NVQ_OK) return s;
    int64_t w_rows[kMaxGroups];
    for (int g = 0; g < G; ++g) w_rows[g] = N;
    s = nvq_grouped_hybrid_quantize(w, K, K, w_rows, G, NVQ_FMT_NVFP4, wc ? NVQ_FMT_MXFP8 : NVQ_FMT_NONE, w_row,
                                    wc ? saved_w_col : nullptr, nullptr, nullptr, stream);
    if (s != NVQ_OK) return s;
    return nvq_grouped_gemm_rows(x_row, w_row, group_rows, G, N, 0, y, N, stream);
}

nvq_status nvq_grouped_linear_bwd_quantize(const void* dy, const int64_t* group_rows, int G, int64_t N,
                                           nvq_qtensor* dy_row, nvq_qtensor* dy_col, nvq_stream stream)
{
    if (!dy_row || !dy_col) return NVQ_ERR_NULL;
    return nvq_grouped_hybrid_quantize(dy, N, N, group_rows, G, NVQ_FMT_MXFP8, NVQ_FMT_MXFP8, dy_row, dy_col, nullptr,
                                       nullptr, stream);
}

nvq_status nvq_grouped_linear_dgrad(const nvq_qtensor* dy_row, const nvq_qtensor* saved_w_col,
                                    const int64_t* group_rows, int G, void* dx, nvq_stream stream)
{
    if (!dy_row || !saved_w_col) return NVQ_ERR_NULL;
    // B = W_col [K][G*N]: group g's contraction slice is columns [g*N, (g+1)*N)
    return nvq_grouped_gemm_rows(dy_row, saved_w_col, group_rows, G, dy_row->cols, 1, dx, saved_w_col->rows, stream);
}

nvq_status nvq_grouped_linear_wgrad(const nvq_qtensor* dy_col, const nvq_qtensor* saved_x_col,
                                    const int64_t* group_rows, int G, void* dw, nvq_stream stream)
{
    if (!dy_col || !saved_x_col) return NVQ_ERR_NULL;
    return nvq_grouped_gemm_wgrad(dy_col, saved_x_col, group_rows, G, dw, saved_x_col->rows, stream);
}

const char* nvq_status_string(nvq_status s)
{
    switch (s) {
        case NVQ_OK: return "ok";
        case NVQ_ERR_NULL: return "null pointer";
        case NVQ_ERR_SHAPE: return "invalid shape";
        case NVQ_ERR_ALIGN: return "misaligned pointer or leading dimension";
        case NVQ_ERR_WORKSPACE: return "workspace too small";
        case NVQ_ERR_UNSUPPORTED: return "unsupported option";
        case NVQ_ERR_CUDA: return "CUDA error";
        case NVQ_ERR_TIMEOUT: return "device wait timed out";
        case NVQ_ERR_BOUNDS: return "device bounds check failed";
    }
    return "unknown status";
}

nvq_status nvq_get_device_status(nvq_stream stream, int32_t* code)
{
    if (!code) return NVQ_ERR_NULL;
    int* status = nullptr;
    if (device_setup(&status) != cudaSuccess) return NVQ_ERR_CUDA;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return NVQ_ERR_CUDA;
    int v = 0, zero = 0;
    if (cudaMemcpy(&v, status, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return NVQ_ERR_CUDA;
    if (cudaMemcpy(status, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return NVQ_ERR_CUDA;
    *code = v;
    return NVQ_OK;
}

int nvq_gemm_pair_available(void)
{
    int* status = nullptr;
    if (device_setup(&status) != cudaSuccess) return -1;
    return (pair_gemm_enabled() && device_pair_ok()) ? 1 : 0;
}

const char* nvq_version(void) { return "nvq 0.2 (sm_103a)"; }

}  // extern "C"
