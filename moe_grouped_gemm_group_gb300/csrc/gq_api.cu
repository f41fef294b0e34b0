// C ABI of the grouped FP8 quantizer and grouped GEMMs: host-side argument
// validation, descriptor checks and kernel launches.  No device memory is
// allocated here; nothing synchronises with the host.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "gq.h"
#include "gq_internal.h"


namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

uint64_t mx_scale_bound(int32_t G, int64_t rows_cap, int64_t cols)
{
    return 512ull * (uint64_t)(cols / 128) * (uint64_t)((rows_cap + 127) / 128 + G);
}

uint64_t nv_scale_bound(int32_t G, int64_t rows_cap, int64_t cols)
{
    return 512ull * (uint64_t)(cols / 64) * (uint64_t)((rows_cap + 127) / 128 + G);
}

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

uint64_t channel_scale_bound(int64_t rows_cap, int64_t cols)
{
    return 4ull * (uint64_t)cols * (uint64_t)(rows_cap / 128);
}

// Checks shared by every call on a token buffer of rows_cap rows.
gq_status check_partition(const int32_t* d_split_sizes, int32_t G, int64_t rows_cap, int64_t cols)
{
    // Rows are TMA tensor-map coordinates (32-bit) in every kernel.
    if (G < 1 || G > GQ_MAX_GROUPS || rows_cap < 0 || rows_cap >= (int64_t(1) << 31) || cols <= 0)
        return GQ_ERR_INVALID_ARG;
    if (cols % 128 != 0)
        return GQ_ERR_ALIGNMENT;
    if (d_split_sizes == nullptr && rows_cap % G != 0)
        return GQ_ERR_ALIGNMENT;
    if ((rows_cap + 127) / 128 + G > (int64_t)INT32_MAX / 2)
        return GQ_ERR_INVALID_ARG;
    return GQ_OK;
}

gq_status cuda_status(cudaError_t e) { return e == cudaSuccess ? GQ_OK : GQ_ERR_CUDA; }

}  // namespace

namespace {

gq_status quantize_impl(const void* x_bf16, int64_t rows_cap, int64_t cols,
                        const int32_t* d_split_sizes, int32_t num_groups, const gq_recipe* recipe,
                        gq_quantized* out, int32_t* d_status, gq_stream_t stream, float* dpart)
{
    if (!recipe || !out || !d_status)
        return GQ_ERR_INVALID_ARG;
    gq_status st = check_partition(d_split_sizes, num_groups, rows_cap, cols);
    if (st != GQ_OK)
        return st;
    if (out->num_groups != num_groups || out->rows_cap != rows_cap || out->cols != cols ||
        out->recipe.kind != recipe->kind)
        return GQ_ERR_SHAPE_MISMATCH;
    const bool live = rows_cap > 0;
    if (live && (!x_bf16 || !aligned16(x_bf16)))
        return x_bf16 ? GQ_ERR_ALIGNMENT : GQ_ERR_INVALID_ARG;

    if (recipe->kind == GQ_RECIPE_MXFP8_1X32) {
        if (!recipe->rowwise && !recipe->colwise)
            return GQ_ERR_INVALID_ARG;
        const uint64_t need = mx_scale_bound(num_groups, rows_cap, cols);
        if (recipe->rowwise) {
            if (live && (!out->row_data || !out->row_scale))
                return GQ_ERR_INVALID_ARG;
            if (live && (!aligned16(out->row_data) || !aligned16(out->row_scale)))
                return GQ_ERR_ALIGNMENT;
            if (out->row_scale_bytes < need)
                return GQ_ERR_INVALID_ARG;
        }
        if (recipe->colwise) {
            if (live && (!out->col_data || !out->col_scale))
                return GQ_ERR_INVALID_ARG;
            if (live && (!aligned16(out->col_data) || !aligned16(out->col_scale)))
                return GQ_ERR_ALIGNMENT;
            if (out->col_scale_bytes < need)
                return GQ_ERR_INVALID_ARG;
        }
        out->recipe = *recipe;
        if (!live)
            return GQ_OK;
        return cuda_status(gq::launch_quant_mx(
            x_bf16, rows_cap, cols, d_split_sizes, num_groups,
            recipe->rowwise ? (uint8_t*)out->row_data : nullptr, (uint8_t*)out->row_scale,
            recipe->colwise ? (uint8_t*)out->col_data : nullptr, (uint8_t*)out->col_scale,
            d_status, (cudaStream_t)stream, dpart));
    }
    if (recipe->kind == GQ_RECIPE_NVFP4_1X16) {
        if (!recipe->rowwise && !recipe->colwise)
            return GQ_ERR_INVALID_ARG;
        const uint64_t need = nv_scale_bound(num_groups, rows_cap, cols);
        if (!out->amax)
            return GQ_ERR_INVALID_ARG;
        if (!aligned4(out->amax))
            return GQ_ERR_ALIGNMENT;
        if (recipe->rowwise) {
            if (live && (!out->row_data || !out->row_scale))
                return GQ_ERR_INVALID_ARG;
            if (live && (!aligned16(out->row_data) || !aligned16(out->row_scale)))
                return GQ_ERR_ALIGNMENT;
            if (out->row_scale_bytes < need)
                return GQ_ERR_INVALID_ARG;
        }
        if (recipe->colwise) {
            if (rows_cap % 32 != 0)
                return GQ_ERR_ALIGNMENT;
            if (live && (!out->col_data || !out->col_scale))
                return GQ_ERR_INVALID_ARG;
            if (live && (!aligned16(out->col_data) || !aligned16(out->col_scale)))
                return GQ_ERR_ALIGNMENT;
            if (out->col_scale_bytes < need)
                return GQ_ERR_INVALID_ARG;
        }
        out->recipe = *recipe;
        if (!live)
            return GQ_OK;
        return cuda_status(gq::launch_quant_nv(
            x_bf16, rows_cap, cols, d_split_sizes, num_groups,
            recipe->rowwise ? (uint8_t*)out->row_data : nullptr, (uint8_t*)out->row_scale,
            recipe->colwise ? (uint8_t*)out->col_data : nullptr, (uint8_t*)out->col_scale, out->amax, d_status,
            (cudaStream_t)stream));
    }
    if (recipe->kind == GQ_RECIPE_CHANNEL128_F32) {
        if (recipe->rowwise || !recipe->colwise)
            return GQ_ERR_UNSUPPORTED;
        if (live && (!out->col_data || !out->col_scale))
            return GQ_ERR_INVALID_ARG;
        if (live && (!aligned16(out->col_data) || !aligned16(out->col_scale)))
            return GQ_ERR_ALIGNMENT;
        if (out->col_scale_bytes < channel_scale_bound(rows_cap, cols))
            return GQ_ERR_INVALID_ARG;
        out->recipe = *recipe;
        if (!live)
            return GQ_OK;
        return cuda_status(gq::launch_quant_channel(
            x_bf16, rows_cap, cols, d_split_sizes, num_groups, recipe->zero_scale,
            (uint8_t*)out->col_data, (float*)out->col_scale, d_status, (cudaStream_t)stream));
    }
    return GQ_ERR_UNSUPPORTED;
}

}  // namespace

extern "C" {

const char* gq_status_string(int32_t status)
{
    switch (status) {
    case GQ_OK: return "GQ_OK";
    case GQ_ERR_INVALID_ARG: return "GQ_ERR_INVALID_ARG: null pointer, bad count or capacity";
    case GQ_ERR_ALIGNMENT: return "GQ_ERR_ALIGNMENT: cols % 128, rows_cap % num_groups or a pointer not 16-byte aligned";
    case GQ_ERR_SPLITS: return "GQ_ERR_SPLITS: a split size is negative, misaligned, or they sum past rows_cap";
    case GQ_ERR_UNSUPPORTED: return "GQ_ERR_UNSUPPORTED: recipe, orientation or dtype combination not provided";
    case GQ_ERR_CUDA: return "GQ_ERR_CUDA: a CUDA runtime call or launch failed";
    case GQ_ERR_TIMEOUT: return "GQ_ERR_TIMEOUT: a device pipeline wait gave up";
    case GQ_ERR_SHAPE_MISMATCH: return "GQ_ERR_SHAPE_MISMATCH: descriptor disagrees with the call";
    default: return "unknown gq_status";
    }
}

int32_t gq_version(void) { return (1 << 16) | 2; }

uint64_t gq_scale_bytes_bound(const gq_recipe* recipe, int32_t num_groups, int64_t rows_cap,
                              int64_t cols)
{
    if (!recipe || num_groups < 1 || rows_cap < 0 || cols <= 0 || cols % 128 != 0)
        return 0;
    if (recipe->kind == GQ_RECIPE_MXFP8_1X32)
        return mx_scale_bound(num_groups, rows_cap, cols);
    if (recipe->kind == GQ_RECIPE_CHANNEL128_F32)
        return channel_scale_bound(rows_cap, cols);
    if (recipe->kind == GQ_RECIPE_NVFP4_1X16)
        return nv_scale_bound(num_groups, rows_cap, cols);
    return 0;
}

gq_status gq_split_scan(const int32_t* d_split_sizes, int32_t num_groups, int64_t rows_cap,
                        int64_t cols, int32_t recipe_kind, int64_t* d_table, int32_t* d_status,
                        gq_stream_t stream)
{
    if (!d_table || !d_status)
        return GQ_ERR_INVALID_ARG;
    if (recipe_kind != GQ_RECIPE_MXFP8_1X32 && recipe_kind != GQ_RECIPE_CHANNEL128_F32 &&
        recipe_kind != GQ_RECIPE_NVFP4_1X16)
        return GQ_ERR_UNSUPPORTED;
    gq_status st = check_partition(d_split_sizes, num_groups, rows_cap, cols);
    if (st != GQ_OK)
        return st;
    const int align = recipe_kind == GQ_RECIPE_CHANNEL128_F32 ? 128 : 32;
    return cuda_status(gq::launch_split_scan(d_split_sizes, num_groups, rows_cap, cols, align,
                                             recipe_kind, d_table, d_status,
                                             (cudaStream_t)stream));
}

gq_status gq_quantize(const void* x_bf16, int64_t rows_cap, int64_t cols,
                      const int32_t* d_split_sizes, int32_t num_groups, const gq_recipe* recipe,
                      gq_quantized* out, int32_t* d_status, gq_stream_t stream)
{
    return quantize_impl(x_bf16, rows_cap, cols, d_split_sizes, num_groups, recipe, out, d_status, stream,
                         nullptr);
}

uint64_t gq_dbias_workspace_bytes(int32_t num_groups, int64_t rows_cap, int64_t cols)
{
    if (num_groups < 1 || rows_cap < 0 || cols <= 0 || cols % 128 != 0)
        return 0;
    return 4ull * (uint64_t)cols * (uint64_t)((rows_cap + 127) / 128 + num_groups);
}

gq_status gq_quantize_dbias(const void* x_bf16, int64_t rows_cap, int64_t cols,
                            const int32_t* d_split_sizes, int32_t num_groups, const gq_recipe* recipe,
                            gq_quantized* out, float* d_dbias, void* d_workspace, uint64_t workspace_bytes,
                            int32_t* d_status, gq_stream_t stream)
{
    if (!recipe || !d_dbias || !d_workspace)
        return GQ_ERR_INVALID_ARG;
    if (recipe->kind != GQ_RECIPE_MXFP8_1X32)
        return GQ_ERR_UNSUPPORTED;
    if (!aligned16(d_dbias) || !aligned16(d_workspace))
        return GQ_ERR_ALIGNMENT;
    if (workspace_bytes < gq_dbias_workspace_bytes(num_groups, rows_cap, cols))
        return GQ_ERR_INVALID_ARG;
    gq_status st = quantize_impl(x_bf16, rows_cap, cols, d_split_sizes, num_groups, recipe, out, d_status,
                                 stream, static_cast<float*>(d_workspace));
    if (st != GQ_OK)
        return st;
    // with L == 0 (rows_cap == 0 included) every group sums no tile: zeros
    return cuda_status(gq::launch_dbias_reduce(d_split_sizes, num_groups, rows_cap, cols,
                                               static_cast<const float*>(d_workspace), d_dbias, d_status,
                                               (cudaStream_t)stream));
}

}  // extern "C"

namespace {

// Checks of one GEMM operand: recipe, orientation, shape and buffers.
gq_status check_operand(const gq_quantized* q, int32_t kind, bool colwise, int32_t G,
                        int64_t rows, int64_t cols)
{
    if (!q)
        return GQ_ERR_INVALID_ARG;
    if (q->recipe.kind != kind)
        return GQ_ERR_UNSUPPORTED;
    if (q->num_groups != G || q->rows_cap != rows || q->cols != cols)
        return GQ_ERR_SHAPE_MISMATCH;
    if (colwise ? !q->recipe.colwise : !q->recipe.rowwise)
        return GQ_ERR_UNSUPPORTED;
    const void* d = colwise ? q->col_data : q->row_data;
    const void* s = colwise ? q->col_scale : q->row_scale;
    if (rows > 0 && (!d || !s))
        return GQ_ERR_INVALID_ARG;
    if (rows > 0 && (!aligned16(d) || !aligned16(s)))
        return GQ_ERR_ALIGNMENT;
    const uint64_t cap = colwise ? q->col_scale_bytes : q->row_scale_bytes;
    const uint64_t need = kind == GQ_RECIPE_MXFP8_1X32   ? mx_scale_bound(G, rows, cols)
                          : kind == GQ_RECIPE_NVFP4_1X16 ? nv_scale_bound(G, rows, cols)
                                                         : channel_scale_bound(rows, cols);
    if (cap < need)
        return GQ_ERR_INVALID_ARG;
    if (kind == GQ_RECIPE_NVFP4_1X16) {
        if (!q->amax)
            return GQ_ERR_INVALID_ARG;
        if (!aligned4(q->amax))
            return GQ_ERR_ALIGNMENT;
        if (colwise && rows % 32 != 0)
            return GQ_ERR_ALIGNMENT;
    }
    return GQ_OK;
}

// An NVFP4 operand as the GEMM reads it: rowwise [rows, cols/2], or
// columnwise stored transposed [cols, rows/2].
gq::NvOperand nv_operand(const gq_quantized* q, bool colwise)
{
    gq::NvOperand o;
    o.data = (const uint8_t*)(colwise ? q->col_data : q->row_data);
    o.scale = (const uint8_t*)(colwise ? q->col_scale : q->row_scale);
    o.amax = q->amax;
    o.rows = colwise ? q->cols : q->rows_cap;
    o.row_bytes = colwise ? q->rows_cap / 2 : q->cols / 2;
    return o;
}

gq::GemmOperand operand(const gq_quantized* q, bool colwise)
{
    gq::GemmOperand o;
    o.data = (const uint8_t*)(colwise ? q->col_data : q->row_data);
    o.scale = colwise ? q->col_scale : q->row_scale;
    o.scale_bytes = colwise ? q->col_scale_bytes : q->row_scale_bytes;
    o.rows = q->rows_cap;
    o.cols = q->cols;
    return o;
}

gq_status check_gemm_common(const int32_t* splits, int32_t G, int64_t rows_cap, int64_t n,
                            int64_t k, const void* out, const int32_t* d_status)
{
    if (!d_status || n <= 0 || k <= 0)
        return GQ_ERR_INVALID_ARG;
    if (n % 128 != 0 || k % 128 != 0)
        return GQ_ERR_ALIGNMENT;
    gq_status st = check_partition(splits, G, rows_cap, 128);
    if (st != GQ_OK)
        return st;
    if (!out)
        return GQ_ERR_INVALID_ARG;
    if (!aligned16(out))
        return GQ_ERR_ALIGNMENT;
    return GQ_OK;
}

}  // namespace

namespace {

gq_status fprop_impl(const gq_quantized* x, const gq_quantized* w, const int32_t* d_split_sizes,
                     int32_t num_groups, int64_t n, int64_t k, void* y, int32_t out_dtype, const void* d_bias,
                     int32_t bias_dtype, int32_t* d_status, gq_stream_t stream,
                     const gq::ActOutput* act = nullptr)
{
    if (!x || !w)
        return GQ_ERR_INVALID_ARG;
    gq_status st = check_gemm_common(d_split_sizes, num_groups, x->rows_cap, n, k, y, d_status);
    if (st != GQ_OK)
        return st;
    if (out_dtype != GQ_DTYPE_F32 && out_dtype != GQ_DTYPE_BF16)
        return GQ_ERR_UNSUPPORTED;
    if (x->recipe.kind == GQ_RECIPE_NVFP4_1X16) {
        if (d_bias || act || n % 256 != 0 || k % 256 != 0)
            return GQ_ERR_UNSUPPORTED;
        if ((st = check_operand(x, GQ_RECIPE_NVFP4_1X16, false, num_groups, x->rows_cap, k)) != GQ_OK)
            return st;
        if ((st = check_operand(w, GQ_RECIPE_NVFP4_1X16, false, num_groups, (int64_t)num_groups * n, k)) !=
            GQ_OK)
            return st;
        if (x->rows_cap == 0)
            return GQ_OK;
        return gq::launch_gemm_nv(gq::NV_FPROP, nv_operand(x, false), nv_operand(w, false), d_split_sizes,
                                  num_groups, x->rows_cap, n, k, y, out_dtype, 0, d_status, (cudaStream_t)stream);
    }
    if ((st = check_operand(x, GQ_RECIPE_MXFP8_1X32, false, num_groups, x->rows_cap, k)) != GQ_OK)
        return st;
    if ((st = check_operand(w, GQ_RECIPE_MXFP8_1X32, false, num_groups, (int64_t)num_groups * n,
                            k)) != GQ_OK)
        return st;
    if (x->rows_cap == 0)
        return GQ_OK;
    return gq::launch_gemm(gq::GEMM_FPROP, operand(x, false), operand(w, false), d_split_sizes,
                           num_groups, x->rows_cap, n, k, y, out_dtype, 0, d_status,
                           (cudaStream_t)stream, nullptr, d_bias, bias_dtype, act);
}

}  // namespace

extern "C" {


gq_status gq_gemm_fprop(const gq_quantized* x, const gq_quantized* w,
                        const int32_t* d_split_sizes, int32_t num_groups, int64_t n, int64_t k,
                        void* y, int32_t out_dtype, int32_t* d_status, gq_stream_t stream)
{
    return fprop_impl(x, w, d_split_sizes, num_groups, n, k, y, out_dtype, nullptr, 0, d_status, stream);
}

gq_status gq_gemm_fprop_bias(const gq_quantized* x, const gq_quantized* w,
                             const int32_t* d_split_sizes, int32_t num_groups, int64_t n, int64_t k,
                             const void* d_bias, int32_t bias_dtype, void* y, int32_t out_dtype,
                             int32_t* d_status, gq_stream_t stream)
{
    if (!d_bias)
        return GQ_ERR_INVALID_ARG;
    if (bias_dtype != GQ_DTYPE_F32 && bias_dtype != GQ_DTYPE_BF16)
        return GQ_ERR_UNSUPPORTED;
    if (!aligned16(d_bias))
        return GQ_ERR_ALIGNMENT;
    return fprop_impl(x, w, d_split_sizes, num_groups, n, k, y, out_dtype, d_bias, bias_dtype, d_status,
                      stream);
}

}  // extern "C"

namespace {

// The fprop with a fused activation + MX quantisation of it (mode 1:
// ScaledSReLU, activation width n; mode 2: ScaledSwiGLU, width n / 2).
gq_status fprop_act_impl(const gq_quantized* x, const gq_quantized* w, const int32_t* d_split_sizes,
                         int32_t num_groups, int64_t n, int64_t k, const void* d_bias, int32_t bias_dtype,
                         const float* d_probs, void* y, int32_t out_dtype, gq_quantized* act_out, int32_t* d_status,
                         gq_stream_t stream, int mode)
{
    if (!x || !act_out || !d_probs)
        return GQ_ERR_INVALID_ARG;
    if (d_bias && bias_dtype != GQ_DTYPE_F32 && bias_dtype != GQ_DTYPE_BF16)
        return GQ_ERR_UNSUPPORTED;
    if ((d_bias && !aligned16(d_bias)) || !aligned16(d_probs))
        return GQ_ERR_ALIGNMENT;
    if (n % 256 != 0)
        return GQ_ERR_UNSUPPORTED;
    const int64_t act_cols = mode == 2 ? n / 2 : n;
    if (act_out->num_groups != num_groups || act_out->rows_cap != x->rows_cap || act_out->cols != act_cols)
        return GQ_ERR_SHAPE_MISMATCH;
    if (act_out->recipe.kind != GQ_RECIPE_MXFP8_1X32 || !act_out->recipe.rowwise || !act_out->recipe.colwise)
        return GQ_ERR_UNSUPPORTED;
    if (x->rows_cap > 0) {
        if (!act_out->row_data || !act_out->row_scale || !act_out->col_data || !act_out->col_scale)
            return GQ_ERR_INVALID_ARG;
        if (!aligned16(act_out->row_data) || !aligned16(act_out->row_scale) || !aligned16(act_out->col_data) ||
            !aligned16(act_out->col_scale))
            return GQ_ERR_ALIGNMENT;
        const uint64_t need = mx_scale_bound(num_groups, x->rows_cap, act_cols);
        if (act_out->row_scale_bytes < need || act_out->col_scale_bytes < need)
            return GQ_ERR_INVALID_ARG;
    }
    const gq::ActOutput act{d_probs, (uint8_t*)act_out->row_data, (uint8_t*)act_out->row_scale,
                            (uint8_t*)act_out->col_data, (uint8_t*)act_out->col_scale, mode};
    return fprop_impl(x, w, d_split_sizes, num_groups, n, k, y, out_dtype, d_bias, bias_dtype, d_status, stream,
                      &act);
}

}  // namespace

extern "C" {

gq_status gq_gemm_fprop_srelu_quant(const gq_quantized* x, const gq_quantized* w,
                                    const int32_t* d_split_sizes, int32_t num_groups, int64_t n, int64_t k,
                                    const void* d_bias, int32_t bias_dtype, const float* d_probs, void* y,
                                    int32_t out_dtype, gq_quantized* act_out, int32_t* d_status,
                                    gq_stream_t stream)
{
    return fprop_act_impl(x, w, d_split_sizes, num_groups, n, k, d_bias, bias_dtype, d_probs, y, out_dtype, act_out,
                          d_status, stream, 1);
}

gq_status gq_gemm_fprop_swiglu_quant(const gq_quantized* x, const gq_quantized* w,
                                     const int32_t* d_split_sizes, int32_t num_groups, int64_t n, int64_t k,
                                     const void* d_bias, int32_t bias_dtype, const float* d_probs, void* y,
                                     int32_t out_dtype, gq_quantized* act_out, int32_t* d_status,
                                     gq_stream_t stream)
{
    return fprop_act_impl(x, w, d_split_sizes, num_groups, n, k, d_bias, bias_dtype, d_probs, y, out_dtype, act_out,
                          d_status, stream, 2);
}

gq_status gq_gemm_dgrad(const gq_quantized* dy, const gq_quantized* w,
                        const int32_t* d_split_sizes, int32_t num_groups, int64_t n, int64_t k,
                        void* dx, int32_t out_dtype, int32_t* d_status, gq_stream_t stream)
{
    if (!dy || !w)
        return GQ_ERR_INVALID_ARG;
    gq_status st = check_gemm_common(d_split_sizes, num_groups, dy->rows_cap, n, k, dx, d_status);
    if (st != GQ_OK)
        return st;
    if (out_dtype != GQ_DTYPE_F32 && out_dtype != GQ_DTYPE_BF16)
        return GQ_ERR_UNSUPPORTED;
    if (dy->recipe.kind == GQ_RECIPE_NVFP4_1X16) {
        if (n % 256 != 0 || k % 256 != 0)
            return GQ_ERR_UNSUPPORTED;
        if ((st = check_operand(dy, GQ_RECIPE_NVFP4_1X16, false, num_groups, dy->rows_cap, n)) != GQ_OK)
            return st;
        if ((st = check_operand(w, GQ_RECIPE_NVFP4_1X16, true, num_groups, (int64_t)num_groups * n, k)) != GQ_OK)
            return st;
        if (dy->rows_cap == 0)
            return GQ_OK;
        return gq::launch_gemm_nv(gq::NV_DGRAD, nv_operand(dy, false), nv_operand(w, true), d_split_sizes,
                                  num_groups, dy->rows_cap, n, k, dx, out_dtype, 0, d_status, (cudaStream_t)stream);
    }
    if ((st = check_operand(dy, GQ_RECIPE_MXFP8_1X32, false, num_groups, dy->rows_cap, n)) != GQ_OK)
        return st;
    if ((st = check_operand(w, GQ_RECIPE_MXFP8_1X32, true, num_groups, (int64_t)num_groups * n,
                            k)) != GQ_OK)
        return st;
    if (dy->rows_cap == 0)
        return GQ_OK;
    return gq::launch_gemm(gq::GEMM_DGRAD, operand(dy, false), operand(w, true), d_split_sizes,
                           num_groups, dy->rows_cap, n, k, dx, out_dtype, 0, d_status,
                           (cudaStream_t)stream);
}

gq_status gq_gemm_wgrad(const gq_quantized* dy, const gq_quantized* x,
                        const int32_t* d_split_sizes, int32_t num_groups, int64_t n, int64_t k,
                        float* dw, int32_t accumulate, void* d_workspace, uint64_t workspace_bytes,
                        int32_t* d_status, gq_stream_t stream)
{
    if (!dy || !x)
        return GQ_ERR_INVALID_ARG;
    gq_status st = check_gemm_common(d_split_sizes, num_groups, dy->rows_cap, n, k, dw, d_status);
    if (st != GQ_OK)
        return st;
    if (accumulate != 0 && accumulate != 1)
        return GQ_ERR_INVALID_ARG;
    if (d_workspace && workspace_bytes < GQ_WGRAD_WORKSPACE_BYTES)
        return GQ_ERR_INVALID_ARG;
    if (d_workspace && !aligned16(d_workspace))
        return GQ_ERR_ALIGNMENT;
    if (dy->recipe.kind != x->recipe.kind)
        return GQ_ERR_UNSUPPORTED;
    const int32_t kind = dy->recipe.kind;
    if (kind != GQ_RECIPE_MXFP8_1X32 && kind != GQ_RECIPE_CHANNEL128_F32 && kind != GQ_RECIPE_NVFP4_1X16)
        return GQ_ERR_UNSUPPORTED;
    if (x->rows_cap != dy->rows_cap)
        return GQ_ERR_SHAPE_MISMATCH;
    if ((st = check_operand(dy, kind, true, num_groups, dy->rows_cap, n)) != GQ_OK)
        return st;
    if ((st = check_operand(x, kind, true, num_groups, x->rows_cap, k)) != GQ_OK)
        return st;
    if (kind == GQ_RECIPE_NVFP4_1X16) {
        if (k % 256 != 0)
            return GQ_ERR_UNSUPPORTED;
        return gq::launch_gemm_nv(gq::NV_WGRAD, nv_operand(dy, true), nv_operand(x, true), d_split_sizes,
                                  num_groups, dy->rows_cap, n, k, dw, GQ_DTYPE_F32, accumulate, d_status,
                                  (cudaStream_t)stream);
    }
    return gq::launch_gemm(kind == GQ_RECIPE_MXFP8_1X32 ? gq::GEMM_WGRAD_MX
                                                        : gq::GEMM_WGRAD_CHANNEL,
                           operand(dy, true), operand(x, true), d_split_sizes, num_groups,
                           dy->rows_cap, n, k, dw, GQ_DTYPE_F32, accumulate, d_status,
                           (cudaStream_t)stream, d_workspace);
}

}  // extern "C"
