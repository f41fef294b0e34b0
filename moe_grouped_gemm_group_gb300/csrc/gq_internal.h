// Host-side declarations shared by the C-ABI layer and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gq.h"

#define GQ_MAX_GROUPS 1024

namespace gq {

// Per-device facts, queried once per device.
struct DeviceInfo {
    int sm_count = 0;
    int cc_major = 0, cc_minor = 0;
    size_t smem_optin = 0;
};
const DeviceInfo& device_info();

// The driver's ID of the current CUDA context (never reused within a
// process), false while no context is current.  Per-context set-up (kernel
// attributes, symbol addresses) is cached under it, so that a new context --
// another one on the same device, or the one after cudaDeviceReset -- gets
// its own set-up.
bool current_context_id(unsigned long long* id);

// Per (kernel, context) set-up, done on the first launch there and cached:
// the dynamic shared-memory limit and the resident blocks per SM.  Later
// launches only enqueue work.
cudaError_t prepare_kernel(const void* fn, int dyn_smem, int threads, int* blocks_per_sm);

// 2-D tensor map over a row-major [rows, cols] buffer of `elem_bytes`-byte
// elements (rows stride = cols * elem_bytes), boxes of box_cols x box_rows
// with the 128-byte swizzle; out-of-range elements read as zero.  False if
// the driver's encoder is unavailable or rejects the map.
bool make_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, int elem_bytes,
                        const void* base, int64_t rows, int64_t cols, int box_cols, int box_rows);

// The same with the 64-byte swizzle (box rows of at most 64 bytes; 16-byte
// chunk c of box row r sits at chunk c ^ ((r >> 1) & 3) of that row).
bool make_tensor_map_2d_sw64(CUtensorMap* map, CUtensorMapDataType dtype, int elem_bytes,
                             const void* base, int64_t rows, int64_t cols, int box_cols,
                             int box_rows);

// The same without swizzle (boxes land row after row in shared memory).
bool make_tensor_map_2d_plain(CUtensorMap* map, CUtensorMapDataType dtype, int elem_bytes,
                              const void* base, int64_t rows, int64_t cols, int box_cols,
                              int box_rows);

inline bool make_map_u8(CUtensorMap* map, const uint8_t* base, int64_t rows, int64_t cols,
                        int box_rows)
{
    return make_tensor_map_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, base, rows, cols, 128,
                              box_rows);
}

// Quantizer launchers (gq_quant.cu).
cudaError_t launch_split_scan(const int32_t* splits, int G, int64_t rows_cap, int64_t cols,
                              int align, int scale_kind, int64_t* table, int32_t* status,
                              cudaStream_t stream);
cudaError_t launch_quant_mx(const void* x, int64_t rows_cap, int64_t cols, const int32_t* splits,
                            int G, uint8_t* row_data, uint8_t* row_scale, uint8_t* col_data,
                            uint8_t* col_scale, int32_t* status, cudaStream_t stream, float* dpart = nullptr);
cudaError_t launch_quant_channel(const void* x, int64_t rows_cap, int64_t cols,
                                 const int32_t* splits, int G, float zero_scale,
                                 uint8_t* col_data, float* col_scale, int32_t* status,
                                 cudaStream_t stream);

// Bias gradient of a grouped buffer from the per-tile column sums that the
// MX quantiser wrote to dpart (gq_quant.cu).
cudaError_t launch_dbias_reduce(const int32_t* splits, int G, int64_t rows_cap, int64_t cols,
                                const float* dpart, float* db, int32_t* status, cudaStream_t stream);

// GEMM launchers (gq_gemm.cu).  Operand buffers are already validated.
struct GemmOperand {
    const uint8_t* data;   // e4m3 codes [rows, cols]
    const void* scale;     // E8M0 swizzled bytes or fp32 per-channel scales
    uint64_t scale_bytes;  // capacity of `scale` (at least the bound for its shape)
    int64_t rows;          // rows of the buffer (rows_cap, or G * n for weights)
    int64_t cols;
};
enum GemmKind { GEMM_FPROP = 0, GEMM_DGRAD = 1, GEMM_WGRAD_MX = 2, GEMM_WGRAD_CHANNEL = 3 };

// Outputs of the fprop with a fused activation + MX quantisation: per-row
// probs and the MX rowwise / columnwise codes and scales of the activation.
// mode 1: ScaledSReLU (activation width n); mode 2: ScaledSwiGLU (width n / 2).
struct ActOutput {
    const float* probs;
    uint8_t* row_data;
    uint8_t* row_scale;
    uint8_t* col_data;
    uint8_t* col_scale;
    int mode = 1;
};

// Output tiles of the k-grouped MX wgrad over G groups of an [n, k] weight:
// G * n/128 * k/256 when the launcher takes 256-wide tiles, else
// G * n/128 * k/128.  The tile-claim counter counts them in 32-bit halves.
int64_t wgrad_mx_tiles(int G, int64_t n, int64_t k);

gq_status launch_gemm(GemmKind kind, const GemmOperand& a, const GemmOperand& b,
                      const int32_t* splits, int G, int64_t rows_cap, int64_t n, int64_t k,
                      void* out, int out_dtype, int accumulate, int32_t* status,
                      cudaStream_t stream, void* workspace = nullptr, const void* bias = nullptr,
                      int bias_dtype = 0, const ActOutput* act = nullptr);

// NVFP4 quantiser and GEMMs (gq_nvfp4.cu).  Operand buffers are already
// validated; the quantiser runs the split scan + amax reset, the per-group
// amax pass and the quantisation pass on `stream`.
cudaError_t launch_quant_nv(const void* x, int64_t rows_cap, int64_t cols, const int32_t* splits, int G,
                            uint8_t* row_data, uint8_t* row_scale, uint8_t* col_data, uint8_t* col_scale, float* amax,
                            int32_t* status, cudaStream_t stream);
struct NvOperand {
    const uint8_t* data;   // packed E2M1 codes, [rows, row_bytes]
    const uint8_t* scale;  // swizzled E4M3 scale atoms
    const float* amax;     // per-group amax, fp32 [G]
    int64_t rows;          // rows of the stored array (rowwise: the buffer's rows; columnwise: its cols)
    int64_t row_bytes;     // bytes per stored row
};
enum NvGemmKind { NV_FPROP = 0, NV_DGRAD = 1, NV_WGRAD = 2 };
gq_status launch_gemm_nv(NvGemmKind kind, const NvOperand& a, const NvOperand& b, const int32_t* splits, int G,
                         int64_t rows_cap, int64_t n, int64_t k, void* out, int out_dtype, int accumulate,
                         int32_t* status, cudaStream_t stream);

}  // namespace gq
