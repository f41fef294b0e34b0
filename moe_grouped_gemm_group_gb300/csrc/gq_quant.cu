// Grouped FP8 quantizer kernels.
//
//  k_split_scan  -- the split-size scan exposed by gq_split_scan.
//  k_quant_mx    -- MXFP8 1x32 rowwise + columnwise in one pass over the live
//                   rows (TransformerEngine issue 3484 layout; PR 3224
//                   per-member extents).
//  k_quant_ch    -- per-channel 128-row fp32-scale cast (DeepGEMM issue 365,
//                   _per_channel_cast_to_fp8).
//
// Work unit: a 128-row x 128-column tile that never straddles two groups
// (groups are scanned in shared memory by every CTA; row tiles are numbered
// group by group).  512 threads = 16 warps; warp (rb, cb) owns the 32 x 32
// sub-block rows [32 rb, 32 rb + 32) x columns [32 cb, 32 cb + 32); lane l
// holds row 32 rb + l of it in 16 registers (32 bf16).  A rowwise block is
// one lane's 32 values (amax in registers); a columnwise block is one column
// of the sub-block (amax by a warp-wide redux.sync).  One 128 x 128 tile
// yields exactly one rowwise and one columnwise 512-byte scale atom, staged
// in shared memory and written with 16-byte stores.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "gq_device.cuh"
#include "gq_internal.h"

namespace gq {
namespace {

constexpr int kQuantThreads = 512;

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// E8M0 byte of a block from the bit pattern of its bf16 amax:
// e = floor(log2 amax) - 8 clamped at -127 -> byte = e + 127 = max(E - 8, 0)
// with E the (bf16 = fp32) biased exponent field; zero and subnormal amax
// give 0.  Finite inputs never reach byte 255.
__device__ __forceinline__ uint32_t e8m0_byte(uint32_t amax_bits)
{
    const int E = (int)((amax_bits >> 7) & 0xffu);
    return (uint32_t)max(E - 8, 0);
}

// 2^-e for the byte above, as an exact fp32 power of two (biased exponent
// 254 - byte lies in [8, 254]).
__device__ __forceinline__ float inv_scale(uint32_t byte) { return __uint_as_float((254u - byte) << 23); }

// Two fp32 values -> two e4m3 bytes (nearest-even, saturating), `a` in the
// low byte.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float a, float b)
{
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ void load_row32(const uint16_t* __restrict__ p, uint32_t (&v)[16])
{
    const uint4* q = reinterpret_cast<const uint4*>(p);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 u = __ldg(q + i);
        v[4 * i + 0] = u.x;
        v[4 * i + 1] = u.y;
        v[4 * i + 2] = u.z;
        v[4 * i + 3] = u.w;
    }
}

__device__ __forceinline__ void store32(uint8_t* p, const uint32_t (&w)[8])
{
    uint4* q = reinterpret_cast<uint4*>(p);
    q[0] = make_uint4(w[0], w[1], w[2], w[3]);
    q[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

// Magnitude bits of element j (0..31) of a lane's packed row.
__device__ __forceinline__ uint32_t mag(const uint32_t (&v)[16], int j)
{
    return (j & 1) ? ((v[j >> 1] >> 16) & 0x7fffu) : (v[j >> 1] & 0x7fffu);
}

__device__ __forceinline__ float elem(const uint32_t (&v)[16], int j)
{
    return (j & 1) ? bf16_hi(v[j >> 1]) : bf16_lo(v[j >> 1]);
}

__global__ void k_split_scan(const int32_t* __restrict__ splits, int G, int64_t rows_cap,
                             int64_t cols, int align, int scale_kind, int64_t* __restrict__ table,
                             int32_t* __restrict__ status)
{
    __shared__ int64_t s_off[GQ_MAX_GROUPS + 1];
    __shared__ int32_t s_tp[GQ_MAX_GROUPS + 1];
    __shared__ int64_t s_w64[32];
    __shared__ int32_t s_w32[32];
    if (load_status(status) != 0)
        return;
    const int err = block_scan_splits(splits, G, rows_cap, align, s_off, s_tp, s_w64, s_w32);
    if (err) {
        if (threadIdx.x == 0)
            set_status(status, err);
        return;
    }
    for (int g = threadIdx.x; g <= G; g += blockDim.x) {
        table[g] = s_off[g];
        table[G + 1 + g] = s_tp[g];
        table[2 * (G + 1) + g] = scale_kind == 0 ? 512 * (cols >> 7) * (int64_t)s_tp[g]
                                                 : 4 * cols * (s_off[g] >> 7);
    }
}

template <bool ROW, bool COL>
__global__ void __launch_bounds__(kQuantThreads, 2)
k_quant_mx(const uint16_t* __restrict__ x, int64_t rows_cap, int64_t cols,
           const int32_t* __restrict__ splits, int G, uint8_t* __restrict__ row_data,
           uint8_t* __restrict__ row_scale, uint8_t* __restrict__ col_data,
           uint8_t* __restrict__ col_scale, int32_t* __restrict__ status)
{
    __shared__ int64_t s_off[GQ_MAX_GROUPS + 1];
    __shared__ int32_t s_tp[GQ_MAX_GROUPS + 1];
    __shared__ int64_t s_w64[32];
    __shared__ int32_t s_w32[32];
    __shared__ __align__(16) uint8_t s_rs[512];
    __shared__ __align__(16) uint8_t s_cs[512];

    if (load_status(status) != 0)
        return;
    const int err = block_scan_splits(splits, G, rows_cap, 32, s_off, s_tp, s_w64, s_w32);
    if (err) {
        if (threadIdx.x == 0)
            set_status(status, err);
        return;
    }

    const int nct = (int)(cols >> 7);
    const int64_t total = (int64_t)s_tp[G] * nct;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rb = warp >> 2, cb = warp & 3;

    for (int64_t t = blockIdx.x; t < total; t += gridDim.x) {
        const int64_t rt = t / nct;
        const int ct = (int)(t - rt * nct);
        const int g = group_of_tile(s_tp, G, rt);
        const int64_t lt = rt - s_tp[g];
        const int64_t m = s_off[g + 1] - s_off[g];
        const int64_t rows_here = min((int64_t)128, m - 128 * lt);   // a multiple of 32
        const bool active = 32 * rb < rows_here;                     // uniform per warp
        const int64_t row = s_off[g] + 128 * lt + 32 * rb + lane;
        const int64_t col0 = (int64_t)ct * 128 + 32 * cb;

        uint32_t rbyte = 0, cbyte = 0;
        if (active) {
            uint32_t v[16];
            load_row32(x + row * cols + col0, v);
            if (ROW) {
                uint32_t mx = 0;
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    mx = __vmaxu2(mx, v[i] & 0x7fff7fffu);
                rbyte = e8m0_byte(max(mx & 0xffffu, mx >> 16));
                const float s = inv_scale(rbyte);
                uint32_t w[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t p0 = cvt_e4m3x2(bf16_lo(v[2 * i]) * s, bf16_hi(v[2 * i]) * s);
                    const uint32_t p1 =
                        cvt_e4m3x2(bf16_lo(v[2 * i + 1]) * s, bf16_hi(v[2 * i + 1]) * s);
                    w[i] = p0 | (p1 << 16);
                }
                store32(row_data + row * cols + col0, w);
            }
            if (COL) {
                float sc[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const uint32_t am = __reduce_max_sync(0xffffffffu, mag(v, j));
                    const uint32_t byte = e8m0_byte(am);
                    if (lane == j)
                        cbyte = byte;
                    sc[j] = elem(v, j) * inv_scale(byte);
                }
                uint32_t w[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t p0 = cvt_e4m3x2(sc[4 * i + 0], sc[4 * i + 1]);
                    const uint32_t p1 = cvt_e4m3x2(sc[4 * i + 2], sc[4 * i + 3]);
                    w[i] = p0 | (p1 << 16);
                }
                store32(col_data + row * cols + col0, w);
            }
        }
        // Scale atoms: rowwise (row 32 rb + lane, block cb); columnwise
        // (channel 32 cb + lane, 32-row block rb).  Inactive warps write the
        // zero entries of a partial last tile.
        s_rs[lane * 16 + rb * 4 + cb] = (uint8_t)rbyte;
        s_cs[lane * 16 + cb * 4 + rb] = (uint8_t)cbyte;
        __syncthreads();
        const int64_t base = 512 * (int64_t)nct * s_tp[g];
        if (ROW && threadIdx.x < 32) {
            const uint4 a = reinterpret_cast<const uint4*>(s_rs)[threadIdx.x];
            reinterpret_cast<uint4*>(row_scale + base + (lt * nct + ct) * 512)[threadIdx.x] = a;
        }
        if (COL && threadIdx.x >= 32 && threadIdx.x < 64) {
            const int64_t T = s_tp[g + 1] - s_tp[g];
            const uint4 a = reinterpret_cast<const uint4*>(s_cs)[threadIdx.x - 32];
            reinterpret_cast<uint4*>(col_scale + base + ((int64_t)ct * T + lt) * 512)[threadIdx.x - 32] = a;
        }
        __syncthreads();
    }
}

__global__ void __launch_bounds__(kQuantThreads, 2)
k_quant_ch(const uint16_t* __restrict__ x, int64_t rows_cap, int64_t cols,
           const int32_t* __restrict__ splits, int G, float zero_scale,
           uint8_t* __restrict__ col_data, float* __restrict__ col_scale,
           int32_t* __restrict__ status)
{
    __shared__ int64_t s_off[GQ_MAX_GROUPS + 1];
    __shared__ int32_t s_tp[GQ_MAX_GROUPS + 1];
    __shared__ int64_t s_w64[32];
    __shared__ int32_t s_w32[32];
    __shared__ uint32_t s_part[4][128];
    __shared__ float s_rcp[128];

    if (load_status(status) != 0)
        return;
    const int err = block_scan_splits(splits, G, rows_cap, 128, s_off, s_tp, s_w64, s_w32);
    if (err) {
        if (threadIdx.x == 0)
            set_status(status, err);
        return;
    }
    // Every group starts on a multiple of 128, so live row block b (rows
    // [128 b, 128 b + 128)) lies inside one group.
    const int nct = (int)(cols >> 7);
    const int64_t nb = s_off[G] >> 7;
    const int64_t total = nb * nct;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rb = warp >> 2, cb = warp & 3;

    for (int64_t t = blockIdx.x; t < total; t += gridDim.x) {
        const int64_t b = t / nct;
        const int ct = (int)(t - b * nct);
        const int64_t row = 128 * b + 32 * rb + lane;
        const int64_t col0 = (int64_t)ct * 128 + 32 * cb;
        uint32_t v[16];
        load_row32(x + row * cols + col0, v);
        uint32_t mine = 0;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const uint32_t am = __reduce_max_sync(0xffffffffu, mag(v, j));
            if (lane == j)
                mine = am;
        }
        s_part[rb][32 * cb + lane] = mine;
        __syncthreads();
        if (threadIdx.x < 128) {
            const int c = threadIdx.x;
            const uint32_t am = max(max(s_part[0][c], s_part[1][c]), max(s_part[2][c], s_part[3][c]));
            float sf = __fdiv_rn(__uint_as_float(am << 16), 448.0f);
            if (sf == 0.0f)
                sf = zero_scale;
            sf = fmaxf(sf, 1e-30f);
            s_rcp[c] = __fdiv_rn(1.0f, sf);
            col_scale[b * cols + (int64_t)ct * 128 + c] = sf;
        }
        __syncthreads();
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int j = 4 * i;
            const float* r = s_rcp + 32 * cb + j;
            const uint32_t p0 = cvt_e4m3x2(__fmul_rn(elem(v, j + 0), r[0]), __fmul_rn(elem(v, j + 1), r[1]));
            const uint32_t p1 = cvt_e4m3x2(__fmul_rn(elem(v, j + 2), r[2]), __fmul_rn(elem(v, j + 3), r[3]));
            w[i] = p0 | (p1 << 16);
        }
        store32(col_data + row * cols + col0, w);
    }
}

int blocks_per_sm_for(const void* fn, int threads)
{
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, 0) != cudaSuccess || n < 1)
        n = 1;
    return n;
}

}  // namespace

cudaError_t launch_split_scan(const int32_t* splits, int G, int64_t rows_cap, int64_t cols,
                              int align, int scale_kind, int64_t* table, int32_t* status,
                              cudaStream_t stream)
{
    k_split_scan<<<1, 1024, 0, stream>>>(splits, G, rows_cap, cols, align, scale_kind, table,
                                         status);
    return cudaGetLastError();
}

cudaError_t launch_quant_mx(const void* x, int64_t rows_cap, int64_t cols, const int32_t* splits,
                            int G, uint8_t* row_data, uint8_t* row_scale, uint8_t* col_data,
                            uint8_t* col_scale, int32_t* status, cudaStream_t stream)
{
    const int64_t tiles_bound = ((rows_cap + 127) / 128 + G) * (cols / 128);
    const auto* xp = static_cast<const uint16_t*>(x);
    const int sms = device_info().sm_count;
    auto grid_for = [&](const void* fn) {
        const int64_t g = (int64_t)sms * blocks_per_sm_for(fn, kQuantThreads);
        return (unsigned)std::max<int64_t>(1, std::min<int64_t>(g, tiles_bound));
    };
    if (row_data && col_data) {
        const void* fn = (const void*)k_quant_mx<true, true>;
        k_quant_mx<true, true><<<grid_for(fn), kQuantThreads, 0, stream>>>(
            xp, rows_cap, cols, splits, G, row_data, row_scale, col_data, col_scale, status);
    } else if (row_data) {
        const void* fn = (const void*)k_quant_mx<true, false>;
        k_quant_mx<true, false><<<grid_for(fn), kQuantThreads, 0, stream>>>(
            xp, rows_cap, cols, splits, G, row_data, row_scale, col_data, col_scale, status);
    } else {
        const void* fn = (const void*)k_quant_mx<false, true>;
        k_quant_mx<false, true><<<grid_for(fn), kQuantThreads, 0, stream>>>(
            xp, rows_cap, cols, splits, G, row_data, row_scale, col_data, col_scale, status);
    }
    return cudaGetLastError();
}

cudaError_t launch_quant_channel(const void* x, int64_t rows_cap, int64_t cols,
                                 const int32_t* splits, int G, float zero_scale,
                                 uint8_t* col_data, float* col_scale, int32_t* status,
                                 cudaStream_t stream)
{
    const int64_t tiles_bound = (rows_cap / 128) * (cols / 128);
    const int sms = device_info().sm_count;
    const int64_t g = (int64_t)sms * blocks_per_sm_for((const void*)k_quant_ch, kQuantThreads);
    const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(g, tiles_bound));
    k_quant_ch<<<grid, kQuantThreads, 0, stream>>>(static_cast<const uint16_t*>(x), rows_cap, cols,
                                                   splits, G, zero_scale, col_data, col_scale,
                                                   status);
    return cudaGetLastError();
}

}  // namespace gq
