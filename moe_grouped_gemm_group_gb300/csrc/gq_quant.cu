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
// group by group).  k_quant_mx runs 16 consumer warps and one producer warp
// that feeds a ring of input tiles by TMA.  Consumer warp (rb, cb) owns the
// 32 x 32 sub-block rows [32 rb, 32 rb + 32) x columns [32 cb, 32 cb + 32);
// lane l holds row 32 rb + l of it in 16 registers (32 bf16).  A rowwise
// block is one lane's 32 values (amax in registers); a columnwise block is one
// column of the sub-block (amax by a warp butterfly that leaves column j's
// amax in lane j).  One 128 x 128 tile yields exactly one rowwise and one
// columnwise 512-byte scale atom.  Codes and atoms are staged in swizzled
// shared memory and leave by TMA stores and bulk copies.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "gq_device.cuh"
#include "gq_internal.h"
#include "gq_ptx.cuh"

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

// Four codes (x0's in the low byte) of (x0, x1, x2, x3) scaled by (s0, s1,
// s2, s3): two packed fp32x2 multiplies (round to nearest, subnormals kept;
// the products are exact, powers of two times bf16 values) and two
// conversions.
__device__ __forceinline__ uint32_t scale_cvt4(float x0, float x1, float x2, float x3, float s0, float s1,
                                               float s2, float s3)
{
    const float2 lo = __fmul2_rn(make_float2(x0, x1), make_float2(s0, s1));
    const float2 hi = __fmul2_rn(make_float2(x2, x3), make_float2(s2, s3));
    return (uint32_t)__nv_cvt_float2_to_fp8x2(lo, __NV_SATFINITE, __NV_E4M3) |
           ((uint32_t)__nv_cvt_float2_to_fp8x2(hi, __NV_SATFINITE, __NV_E4M3) << 16);
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
        table[2 * (G + 1) + g] = scale_kind == 0   ? 512 * (cols >> 7) * (int64_t)s_tp[g]
                                 : scale_kind == 2 ? 512 * (cols >> 6) * (int64_t)s_tp[g]
                                                   : 4 * cols * (s_off[g] >> 7);
    }
}

// Shared-memory plan of k_quant_mx: a ring of kQStages input tiles, each a
// 128-row x 128-column bf16 tile loaded by TMA as two 128-byte-swizzled boxes
// of [128 rows][64 columns]; two output staging buffers, each holding the
// tile's rowwise and columnwise codes (128-byte-swizzled [128 rows][128 B])
// and its two 512-byte scale atoms; the column-scale broadcast area;
// barriers; the split scan.
// Ring depth and CTAs per SM (tuning knobs; the defaults are the measured best).
#ifndef GQ_Q_STAGES
#define GQ_Q_STAGES 4
#endif
#ifndef GQ_Q_MINB
#define GQ_Q_MINB 1
#endif
constexpr int kQStages = GQ_Q_STAGES;
constexpr int kQTile = 128 * 128 * 2;
constexpr int kQOut = 128 * 128;                       // one orientation's codes
constexpr int kQStageOut = 2 * kQOut + 1024;           // row codes, col codes, 2 atoms
constexpr int kQConsumers = 512;                       // 16 consumer warps
constexpr int kQThreadsMx = kQConsumers + 32;          // + 1 producer warp
constexpr int kQScanBytes = (GQ_MAX_GROUPS + 1) * 8 + (GQ_MAX_GROUPS + 2) * 4 + 32 * 8 + 32 * 4;
constexpr int kQDsum = 2 * 4 * 128 * 4;                // bias-grad column sums [2][4 row blocks][128]
constexpr int kQSmem = 1024 + kQStages * kQTile + 2 * kQStageOut + 16 * 32 * 4 + 8 * 2 * kQStages + 16 +
                       kQScanBytes + kQDsum;

// A CTA's walk over the tiles t = blockIdx.x + i * gridDim.x, in increasing
// order: row tile rt, column tile ct, the group g that owns rt, and the ring
// stage s with its phase, each advanced incrementally (no division and no
// search per tile).  `g` stays valid while rt < s_tp[G], i.e. while tiles
// remain.
struct QTileWalk {
    int64_t rt, step_rt;
    int ct, step_ct, nct, g, s;
    uint32_t ph;

    __device__ __forceinline__ void init(const int32_t* s_tp, int G, int nct_)
    {
        nct = nct_;
        rt = blockIdx.x / nct;
        ct = (int)(blockIdx.x % nct);
        step_rt = gridDim.x / nct;
        step_ct = (int)(gridDim.x % nct);
        g = rt < s_tp[G] ? group_of_tile(s_tp, G, rt) : G - 1;
        s = 0;
        ph = 0;
    }

    __device__ __forceinline__ void next(const int32_t* s_tp, int G)
    {
        rt += step_rt;
        ct += step_ct;
        if (ct >= nct) {
            ct -= nct;
            ++rt;
        }
        while (g < G - 1 && s_tp[g + 1] <= rt)
            ++g;
        if (++s == kQStages) {
            s = 0;
            ph ^= 1u;
        }
    }
};

// Output tensor maps of k_quant_mx: codes of one orientation as [rows, cols]
// uint8 with 128-byte swizzle, boxes of 128 columns x 128 rows (whole tiles)
// and 128 columns x 32 rows (the live part of a group's last tile).
struct QuantOutMaps {
    CUtensorMap row128, row32, col128, col32;
};

// DBIAS: also the bias gradient's per-tile column sums of the live rows,
// written to dpart[global row tile][cols] (fp32, fixed summation order).
template <bool ROW, bool COL, bool DBIAS>
__global__ void __launch_bounds__(kQThreadsMx, GQ_Q_MINB)
k_quant_mx(const __grid_constant__ CUtensorMap tma_x, const __grid_constant__ QuantOutMaps om,
           int64_t rows_cap, int64_t cols, const int32_t* __restrict__ splits, int G,
           uint8_t* __restrict__ row_scale, uint8_t* __restrict__ col_scale,
           float* __restrict__ dpart, int32_t* __restrict__ status)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint8_t* tiles = base;
    uint8_t* outs = tiles + kQStages * kQTile;                       // [2][kQStageOut]
    float* s_inv = reinterpret_cast<float*>(outs + 2 * kQStageOut);  // [16 warps][32] column 2^-e
    uint64_t* full = reinterpret_cast<uint64_t*>(s_inv + 16 * 32);
    uint64_t* empty = full + kQStages;
    volatile int* abort = reinterpret_cast<volatile int*>(empty + kQStages);
    int64_t* s_off = reinterpret_cast<int64_t*>(empty + kQStages + 2);
    int32_t* s_tp = reinterpret_cast<int32_t*>(s_off + GQ_MAX_GROUPS + 1);
    int64_t* s_w64 = reinterpret_cast<int64_t*>(s_tp + GQ_MAX_GROUPS + 2);
    int32_t* s_w32 = reinterpret_cast<int32_t*>(s_w64 + 32);
    float* s_dsum = reinterpret_cast<float*>(s_w32 + 32);               // [2][4][128]

    if (load_status(status) != 0)
        return;
    const int err = block_scan_splits(splits, G, rows_cap, 32, s_off, s_tp, s_w64, s_w32);
    if (err) {
        if (threadIdx.x == 0)
            set_status(status, err);
        return;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < kQStages; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], kQConsumers / 32);
        }
        *abort = 0;
        ptx::fence_barrier_init();
    }
    __syncthreads();

    const int nct = (int)(cols >> 7);
    const int64_t total = (int64_t)s_tp[G] * nct;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp == kQConsumers / 32) {
        // ------------------------------------------------------ producer --
        if (lane == 0) {
            ptx::prefetch_tmap(&tma_x);
            int64_t it = 0;
            QTileWalk wk;
            wk.init(s_tp, G, nct);
            for (int64_t t = blockIdx.x; t < total && !*abort; t += gridDim.x, ++it, wk.next(s_tp, G)) {
                const int s = wk.s;
                const uint32_t ph = wk.ph;
                if (!ptx::mbar_wait(&empty[s], ph ^ 1u, abort, status))
                    break;
                const int64_t rt = wk.rt;
                const int ct = wk.ct;
                const int g = wk.g;
                const int32_t row0 = (int32_t)(s_off[g] + 128 * (rt - s_tp[g]));
                ptx::mbar_arrive_expect_tx(&full[s], kQTile);
                ptx::tma_load_2d(tiles + s * kQTile, &tma_x, &full[s], ct * 128, row0);
                ptx::tma_load_2d(tiles + s * kQTile + kQTile / 2, &tma_x, &full[s], ct * 128 + 64, row0);
            }
            // every issued load lands before the CTA leaves
            volatile int no_abort = 0;
            for (int64_t q = it - kQStages < 0 ? 0 : it - kQStages; q < it; ++q)
                if (!ptx::mbar_wait(&full[q % kQStages], (uint32_t)((q / kQStages) & 1), &no_abort, status))
                    break;
        }
        return;
    }

    // ---------------------------------------------------------- consumers --
    // Each tile's codes and scale atoms are staged in shared memory (double
    // buffered) and leave as whole 128-byte lines: TMA stores for the codes,
    // bulk copies for the atoms, all issued by consumer thread 0 after the
    // consumers' barrier.  Before that barrier thread 0 waits until the
    // previous tile's stores have read their buffer, which frees the buffer
    // the next tile writes.
    const int rb = warp >> 2, cb = warp & 3;
    const uint32_t r_in_tile = 32 * rb + lane;
    const bool lead = threadIdx.x == 0;
    int64_t it = 0;
    QTileWalk wk;
    wk.init(s_tp, G, nct);
    for (int64_t t = blockIdx.x; t < total; t += gridDim.x, ++it, wk.next(s_tp, G)) {
        const int s = wk.s;
        const uint32_t ph = wk.ph;
        const int64_t rt = wk.rt;
        const int ct = wk.ct;
        const int g = wk.g;
        const int64_t lt = rt - s_tp[g];
        const int64_t m = s_off[g + 1] - s_off[g];
        const int rows_here = (int)min((int64_t)128, m - 128 * lt);   // a multiple of 32
        const bool active = 32 * rb < rows_here;                     // uniform per warp
        uint8_t* ob = outs + (it & 1) * kQStageOut;
        const uint32_t rd_box = ptx::smem_addr(ob), cd_box = ptx::smem_addr(ob + kQOut);
        uint8_t* atoms = ob + 2 * kQOut;                                 // [row 512 | col 512]

        const bool ok = ptx::mbar_wait(&full[s], ph, abort, status);
        uint32_t v[16];
        if (ok) {
            // row r_in_tile, columns 32 cb .. 32 cb + 31: box cb / 2, chunks 4 (cb % 2) + i
            const uint32_t box = ptx::smem_addr(tiles + s * kQTile + (cb >> 1) * (kQTile / 2));
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 u = ptx::lds128(box + ptx::swz128(r_in_tile, 4 * (cb & 1) + i));
                v[4 * i + 0] = u.x;
                v[4 * i + 1] = u.y;
                v[4 * i + 2] = u.z;
                v[4 * i + 3] = u.w;
            }
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive(&empty[s]);
        }
        uint32_t rbyte = 0, cbyte = 0;
        float csum = 0.f;                                // bias grad: this lane's column over the warp's rows
        if (ok && active) {
            // magnitudes (sign bits cleared), two bf16 per register
            uint32_t mg[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                mg[i] = v[i] & 0x7fff7fffu;
            float xf[32];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                xf[2 * i] = bf16_lo(v[i]);
                xf[2 * i + 1] = bf16_hi(v[i]);
            }
            if (ROW) {
                uint32_t mx = mg[0];
#pragma unroll
                for (int i = 1; i < 16; ++i)
                    mx = __vmaxu2(mx, mg[i]);
                rbyte = e8m0_byte(max(mx & 0xffffu, mx >> 16));
                const float sc = inv_scale(rbyte);
                uint32_t w[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    w[i] = scale_cvt4(xf[4 * i], xf[4 * i + 1], xf[4 * i + 2], xf[4 * i + 3], sc, sc, sc, sc);
                // 32 codes = 16-byte chunks 2 cb and 2 cb + 1 of the row
                ptx::sts128(rd_box + ptx::swz128(r_in_tile, 2 * cb), make_uint4(w[0], w[1], w[2], w[3]));
                ptx::sts128(rd_box + ptx::swz128(r_in_tile, 2 * cb + 1), make_uint4(w[4], w[5], w[6], w[7]));
            }
            if (COL) {
                // Transpose-max across the warp: after exchanging half of the
                // remaining columns with lane ^ 16, ^ 8, ^ 4, ^ 2, ^ 1, lane j
                // holds the max over the 32 rows of column j.
                uint32_t red[8];
                const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2, b0 = lane & 1;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t send = b4 ? mg[i] : mg[i + 8];
                    const uint32_t keep = b4 ? mg[i + 8] : mg[i];
                    red[i] = __vmaxu2(keep, __shfl_xor_sync(0xffffffffu, send, 16));
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t send = b3 ? red[i] : red[i + 4];
                    const uint32_t keep = b3 ? red[i + 4] : red[i];
                    red[i] = __vmaxu2(keep, __shfl_xor_sync(0xffffffffu, send, 8));
                }
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const uint32_t send = b2 ? red[i] : red[i + 2];
                    const uint32_t keep = b2 ? red[i + 2] : red[i];
                    red[i] = __vmaxu2(keep, __shfl_xor_sync(0xffffffffu, send, 4));
                }
                {
                    const uint32_t send = b1 ? red[0] : red[1];
                    const uint32_t keep = b1 ? red[1] : red[0];
                    red[0] = __vmaxu2(keep, __shfl_xor_sync(0xffffffffu, send, 2));
                }
                const uint32_t pairmax = __vmaxu2(red[0], __shfl_xor_sync(0xffffffffu, red[0], 1));
                cbyte = e8m0_byte(b0 ? (pairmax >> 16) : (pairmax & 0xffffu));
                // broadcast the 32 column scales through shared memory
                float* inv = s_inv + warp * 32;
                inv[lane] = inv_scale(cbyte);
                __syncwarp();
                float sc[32];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 f = reinterpret_cast<const float4*>(inv)[i];
                    sc[4 * i] = f.x;
                    sc[4 * i + 1] = f.y;
                    sc[4 * i + 2] = f.z;
                    sc[4 * i + 3] = f.w;
                }
                __syncwarp();
                uint32_t w[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    w[i] = scale_cvt4(xf[4 * i], xf[4 * i + 1], xf[4 * i + 2], xf[4 * i + 3], sc[4 * i],
                                      sc[4 * i + 1], sc[4 * i + 2], sc[4 * i + 3]);
                ptx::sts128(cd_box + ptx::swz128(r_in_tile, 2 * cb), make_uint4(w[0], w[1], w[2], w[3]));
                ptx::sts128(cd_box + ptx::swz128(r_in_tile, 2 * cb + 1), make_uint4(w[4], w[5], w[6], w[7]));
            }
            if (DBIAS) {
                // Transposed butterfly: after exchanging half of the remaining
                // columns with lane ^ 16, ^ 8, ^ 4, ^ 2, ^ 1 (adding what comes
                // back), lane j holds the sum of column j over the 32 rows, in
                // an order fixed by the lane bits.
                const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2, b0 = lane & 1;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float send = b4 ? xf[i] : xf[i + 16];
                    const float keep = b4 ? xf[i + 16] : xf[i];
                    xf[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float send = b3 ? xf[i] : xf[i + 8];
                    const float keep = b3 ? xf[i + 8] : xf[i];
                    xf[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float send = b2 ? xf[i] : xf[i + 4];
                    const float keep = b2 ? xf[i + 4] : xf[i];
                    xf[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
                }
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const float send = b1 ? xf[i] : xf[i + 2];
                    const float keep = b1 ? xf[i + 2] : xf[i];
                    xf[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
                }
                {
                    const float send = b0 ? xf[0] : xf[1];
                    const float keep = b0 ? xf[1] : xf[0];
                    csum = keep + __shfl_xor_sync(0xffffffffu, send, 1);
                }
            }
        }
        if (DBIAS)
            s_dsum[(it & 1) * 512 + rb * 128 + cb * 32 + lane] = csum;
        // Scale atoms: rowwise (row 32 rb + lane, block cb), columnwise
        // (channel 32 cb + lane, 32-row block rb); inactive warps write the
        // zero entries of a partial last tile.  16 warps cover each atom once.
        atoms[lane * 16 + rb * 4 + cb] = (uint8_t)rbyte;
        atoms[512 + lane * 16 + cb * 4 + rb] = (uint8_t)cbyte;
        ptx::fence_proxy_async_smem();
        if (lead)
            ptx::bulk_wait_read_all();      // the previous tile's stores have read their buffer
        if (ptx::named_barrier_or(1, kQConsumers, !ok))
            break;
        if (DBIAS && threadIdx.x < 128) {
            // the tile's column sums: its four 32-row blocks, added in order
            const float* d = s_dsum + (it & 1) * 512 + threadIdx.x;
            dpart[(s_tp[g] + lt) * cols + ct * 128 + threadIdx.x] = ((d[0] + d[128]) + d[256]) + d[384];
        }
        if (lead) {
            const int32_t row0 = (int32_t)(s_off[g] + 128 * lt);
            const int32_t x = ct * 128;
            const int64_t sbase = 512 * (int64_t)nct * s_tp[g];
            if (ROW) {
                if (rows_here == 128)
                    ptx::tma_store_2d(&om.row128, ob, x, row0);
                else
                    for (int k = 0; k < rows_here / 32; ++k)
                        ptx::tma_store_2d(&om.row32, ob + k * 32 * 128, x, row0 + 32 * k);
                ptx::bulk_store(row_scale + sbase + (lt * nct + ct) * 512, atoms, 512);
            }
            if (COL) {
                if (rows_here == 128)
                    ptx::tma_store_2d(&om.col128, ob + kQOut, x, row0);
                else
                    for (int k = 0; k < rows_here / 32; ++k)
                        ptx::tma_store_2d(&om.col32, ob + kQOut + k * 32 * 128, x, row0 + 32 * k);
                const int64_t T = s_tp[g + 1] - s_tp[g];
                ptx::bulk_store(col_scale + sbase + ((int64_t)ct * T + lt) * 512, atoms + 512, 512);
            }
            ptx::bulk_commit_group();
        }
    }
    if (lead)
        ptx::bulk_wait_all();
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

// Bias gradient from the per-tile column sums: db[g][c] = sum over the
// group's row tiles, in tile order, of dpart[tile][c]; empty groups (and
// L == 0) get 0.
__global__ void __launch_bounds__(256)
k_dbias_reduce(const int32_t* __restrict__ splits, int G, int64_t rows_cap, int64_t cols,
               const float* __restrict__ dpart, float* __restrict__ db, int32_t* __restrict__ status)
{
    __shared__ int64_t s_off[GQ_MAX_GROUPS + 1];
    __shared__ int32_t s_tp[GQ_MAX_GROUPS + 1];
    __shared__ int64_t s_w64[32];
    __shared__ int32_t s_w32[32];
    if (load_status(status) != 0)
        return;
    const int err = block_scan_splits(splits, G, rows_cap, 32, s_off, s_tp, s_w64, s_w32);
    if (err) {
        if (threadIdx.x == 0)
            set_status(status, err);
        return;
    }
    const int64_t n = (int64_t)G * cols;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int g = (int)(i / cols);
        const int64_t c = i - (int64_t)g * cols;
        float acc = 0.f;
        for (int64_t t = s_tp[g]; t < s_tp[g + 1]; ++t)
            acc += dpart[t * cols + c];
        db[i] = acc;
    }
}

int blocks_per_sm_for(const void* fn, int threads)
{
    int n = 1;
    if (prepare_kernel(fn, 0, threads, &n) != cudaSuccess)
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
                            uint8_t* col_scale, int32_t* status, cudaStream_t stream, float* dpart)
{
    CUtensorMap map;
    QuantOutMaps om;
    if (!make_tensor_map_2d(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, rows_cap, cols, 64, 128))
        return cudaErrorInvalidValue;
    // unused orientations get a valid (never used) map
    const uint8_t* rd = row_data ? row_data : col_data;
    const uint8_t* cd = col_data ? col_data : row_data;
    if (!make_map_u8(&om.row128, rd, rows_cap, cols, 128) || !make_map_u8(&om.row32, rd, rows_cap, cols, 32) ||
        !make_map_u8(&om.col128, cd, rows_cap, cols, 128) || !make_map_u8(&om.col32, cd, rows_cap, cols, 32))
        return cudaErrorInvalidValue;
    const int64_t tiles_bound = ((rows_cap + 127) / 128 + G) * (cols / 128);
    const int sms = device_info().sm_count;
    auto go = [&](auto kernel) {
        int per_sm = 1;
        const cudaError_t e = prepare_kernel(reinterpret_cast<const void*>(kernel), kQSmem, kQThreadsMx, &per_sm);
        if (e != cudaSuccess)
            return e;
        const int64_t grid = std::max<int64_t>(1, std::min<int64_t>((int64_t)sms * per_sm, tiles_bound));
        kernel<<<(unsigned)grid, kQThreadsMx, kQSmem, stream>>>(map, om, rows_cap, cols, splits, G, row_scale,
                                                                col_scale, dpart, status);
        return cudaGetLastError();
    };
    if (dpart) {
        if (row_data && col_data)
            return go(k_quant_mx<true, true, true>);
        if (row_data)
            return go(k_quant_mx<true, false, true>);
        return go(k_quant_mx<false, true, true>);
    }
    if (row_data && col_data)
        return go(k_quant_mx<true, true, false>);
    if (row_data)
        return go(k_quant_mx<true, false, false>);
    return go(k_quant_mx<false, true, false>);
}

cudaError_t launch_dbias_reduce(const int32_t* splits, int G, int64_t rows_cap, int64_t cols,
                                const float* dpart, float* db, int32_t* status, cudaStream_t stream)
{
    const int64_t n = (int64_t)G * cols;
    const int64_t cap = (int64_t)device_info().sm_count * 4;
    const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>((n + 255) / 256, cap));
    k_dbias_reduce<<<grid, 256, 0, stream>>>(splits, G, rows_cap, cols, dpart, db, status);
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
