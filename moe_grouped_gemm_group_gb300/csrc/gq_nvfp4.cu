// NVFP4 grouped quantiser and grouped GEMMs on the 5th-generation tensor core
// (tcgen05, sm_103a).
//
// The pages name NVFP4 as a second quantiser of the same grouped code paths
// (TransformerEngine PR 3224) without defining it; this is the public NVFP4
// format:
//   codes   FP4 E2M1, two a byte, the element with the even index in the low
//           nibble;
//   blocks  16 consecutive elements along the contraction axis, one E4M3
//           scale byte each;
//   groups  one fp32 second-level scale S_g = 2688 / amax_g (2688 = 448 * 6),
//           amax_g the largest |x| over the group's live rows; S_g = 1 when
//           amax_g == 0, clamped to FLT_MAX.
// Per block, fp32 op by op: s = (amax_b / 6) * S_g; sf = e4m3(s) (nearest
// even, saturating); m = S_g / sf (0 when sf == 0, clamped to FLT_MAX);
// codes = e2m1(x * m) (nearest even, saturating).  A code stands for
// e2m1 * sf / S_g; the GEMMs apply sf inside the MMA and 1 / (S_a S_b) to
// the fp32 accumulator.
//
// Layouts.  The tensor core takes packed 4-bit operands K-major only, so
// every operand is stored with its contraction axis contiguous:
//   rowwise codes     [rows_cap, cols/2]
//   columnwise codes  [cols, rows_cap/2]: row c holds column c's codes,
//                     quantised in blocks of 16 rows
//   scale atoms       the 512-byte [32][4][4] atom of the MX layout with 16
//                     elements a scale, so an atom covers 128 rows (or
//                     channels) x 64 elements; group g's region starts at
//                     byte 512 * (cols/64) * (T_0 + ... + T_{g-1}),
//                     T_h = ceil(m_h / 128); rowwise atoms are ordered
//                     [128-row tile][64-column block], columnwise atoms
//                     [128-column tile][64-row block] with the group's 2 T_g
//                     row blocks the inner stride.  Entries that cover no
//                     live row are 0.
//
//   fprop  Y_g  = X_g W_g^T   A = X rowwise, B = W_g rowwise
//   dgrad  dX_g = dY_g W_g    A = dY rowwise, B = W columnwise ([k, G n/2])
//   wgrad  dW_g = dY_g^T X_g  A = dY columnwise, B = X columnwise, over the
//                             group's live rows: a group's last 256-row
//                             k-tile issues only the MMAs of its live 64-row
//                             blocks, and inside a half-live block the
//                             scales of the dead 16-row blocks are 0, so
//                             rows past the group never reach the result.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cfloat>
#include <cstdint>

#include "gq_internal.h"
#include "gq_ptx.cuh"

namespace gq {
namespace {

// ------------------------------------------------------------------------ //
// Element and block arithmetic                                              //
// ------------------------------------------------------------------------ //

__device__ __forceinline__ float nv_global_scale(float amax)
{
    if (amax == 0.f)
        return 1.f;
    return fminf(__fdiv_rn(2688.f, amax), FLT_MAX);
}

// 1 / (S_a S_b), the factor that turns the accumulator of E2M1 x E4M3-scaled
// products into the product of the dequantised operands.
__device__ __forceinline__ float nv_alpha(float amax_a, float amax_b)
{
    return __fmul_rn(__frcp_rn(nv_global_scale(amax_a)), __frcp_rn(nv_global_scale(amax_b)));
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// amax / 6 rounded to nearest even for a bf16 amax, without a division:
// q1 = amax * RN(1/6), then one correction step q1 + (amax - 6 q1) * RN(1/6)
// with fused multiply-adds (Markstein's correction of a reciprocal product).
// Checked against the correctly rounded quotient for every finite bf16
// magnitude, subnormals included.
__device__ __forceinline__ float div6_bf16(float amax)
{
    const float y = 0x1.555556p-3f;               // RN(1/6)
    const float q1 = __fmul_rn(amax, y);
    const float r = __fmaf_rn(-q1, 6.f, amax);
    return __fmaf_rn(r, y, q1);
}

// The quantiser's per-tile table m[sf] = S_g / sf (0 for sf = 0, clamped to
// FLT_MAX) over the 127 non-negative finite E4M3 bytes, so that a block
// needs no division.
__device__ __forceinline__ float nv_encode_mult(float S, uint32_t sf)
{
    if (sf == 0)
        return 0.f;
    const float d = __half2float(__half(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)sf, __NV_E4M3)));
    return fminf(__fdiv_rn(S, d), FLT_MAX);
}

// Eight values as E2M1 codes in one word, element 2i of the pairs in nibble
// 2i (round to nearest even, saturating): the converting instruction puts its
// first source in the high nibble of its byte.
__device__ __forceinline__ uint32_t e2m1x8(float2 a, float2 b, float2 c, float2 d)
{
    uint32_t w;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(w)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y), "f"(d.x), "f"(d.y));
    return w;
}

// Halfwise maximum of two bf16 pairs (non-negative values: exact).
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b)
{
    const __nv_bfloat162 r = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&a),
                                     *reinterpret_cast<const __nv_bfloat162*>(&b));
    return *reinterpret_cast<const uint32_t*>(&r);
}

// One block of 16 values whose amax (an fp32 widened from bf16) is known:
// its E4M3 scale byte and its 16 codes (element i in nibble i of the 64-bit
// word, i.e. byte i / 2, low nibble for even i).
__device__ __forceinline__ uint32_t nv_encode16_t(const float (&x)[16], float amax, float S, const float* mtab,
                                                  uint2& codes)
{
    const float s = __fmul_rn(div6_bf16(amax), S);
    const uint32_t sf = __nv_cvt_float_to_fp8(s, __NV_SATFINITE, __NV_E4M3);
    const float m = mtab[sf];
    float2 p[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        p[i] = __fmul2_rn(make_float2(x[2 * i], x[2 * i + 1]), make_float2(m, m));
    codes = make_uint2(e2m1x8(p[0], p[1], p[2], p[3]), e2m1x8(p[4], p[5], p[6], p[7]));
    return sf;
}

// Largest bf16 magnitude among the 2 x 4 halves of two 16-byte words, as fp32.
__device__ __forceinline__ float amax16_bf16(const uint4& a, const uint4& b)
{
    constexpr uint32_t M = 0x7fff7fffu;
    uint32_t m = bmax2(bmax2(a.x & M, a.y & M), bmax2(a.z & M, a.w & M));
    m = bmax2(m, bmax2(bmax2(b.x & M, b.y & M), bmax2(b.z & M, b.w & M)));
    return __uint_as_float(max(m & 0xffffu, m >> 16) << 16);
}

// Largest g in [0, G) with s_off[g] <= r: the group that owns live row r
// (an empty group shares its offset with the next group and loses to it).
__device__ __forceinline__ int group_of_row(const int32_t* s_off, int G, int64_t r)
{
    int lo = 0, hi = G - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)s_off[mid] <= r)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

constexpr int kScanBytes = (GQ_MAX_GROUPS + 1) * 4 + (GQ_MAX_GROUPS + 2) * 4 + 8 + 32 * 8 + 64 * 4;

struct Scan {
    int32_t* off;
    int32_t* tp;
    int64_t* w64;
    int32_t* w32;
};

__device__ __forceinline__ Scan carve_scan(uint8_t* p)
{
    Scan s;
    s.off = reinterpret_cast<int32_t*>(p);
    s.tp = s.off + GQ_MAX_GROUPS + 1;
    s.w64 = reinterpret_cast<int64_t*>((reinterpret_cast<uintptr_t>(s.tp + GQ_MAX_GROUPS + 2) + 7) & ~uintptr_t(7));
    s.w32 = reinterpret_cast<int32_t*>(s.w64 + 32);
    return s;
}

// ------------------------------------------------------------------------ //
// Quantiser                                                                 //
// ------------------------------------------------------------------------ //

// Split scan (errors go to the status word) and amax[g] = 0.  One CTA.
__global__ void __launch_bounds__(256) k_nv_prepare(const int32_t* splits, int G, int64_t rows_cap,
                                                    float* amax, int32_t* status)
{
    __shared__ __align__(16) uint8_t scan_raw[kScanBytes];
    if (load_status(status) != 0)
        return;
    const Scan sc = carve_scan(scan_raw);
    const int err = block_scan_splits(splits, G, rows_cap, 32, sc.off, sc.tp, sc.w64, sc.w32);
    if (err) {
        if (threadIdx.x == 0)
            set_status(status, err);
        return;
    }
    for (int g = threadIdx.x; g < G; g += blockDim.x)
        amax[g] = 0.f;
}

// amax[g] = largest |x| over group g's live rows.  Work unit: a 32-row block
// (inside one group: splits are multiples of 32) x all columns; the CTA's
// maximum of the bf16 magnitudes (compared as integers) goes to amax[g] by
// an atomic max on the fp32 bit pattern.
__global__ void __launch_bounds__(256) k_nv_amax(const uint16_t* __restrict__ x, int64_t rows_cap, int64_t cols,
                                                 const int32_t* splits, int G, float* amax, int32_t* status)
{
    __shared__ __align__(16) uint8_t scan_raw[kScanBytes];
    __shared__ uint32_t s_red[8];
    if (load_status(status) != 0)
        return;
    const Scan sc = carve_scan(scan_raw);
    if (block_scan_splits(splits, G, rows_cap, 32, sc.off, sc.tp, sc.w64, sc.w32))
        return;                                  // reported by k_nv_prepare
    const int64_t nblk = (int64_t)sc.off[G] / 32;
    const int64_t chunks = 32 * cols / 8;        // 16-byte chunks of a 32-row block
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int64_t blk = blockIdx.x; blk < nblk; blk += gridDim.x) {
        const uint4* src = reinterpret_cast<const uint4*>(x + 32 * blk * cols);
        uint32_t mx = 0;
#pragma unroll 8
        for (int64_t i = tid; i < chunks; i += 256) {
            const uint4 v = __ldg(src + i);
            mx = max(mx, max(max(v.x & 0x7fffu, v.x >> 16 & 0x7fffu), max(v.y & 0x7fffu, v.y >> 16 & 0x7fffu)));
            mx = max(mx, max(max(v.z & 0x7fffu, v.z >> 16 & 0x7fffu), max(v.w & 0x7fffu, v.w >> 16 & 0x7fffu)));
        }
#pragma unroll
        for (int d = 16; d > 0; d >>= 1)
            mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, d));
        if (lane == 0)
            s_red[warp] = mx;
        __syncthreads();
        if (tid == 0) {
            uint32_t m = s_red[0];
            for (int w = 1; w < 8; ++w)
                m = max(m, s_red[w]);
            const int g = group_of_row(sc.off, G, 32 * blk);
            if (m != 0)
                atomicMax(reinterpret_cast<unsigned int*>(amax + g), m << 16);
        }
        __syncthreads();
    }
}

// Shared-memory plan of k_nv_quant: a ring of kNqStages bf16 input tiles
// (128 rows x 128 columns, two 128-byte-swizzled TMA boxes of [128 rows][64
// columns]) with the tile's table m[sf]; two output staging buffers (the
// columnwise codes and the tile's four atoms); the ring's barriers; the
// split scan.
constexpr int kNqStages = 5;
constexpr int kNqTile = 128 * 128 * 2;
constexpr int kNqConsumers = 512;                     // 16 consumer warps
constexpr int kNqThreads = kNqConsumers + 32;         // + 1 producer warp
// columnwise code staging: [16-row block b][column c] x 8 bytes, rows of
// 1056 bytes (1024 + 32 of padding: the read-out's column groups of
// different blocks then fall on different banks)
constexpr int kNqStagePitch = 1024 + 32;
constexpr int kNqOut = 8 * kNqStagePitch + 4 * 512;
constexpr int kNqSmem = 1024 + kNqStages * kNqTile + kNqStages * 512 + 2 * kNqOut + kNqStages * 32 +
                        2 * 8 * kNqStages + 16 + kScanBytes;

// Tile order of the quantiser (tuning knob): tiles are walked in bands of
// GQ_NQ_BAND row tiles, row tile fastest inside a band, so that the CTAs
// working at the same time cover a few row tiles x many column tiles: the
// rowwise codes (64 bytes a row per tile) and the transposed columnwise codes
// (64 bytes a column per tile) both leave in runs of adjacent segments.
#ifndef GQ_NQ_BAND
#define GQ_NQ_BAND 8
#endif
constexpr int kNqBand = GQ_NQ_BAND;

// One 128 x 128 tile of one group (the group's own 128-row tiles, so one S_g
// per tile).  32 bytes: the producer decodes each tile once and hands it to
// the consumers with the stage.
struct NqTile {
    int g;
    int rows;          // live rows (a multiple of 32)
    int64_t mt, ct;    // row tile in the group, column tile
    int64_t row0;      // first buffer row
};
static_assert(sizeof(NqTile) == 32, "tile record size");

__device__ __forceinline__ NqTile nq_tile(const Scan& sc, int G, int64_t nct, int64_t t)
{
    NqTile q;
    const int64_t band = t / (kNqBand * nct);
    const int64_t rt0 = band * kNqBand;
    const int64_t nb = min((int64_t)kNqBand, (int64_t)sc.tp[G] - rt0);     // row tiles of this band
    const int64_t u = t - band * kNqBand * nct;
    const int64_t rt = rt0 + u % nb;
    q.ct = u / nb;
    q.g = group_of_tile(sc.tp, G, rt);
    q.mt = rt - sc.tp[q.g];
    q.rows = (int)min((int64_t)128, (int64_t)(sc.off[q.g + 1] - sc.off[q.g]) - 128 * q.mt);
    q.row0 = sc.off[q.g] + 128 * q.mt;
    return q;
}

// Byte address of bf16 element (r, 4 p') of a 128-byte-swizzled tile, for the
// 4-byte column pair p (columns 2 p, 2 p + 1) of row r.
__device__ __forceinline__ uint32_t nq_pair_addr(uint32_t tile, int r, int p)
{
    const int h = p >> 5, j = (p & 31) >> 2;
    return tile + h * 16384 + r * 128 + ((j ^ (r & 7)) << 4) + 4 * (p & 3);
}

// Warp roles: warp 16 is the producer -- per tile it waits for a free stage,
// writes the tile's m[sf] table (its 32 lanes), and lane 0 issues the TMA
// loads of the tile's live rows (whole 128-row boxes, or 32-row boxes for a
// group's last tile, so rows past the live total are never read).  Warps
// 0..15 are the consumers: rowwise items (row, 16-column block) send their 8
// code bytes straight to global memory; columnwise items (column pair,
// 16-row block) stage theirs; one named barrier per tile, after which the
// stage goes back to the producer and the staged codes and atoms leave as
// 16-byte chunks (double-buffered staging, so one barrier suffices).
template <bool ROW, bool COL>
__global__ void __launch_bounds__(kNqThreads, 1)
k_nv_quant(const __grid_constant__ CUtensorMap map128, const __grid_constant__ CUtensorMap map32, int64_t rows_cap,
           int64_t cols, const int32_t* splits, int G, const float* __restrict__ amax, uint8_t* row_data,
           uint8_t* row_scale, uint8_t* col_data, uint8_t* col_scale, int32_t* status)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* mtabs = reinterpret_cast<float*>(tiles + kNqStages * kNqTile);     // [stage][128]
    uint8_t* outs = reinterpret_cast<uint8_t*>(mtabs + kNqStages * 128);     // [2][ccodes | atoms]
    NqTile* infos = reinterpret_cast<NqTile*>(outs + 2 * kNqOut);            // [stage]
    uint64_t* full = reinterpret_cast<uint64_t*>(infos + kNqStages);
    uint64_t* empty = full + kNqStages;
    volatile int* abort = reinterpret_cast<volatile int*>(empty + kNqStages);
    if (load_status(status) != 0)
        return;
    const Scan sc = carve_scan(reinterpret_cast<uint8_t*>(empty + kNqStages) + 16);
    if (block_scan_splits(splits, G, rows_cap, 32, sc.off, sc.tp, sc.w64, sc.w32))
        return;                                  // reported by k_nv_prepare
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < kNqStages; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        *abort = 0;
        ptx::fence_barrier_init();
    }
    __syncthreads();
    const int64_t nct = cols / 128;
    const int64_t ntiles = (int64_t)sc.tp[G] * nct;

    if (warp == kNqConsumers / 32) {
        // ------------------------------------------------------- producer --
        if (lane == 0) {
            ptx::prefetch_tmap(&map128);
            ptx::prefetch_tmap(&map32);
        }
        int s = 0;
        uint32_t ph = 0;
        int64_t issued = 0;
        for (int64_t t = blockIdx.x; t < ntiles && !*abort; t += gridDim.x) {
            if (!ptx::mbar_wait_warp(&empty[s], ph ^ 1u, abort, status))
                break;
            const NqTile q = nq_tile(sc, G, nct, t);
            const float S = nv_global_scale(__ldg(amax + q.g));
            // entry 127 (an E4M3 NaN byte, never a scale) carries S_g itself
            for (int e = lane; e < 128; e += 32)
                mtabs[s * 128 + e] = e == 127 ? S : nv_encode_mult(S, (uint32_t)e);
            if (lane == 0)
                infos[s] = q;
            __syncwarp();
            if (lane == 0) {
                uint8_t* dst = tiles + s * kNqTile;
                ptx::mbar_arrive_expect_tx(&full[s], (uint32_t)(q.rows * 256));
                const int32_t x0 = (int32_t)(q.ct * 128);
                if (q.rows == 128) {
                    ptx::tma_load_2d(dst, &map128, &full[s], x0, (int32_t)q.row0);
                    ptx::tma_load_2d(dst + 16384, &map128, &full[s], x0 + 64, (int32_t)q.row0);
                } else {
                    for (int r = 0; r < q.rows; r += 32) {
                        ptx::tma_load_2d(dst + r * 128, &map32, &full[s], x0, (int32_t)(q.row0 + r));
                        ptx::tma_load_2d(dst + 16384 + r * 128, &map32, &full[s], x0 + 64, (int32_t)(q.row0 + r));
                    }
                }
            }
            ++issued;
            if (++s == kNqStages) {
                s = 0;
                ph ^= 1u;
            }
        }
        if (lane == 0) {
            // loads in flight after an abort land before the CTA leaves
            volatile int no_abort = 0;
            for (int64_t k = issued - kNqStages < 0 ? 0 : issued - kNqStages; k < issued; ++k)
                if (!ptx::mbar_wait(&full[k % kNqStages], (uint32_t)((k / kNqStages) & 1), &no_abort, status))
                    break;
        }
        return;
    }

    // ---------------------------------------------------------- consumers --
    int s = 0, ob = 0;
    uint32_t ph = 0;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const bool ok = ptx::mbar_wait_warp(&full[s], ph, abort, status);
        if (ptx::named_barrier_or(1, kNqConsumers, !ok))
            break;
        const NqTile q = infos[s];
        const int rows = q.rows;
        const uint32_t tile = ptx::smem_addr(tiles + s * kNqTile);
        const float* mtab = mtabs + s * 128;
        const float S = mtab[127];
        uint8_t* ccodes = outs + ob * kNqOut;
        uint8_t* atoms = ccodes + 8 * kNqStagePitch;
        if (ROW) {
            for (int i = tid; i < 128 * 8; i += kNqConsumers) {
                // row r, 16-column block jb: a warp takes 8 consecutive rows x 4
                // blocks, so each quarter-warp's 16-byte reads hit 8 different
                // swizzled chunks (no bank conflict)
                const int w = i >> 5, l = i & 31;
                const int r = (w & 15) * 8 + (l & 7), jb = (w >> 4) * 4 + (l >> 3);
                uint32_t sf = 0;
                if (r < rows) {
                    const int h = jb >> 2, j = 2 * (jb & 3);
                    const uint32_t rowa = tile + h * 16384 + r * 128;
                    const uint4 a = ptx::lds128(rowa + ((j ^ (r & 7)) << 4));
                    const uint4 b = ptx::lds128(rowa + (((j + 1) ^ (r & 7)) << 4));
                    const float v[16] = {bf16_lo(a.x), bf16_hi(a.x), bf16_lo(a.y), bf16_hi(a.y),
                                         bf16_lo(a.z), bf16_hi(a.z), bf16_lo(a.w), bf16_hi(a.w),
                                         bf16_lo(b.x), bf16_hi(b.x), bf16_lo(b.y), bf16_hi(b.y),
                                         bf16_lo(b.z), bf16_hi(b.z), bf16_lo(b.w), bf16_hi(b.w)};
                    uint2 cw;
                    sf = nv_encode16_t(v, amax16_bf16(a, b), S, mtab, cw);
                    *reinterpret_cast<uint2*>(row_data + (q.row0 + r) * (cols / 2) + q.ct * 64 + jb * 8) = cw;
                }
                atoms[(jb >> 2) * 512 + (r & 31) * 16 + (r >> 5) * 4 + (jb & 3)] = (uint8_t)sf;
            }
        }
        if (COL) {
            const int p = tid & 63, b = tid >> 6;      // column pair, 16-row block (512 items)
            uint32_t sf0 = 0, sf1 = 0;
            if (16 * b < rows) {
                float v0[16], v1[16];
                uint32_t m = 0;
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    uint32_t wd;
                    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(wd) : "r"(nq_pair_addr(tile, 16 * b + k, p)));
                    v0[k] = bf16_lo(wd);
                    v1[k] = bf16_hi(wd);
                    m = bmax2(m, wd & 0x7fff7fffu);
                }
                uint2 c0, c1;
                sf0 = nv_encode16_t(v0, __uint_as_float((m & 0xffffu) << 16), S, mtab, c0);
                sf1 = nv_encode16_t(v1, __uint_as_float(m & 0xffff0000u), S, mtab, c1);
                *reinterpret_cast<uint4*>(ccodes + b * kNqStagePitch + 16 * p) = make_uint4(c0.x, c0.y, c1.x, c1.y);
            }
            const int c = 2 * p;
            atoms[(2 + (b >> 2)) * 512 + (c & 31) * 16 + (c >> 5) * 4 + (b & 3)] = (uint8_t)sf0;
            atoms[(2 + (b >> 2)) * 512 + ((c + 1) & 31) * 16 + ((c + 1) >> 5) * 4 + (b & 3)] = (uint8_t)sf1;
        }
        ptx::named_barrier_or(1, kNqConsumers, 0);
        if (tid == 0)
            ptx::mbar_arrive(&empty[s]);
        const int64_t sb = 512 * (cols / 64) * (int64_t)sc.tp[q.g];
        if (ROW && tid < 64)
            *reinterpret_cast<uint4*>(row_scale + sb + (q.mt * (cols / 64) + 2 * q.ct) * 512 + tid * 16) =
                *reinterpret_cast<const uint4*>(atoms + tid * 16);
        if (COL) {
            const int64_t T = sc.tp[q.g + 1] - sc.tp[q.g];
            const int nch = rows / 32;                 // 16-byte chunks of a column (rows / 2 bytes)
            for (int i = tid; i < 128 * nch; i += kNqConsumers) {
                const int c = i / nch, ch = i - c * nch;  // chunk ch = blocks 2 ch, 2 ch + 1
                const uint2 lo = *reinterpret_cast<const uint2*>(ccodes + (2 * ch) * kNqStagePitch + 8 * c);
                const uint2 hi = *reinterpret_cast<const uint2*>(ccodes + (2 * ch + 1) * kNqStagePitch + 8 * c);
                *reinterpret_cast<uint4*>(col_data + (q.ct * 128 + c) * (rows_cap / 2) + q.row0 / 2 + ch * 16) =
                    make_uint4(lo.x, lo.y, hi.x, hi.y);
            }
            if (tid >= 64 && tid < 128)
                *reinterpret_cast<uint4*>(col_scale + sb + (q.ct * 2 * T + 2 * q.mt) * 512 + (tid - 64) * 16) =
                    *reinterpret_cast<const uint4*>(atoms + 1024 + (tid - 64) * 16);
        }
        ob ^= 1;
        if (++s == kNqStages) {
            s = 0;
            ph ^= 1u;
        }
    }
}

// ------------------------------------------------------------------------ //
// GEMM                                                                      //
// ------------------------------------------------------------------------ //

// D(tmem) (+)= A(smem) * B(smem), E2M1 x E2M1 -> f32, with one UE4M3 scale
// per 16 elements of A and B read from TMEM (4 per row per instruction).
__device__ __forceinline__ void tc_mma_nvf4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                            uint32_t sfb, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X"
        " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)
        : "memory");
}

// Instruction descriptor of kind::mxf4nvf4: E2M1 A and B (format 1 at bits
// 7-9 and 10-12), both K-major, N >> 3 at bit 17, scale type UE4M3 (bit 23
// clear), M >> 4 at bit 24, scale-factor selectors 0.
__host__ __device__ constexpr uint32_t idesc_nvf4(uint32_t m, uint32_t n)
{
    return (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

struct NvArgs {
    const int32_t* splits;
    int G;
    int64_t rows_cap;
    int64_t n, k;
    const uint8_t* sfa;
    const uint8_t* sfb;
    const float* amax_a;
    const float* amax_b;
    void* out;
    int accumulate;
    int32_t* status;
};

template <int KIND>
struct NvShape {
    static constexpr int A_BYTES = 128 * 128;       // 128 rows x 256 codes
    static constexpr int B_BYTES = 256 * 128;       // 256 rows x 256 codes
    static constexpr int SFA_BYTES = 4 * 512;       // one atom per 64-deep MMA
    static constexpr int SFB_BYTES = 8 * 512;       // [128-row half of B][64-deep MMA]
    static constexpr int STAGE = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
    // output boxes: one per epilogue warp (fp32 32 x 32 with the 128-byte
    // swizzle for wgrad, 32 rows x 64 bytes with the 64-byte swizzle else)
    static constexpr int BOX = KIND == NV_WGRAD ? 4096 : 2048;
    static constexpr int OUT_BYTES = 8 * BOX;
    static constexpr int BAR_BYTES = 8 * (2 * 8 + 3) + 16;
    static constexpr int STAGES_FIT = (227 * 1024 - 1024 - OUT_BYTES - kScanBytes - BAR_BYTES) / STAGE;
    static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
    static constexpr int SMEM = 1024 + STAGES * STAGE + OUT_BYTES + BAR_BYTES + kScanBytes;
    static constexpr int THREADS = 128 + 32 * 8;
    // TMEM: accumulator in columns [0, 256); scale atoms of a k-tile (A: 4
    // atoms = 16 columns, B: 8 atoms = 32 columns) in one of 4 slots after it
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t SF_COL = 256;
    static constexpr uint32_t SF_STRIDE = 48;
    static constexpr uint32_t SF_SLOTS = 4;
    static_assert(STAGES >= 2, "pipeline needs two stages");
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
    static_assert(SF_COL + SF_SLOTS * SF_STRIDE <= TMEM_COLS, "TMEM budget");
};

struct NvTile {
    int g;
    int64_t row0;     // fprop/dgrad: first row of the tile; wgrad: first row of the group
    int rows;         // fprop/dgrad: live rows of the tile
    int64_t mt;       // fprop/dgrad: row tile in the group; wgrad: 128-row tile of n
    int64_t col0;     // first output column
    int nk;           // 256-deep k-tiles
    int last_mma;     // MMAs (64-deep) of the last k-tile
    int64_t T;        // 128-row tiles of the group
    bool skip;        // wgrad, empty group, accumulate: nothing to do
};

template <int KIND>
__device__ __forceinline__ int64_t nv_tile_count(const NvArgs& p, const int32_t* s_tp)
{
    if (KIND == NV_FPROP)
        return (int64_t)s_tp[p.G] * (p.n / 256);
    if (KIND == NV_DGRAD)
        return (int64_t)s_tp[p.G] * (p.k / 256);
    return (int64_t)p.G * (p.n / 128) * (p.k / 256);
}

template <int KIND>
__device__ __forceinline__ NvTile nv_decode(const NvArgs& p, const int32_t* s_off, const int32_t* s_tp, int64_t tile)
{
    NvTile t;
    if (KIND != NV_WGRAD) {
        const int64_t nnt = (KIND == NV_FPROP ? p.n : p.k) / 256;
        const int64_t rt = tile / nnt;
        t.g = group_of_tile(s_tp, p.G, rt);
        t.mt = rt - s_tp[t.g];
        const int64_t m = s_off[t.g + 1] - s_off[t.g];
        t.row0 = s_off[t.g] + 128 * t.mt;
        t.rows = (int)min((int64_t)128, m - 128 * t.mt);
        t.col0 = (tile - rt * nnt) * 256;
        t.nk = (int)((KIND == NV_FPROP ? p.k : p.n) / 256);
        t.last_mma = 4;
        t.T = s_tp[t.g + 1] - s_tp[t.g];
        t.skip = false;
    } else {
        const int64_t nkt = p.k / 256;
        const int64_t per_group = (p.n / 128) * nkt;
        t.g = (int)(tile / per_group);
        const int64_t rem = tile - t.g * per_group;
        t.mt = rem / nkt;
        t.col0 = (rem - t.mt * nkt) * 256;
        const int64_t m = s_off[t.g + 1] - s_off[t.g];
        t.row0 = s_off[t.g];
        t.rows = 128;
        t.nk = (int)((m + 255) / 256);
        const int nb64 = (int)((m + 63) / 64);
        t.last_mma = t.nk > 0 ? nb64 - 4 * (t.nk - 1) : 0;
        t.T = s_tp[t.g + 1] - s_tp[t.g];
        t.skip = (m == 0) && p.accumulate;
    }
    return t;
}

template <int KIND, bool OUT_BF16>
__global__ void __launch_bounds__(NvShape<KIND>::THREADS, 1)
k_gemm_nv(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
          const __grid_constant__ CUtensorMap tma_o, const NvArgs p)
{
    using S = NvShape<KIND>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = base;
    uint8_t* sB = sA + S::STAGES * S::A_BYTES;
    uint8_t* sOut = sB + S::STAGES * S::B_BYTES;
    uint8_t* sSFA = sOut + S::OUT_BYTES;
    uint8_t* sSFB = sSFA + S::STAGES * S::SFA_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(sSFB + S::STAGES * S::SFB_BYTES);
    uint64_t* empty = full + 8;
    uint64_t* tfull = empty + 8;
    uint64_t* tempty = tfull + 1;
    uint64_t* drain = tempty + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const Scan sc = carve_scan(reinterpret_cast<uint8_t*>(tmem_slot + 4));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (load_status(p.status) != 0)
        return;
    const int err = block_scan_splits(p.splits, p.G, p.rows_cap, 32, sc.off, sc.tp, sc.w64, sc.w32);
    if (err) {
        if (threadIdx.x == 0)
            set_status(p.status, err);
        return;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < S::STAGES; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        ptx::mbar_init(tfull, 1);
        ptx::mbar_init(tempty, 8);
        ptx::mbar_init(drain, 1);
        *abort = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(tmem_slot, S::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tma_a);
        ptx::prefetch_tmap(&tma_b);
        ptx::prefetch_tmap(&tma_o);
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int64_t ntiles = nv_tile_count<KIND>(p, sc.tp);

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer --
        int64_t issued = 0;
        int ps = 0;
        uint32_t pph = 0;
        bool ok = true;
        for (int64_t tile = blockIdx.x; tile < ntiles && ok && !*abort; tile += gridDim.x) {
            const NvTile t = nv_decode<KIND>(p, sc.off, sc.tp, tile);
            if (t.skip || t.nk == 0)
                continue;
            for (int kt = 0; kt < t.nk; ++kt, ++issued) {
                if (!ptx::mbar_wait(&empty[ps], pph ^ 1u, abort, p.status)) {
                    ok = false;
                    break;
                }
                const int s = ps;
                if (++ps == S::STAGES) {
                    ps = 0;
                    pph ^= 1u;
                }
                const int nm = (KIND == NV_WGRAD && kt == t.nk - 1) ? t.last_mma : 4;
                uint64_t* bar = &full[s];
                ptx::mbar_arrive_expect_tx(bar, (uint32_t)(S::A_BYTES + S::B_BYTES + 3 * 512 * nm));
                uint8_t* sa = sA + s * S::A_BYTES;
                uint8_t* sb = sB + s * S::B_BYTES;
                uint8_t* ssfa = sSFA + s * S::SFA_BYTES;
                uint8_t* ssfb = sSFB + s * S::SFB_BYTES;
                if (KIND == NV_FPROP) {
                    const int64_t kb = p.k / 64;                          // 64-column blocks of X and W
                    ptx::tma_load_2d(sa, &tma_a, bar, kt * 128, (int32_t)t.row0);
                    ptx::tma_load_2d(sb, &tma_b, bar, kt * 128, (int32_t)(t.g * p.n + t.col0));
                    ptx::bulk_load(ssfa, p.sfa + 512 * (kb * sc.tp[t.g] + t.mt * kb + 4 * kt), 2048, bar);
                    const int64_t wb = kb * (int64_t)t.g * (p.n / 128);
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        ptx::bulk_load(ssfb + 2048 * h, p.sfb + 512 * (wb + (t.col0 / 128 + h) * kb + 4 * kt), 2048,
                                       bar);
                } else if (KIND == NV_DGRAD) {
                    const int64_t nb = p.n / 64;                          // 64-column blocks of dY, row blocks of W
                    ptx::tma_load_2d(sa, &tma_a, bar, kt * 128, (int32_t)t.row0);
                    ptx::tma_load_2d(sb, &tma_b, bar, (int32_t)(t.g * (p.n / 2) + kt * 128), (int32_t)t.col0);
                    ptx::bulk_load(ssfa, p.sfa + 512 * (nb * sc.tp[t.g] + t.mt * nb + 4 * kt), 2048, bar);
                    const int64_t wb = (p.k / 64) * (int64_t)t.g * (p.n / 128);
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        ptx::bulk_load(ssfb + 2048 * h, p.sfb + 512 * (wb + (t.col0 / 128 + h) * nb + 4 * kt), 2048,
                                       bar);
                } else {
                    const int32_t x0 = (int32_t)(t.row0 / 2 + 128 * kt);    // byte of the k-tile's first row
                    const int64_t T2 = 2 * t.T;                             // 64-row blocks of the group
                    ptx::tma_load_2d(sa, &tma_a, bar, x0, (int32_t)(t.mt * 128));
                    ptx::tma_load_2d(sb, &tma_b, bar, x0, (int32_t)t.col0);
                    ptx::bulk_load(ssfa, p.sfa + 512 * ((p.n / 64) * sc.tp[t.g] + t.mt * T2 + 4 * kt),
                                   (uint32_t)(512 * nm), bar);
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        ptx::bulk_load(ssfb + 2048 * h,
                                       p.sfb + 512 * ((p.k / 64) * sc.tp[t.g] + (t.col0 / 128 + h) * T2 + 4 * kt),
                                       (uint32_t)(512 * nm), bar);
                }
            }
        }
        volatile int no_abort = 0;
        for (int64_t q = issued - S::STAGES < 0 ? 0 : issued - S::STAGES; q < issued; ++q)
            if (!ptx::mbar_wait(&full[q % S::STAGES], (uint32_t)((q / S::STAGES) & 1), &no_abort, p.status))
                break;
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------- MMA issuer --
        const uint64_t a_desc0 = ptx::smem_desc(ptx::smem_addr(sA), 16, 1024, 2);
        const uint64_t b_desc0 = ptx::smem_desc(ptx::smem_addr(sB), 16, 1024, 2);
        const uint64_t sfa_desc0 = ptx::smem_desc(ptx::smem_addr(sSFA), 0, 128, 0);
        const uint64_t sfb_desc0 = ptx::smem_desc(ptx::smem_addr(sSFB), 0, 128, 0);
        constexpr uint32_t idesc = idesc_nvf4(128, 256);
        int s = 0;
        uint32_t ph = 0, slot = 0;
        int64_t tiles_done = 0;
        bool ok = true;
        for (int64_t tile = blockIdx.x; tile < ntiles && ok && !*abort; tile += gridDim.x) {
            const NvTile t = nv_decode<KIND>(p, sc.off, sc.tp, tile);
            if (t.skip || t.nk == 0)
                continue;
            if (!ptx::mbar_wait(tempty, (uint32_t)((tiles_done & 1) ^ 1), abort, p.status))
                break;
            ptx::tc_fence_after_sync();
            for (int kt = 0; kt < t.nk; ++kt) {
                if (!ptx::mbar_wait(&full[s], ph, abort, p.status)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after_sync();
                const int nm = (KIND == NV_WGRAD && kt == t.nk - 1) ? t.last_mma : 4;
                const uint32_t sfa_t = tmem + S::SF_COL + slot * S::SF_STRIDE;
                const uint32_t sfb_t = sfa_t + 16;
                for (int j = 0; j < nm; ++j) {
                    ptx::tc_cp_sf_atom(sfa_t + 4 * j, sfa_desc0 + (uint64_t)((s * S::SFA_BYTES + 512 * j) >> 4));
                    ptx::tc_cp_sf_atom(sfb_t + 8 * j, sfb_desc0 + (uint64_t)((s * S::SFB_BYTES + 512 * j) >> 4));
                    ptx::tc_cp_sf_atom(sfb_t + 8 * j + 4,
                                       sfb_desc0 + (uint64_t)((s * S::SFB_BYTES + 2048 + 512 * j) >> 4));
                }
                const uint64_t ad = a_desc0 + (uint64_t)(s * (S::A_BYTES >> 4));
                const uint64_t bd = b_desc0 + (uint64_t)(s * (S::B_BYTES >> 4));
                for (int j = 0; j < nm; ++j)          // K = 64 codes = 32 bytes along the swizzled row
                    tc_mma_nvf4(tmem, ad + 2u * j, bd + 2u * j, idesc, sfa_t + 4 * j, sfb_t + 8 * j, (kt | j) != 0);
                ptx::tc_commit(&empty[s]);
                if (++s == S::STAGES) {
                    s = 0;
                    ph ^= 1u;
                }
                slot = (slot + 1) & (S::SF_SLOTS - 1);
            }
            if (!ok)
                break;
            ptx::tc_commit(tfull);
            ++tiles_done;
        }
        ptx::tc_commit(drain);
        volatile int no_abort = 0;
        ptx::mbar_wait(drain, 0, &no_abort, p.status);
    } else if (warp >= 4) {
        // --------------------------------------------------- epilogue --
        // The accumulator (128 x 256 fp32) fills the TMEM columns it has, so
        // each of the 8 warps drains its lane quadrant's 32 rows x 128
        // columns into registers at once and hands TMEM back; the next
        // tile's MMAs overlap the scaling by 1 / (S_a S_b) and the stores.
        // Each warp then writes its rows through its own box in shared
        // memory that lane 0 hands to the TMA unit.
        const int q = warp & 3, h = (warp - 4) >> 2;
        uint8_t* box = sOut + (warp - 4) * S::BOX;
        const uint32_t box_addr = ptx::smem_addr(box);
        int64_t tiles_done = 0;
        for (int64_t tile = blockIdx.x; tile < ntiles && !*abort; tile += gridDim.x) {
            const NvTile t = nv_decode<KIND>(p, sc.off, sc.tp, tile);
            if (t.skip || (KIND != NV_WGRAD && t.nk == 0))
                continue;
            uint32_t v[4][32];
            if (t.nk > 0) {
                if (!ptx::mbar_wait_warp(tfull, (uint32_t)(tiles_done & 1), abort, p.status))
                    break;
                ptx::tc_fence_after_sync();
                const uint32_t tb = tmem + ((uint32_t)(32 * q) << 16) + 128 * h;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
                    ptx::tmem_ld_32x32(tb + 32 * cc, v[cc]);
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
                    ptx::tmem_wait_ld(v[cc]);
                ptx::tc_fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    ptx::mbar_arrive(tempty);
                ++tiles_done;
                const float alpha = nv_alpha(__ldg(p.amax_a + t.g), __ldg(p.amax_b + t.g));
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        v[cc][i] = __float_as_uint(__fmul_rn(__uint_as_float(v[cc][i]), alpha));
            } else {                                      // wgrad of an empty group: dW_g = 0
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        v[cc][i] = 0u;
            }
            if (KIND == NV_WGRAD) {
                const int32_t orow = (int32_t)((int64_t)t.g * p.n + t.mt * 128 + 32 * q);
                const int32_t ocol = (int32_t)(t.col0 + 128 * h);
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    if (lane == 0)
                        ptx::bulk_wait_read_all();    // the last box's store has read it
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        ptx::sts128(box_addr + ptx::swz128(lane, j),
                                    make_uint4(v[b][4 * j], v[b][4 * j + 1], v[b][4 * j + 2], v[b][4 * j + 3]));
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if (p.accumulate)
                            ptx::tma_reduce_add_2d(&tma_o, box, ocol + 32 * b, orow);
                        else
                            ptx::tma_store_2d(&tma_o, box, ocol + 32 * b, orow);
                        ptx::bulk_commit_group();
                    }
                }
            } else {
                if (32 * q >= t.rows)
                    continue;
                // 32 rows x 64 bytes (64-byte swizzle) per box
                constexpr int CW = OUT_BF16 ? 32 : 16;
                constexpr int NBOX = 128 / CW;
                const uint32_t row_addr = box_addr + 64 * lane;
                const uint32_t sw = (lane >> 1) & 3;
                const int32_t orow = (int32_t)(t.row0 + 32 * q);
                const int32_t ocol = (int32_t)(t.col0 + 128 * h);
#pragma unroll
                for (int b = 0; b < NBOX; ++b) {
                    if (lane == 0)
                        ptx::bulk_wait_read_all();
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint4 val;
                        if (OUT_BF16) {
                            const uint32_t* src = &v[b][8 * j];
                            uint32_t w[4];
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const __nv_bfloat162 hv = __floats2bfloat162_rn(__uint_as_float(src[2 * i]),
                                                                                __uint_as_float(src[2 * i + 1]));
                                w[i] = *reinterpret_cast<const uint32_t*>(&hv);
                            }
                            val = make_uint4(w[0], w[1], w[2], w[3]);
                        } else {
                            const uint32_t* src = &v[b >> 1][16 * (b & 1) + 4 * j];
                            val = make_uint4(src[0], src[1], src[2], src[3]);
                        }
                        ptx::sts128(row_addr + ((j ^ sw) << 4), val);
                    }
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        ptx::tma_store_2d(&tma_o, box, ocol + CW * b, orow);
                        ptx::bulk_commit_group();
                    }
                }
            }
        }
        if (lane == 0)
            ptx::bulk_wait_all();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, S::TMEM_COLS);
    }
}

// Zero-fill of dW for a wgrad over an empty buffer.
__global__ void k_nv_zero_fill(float* __restrict__ out, int64_t count, const int32_t* status)
{
    if (load_status(status) != 0)
        return;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < count; i += (int64_t)gridDim.x * blockDim.x)
        out[i] = 0.f;
}

template <int KIND, bool OUT_BF16>
gq_status run_nv(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mo, const NvArgs& args,
                 int64_t tiles_bound, cudaStream_t stream)
{
    using S = NvShape<KIND>;
    auto kernel = k_gemm_nv<KIND, OUT_BF16>;
    if (prepare_kernel(reinterpret_cast<const void*>(kernel), S::SMEM, 0, nullptr) != cudaSuccess)
        return GQ_ERR_CUDA;
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(tiles_bound, device_info().sm_count));
    kernel<<<(unsigned)grid, S::THREADS, S::SMEM, stream>>>(ma, mb, mo, args);
    return cudaGetLastError() == cudaSuccess ? GQ_OK : GQ_ERR_CUDA;
}

}  // namespace

cudaError_t launch_quant_nv(const void* x, int64_t rows_cap, int64_t cols, const int32_t* splits, int G,
                            uint8_t* row_data, uint8_t* row_scale, uint8_t* col_data, uint8_t* col_scale, float* amax,
                            int32_t* status, cudaStream_t stream)
{
    const uint16_t* xb = static_cast<const uint16_t*>(x);
    k_nv_prepare<<<1, 256, 0, stream>>>(splits, G, rows_cap, amax, status);
    if (cudaGetLastError() != cudaSuccess)
        return cudaErrorLaunchFailure;
    const int sms = device_info().sm_count;
    const int64_t blk_bound = rows_cap / 32 + 1;
    k_nv_amax<<<(unsigned)std::max<int64_t>(1, std::min<int64_t>(blk_bound, 4 * (int64_t)sms)), 256, 0, stream>>>(
        xb, rows_cap, cols, splits, G, amax, status);
    if (cudaGetLastError() != cudaSuccess)
        return cudaErrorLaunchFailure;
    CUtensorMap m128, m32;
    if (!make_tensor_map_2d(&m128, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, rows_cap, cols, 64, 128) ||
        !make_tensor_map_2d(&m32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, rows_cap, cols, 64, 32))
        return cudaErrorInvalidValue;
    const void* fn = row_data && col_data ? reinterpret_cast<const void*>(k_nv_quant<true, true>)
                     : row_data           ? reinterpret_cast<const void*>(k_nv_quant<true, false>)
                                          : reinterpret_cast<const void*>(k_nv_quant<false, true>);
    const cudaError_t e = prepare_kernel(fn, kNqSmem, kNqThreads, nullptr);
    if (e != cudaSuccess)
        return e;
    const int64_t tiles_bound = ((rows_cap + 127) / 128 + G) * (cols / 128);
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>((int64_t)sms, tiles_bound));
    if (row_data && col_data)
        k_nv_quant<true, true><<<(unsigned)grid, kNqThreads, kNqSmem, stream>>>(
            m128, m32, rows_cap, cols, splits, G, amax, row_data, row_scale, col_data, col_scale, status);
    else if (row_data)
        k_nv_quant<true, false><<<(unsigned)grid, kNqThreads, kNqSmem, stream>>>(
            m128, m32, rows_cap, cols, splits, G, amax, row_data, row_scale, col_data, col_scale, status);
    else
        k_nv_quant<false, true><<<(unsigned)grid, kNqThreads, kNqSmem, stream>>>(
            m128, m32, rows_cap, cols, splits, G, amax, row_data, row_scale, col_data, col_scale, status);
    return cudaGetLastError();
}

gq_status launch_gemm_nv(NvGemmKind kind, const NvOperand& a, const NvOperand& b, const int32_t* splits, int G,
                         int64_t rows_cap, int64_t n, int64_t k, void* out, int out_dtype, int accumulate,
                         int32_t* status, cudaStream_t stream)
{
    NvArgs args;
    args.splits = splits;
    args.G = G;
    args.rows_cap = rows_cap;
    args.n = n;
    args.k = k;
    args.sfa = a.scale;
    args.sfb = b.scale;
    args.amax_a = a.amax;
    args.amax_b = b.amax;
    args.out = out;
    args.accumulate = accumulate;
    args.status = status;
    if (rows_cap >= (int64_t(1) << 31) || a.rows >= (int64_t(1) << 31) || b.rows >= (int64_t(1) << 31))
        return GQ_ERR_INVALID_ARG;
    if (rows_cap == 0) {
        if (kind == NV_WGRAD && !accumulate) {
            k_nv_zero_fill<<<256, 256, 0, stream>>>(static_cast<float*>(out), (int64_t)G * n * k, status);
            return cudaGetLastError() == cudaSuccess ? GQ_OK : GQ_ERR_CUDA;
        }
        return GQ_OK;
    }
    CUtensorMap ma, mb, mo;
    if (!make_map_u8(&ma, a.data, a.rows, a.row_bytes, 128) ||
        !make_map_u8(&mb, b.data, b.rows, b.row_bytes, 256))
        return GQ_ERR_CUDA;
    if (kind == NV_WGRAD) {
        if (!make_tensor_map_2d(&mo, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, out, (int64_t)G * n, k, 32, 32))
            return GQ_ERR_CUDA;
        return run_nv<NV_WGRAD, false>(ma, mb, mo, args, (int64_t)G * (n / 128) * (k / 256), stream);
    }
    const int64_t n_out = kind == NV_FPROP ? n : k;
    const bool bf16 = out_dtype == GQ_DTYPE_BF16;
    if (!make_tensor_map_2d_sw64(&mo, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                                 bf16 ? 2 : 4, out, rows_cap, n_out, bf16 ? 32 : 16, 32))
        return GQ_ERR_CUDA;
    const int64_t bound = ((rows_cap + 127) / 128 + G) * (n_out / 256);
    if (kind == NV_FPROP)
        return bf16 ? run_nv<NV_FPROP, true>(ma, mb, mo, args, bound, stream)
                    : run_nv<NV_FPROP, false>(ma, mb, mo, args, bound, stream);
    return bf16 ? run_nv<NV_DGRAD, true>(ma, mb, mo, args, bound, stream)
                : run_nv<NV_DGRAD, false>(ma, mb, mo, args, bound, stream);
}

}  // namespace gq
