// Grouped FP8 GEMMs on the 5th-generation tensor core (tcgen05, sm_103a).
//
//  fprop  Y_g  = X_g W_g^T      A = X rowwise (K-major), B = W_g rowwise (K-major)
//  dgrad  dX_g = dY_g W_g       A = dY rowwise (K-major), B = W_g columnwise (MN-major)
//  wgrad  dW_g = dY_g^T X_g     A = dY columnwise (MN-major), B = X columnwise (MN-major),
//                               contracting over group g's live rows only
//
// (TransformerEngine issue 3484: forward and dgrad have M as a free
// dimension, the wgrad contracts over the token axis; DeepGEMM issue 365:
// the k-grouped wgrad with per-channel 128-row fp32 scales.)
//
// One persistent CTA per SM walks a static tile list (tile = blockIdx.x +
// i * gridDim.x).  Warp roles:
//   warp 0 (one thread)  TMA producer: operand tiles by 2-D tensor maps with
//                        128-byte swizzle, 512-byte E8M0 scale atoms by bulk
//                        copies, into a ring of shared-memory stages;
//   warp 1 (one thread)  MMA issuer: copies the scale atoms to TMEM
//                        (tcgen05.cp), issues block-scaled MMAs
//                        (kind::mxf8f6f4, M = 128, N = BN, K = 32 per
//                        instruction, 4 per 128-deep k-tile), commits stages
//                        back to the producer and finished accumulators to
//                        the epilogue;
//   warps 4..7           epilogue: TMEM -> registers -> global, one output
//                        row per thread.
// Accumulators live in TMEM (double-buffered for BN = 128) so the epilogue of
// one tile overlaps the MMAs of the next.  Each output element is produced
// by one CTA with a fixed contraction order: results are deterministic.
//
// The wgrad's last k-tile of a group with m_g % 128 != 0 issues only
// m_g % 128 / 32 of its four MMAs, so rows past the group (the next group's
// tokens, padding, or out-of-range zero fill) never enter a contraction.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <mutex>
#include <type_traits>

#include "gq_internal.h"
#include "gq_ptx.cuh"

namespace gq {
namespace {

constexpr int BM = 128;     // MMA M (rows of the A side)
// L2 prefetch distance of the producers, in k-tiles (tuning knob; 0 = off):
// the operand boxes of k-tile kt + PF are prefetched into L2 when k-tile kt
// is loaded, so that first-touch DRAM latency hides behind the smem ring.
#ifndef GQ_PF_DIST
#define GQ_PF_DIST 0
#endif
constexpr int PF_DIST = GQ_PF_DIST;
constexpr int BK = 128;     // k-tile depth in elements (= bytes for e4m3)
constexpr int kSmemLimit = 227 * 1024;
constexpr int kEpiBox = 32 * 64;   // fprop/dgrad output box per epilogue warp (BN = 256)

struct GemmArgs {
    const int32_t* splits;
    int G;
    int64_t rows_cap;
    int64_t n, k;             // the API's n and k
    const uint8_t* sfa;       // scale base of the A-side operand
    const uint8_t* sfb;       // scale base of the B-side operand
    void* out;
    int accumulate;
    int32_t* status;
    // k-grouped MX wgrad only: tile-claim counter (low 32 bits: tiles taken
    // from the front of the run-time order, high 32 bits: from the back), or
    // null for the static round-robin order; CTAs below front_ctas claim
    // from the front
    unsigned long long* claim = nullptr;
    int front_ctas = 0;
    // fprop only: per-group bias [G, n] (fp32, or bf16 when bias_bf16),
    // added to every live row of the group before the output conversion
    const void* bias = nullptr;
    int bias_bf16 = 0;
    // fprop with the fused activation (the ACT kernels): per-row probs, and
    // the MXFP8 rowwise / columnwise codes [R, n] and grouped swizzled scale
    // atoms of probs[r] * relu(y)^2
    const float* act_probs = nullptr;
    uint8_t* act_row = nullptr;
    uint8_t* act_row_scale = nullptr;
    uint8_t* act_col = nullptr;
    uint8_t* act_col_scale = nullptr;
    // ScaledSwiGLU (ACT == 2): columns of the activation, n / 2; the fc1
    // output's gate half is [0, act_half), its linear half [act_half, n)
    int64_t act_half = 0;
};

// Four consecutive bias values of group row `g`, column `col` (col % 4 == 0).
__device__ __forceinline__ float4 load_bias4(const GemmArgs& p, int g, int64_t col)
{
    const int64_t i = (int64_t)g * p.n + col;
    if (p.bias_bf16) {
        const uint2 u = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p.bias) + i));
        return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                           __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
    }
    return __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(p.bias) + i));
}

// v[i] += bias for the 32 columns [col, col + 32) of group g.
__device__ __forceinline__ void add_bias32(const GemmArgs& p, int g, int64_t col, uint32_t (&v)[32])
{
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
        const float4 b = load_bias4(p, g, col + i);
        v[i] = __float_as_uint(__uint_as_float(v[i]) + b.x);
        v[i + 1] = __float_as_uint(__uint_as_float(v[i + 1]) + b.y);
        v[i + 2] = __float_as_uint(__uint_as_float(v[i + 2]) + b.z);
        v[i + 3] = __float_as_uint(__uint_as_float(v[i + 3]) + b.w);
    }
}

// Output box slots per epilogue warp of the wide wgrad (tuning knob): more
// slots keep more of the old main grad in flight per CTA but leave room for
// fewer pipeline stages.
#ifndef GQ_WG_SLOTS
#define GQ_WG_SLOTS 2
#endif
constexpr int kWgSlots = GQ_WG_SLOTS;

// How the accumulating wide wgrad moves a tile into the main grad.  Each
// warp's share is four 32-column boxes; either all four go by load + add +
// store, or boxes 1 and 3 go by TMA reduce-add and the others by load + add
// + store.  Measured on a 3.8 GB fp32 buffer: when every SM carries main-grad
// traffic, load + add + store alone reaches the copy rate and mixes fall
// short of it; when only half of the SMs do (the others busy with long
// contractions), load + add + store alone and reduce-add alone each move
// about 70% of the copy rate and mixes more (the reduce-adds hold no load in
// flight): 79% with half the boxes by reduce-add, ~100% with 10-12 of 16.  In
// the kernel itself, beside the long contractions, half is the fastest share
// (one or three boxes in four by reduce-add are slower).  So the kernel mixes
// when the split sizes are skewed: when the largest group holds at least
// GQ_WG_MIX_SKEW times the mean live group (tuning knob; 0 = always mix, a
// huge value = never).
#ifndef GQ_WG_MIX_SKEW
#define GQ_WG_MIX_SKEW 4
#endif
constexpr int64_t kWgMixSkew = GQ_WG_MIX_SKEW;

// Share of the wgrad's CTAs (percent) that claim tiles from the largest
// groups down in the run-time order; the others start from the smallest
// (tuning knob).
#ifndef GQ_WG_FRONT_PCT
#define GQ_WG_FRONT_PCT 40
#endif
constexpr int kWgFrontPct = GQ_WG_FRONT_PCT;

// x-operand bytes of a group above which the wgrad walks its tiles column by
// column (see decode_tile).
#ifndef GQ_WG_COLUMN_ORDER_MB
#define GQ_WG_COLUMN_ORDER_MB 32
#endif
constexpr int64_t kWgColumnOrderBytes = (int64_t)GQ_WG_COLUMN_ORDER_MB << 20;

// Depth of the shared-memory ring through which the producer passes claimed
// tiles to the MMA issuer and the epilogue warps.
constexpr int kTileRing = 8;

template <int KIND, int BN>
struct MxShape {
    // BN = 128: 4 epilogue warps, one row per thread; BN = 256: 8 epilogue
    // warps (two per TMEM lane quadrant, 128 columns each).
    static constexpr int EPI_WARPS = BN == 256 ? 8 : 4;
    static constexpr int THREADS = 128 + 32 * EPI_WARPS;
    static constexpr int A_BYTES = BM * BK;
    static constexpr int B_BYTES = BN * BK;
    static constexpr int SFA_BYTES = 512;
    static constexpr int SFB_BYTES = 512 * (BN / 128);
    static constexpr int STAGE = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
    // wgrad sends its fp32 output through 64 KB of shared memory on the way
    // to a TMA store or reduce-add: a ring of four 128 x 32 boxes for
    // BN = 128, a ring of kWgSlots 32 x 32 boxes per epilogue warp for
    // BN = 256.  fprop/dgrad with BN = 256 stage their output too: each of
    // the 8 epilogue warps owns a 2 KB box of 32 rows x 64 bytes (64-byte
    // swizzle).
    static constexpr int OUT_BYTES = KIND == GEMM_WGRAD_MX ? (BN == 256 ? 8 * kWgSlots * 32 * 128 : 4 * BM * 128)
                                     : (BN == 256 ? kEpiBox * 8 : 0);
    static constexpr int ACC = BN == 128 ? 2 : 1;                    // TMEM accumulator buffers
    // Scale factors rotate through SF_SLOTS column groups, so that the copy
    // for k-tile i + 1 never overwrites columns the MMAs of k-tile i still
    // read (one shared slot would serialise the tensor pipe every k-tile).
    static constexpr uint32_t SF_SLOTS = 8;
    static constexpr uint32_t SF_STRIDE = 4 + BN / 32;                // A atom + B atoms
    static constexpr uint32_t SFA_COL = ACC * BN;                     // TMEM column of A scales, slot 0
    static constexpr uint32_t SFB_COL = SFA_COL + 4;                  // TMEM column of B scales, slot 0
    static constexpr uint32_t TMEM_COLS = 512;
    // wgrad adds the groups in decreasing order of size and the tile ring
    static constexpr int SCAN_BYTES = (GQ_MAX_GROUPS + 1) * 4 + (GQ_MAX_GROUPS + 2) * 4 + 8 + 32 * 8 + 32 * 4 +
                                      (KIND == GEMM_WGRAD_MX ? (GQ_MAX_GROUPS + kTileRing) * 4 : 0);
    // wide wgrad: one barrier per output box slot (8 warps x 2) for the TMA
    // loads of the old main grad
    static constexpr int OUT_BARS = (KIND == GEMM_WGRAD_MX && BN == 256) ? 8 * kWgSlots : 0;
    // wgrad: full / empty barriers of the claimed-tile ring
    static constexpr int RING_BARS = KIND == GEMM_WGRAD_MX ? 2 * kTileRing : 0;
    static constexpr int BAR_BYTES = 8 * (2 * 8 + 2 * ACC + 1 + OUT_BARS + RING_BARS) + 16;
    static constexpr int STAGES_FIT = (kSmemLimit - 1024 - OUT_BYTES - SCAN_BYTES - BAR_BYTES) / STAGE;
    static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
    static constexpr int SMEM = 1024 + STAGES * STAGE + OUT_BYTES + BAR_BYTES + SCAN_BYTES;
    static_assert(STAGES >= 2, "pipeline needs two stages");
    static_assert(kWgSlots == 2 || kWgSlots == 3, "wgrad box slots");
    static_assert((SF_SLOTS & (SF_SLOTS - 1)) == 0, "scale slots: a power of two");
    static_assert(SMEM <= kSmemLimit, "shared memory budget");
    static_assert(SFA_COL + SF_SLOTS * SF_STRIDE <= TMEM_COLS, "TMEM budget");
};

// Shared-memory carve-up common to the GEMM kernels.
struct Carve {
    uint8_t* a;
    uint8_t* b;
    uint8_t* out;         // output staging tile (wgrad), 1024-aligned
    uint8_t* sfa;
    uint8_t* sfb;
    uint64_t* full;
    uint64_t* empty;
    uint64_t* tfull;
    uint64_t* tempty;
    uint64_t* drain;
    uint64_t* obar;       // output-box load barriers (wide wgrad)
    uint32_t* tmem_base;
    volatile int* abort;
    int32_t* s_off;       // group row offsets (rows_cap < 2^31 on every GEMM call)
    int32_t* s_tp;
    int64_t* s_w64;
    int32_t* s_w32;
};

__device__ __forceinline__ Carve carve(uint8_t* raw, int stages, int a_bytes, int b_bytes,
                                       int sfa_bytes, int sfb_bytes, int acc, int out_bytes = 0,
                                       int out_bars = 0)
{
    Carve c;
    uint8_t* p = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) &
                                            ~uintptr_t(1023));
    c.a = p;
    p += stages * a_bytes;
    c.b = p;
    p += stages * b_bytes;
    c.out = p;
    p += out_bytes;
    c.sfa = p;
    p += stages * sfa_bytes;
    c.sfb = p;
    p += stages * sfb_bytes;
    p = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 7) & ~uintptr_t(7));
    c.full = reinterpret_cast<uint64_t*>(p);
    c.empty = c.full + 8;
    c.tfull = c.empty + 8;
    c.tempty = c.tfull + acc;
    c.drain = c.tempty + acc;
    c.obar = c.drain + 1;
    c.tmem_base = reinterpret_cast<uint32_t*>(c.obar + out_bars);
    c.abort = reinterpret_cast<volatile int*>(c.tmem_base + 1);
    c.s_off = reinterpret_cast<int32_t*>(c.tmem_base + 4);
    c.s_tp = c.s_off + GQ_MAX_GROUPS + 1;
    c.s_w64 = reinterpret_cast<int64_t*>((reinterpret_cast<uintptr_t>(c.s_tp + GQ_MAX_GROUPS + 2) + 7) &
                                         ~uintptr_t(7));
    c.s_w32 = reinterpret_cast<int32_t*>(c.s_w64 + 32);
    return c;
}

// One output tile of a grouped GEMM.
struct Tile {
    int g;            // group
    int64_t row0;     // fprop/dgrad: first token row of the tile; wgrad: first token row of the group
    int rows;         // fprop/dgrad: live rows in the tile (a multiple of 32)
    int64_t mt;       // fprop/dgrad: row tile inside the group; wgrad: 128-row tile of n
    int64_t col0;     // first output column
    int nk;           // k-tiles
    int last_sub;     // K = 32 steps in the last k-tile (wgrad), else 4
    int T;            // 128-row tiles of the group
    bool skip;        // nothing to do (empty group, accumulate)
};

template <int KIND, int BN>
__device__ __forceinline__ int64_t tile_count(const GemmArgs& p, const int32_t* s_tp)
{
    if (KIND == GEMM_FPROP)
        return (int64_t)s_tp[p.G] * (p.n / BN);
    if (KIND == GEMM_DGRAD)
        return (int64_t)s_tp[p.G] * (p.k / BN);
    return (int64_t)p.G * (p.n / BM) * (p.k / BN);
}

template <int KIND, int BN>
__device__ __forceinline__ Tile decode_tile(const GemmArgs& p, const int32_t* s_off,
                                            const int32_t* s_tp, int64_t tile,
                                            const int32_t* ord = nullptr)
{
    Tile t;
    if (KIND == GEMM_FPROP || KIND == GEMM_DGRAD) {
        const int64_t nnt = (KIND == GEMM_FPROP ? p.n : p.k) / BN;
        const int64_t rt = tile / nnt;
        const int64_t nt = tile - rt * nnt;
        t.g = group_of_tile(s_tp, p.G, rt);
        t.mt = rt - s_tp[t.g];
        const int64_t m = s_off[t.g + 1] - s_off[t.g];
        t.row0 = s_off[t.g] + 128 * t.mt;
        t.rows = (int)min((int64_t)128, m - 128 * t.mt);
        t.col0 = nt * BN;
        t.nk = (int)((KIND == GEMM_FPROP ? p.k : p.n) / BK);
        t.last_sub = 4;
        t.T = s_tp[t.g + 1] - s_tp[t.g];
        t.skip = false;
    } else {
        const int64_t nkt = p.k / BN;
        const int64_t per_group = (p.n / BM) * nkt;
        const int64_t gi = tile / per_group;              // position in the group order
        t.g = ord ? ord[gi] : (int)gi;
        const int64_t rem = tile - gi * per_group;
        const int64_t m = s_off[t.g + 1] - s_off[t.g];
        // Tiles running at the same time share operand columns through L2.
        // By default they walk the output row by row (whole main-grad rows
        // at a time), which re-reads the group's x columns once per wave of
        // tiles; for a group whose x operand outgrows L2's share and is the
        // larger of the two, they walk column by column instead, so that
        // the smaller dy operand is the one read again.
        if (p.k > p.n && m * p.k > kWgColumnOrderBytes) {
            const int64_t nmt = p.n / BM;
            t.mt = rem % nmt;
            t.col0 = (rem / nmt) * BN;
        } else {
            t.mt = rem / nkt;
            t.col0 = (rem - t.mt * nkt) * BN;
        }
        t.row0 = s_off[t.g];
        t.rows = 128;
        t.nk = (int)((m + 127) / 128);
        t.last_sub = t.nk > 0 ? (int)((m - 128 * (int64_t)(t.nk - 1)) / 32) : 0;
        t.T = s_tp[t.g + 1] - s_tp[t.g];
        t.skip = (m == 0) && p.accumulate;
    }
    return t;
}

__device__ __forceinline__ void store_row_f32(float* dst, const uint32_t (&r)[32])
{
    float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
    for (int i = 0; i < 8; ++i)
        d[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                           __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
}

__device__ __forceinline__ void store_row_bf16(uint16_t* dst, const uint32_t (&r)[32])
{
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(r[8 * i + 2 * j]),
                                                           __uint_as_float(r[8 * i + 2 * j + 1]));
            w[j] = *reinterpret_cast<const uint32_t*>(&h);
        }
        d[i] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// One claim from the wgrad's tile-claim counter: the next tile from the front
// (or back) of the run-time order, or -1 once the two ends have met.  Every
// tile is handed out exactly once: a claim is granted only while the claims
// granted so far, from both ends, number fewer than ntiles.
__device__ __forceinline__ int64_t claim_tile(unsigned long long* claim, bool front, int64_t ntiles)
{
    const unsigned long long old = atomicAdd(claim, front ? 1ull : (1ull << 32));
    const int64_t f = (int64_t)(old & 0xffffffffull), b = (int64_t)(old >> 32);
    if (f + b >= ntiles)
        return -1;
    return front ? f : ntiles - 1 - b;
}

// Producer side of the claimed-tile ring: entry q gets `tile` (-1 ends the
// sequence).  False if the wait for a free entry gave up.
__device__ __forceinline__ bool ring_put(uint64_t* full, uint64_t* empty, int32_t* ring, int64_t& q,
                                         int64_t tile, volatile int* abort, int32_t* status)
{
    const int e = (int)(q % kTileRing);
    if (!ptx::mbar_wait(&empty[e], (uint32_t)(((q / kTileRing) & 1) ^ 1), abort, status))
        return false;
    *reinterpret_cast<volatile int32_t*>(&ring[e]) = (int32_t)tile;
    ptx::mbar_arrive(&full[e]);
    ++q;
    return true;
}

// Consumer side: entry q of the ring, -1 at the end of the sequence or when
// the wait gave up.  WARP: the whole warp calls it and gets the same value,
// and one arrival per warp frees the entry.
template <bool WARP>
__device__ __forceinline__ int64_t ring_get(uint64_t* full, uint64_t* empty, const int32_t* ring, int64_t& q,
                                            volatile int* abort, int32_t* status)
{
    const int e = (int)(q % kTileRing);
    const uint32_t par = (uint32_t)((q / kTileRing) & 1);
    const bool ok = WARP ? ptx::mbar_wait_warp(&full[e], par, abort, status)
                         : ptx::mbar_wait(&full[e], par, abort, status);
    if (!ok)
        return -1;
    const int64_t tile = *reinterpret_cast<const volatile int32_t*>(&ring[e]);
    if (WARP)
        __syncwarp();
    if (!WARP || (threadIdx.x & 31) == 0)
        ptx::mbar_arrive(&empty[e]);
    ++q;
    return tile;
}

// E8M0 byte of a block from its fp32 amax: max(E - 8, 0) with E the biased
// exponent field (floor(log2 amax) - 8, clamped at -127; zero and subnormal
// amax give 0), and 2^-e for that byte as an exact fp32 power of two.
__device__ __forceinline__ uint32_t e8m0_of_f32(float amax)
{
    const int E = (int)((__float_as_uint(amax) >> 23) & 0xffu);
    return (uint32_t)max(E - 8, 0);
}

__device__ __forceinline__ float inv_scale_of(uint32_t byte) { return __uint_as_float((254u - byte) << 23); }

// Four e4m3 codes (x0's in the low byte) of x * s, rounded to nearest even
// and saturated; the products are exact (s is a power of two).
__device__ __forceinline__ uint32_t codes4(float x0, float x1, float x2, float x3, float s0, float s1, float s2,
                                          float s3)
{
    const float2 lo = __fmul2_rn(make_float2(x0, x1), make_float2(s0, s1));
    const float2 hi = __fmul2_rn(make_float2(x2, x3), make_float2(s2, s3));
    return (uint32_t)__nv_cvt_float2_to_fp8x2(lo, __NV_SATFINITE, __NV_E4M3) |
           ((uint32_t)__nv_cvt_float2_to_fp8x2(hi, __NV_SATFINITE, __NV_E4M3) << 16);
}

// Transposed butterfly maximum of a warp's 32 x 32 fp32 block (lane = row,
// x[i] = column i) on the magnitudes' bit patterns: lane j ends with the
// largest |value| of column j.
__device__ __forceinline__ uint32_t warp_colmax(const uint32_t (&x)[32], int lane)
{
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2, b0 = lane & 1;
    uint32_t m[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t send = (b4 ? x[i] : x[i + 16]) & 0x7fffffffu;
        const uint32_t keep = (b4 ? x[i + 16] : x[i]) & 0x7fffffffu;
        m[i] = max(keep, __shfl_xor_sync(0xffffffffu, send, 16));
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t send = b3 ? m[i] : m[i + 8];
        const uint32_t keep = b3 ? m[i + 8] : m[i];
        m[i] = max(keep, __shfl_xor_sync(0xffffffffu, send, 8));
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t send = b2 ? m[i] : m[i + 4];
        const uint32_t keep = b2 ? m[i + 4] : m[i];
        m[i] = max(keep, __shfl_xor_sync(0xffffffffu, send, 4));
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const uint32_t send = b1 ? m[i] : m[i + 2];
        const uint32_t keep = b1 ? m[i + 2] : m[i];
        m[i] = max(keep, __shfl_xor_sync(0xffffffffu, send, 2));
    }
    return max(b0 ? m[1] : m[0], __shfl_xor_sync(0xffffffffu, b0 ? m[0] : m[1], 1));
}

// The fused ScaledSReLU of one epilogue warp: its 32 rows (lane = row, one
// 32-row block of the group) x 128 columns of the fp32 result, one 32-column
// chunk at a time.  a = probs[r] * relu(y)^2 in fp32 (t = max(y, 0); t = t *
// t; a = t * p), then MXFP8 1x32 codes and E8M0 scales of a, rowwise (blocks
// of 32 columns) and columnwise (the warp's 32 rows), written to the grouped
// layout of a [R, n] buffer: atoms of group g at 512 * (n/128) * (tiles
// before g), rowwise [row tile][column block], columnwise [column
// block][row tile], byte (r % 32) * 16 + (r / 32) * 4 + j.

// Where one warp's activation scale bytes go.
struct ActAtoms {
    uint8_t* row;     // this lane's 32-bit word (or 16-bit half) of the rowwise atom
    uint8_t* col;     // this lane's first byte of the columnwise atom
};

// Atoms of the activation columns [c0, c0 + 128) of tile t (SReLU: c0 =
// col0 + 128 h of the [R, n] buffer; SwiGLU: the 128-column block holding the
// warp's 64 columns of the [R, n/2] buffer), for rows 32 q + lane.
__device__ __forceinline__ ActAtoms act_atoms(const GemmArgs& p, const Tile& t, const int32_t* s_tp, int64_t width,
                                              int64_t c0, int q, int lane)
{
    const int64_t nb = width / 128;
    const int64_t cb = c0 / 128;
    const int64_t sb = 512 * nb * (int64_t)s_tp[t.g];
    ActAtoms a;
    a.row = p.act_row_scale + sb + (t.mt * nb + cb) * 512 + lane * 16 + q * 4;
    a.col = p.act_col_scale + sb + (cb * t.T + t.mt) * 512 + lane * 16 + q;
    return a;
}

// MX codes of one 32-column block x of the warp's rows (lane = row) into
// row `row`, columns [col, col + 32) of the rowwise and columnwise code
// buffers of width `width`; the column scale byte goes to *cbyte, the row
// scale byte is returned.
__device__ __forceinline__ uint32_t act_block_codes(const GemmArgs& p, int64_t row, int64_t col, int64_t width,
                                                    uint32_t amax_r, uint8_t* cbyte_at, int lane,
                                                    const uint32_t (&x)[32])
{
    const uint32_t rb = e8m0_of_f32(__uint_as_float(amax_r));
    const float rs = inv_scale_of(rb);
    {
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            w[i] = codes4(__uint_as_float(x[4 * i]), __uint_as_float(x[4 * i + 1]), __uint_as_float(x[4 * i + 2]),
                          __uint_as_float(x[4 * i + 3]), rs, rs, rs, rs);
        uint4* dst = reinterpret_cast<uint4*>(p.act_row + row * width + col);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
    const uint32_t cbyte = e8m0_of_f32(__uint_as_float(warp_colmax(x, lane)));
    *cbyte_at = (uint8_t)cbyte;
    const float csc = inv_scale_of(cbyte);
    {
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            w[i] = codes4(__uint_as_float(x[4 * i]), __uint_as_float(x[4 * i + 1]), __uint_as_float(x[4 * i + 2]),
                          __uint_as_float(x[4 * i + 3]), __shfl_sync(0xffffffffu, csc, 4 * i),
                          __shfl_sync(0xffffffffu, csc, 4 * i + 1), __shfl_sync(0xffffffffu, csc, 4 * i + 2),
                          __shfl_sync(0xffffffffu, csc, 4 * i + 3));
        uint4* dst = reinterpret_cast<uint4*>(p.act_col + row * width + col);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
    return rb;
}

// ScaledSReLU of chunk x (in place), then its codes; returns the row scale byte.
__device__ __forceinline__ uint32_t act_srelu_chunk(const GemmArgs& p, int64_t row, int64_t col, float pr,
                                                    uint8_t* cbyte_at, int lane, uint32_t (&x)[32])
{
    uint32_t amax_r = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        float y = __uint_as_float(x[i]);
        y = y > 0.f ? y : 0.f;
        const float a = __fmul_rn(__fmul_rn(y, y), pr);
        x[i] = __float_as_uint(a);
        amax_r = max(amax_r, __float_as_uint(a) & 0x7fffffffu);
    }
    return act_block_codes(p, row, col, p.n, amax_r, cbyte_at, lane, x);
}

// exp for the fused ScaledSwiGLU, this library's own: the argument clamped
// to [-87, 88], reduced by ln 2 in the Cody-Waite way (n = rint(x log2 e);
// r = x - n ln2_hi - n ln2_lo, ln2_hi holding 16 bits so that n ln2_hi is
// exact), the degree-7 Taylor polynomial of exp(r) in Horner form with fused
// multiply-adds, and an exact scaling by 2^n.  Every step is one correctly
// rounded fp32 operation.
__device__ __forceinline__ float act_exp(float x)
{
    x = fminf(fmaxf(x, -87.f), 88.f);
    const float n = rintf(__fmul_rn(x, 0x1.715476p+0f));
    float r = __fmaf_rn(n, -0x1.62e4p-1f, x);
    r = __fmaf_rn(n, -0x1.7f7d1cp-20f, r);
    float y = 0x1.a01a02p-13f;
    y = __fmaf_rn(y, r, 0x1.6c16c2p-10f);
    y = __fmaf_rn(y, r, 0x1.111112p-7f);
    y = __fmaf_rn(y, r, 0x1.555556p-5f);
    y = __fmaf_rn(y, r, 0x1.555556p-3f);
    y = __fmaf_rn(y, r, 0.5f);
    y = __fmaf_rn(y, r, 1.f);
    y = __fmaf_rn(y, r, 1.f);
    return __fmul_rn(y, __int_as_float(((int)n + 127) << 23));
}

// silu(x) = x / (1 + exp(-x)), fp32 op by op.
__device__ __forceinline__ float act_silu(float x) { return __fdiv_rn(x, __fadd_rn(1.f, act_exp(-x))); }

// The fused ScaledSwiGLU of one epilogue warp, one 32-column output block at
// a time: gate columns g and the matching linear columns l of its 32 rows
// (lane = row, one 32-row block of the group).  a = (silu(g) * l) * probs[r]
// in fp32 op by op (into g), then MXFP8 1x32 codes and E8M0 scales of a,
// rowwise and columnwise, at output columns [col, col + 32) of the [R,
// act_half] buffer; returns the row scale byte.
__device__ __forceinline__ uint32_t act_glu_chunk(const GemmArgs& p, int64_t row, int64_t col, float pr,
                                                  uint8_t* cbyte_at, int lane, uint32_t (&g)[32],
                                                  const uint32_t (&l)[32])
{
    uint32_t amax_r = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const float a = __fmul_rn(__fmul_rn(act_silu(__uint_as_float(g[i])), __uint_as_float(l[i])), pr);
        g[i] = __float_as_uint(a);
        amax_r = max(amax_r, __float_as_uint(a) & 0x7fffffffu);
    }
    return act_block_codes(p, row, col, p.act_half, amax_r, cbyte_at, lane, g);
}

// Wait for the TMA writes of the last min(stages, issued) issued stages, so
// that none lands after the CTA has left (bounded; used on every exit path).
__device__ __forceinline__ void drain_loads(uint64_t* full, int stages, int64_t issued,
                                            int32_t* status)
{
    volatile int no_abort = 0;
    for (int64_t q = issued - stages < 0 ? 0 : issued - stages; q < issued; ++q)
        if (!ptx::mbar_wait(&full[q % stages], (uint32_t)((q / stages) & 1), &no_abort, status))
            break;
}

// ------------------------------------------------------------------------ //
// MXFP8 grouped GEMM (fprop, dgrad, wgrad)                                  //
// ------------------------------------------------------------------------ //

// ACT (fprop, BN = 256 only): the epilogue also writes the MX-quantised
// activation of the result -- 1: ScaledSReLU (act_quant_warp); 2:
// ScaledSwiGLU (act_glu_warp), where a tile holds 128 gate columns [c, c +
// 128) and the 128 matching linear columns [act_half + c, ...), c = col0 / 2,
// loaded as two 128-row boxes of W_g.
template <int KIND, int BN, bool OUT_BF16, int ACT = 0>
__global__ void __launch_bounds__(MxShape<KIND, BN>::THREADS, 1)
k_gemm_mx(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
          const __grid_constant__ CUtensorMap tma_o, const GemmArgs p)
{
    using S = MxShape<KIND, BN>;
    constexpr bool A_MN = (KIND == GEMM_WGRAD_MX);
    constexpr bool B_MN = (KIND != GEMM_FPROP);
    extern __shared__ uint8_t smem_raw[];
    const Carve c = carve(smem_raw, S::STAGES, S::A_BYTES, S::B_BYTES, S::SFA_BYTES, S::SFB_BYTES,
                          S::ACC, S::OUT_BYTES, S::OUT_BARS + S::RING_BARS);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (load_status(p.status) != 0)
        return;
    const int err = block_scan_splits(p.splits, p.G, p.rows_cap, 32, c.s_off, c.s_tp, c.s_w64,
                                      c.s_w32);
    if (err) {
        if (threadIdx.x == 0)
            set_status(p.status, err);
        return;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < S::STAGES; ++s) {
            ptx::mbar_init(&c.full[s], 1);
            ptx::mbar_init(&c.empty[s], 1);
        }
        for (int a = 0; a < S::ACC; ++a) {
            ptx::mbar_init(&c.tfull[a], 1);
            ptx::mbar_init(&c.tempty[a], S::EPI_WARPS);
        }
        ptx::mbar_init(c.drain, 1);
        for (int b = 0; b < S::OUT_BARS; ++b)
            ptx::mbar_init(&c.obar[b], 1);
        for (int b = 0; b < S::RING_BARS / 2; ++b) {
            ptx::mbar_init(&c.obar[S::OUT_BARS + b], 1);                        // full
            ptx::mbar_init(&c.obar[S::OUT_BARS + kTileRing + b], 1 + S::EPI_WARPS);  // empty
        }
        *c.abort = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(c.tmem_base, S::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tma_a);
        ptx::prefetch_tmap(&tma_b);
        if (KIND == GEMM_WGRAD_MX || BN == 256)
            ptx::prefetch_tmap(&tma_o);
    }
    // k-grouped wgrad with a claim counter: tiles are handed out at run time,
    // in the order of the groups sorted by decreasing size (ties by index);
    // the producer claims and the other roles read the claims from the ring
    const bool dyn = KIND == GEMM_WGRAD_MX && p.claim != nullptr;
    int32_t* s_ord = c.s_w32 + 32;
    int32_t* s_ring = s_ord + GQ_MAX_GROUPS;
    uint64_t* ring_full = c.obar + S::OUT_BARS;
    uint64_t* ring_empty = ring_full + kTileRing;
    const int32_t* ord = dyn ? s_ord : nullptr;
    if (dyn) {
        for (int g = threadIdx.x; g < p.G; g += blockDim.x) {
            const int32_t mg = c.s_off[g + 1] - c.s_off[g];
            int r = 0;
            for (int o = 0; o < p.G; ++o) {
                const int32_t mo = c.s_off[o + 1] - c.s_off[o];
                r += (mo > mg) || (mo == mg && o < g);
            }
            s_ord[r] = g;
        }
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *c.tmem_base;
    const int64_t ntiles = tile_count<KIND, BN>(p, c.s_tp);

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer --
        int64_t issued = 0, cursor = blockIdx.x, rq = 0;
        int ps = 0;                                       // stage of the next load, its phase
        uint32_t pph = 0;
        const bool front = (int)blockIdx.x < p.front_ctas;
        // Run-time order: with accumulate, the empty groups (last in the
        // size order) have nothing to do and stay out of the claims.  The
        // next claim is issued while the current tile's loads go out, so its
        // round trip is hidden.
        int64_t nclaim = ntiles, claimed = -1;
        if (dyn) {
            if (p.accumulate) {
                int live = 0;
                for (int g = 0; g < p.G; ++g)
                    live += c.s_off[g + 1] > c.s_off[g];
                nclaim = (int64_t)live * (ntiles / p.G);
            }
            claimed = claim_tile(p.claim, front, nclaim);
        }
        while (!*c.abort) {
            int64_t tile;
            if (!dyn) {
                tile = cursor;
                cursor += gridDim.x;
                if (tile >= ntiles)
                    break;
            } else {
                tile = claimed;
                if (tile >= 0)
                    claimed = claim_tile(p.claim, front, nclaim);
                if (tile >= 0 && decode_tile<KIND, BN>(p, c.s_off, c.s_tp, tile, ord).skip)
                    continue;
                if (!ring_put(ring_full, ring_empty, s_ring, rq, tile, c.abort, p.status) || tile < 0)
                    break;
            }
            const Tile t = decode_tile<KIND, BN>(p, c.s_off, c.s_tp, tile, ord);
            if (t.skip || t.nk == 0)
                continue;
            for (int kt = 0; kt < t.nk; ++kt, ++issued) {
                const int s = ps;
                if (!ptx::mbar_wait(&c.empty[s], pph ^ 1u, c.abort, p.status))
                    break;
                if (++ps == S::STAGES) {
                    ps = 0;
                    pph ^= 1u;
                }
                uint64_t* bar = &c.full[s];
                ptx::mbar_arrive_expect_tx(bar, S::STAGE);
                uint8_t* sa = c.a + s * S::A_BYTES;
                uint8_t* sb = c.b + s * S::B_BYTES;
                uint8_t* ssfa = c.sfa + s * S::SFA_BYTES;
                uint8_t* ssfb = c.sfb + s * S::SFB_BYTES;
                if (PF_DIST > 0 && kt + PF_DIST < t.nk) {
                    const int kp = kt + PF_DIST;
                    if (KIND == GEMM_FPROP) {
                        ptx::tma_prefetch_l2_2d(&tma_a, kp * BK, (int32_t)t.row0);
                        ptx::tma_prefetch_l2_2d(&tma_b, kp * BK, (int32_t)(t.g * p.n + t.col0));
                    } else if (KIND == GEMM_DGRAD) {
                        ptx::tma_prefetch_l2_2d(&tma_a, kp * BK, (int32_t)t.row0);
#pragma unroll
                        for (int j = 0; j < BN / 128; ++j)
                            ptx::tma_prefetch_l2_2d(&tma_b, (int32_t)(t.col0 + 128 * j), (int32_t)(t.g * p.n + kp * BK));
                    } else {
                        const int32_t rp = (int32_t)(t.row0 + (int64_t)kp * BK);
                        ptx::tma_prefetch_l2_2d(&tma_a, (int32_t)(t.mt * BM), rp);
#pragma unroll
                        for (int j = 0; j < BN / 128; ++j)
                            ptx::tma_prefetch_l2_2d(&tma_b, (int32_t)(t.col0 + 128 * j), rp);
                    }
                }
                if (KIND == GEMM_FPROP) {
                    const int64_t kb = p.k / 128;
                    ptx::tma_load_2d(sa, &tma_a, bar, kt * BK, (int32_t)t.row0);
                    // ScaledSwiGLU: the tile's gate rows and its linear rows of W_g
                    const int64_t gc = t.col0 / 2;
                    if (ACT == 2) {
                        ptx::tma_load_2d(sb, &tma_b, bar, kt * BK, (int32_t)(t.g * p.n + gc));
                        ptx::tma_load_2d(sb + 16384, &tma_b, bar, kt * BK, (int32_t)(t.g * p.n + p.act_half + gc));
                    } else {
                        ptx::tma_load_2d(sb, &tma_b, bar, kt * BK, (int32_t)(t.g * p.n + t.col0));
                    }
                    ptx::bulk_load(ssfa, p.sfa + 512 * (kb * c.s_tp[t.g] + t.mt * kb + kt), 512, bar);
                    const int64_t wbase = kb * (int64_t)t.g * (p.n / 128);
#pragma unroll
                    for (int j = 0; j < BN / 128; ++j) {
                        const int64_t ntile = ACT == 2 ? (j == 0 ? gc : p.act_half + gc) / 128 : t.col0 / 128 + j;
                        ptx::bulk_load(ssfb + 512 * j, p.sfb + 512 * (wbase + ntile * kb + kt), 512, bar);
                    }
                } else if (KIND == GEMM_DGRAD) {
                    const int64_t nb = p.n / 128;
                    ptx::tma_load_2d(sa, &tma_a, bar, kt * BK, (int32_t)t.row0);
#pragma unroll
                    for (int j = 0; j < BN / 128; ++j)
                        ptx::tma_load_2d(sb + 16384 * j, &tma_b, bar, (int32_t)(t.col0 + 128 * j),
                                         (int32_t)(t.g * p.n + kt * BK));
                    ptx::bulk_load(ssfa, p.sfa + 512 * (nb * c.s_tp[t.g] + t.mt * nb + kt), 512, bar);
                    const int64_t wbase = (p.k / 128) * (int64_t)t.g * nb;
#pragma unroll
                    for (int j = 0; j < BN / 128; ++j)
                        ptx::bulk_load(ssfb + 512 * j,
                                       p.sfb + 512 * (wbase + (t.col0 / 128 + j) * nb + kt), 512, bar);
                } else {
                    const int32_t r = (int32_t)(t.row0 + (int64_t)kt * BK);
                    ptx::tma_load_2d(sa, &tma_a, bar, (int32_t)(t.mt * BM), r);
#pragma unroll
                    for (int j = 0; j < BN / 128; ++j)
                        ptx::tma_load_2d(sb + 16384 * j, &tma_b, bar, (int32_t)(t.col0 + 128 * j), r);
                    ptx::bulk_load(ssfa,
                                   p.sfa + 512 * ((p.n / 128) * c.s_tp[t.g] + t.mt * t.T + kt), 512,
                                   bar);
#pragma unroll
                    for (int j = 0; j < BN / 128; ++j)
                        ptx::bulk_load(ssfb + 512 * j,
                                       p.sfb + 512 * ((p.k / 128) * c.s_tp[t.g] +
                                                      (t.col0 / 128 + j) * t.T + kt),
                                       512, bar);
                }
            }
        }
        drain_loads(c.full, S::STAGES, issued, p.status);
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------- MMA issuer --
        // Stage, phase and scale slot advance by one per k-tile.  Descriptors
        // of stage 0 are built once and stepped by the stage size: their
        // address field counts 16-byte units and stays inside its 14 bits
        // (shared memory ends below 256 KB).
        const uint64_t a_desc0 = A_MN ? ptx::smem_desc(ptx::smem_addr(c.a), 16384, 1024, 2)
                                      : ptx::smem_desc(ptx::smem_addr(c.a), 16, 1024, 2);
        const uint64_t b_desc0 = B_MN ? ptx::smem_desc(ptx::smem_addr(c.b), 16384, 1024, 2)
                                      : ptx::smem_desc(ptx::smem_addr(c.b), 16, 1024, 2);
        const uint64_t sfa_desc0 = ptx::smem_desc(ptx::smem_addr(c.sfa), 0, 128, 0);
        const uint64_t sfb_desc0 = ptx::smem_desc(ptx::smem_addr(c.sfb), 0, 128, 0);
        int s = 0;
        uint32_t ph = 0, sf_slot = 0;
        int64_t tiles_done = 0, cursor = blockIdx.x, rq = 0;
        while (!*c.abort) {
            int64_t tile;
            if (!dyn) {
                tile = cursor;
                cursor += gridDim.x;
                if (tile >= ntiles)
                    break;
            } else if ((tile = ring_get<false>(ring_full, ring_empty, s_ring, rq, c.abort, p.status)) < 0) {
                break;
            }
            const Tile t = decode_tile<KIND, BN>(p, c.s_off, c.s_tp, tile, ord);
            if (t.skip || t.nk == 0)
                continue;
            const int acc = (int)(tiles_done % S::ACC);
            const uint32_t acc_ph = (uint32_t)((tiles_done / S::ACC) & 1);
            if (!ptx::mbar_wait(&c.tempty[acc], acc_ph ^ 1u, c.abort, p.status))
                break;
            ptx::tc_fence_after_sync();
            const uint32_t d = tmem + acc * BN;
            bool ok = true;
            for (int kt = 0; kt < t.nk; ++kt) {
                if (!ptx::mbar_wait(&c.full[s], ph, c.abort, p.status)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after_sync();
                const uint32_t sfa_t = tmem + S::SFA_COL + sf_slot * S::SF_STRIDE;
                const uint32_t sfb_t = tmem + S::SFB_COL + sf_slot * S::SF_STRIDE;
                ptx::tc_cp_sf_atom(sfa_t, sfa_desc0 + (uint64_t)(s * (S::SFA_BYTES >> 4)));
#pragma unroll
                for (int j = 0; j < BN / 128; ++j)
                    ptx::tc_cp_sf_atom(sfb_t + 4 * j, sfb_desc0 + (uint64_t)((s * S::SFB_BYTES + 512 * j) >> 4));
                const uint64_t ad = a_desc0 + (uint64_t)(s * (S::A_BYTES >> 4));
                const uint64_t bd = b_desc0 + (uint64_t)(s * (S::B_BYTES >> 4));
                // the wgrad's last k-tile may hold fewer than 128 live rows
                const int nsub = (KIND == GEMM_WGRAD_MX && kt == t.nk - 1) ? t.last_sub : 4;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (KIND == GEMM_WGRAD_MX && j >= nsub)
                        break;
                    // K-major: step 32 bytes along the swizzled 128-byte row;
                    // MN-major: step 32 rows of 128 bytes (16-byte units).
                    const uint64_t a_step = A_MN ? 256u * j : 2u * j;
                    const uint64_t b_step = B_MN ? 256u * j : 2u * j;
                    ptx::tc_mma_mxf8(d, ad + a_step, bd + b_step, ptx::idesc_mxf8(BM, BN, A_MN, B_MN, (uint32_t)j),
                                     sfa_t, sfb_t, (kt | j) != 0);
                }
                ptx::tc_commit(&c.empty[s]);
                if (++s == S::STAGES) {
                    s = 0;
                    ph ^= 1u;
                }
                sf_slot = (sf_slot + 1) & (S::SF_SLOTS - 1);
            }
            if (!ok)
                break;
            ptx::tc_commit(&c.tfull[acc]);
            ++tiles_done;
        }
        ptx::tc_commit(c.drain);
        volatile int no_abort = 0;
        ptx::mbar_wait(c.drain, 0, &no_abort, p.status);
    } else if (warp >= 4 && KIND == GEMM_WGRAD_MX && BN == 256) {
        // ------------------------------------- wgrad epilogue, 256 columns --
        // One accumulator fills TMEM, so the tile is drained into registers
        // at once (each of 8 warps takes its lane quadrant's 32 rows x 128
        // columns) and TMEM goes back to the MMA issuer before any byte moves
        // to the main grad: the next tile's MMAs overlap this tile's memory
        // traffic, which is what bounds the k-grouped wgrad.  Each warp sends
        // its rows as four 4 KB boxes (32 rows x 32 fp32, 128-byte swizzle)
        // through kWgSlots shared-memory slots that lane 0 hands to the TMA
        // unit.
        //   accumulate == 0: plain TMA stores.
        //   accumulate == 1: with skewed splits (kWgMixSkew) boxes 1 and 3 go
        //     by TMA reduce-add (the TMA unit adds them into the main grad at
        //     L2), the others by load + add + store: the old main-grad box
        //     comes in by TMA
        //     load, the warp adds its registers to it in place and TMA-stores
        //     the sum.  Either way one round-to-nearest fp32 add per element,
        //     so repeated calls are bitwise identical.  The loads run as one
        //     continuous stream across tiles: once a slot's store (and the
        //     reduce-add staged in the same slot after it) has read it, the
        //     slot is refilled with the load-add-store box kWgSlots further
        //     on in the warp's sequence -- in the next tile when the current
        //     one runs out, whose coordinates the warp takes one tile ahead.
        //     So kWgSlots loads stay in flight per warp whether the tile's
        //     contraction was long or short.
        constexpr int WBOX = 32 * 128;
        const int q = warp & 3, h = (warp - 4) >> 2, w = warp - 4;
        constexpr int WS = kWgSlots;
        static_assert(WS <= 2, "a refill reaches at most one tile ahead");
        uint8_t* ring = c.out + w * WS * WBOX;
        const uint32_t ring_addr = ptx::smem_addr(ring);
        uint64_t* lbar = c.obar + WS * w;                 // load barrier of each slot
        // per slot, bit s of lph is the parity of its next load completion
        // and bit s of lpend says whether a load into it is in flight (lane
        // 0's copy); load-add-store box k (counted over the call) uses slot
        // k % WS, a plain-store box k (accumulate == 0) likewise
        uint32_t lph = 0u, lpend = 0u;
        uint32_t tiles_done = 0, boxes = 0;      // only their parity / residue matters
        bool stop = false;
        int64_t cursor = blockIdx.x, rq = 0;
        const bool acc = p.accumulate != 0;
        // the warp's next tile with work (an empty group with accumulate is
        // skipped), or -1 at the end of the sequence or when a wait gave up
        auto next_tile = [&]() -> int64_t {
            for (;;) {
                int64_t tile;
                if (!dyn) {
                    tile = cursor;
                    cursor += gridDim.x;
                    if (tile >= ntiles)
                        return -1;
                } else if ((tile = ring_get<true>(ring_full, ring_empty, s_ring, rq, c.abort, p.status)) < 0) {
                    return -1;
                }
                if (!decode_tile<KIND, BN>(p, c.s_off, c.s_tp, tile, ord).skip)
                    return tile;
            }
        };
        // main-grad coordinates of box b (0..3) of tile t
        auto box_row = [&](const Tile& t) { return (int32_t)((int64_t)t.g * p.n + t.mt * BM + 32 * q); };
        auto box_col = [&](const Tile& t, int b) { return (int32_t)(t.col0 + 128 * h + 32 * b); };
        auto issue_load = [&](int slot, int32_t col, int32_t row) {     // lane 0
            ptx::mbar_arrive_expect_tx(&lbar[slot], WBOX);
            ptx::tma_load_2d(ring + slot * WBOX, &tma_o, &lbar[slot], col, row);
            lpend |= 1u << slot;
        };
        // MIX: boxes 1 and 3 of a warp's share go by reduce-add; NR
        // load-add-store boxes a tile, the j-th of them at box rmw_pos(j)
        auto epilogue = [&](auto mix_c) {
            constexpr bool MIX = decltype(mix_c)::value;
            constexpr int NR = MIX ? 2 : 4;
            auto rmw_pos = [](int j) { return MIX ? 2 * j : j; };
            int64_t cur = next_tile();
            if (acc && cur >= 0 && lane == 0) {
                const Tile t0 = decode_tile<KIND, BN>(p, c.s_off, c.s_tp, cur, ord);
                for (int j = 0; j < WS; ++j)
                    issue_load(j, box_col(t0, rmw_pos(j)), box_row(t0));
            }
            while (cur >= 0 && !stop && !*c.abort) {
                const Tile t = decode_tile<KIND, BN>(p, c.s_off, c.s_tp, cur, ord);
                const int32_t orow = box_row(t), ocol = box_col(t, 0);
                uint32_t v[4][32];
                if (t.nk > 0) {
                    if (!ptx::mbar_wait_warp(&c.tfull[0], tiles_done & 1u, c.abort, p.status))
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
                        ptx::mbar_arrive(&c.tempty[0]);
                    ++tiles_done;
                } else {                                      // empty group, accumulate = 0: dW_g = 0
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc)
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            v[cc][i] = 0u;
                }
                // one tile ahead (taken once this tile's MMAs are done, so the
                // producer has long handed it out): the refills of the last
                // boxes go to its first boxes
                const int64_t nxt = next_tile();
                int32_t nrow = 0, ncol = 0;
                if (nxt >= 0) {
                    const Tile tn = decode_tile<KIND, BN>(p, c.s_off, c.s_tp, nxt, ord);
                    nrow = box_row(tn);
                    ncol = box_col(tn, 0);
                }
                if (!acc) {
#pragma unroll
                    for (int b = 0; b < 4; ++b, ++boxes) {
                        const int slot = (int)(boxes % (uint32_t)WS);
                        const uint32_t box = ring_addr + slot * WBOX;
                        if (lane == 0) {                      // the store WS boxes back read this slot
                            if (WS == 2)
                                asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
                            else
                                asm volatile("cp.async.bulk.wait_group.read 2;" ::: "memory");
                        }
                        __syncwarp();
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            ptx::sts128(box + ptx::swz128(lane, j),
                                        make_uint4(v[b][4 * j], v[b][4 * j + 1], v[b][4 * j + 2], v[b][4 * j + 3]));
                        ptx::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            ptx::tma_store_2d(&tma_o, ring + slot * WBOX, ocol + 32 * b, orow);
                            ptx::bulk_commit_group();
                        }
                    }
                    cur = nxt;
                    continue;
                }
#pragma unroll
                for (int j = 0; j < NR; ++j, ++boxes) {
                    const int b = rmw_pos(j);
                    const int slot = (int)(boxes % (uint32_t)WS);
                    const uint32_t box = ring_addr + slot * WBOX;
                    if (!ptx::mbar_wait_warp(&lbar[slot], (lph >> slot) & 1u, c.abort, p.status)) {
                        stop = true;
                        break;
                    }
                    lph ^= 1u << slot;
                    lpend &= ~(1u << slot);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint4 o = ptx::lds128(box + ptx::swz128(lane, i));
                        ptx::sts128(box + ptx::swz128(lane, i),
                                    make_uint4(__float_as_uint(__uint_as_float(o.x) + __uint_as_float(v[b][4 * i])),
                                               __float_as_uint(__uint_as_float(o.y) + __uint_as_float(v[b][4 * i + 1])),
                                               __float_as_uint(__uint_as_float(o.z) + __uint_as_float(v[b][4 * i + 2])),
                                               __float_as_uint(__uint_as_float(o.w) + __uint_as_float(v[b][4 * i + 3]))));
                    }
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        ptx::tma_store_2d(&tma_o, ring + slot * WBOX, ocol + 32 * b, orow);
                        ptx::bulk_commit_group();
                    }
                    if constexpr (MIX) {
                        // box b + 1 goes by reduce-add, staged in this slot once
                        // the store has read it
                        if (lane == 0)
                            asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                        __syncwarp();
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            ptx::sts128(box + ptx::swz128(lane, i),
                                        make_uint4(v[b + 1][4 * i], v[b + 1][4 * i + 1], v[b + 1][4 * i + 2],
                                                   v[b + 1][4 * i + 3]));
                        ptx::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            ptx::tma_reduce_add_2d(&tma_o, ring + slot * WBOX, ocol + 32 * (b + 1), orow);
                            ptx::bulk_commit_group();
                        }
                    }
                    // refill the slot with the load-add-store box WS further on,
                    // once what was staged in it has been read
                    if (lane == 0 && (j + WS < NR || nxt >= 0)) {
                        asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                        if (j + WS < NR)
                            issue_load(slot, ocol + 32 * rmw_pos(j + WS), orow);
                        else
                            issue_load(slot, ncol + 32 * rmw_pos(j + WS - NR), nrow);
                    }
                }
                cur = nxt;
            }
        };
        // skewed splits: the largest group against the mean live group
        int32_t mmax = 0, live = 0;
        for (int g = lane; g < p.G; g += 32) {
            const int32_t m = c.s_off[g + 1] - c.s_off[g];
            mmax = max(mmax, m);
            live += m > 0;
        }
        mmax = __reduce_max_sync(0xffffffffu, mmax);
        live = __reduce_add_sync(0xffffffffu, live);
        const bool mix = acc && (int64_t)mmax * live >= kWgMixSkew * (int64_t)c.s_off[p.G];
        if (mix)
            epilogue(std::integral_constant<bool, true>{});
        else
            epilogue(std::integral_constant<bool, false>{});
        if (lane == 0) {
            // loads still in flight (an abort) land before the CTA leaves
            volatile int no_abort = 0;
            for (int sl = 0; sl < WS; ++sl)
                if ((lpend >> sl) & 1u)
                    ptx::mbar_wait(&lbar[sl], (lph >> sl) & 1u, &no_abort, p.status);
            ptx::bulk_wait_all();
        }
    } else if (warp >= 4 && KIND == GEMM_WGRAD_MX) {
        // ------------------------------------------------ wgrad epilogue --
        // The tile's fp32 result leaves through 128 x 32 boxes in shared
        // memory (128-byte swizzle): the epilogue threads copy TMEM columns
        // into a box and one lead thread hands it to the TMA unit -- a plain
        // store (accumulate == 0) or a reduction that adds it into the main
        // grad at L2 (accumulate == 1), one add per element, so repeated
        // calls are bitwise identical.  No old value passes through the SM.
        // 4 warps (BN = 128), one ring of four boxes; the warps meet on named
        // barrier 1.
        constexpr int HALVES = S::EPI_WARPS / 4;
        constexpr int SLOTS = 4 / HALVES;                 // boxes per ring
        constexpr int BOX = BM * 128;
        const int q = warp & 3, h = (warp - 4) >> 2;
        const uint32_t r = 32 * q + lane;
        const bool lead = lane == 0 && q == 0;
        const int bar_id = 1 + h;
        uint8_t* ring = c.out + h * SLOTS * BOX;
        int64_t tiles_done = 0, q_proc = 0;
        bool stop = false;
        int64_t cursor = blockIdx.x, rq = 0;
        while (!stop) {
            int64_t tile;
            if (!dyn) {
                tile = cursor;
                cursor += gridDim.x;
                if (tile >= ntiles)
                    break;
            } else {
                tile = ring_get<true>(ring_full, ring_empty, s_ring, rq, c.abort, p.status);
                // every warp of the half reads the same entry; leave together
                if (ptx::named_barrier_or(bar_id, 128, tile < 0))
                    break;
            }
            const Tile t = decode_tile<KIND, BN>(p, c.s_off, c.s_tp, tile, ord);
            if (t.skip)
                continue;
            const int32_t orow = (int32_t)((int64_t)t.g * p.n + t.mt * BM);
            bool ok = true;
            if (t.nk > 0) {
                ok = ptx::mbar_wait(&c.tfull[tiles_done % S::ACC], (uint32_t)((tiles_done / S::ACC) & 1),
                                    c.abort, p.status);
                if (ok)
                    ptx::tc_fence_after_sync();
            }
            const uint32_t tb = tmem + ((uint32_t)(32 * q) << 16) +
                                (uint32_t)(tiles_done % S::ACC) * BN + 128 * h;
#pragma unroll 1
            for (int cc = 0; cc < 4; ++cc, ++q_proc) {        // each half: 128 columns
                const int slot = (int)(q_proc % SLOTS);
                if (lead) {
                    // the store of box q_proc - SLOTS read this slot; newer ones may pend
                    if (SLOTS == 4)
                        asm volatile("cp.async.bulk.wait_group.read 3;" ::: "memory");
                    else
                        asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
                }
                if (ptx::named_barrier_or(bar_id, 128, !ok)) {
                    stop = true;
                    break;
                }
                uint32_t v[32];
                if (t.nk > 0) {
                    ptx::tmem_ld_32x32(tb + 32 * cc, v);
                    ptx::tmem_wait_ld(v);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        v[i] = 0u;
                }
                const uint32_t box = ptx::smem_addr(ring + slot * BOX);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    ptx::sts128(box + ptx::swz128(r, j), make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
                ptx::fence_proxy_async_smem();
                ptx::named_barrier_or(bar_id, 128, 0);
                if (lead) {
                    const int32_t col = (int32_t)(t.col0 + 128 * h + 32 * cc);
                    if (p.accumulate)
                        ptx::tma_reduce_add_2d(&tma_o, ring + slot * BOX, col, orow);
                    else
                        ptx::tma_store_2d(&tma_o, ring + slot * BOX, col, orow);
                    ptx::bulk_commit_group();
                }
            }
            if (t.nk > 0 && !stop) {
                ptx::tc_fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    ptx::mbar_arrive(&c.tempty[tiles_done % S::ACC]);
                ++tiles_done;
            }
        }
        if (lead)
            ptx::bulk_wait_all();
    } else if (warp >= 4 && BN == 256 && KIND != GEMM_WGRAD_MX) {
        // ------------------------------ fprop/dgrad epilogue, 256 columns --
        // One accumulator fills TMEM, so it is drained into registers (each
        // of 8 warps takes its lane quadrant's 32 rows x 128 columns) and
        // handed back at once; the next tile's MMAs overlap the stores.  Each
        // warp then writes its rows through its own 2 KB box in shared memory
        // (32 rows x 64 bytes, 64-byte swizzle) that lane 0 hands to the TMA
        // unit, box after box: whole 64-byte row segments reach L2 instead of
        // 16-byte pieces of 32 rows per store instruction.  The 32 rows of a
        // warp are all live or all past the group's end (group sizes are
        // multiples of 32), so a box is never partial.
        constexpr int CW = OUT_BF16 ? 32 : 16;           // output columns per box
        constexpr int NBOX = 128 / CW;
        const int q = warp & 3, h = (warp - 4) >> 2;
        uint8_t* box = c.out + (warp - 4) * kEpiBox;
        const uint32_t box_addr = ptx::smem_addr(box);
        const uint32_t row_addr = box_addr + 64 * lane;  // this lane's row of the box
        const uint32_t sw = (lane >> 1) & 3;             // 64-byte swizzle of that row
        int64_t tiles_done = 0;
        for (int64_t tile = blockIdx.x; tile < ntiles && !*c.abort; tile += gridDim.x) {
            const Tile t = decode_tile<KIND, BN>(p, c.s_off, c.s_tp, tile);
            if (t.skip || t.nk == 0)
                continue;
            if (!ptx::mbar_wait_warp(&c.tfull[0], (uint32_t)(tiles_done & 1), c.abort, p.status))
                break;
            ptx::tc_fence_after_sync();
            uint32_t v[4][32];
            // columns of TMEM chunk cc (32 wide) in Y: 128 h + 32 cc of the
            // tile, or for ScaledSwiGLU the warp's 64 gate columns (cc = 0, 1)
            // and the matching 64 linear columns (cc = 2, 3)
            const int64_t gc = t.col0 / 2;
            auto tmem_col = [&](int cc) -> uint32_t {
                return ACT == 2 ? (uint32_t)((cc < 2 ? 0 : 128) + 64 * h + 32 * (cc & 1)) : (uint32_t)(128 * h + 32 * cc);
            };
            auto y_col = [&](int cc) -> int32_t {
                return ACT == 2 ? (int32_t)((cc < 2 ? 0 : p.act_half) + gc + 64 * h + 32 * (cc & 1))
                                : (int32_t)(t.col0 + 128 * h + 32 * cc);
            };
            const uint32_t tb = tmem + ((uint32_t)(32 * q) << 16);
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
                ptx::tmem_ld_32x32(tb + tmem_col(cc), v[cc]);
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
                ptx::tmem_wait_ld(v[cc]);
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive(&c.tempty[0]);
            ++tiles_done;
            // the activation's scale atoms (SwiGLU: the [R, n / 2] buffer's
            // 128-column block holding the warp's 64 columns gc + 64 h)
            ActAtoms at{};
            if constexpr (ACT == 1)
                at = act_atoms(p, t, c.s_tp, p.n, t.col0 + 128 * h, q, lane);
            if constexpr (ACT == 2)
                at = act_atoms(p, t, c.s_tp, p.act_half, gc, q, lane);
            if (32 * q >= t.rows) {
                // rows past the group's end: only the zero entries of the atoms
                if constexpr (ACT == 1) {
                    *reinterpret_cast<uint32_t*>(at.row) = 0u;
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc)
                        at.col[cc * 4] = 0;
                }
                if constexpr (ACT == 2) {
                    *reinterpret_cast<uint16_t*>(at.row + 2 * h) = 0;
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc)
                        at.col[(2 * h + cc) * 4] = 0;
                }
                continue;
            }
            const int32_t orow = (int32_t)(t.row0 + 32 * q);
            // box b of the warp's output (bf16: TMEM chunk b; fp32: half b & 1
            // of chunk b >> 1) through the warp's staging box
            auto store_box = [&](int b) {
                // bias of the box's columns, added just before they are converted
                if (KIND == GEMM_FPROP && p.bias && (OUT_BF16 || (b & 1) == 0))
                    add_bias32(p, t.g, y_col(OUT_BF16 ? b : b >> 1), v[OUT_BF16 ? b : b >> 1]);
                if (lane == 0)
                    ptx::bulk_wait_read_all();           // the last box's store has read it
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
                    ptx::tma_store_2d(&tma_o, box, OUT_BF16 ? y_col(b) : y_col(b >> 1) + 16 * (b & 1), orow);
                    ptx::bulk_commit_group();
                }
            };
            // the pre-activation Y of TMEM chunk cc
            auto store_chunk = [&](int cc) {
                if (OUT_BF16) {
                    store_box(cc);
                } else {
                    store_box(2 * cc);
                    store_box(2 * cc + 1);
                }
            };
            if constexpr (ACT == 0) {
#pragma unroll
                for (int b = 0; b < NBOX; ++b)
                    store_box(b);
            } else {
                // chunk by chunk: Y, then the activation's codes and scales,
                // so that a chunk's registers are free once it is done
                const int64_t row = t.row0 + 32 * q + lane;
                const float pr = __ldg(p.act_probs + row);
                uint32_t rword = 0;
                if constexpr (ACT == 1) {
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        store_chunk(cc);
                        rword |= act_srelu_chunk(p, row, t.col0 + 128 * h + 32 * cc, pr, at.col + cc * 4, lane,
                                                 v[cc]) << (8 * cc);
                    }
                    *reinterpret_cast<uint32_t*>(at.row) = rword;
                } else {
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        store_chunk(j);
                        store_chunk(j + 2);
                        rword |= act_glu_chunk(p, row, gc + 64 * h + 32 * j, pr, at.col + (2 * h + j) * 4, lane, v[j],
                                               v[j + 2]) << (8 * j);
                    }
                    *reinterpret_cast<uint16_t*>(at.row + 2 * h) = (uint16_t)rword;
                }
            }
        }
        if (lane == 0)
            ptx::bulk_wait_all();
    } else if (warp >= 4 && BN == 128 && KIND != GEMM_WGRAD_MX) {
        // ------------------------------------------ fprop/dgrad epilogue --
        const int q = warp & 3;
        const int r = 32 * q + lane;        // row of the tile this thread writes
        int64_t tiles_done = 0;
        for (int64_t tile = blockIdx.x; tile < ntiles && !*c.abort; tile += gridDim.x) {
            const Tile t = decode_tile<KIND, BN>(p, c.s_off, c.s_tp, tile);
            if (t.skip)
                continue;
            float* out32 = nullptr;
            uint16_t* out16 = nullptr;
            const int64_t ld = KIND == GEMM_FPROP ? p.n : p.k;
            if (OUT_BF16)
                out16 = static_cast<uint16_t*>(p.out) + (t.row0 + r) * ld + t.col0;
            else
                out32 = static_cast<float*>(p.out) + (t.row0 + r) * ld + t.col0;
            const int acc = (int)(tiles_done % S::ACC);
            const uint32_t acc_ph = (uint32_t)((tiles_done / S::ACC) & 1);
            if (!ptx::mbar_wait(&c.tfull[acc], acc_ph, c.abort, p.status))
                break;
            ptx::tc_fence_after_sync();
            const bool live = r < t.rows;
            const uint32_t base = tmem + ((uint32_t)(32 * q) << 16) + acc * BN;
#pragma unroll 1
            for (int cc = 0; cc < BN / 32; ++cc) {
                uint32_t v[32];
                ptx::tmem_ld_32x32(base + 32 * cc, v);
                ptx::tmem_wait_ld(v);
                if (live) {
                    if (KIND == GEMM_FPROP && p.bias)
                        add_bias32(p, t.g, t.col0 + 32 * cc, v);
                    if (OUT_BF16)
                        store_row_bf16(out16 + 32 * cc, v);
                    else
                        store_row_f32(out32 + 32 * cc, v);
                }
            }
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive(&c.tempty[acc]);
            ++tiles_done;
        }
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, S::TMEM_COLS);
    }
}

// Whether fprop/dgrad use single-CTA 128 x 256 tiles where the output width
// allows (tuning knob).
#ifndef GQ_WIDE
#define GQ_WIDE 1
#endif
constexpr bool kWideTiles = GQ_WIDE != 0;

// ------------------------------------------------------------------------ //
// Per-channel 128-row fp32-scale k-grouped wgrad                            //
// ------------------------------------------------------------------------ //
//
// dW_g[i, j] = sum_b sfA[b, i] sfB[b, j] sum_{t in block b} qA[t, i] qB[t, j]
// Each 128-token block's unscaled partial (kind::f8f6f4) goes to one of two
// TMEM buffers; the epilogue (two warpgroups, 64 columns each) promotes it
// by the outer product of the block's channel scales into fp32 registers.
// The partial buffer is handed back only after its tcgen05.ld has completed
// (commit -> full, wait::ld -> fence -> arrive empty), so a partial is never
// overwritten while being read.

struct ChShape {
    static constexpr int BN = 128;
    static constexpr int A_BYTES = BM * BK;
    static constexpr int B_BYTES = BN * BK;
    static constexpr int STAGE = A_BYTES + B_BYTES;
    static constexpr int PBUF = 2;
    static constexpr uint32_t TMEM_COLS = 256;
    static constexpr int SCAN_BYTES = MxShape<GEMM_FPROP, 128>::SCAN_BYTES;
    static constexpr int BAR_BYTES = 8 * (2 * 8 + 2 * PBUF + 1) + 16;
    static constexpr int STAGES = 6;
    static constexpr int SMEM = 1024 + STAGES * STAGE + BAR_BYTES + SCAN_BYTES;
    static_assert(SMEM <= kSmemLimit, "shared memory budget");
};

__global__ void __launch_bounds__(384, 1)
k_gemm_wgrad_channel(const __grid_constant__ CUtensorMap tma_a,
                     const __grid_constant__ CUtensorMap tma_b, const GemmArgs p)
{
    using S = ChShape;
    constexpr int BN = S::BN;
    extern __shared__ uint8_t smem_raw[];
    const Carve c = carve(smem_raw, S::STAGES, S::A_BYTES, S::B_BYTES, 0, 0, S::PBUF);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float* sfa = reinterpret_cast<const float*>(p.sfa);
    const float* sfb = reinterpret_cast<const float*>(p.sfb);

    if (load_status(p.status) != 0)
        return;
    const int err = block_scan_splits(p.splits, p.G, p.rows_cap, 128, c.s_off, c.s_tp, c.s_w64,
                                      c.s_w32);
    if (err) {
        if (threadIdx.x == 0)
            set_status(p.status, err);
        return;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < S::STAGES; ++s) {
            ptx::mbar_init(&c.full[s], 1);
            ptx::mbar_init(&c.empty[s], 1);
        }
        for (int a = 0; a < S::PBUF; ++a) {
            ptx::mbar_init(&c.tfull[a], 1);
            ptx::mbar_init(&c.tempty[a], 8);
        }
        ptx::mbar_init(c.drain, 1);
        *c.abort = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(c.tmem_base, S::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tma_a);
        ptx::prefetch_tmap(&tma_b);
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *c.tmem_base;
    const int64_t ntiles = tile_count<GEMM_WGRAD_CHANNEL, BN>(p, c.s_tp);

    if (warp == 0 && lane == 0) {
        int64_t issued = 0;
        for (int64_t tile = blockIdx.x; tile < ntiles && !*c.abort; tile += gridDim.x) {
            const Tile t = decode_tile<GEMM_WGRAD_CHANNEL, BN>(p, c.s_off, c.s_tp, tile);
            if (t.skip || t.nk == 0)
                continue;
            for (int kt = 0; kt < t.nk; ++kt, ++issued) {
                const int s = (int)(issued % S::STAGES);
                const uint32_t ph = (uint32_t)((issued / S::STAGES) & 1);
                if (!ptx::mbar_wait(&c.empty[s], ph ^ 1u, c.abort, p.status))
                    break;
                uint64_t* bar = &c.full[s];
                ptx::mbar_arrive_expect_tx(bar, S::STAGE);
                const int32_t r = (int32_t)(t.row0 + (int64_t)kt * BK);
                ptx::tma_load_2d(c.a + s * S::A_BYTES, &tma_a, bar, (int32_t)(t.mt * BM), r);
                ptx::tma_load_2d(c.b + s * S::B_BYTES, &tma_b, bar, (int32_t)t.col0, r);
            }
        }
        drain_loads(c.full, S::STAGES, issued, p.status);
    } else if (warp == 1 && lane == 0) {
        int64_t consumed = 0, parts = 0;
        constexpr uint32_t idesc = ptx::idesc_f8(BM, BN, 1, 1);
        for (int64_t tile = blockIdx.x; tile < ntiles && !*c.abort; tile += gridDim.x) {
            const Tile t = decode_tile<GEMM_WGRAD_CHANNEL, BN>(p, c.s_off, c.s_tp, tile);
            if (t.skip || t.nk == 0)
                continue;
            bool ok = true;
            for (int kt = 0; kt < t.nk && ok; ++kt, ++consumed, ++parts) {
                const int pb = (int)(parts % S::PBUF);
                const uint32_t pph = (uint32_t)((parts / S::PBUF) & 1);
                const int s = (int)(consumed % S::STAGES);
                const uint32_t ph = (uint32_t)((consumed / S::STAGES) & 1);
                if (!ptx::mbar_wait(&c.tempty[pb], pph ^ 1u, c.abort, p.status) ||
                    !ptx::mbar_wait(&c.full[s], ph, c.abort, p.status)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after_sync();
                const uint32_t a_addr = ptx::smem_addr(c.a + s * S::A_BYTES);
                const uint32_t b_addr = ptx::smem_addr(c.b + s * S::B_BYTES);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    ptx::tc_mma_f8(tmem + pb * BN, ptx::smem_desc(a_addr + 4096 * j, 16384, 1024, 2),
                                   ptx::smem_desc(b_addr + 4096 * j, 16384, 1024, 2), idesc, j != 0);
                ptx::tc_commit(&c.empty[s]);
                ptx::tc_commit(&c.tfull[pb]);
            }
            if (!ok)
                break;
        }
        ptx::tc_commit(c.drain);
        volatile int no_abort = 0;
        ptx::mbar_wait(c.drain, 0, &no_abort, p.status);
    } else if (warp >= 4) {
        const int q = warp & 3, h = (warp - 4) >> 2;
        const int r = 32 * q + lane;
        int64_t parts = 0;
        for (int64_t tile = blockIdx.x; tile < ntiles && !*c.abort; tile += gridDim.x) {
            const Tile t = decode_tile<GEMM_WGRAD_CHANNEL, BN>(p, c.s_off, c.s_tp, tile);
            if (t.skip)
                continue;
            const int64_t n_row = t.mt * BM + r;                       // output row (channel of dY)
            const int64_t col = t.col0 + 64 * h;                       // first output column
            float* out = static_cast<float*>(p.out) + ((int64_t)t.g * p.n + n_row) * p.k + col;
            float acc[64];
#pragma unroll
            for (int i = 0; i < 64; ++i)
                acc[i] = 0.f;
            bool ok = true;
            for (int kt = 0; kt < t.nk; ++kt, ++parts) {
                const int pb = (int)(parts % S::PBUF);
                const uint32_t pph = (uint32_t)((parts / S::PBUF) & 1);
                if (!ptx::mbar_wait(&c.tfull[pb], pph, c.abort, p.status)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after_sync();
                const uint32_t base = tmem + ((uint32_t)(32 * q) << 16) + pb * BN + 64 * h;
                uint32_t v0[32], v1[32];
                ptx::tmem_ld_32x32(base, v0);
                ptx::tmem_ld_32x32(base + 32, v1);
                ptx::tmem_wait_ld(v0);
                ptx::tmem_wait_ld(v1);
                ptx::tc_fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    ptx::mbar_arrive(&c.tempty[pb]);
                const int64_t b = (t.row0 >> 7) + kt;                    // global 128-row block
                const float sa = __ldg(sfa + b * p.n + n_row);
                const float4* sb4 = reinterpret_cast<const float4*>(sfb + b * p.k + col);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 s = __ldg(sb4 + i);
                    acc[4 * i + 0] = fmaf(sa * s.x, __uint_as_float(v0[4 * i + 0]), acc[4 * i + 0]);
                    acc[4 * i + 1] = fmaf(sa * s.y, __uint_as_float(v0[4 * i + 1]), acc[4 * i + 1]);
                    acc[4 * i + 2] = fmaf(sa * s.z, __uint_as_float(v0[4 * i + 2]), acc[4 * i + 2]);
                    acc[4 * i + 3] = fmaf(sa * s.w, __uint_as_float(v0[4 * i + 3]), acc[4 * i + 3]);
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 s = __ldg(sb4 + 8 + i);
                    acc[32 + 4 * i + 0] = fmaf(sa * s.x, __uint_as_float(v1[4 * i + 0]), acc[32 + 4 * i + 0]);
                    acc[32 + 4 * i + 1] = fmaf(sa * s.y, __uint_as_float(v1[4 * i + 1]), acc[32 + 4 * i + 1]);
                    acc[32 + 4 * i + 2] = fmaf(sa * s.z, __uint_as_float(v1[4 * i + 2]), acc[32 + 4 * i + 2]);
                    acc[32 + 4 * i + 3] = fmaf(sa * s.w, __uint_as_float(v1[4 * i + 3]), acc[32 + 4 * i + 3]);
                }
            }
            if (!ok)
                break;
            float4* o = reinterpret_cast<float4*>(out);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float4 v = make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
                if (p.accumulate) {
                    const float4 old = o[i];
                    v = make_float4(old.x + v.x, old.y + v.y, old.z + v.z, old.w + v.w);
                }
                o[i] = v;
            }
        }
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, S::TMEM_COLS);
    }
}

// Zero-fill of dW for a wgrad over an empty buffer (no operand to map).
__global__ void k_zero_fill(float* __restrict__ out, int64_t count, const int32_t* status)
{
    if (load_status(status) != 0)
        return;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < count;
         i += (int64_t)gridDim.x * blockDim.x)
        out[i] = 0.f;
}

// ------------------------------------------------------------------------ //
// Host side                                                                 //
// ------------------------------------------------------------------------ //

template <typename Kernel>
cudaError_t prepare(Kernel kernel, int smem)
{
    return prepare_kernel(reinterpret_cast<const void*>(kernel), smem, 0, nullptr);
}

template <int KIND, int BN, bool OUT_BF16, int ACT = 0>
gq_status run_mx(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mo,
                 const GemmArgs& args, int64_t tiles_bound, cudaStream_t stream)
{
    using S = MxShape<KIND, BN>;
    auto kernel = k_gemm_mx<KIND, BN, OUT_BF16, ACT>;
    if (prepare(kernel, S::SMEM) != cudaSuccess)
        return GQ_ERR_CUDA;
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(tiles_bound, device_info().sm_count));
    GemmArgs a = args;
    a.front_ctas = (int)(grid * kWgFrontPct / 100);
    kernel<<<(unsigned)grid, S::THREADS, S::SMEM, stream>>>(ma, mb, mo, a);
    return cudaGetLastError() == cudaSuccess ? GQ_OK : GQ_ERR_CUDA;
}

}  // namespace

int64_t wgrad_mx_tiles(int G, int64_t n, int64_t k)
{
    const bool wide = kWideTiles && k % 256 == 0;
    return (int64_t)G * (n / 128) * (k / (wide ? 256 : 128));
}

gq_status launch_gemm(GemmKind kind, const GemmOperand& a, const GemmOperand& b,
                      const int32_t* splits, int G, int64_t rows_cap, int64_t n, int64_t k,
                      void* out, int out_dtype, int accumulate, int32_t* status,
                      cudaStream_t stream, void* workspace, const void* bias, int bias_dtype,
                      const ActOutput* act)
{
    GemmArgs args;
    args.bias = bias;
    args.bias_bf16 = bias_dtype == GQ_DTYPE_BF16;
    if (act) {
        args.act_probs = act->probs;
        args.act_row = act->row_data;
        args.act_row_scale = act->row_scale;
        args.act_col = act->col_data;
        args.act_col_scale = act->col_scale;
        args.act_half = act->mode == 2 ? n / 2 : 0;
    }
    args.splits = splits;
    args.G = G;
    args.rows_cap = rows_cap;
    args.n = n;
    args.k = k;
    args.sfa = static_cast<const uint8_t*>(a.scale);
    args.sfb = static_cast<const uint8_t*>(b.scale);
    args.out = out;
    args.accumulate = accumulate;
    args.status = status;

    if (rows_cap >= (int64_t(1) << 31) || b.rows >= (int64_t(1) << 31))
        return GQ_ERR_INVALID_ARG;
    if (rows_cap == 0) {            // wgrad over an empty buffer: dW = 0 or unchanged
        if (!accumulate) {
            k_zero_fill<<<256, 256, 0, stream>>>(static_cast<float*>(out), (int64_t)G * n * k, status);
            return cudaGetLastError() == cudaSuccess ? GQ_OK : GQ_ERR_CUDA;
        }
        return GQ_OK;
    }
    CUtensorMap ma, mb;
    switch (kind) {
    case GEMM_FPROP:
    case GEMM_DGRAD: {
        const int64_t n_out = kind == GEMM_FPROP ? n : k;
        if (!make_map_u8(&ma, a.data, a.rows, a.cols, 128) || !make_map_u8(&mb, b.data, b.rows, b.cols, 128))
            return GQ_ERR_CUDA;
        if (act && (kind != GEMM_FPROP || !kWideTiles || n_out % 256 != 0))
            return GQ_ERR_UNSUPPORTED;
        if (kWideTiles && n_out % 256 == 0) {
            // 128 x 256 tiles: B of fprop travels as one 256-row box (two
            // 128-row boxes, gate and linear rows, for ScaledSwiGLU)
            if (kind == GEMM_FPROP && !(act && act->mode == 2) && !make_map_u8(&mb, b.data, b.rows, b.cols, 256))
                return GQ_ERR_CUDA;
            // the output leaves in 32-row boxes of 64 bytes per row
            const bool bf16 = out_dtype == GQ_DTYPE_BF16;
            CUtensorMap mo;
            if (!make_tensor_map_2d_sw64(&mo, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                                         bf16 ? 2 : 4, out, rows_cap, n_out, bf16 ? 32 : 16, 32))
                return GQ_ERR_CUDA;
            const int64_t bound = ((rows_cap + 127) / 128 + G) * (n_out / 256);
            if (kind == GEMM_FPROP && act && act->mode == 2)
                return bf16 ? run_mx<GEMM_FPROP, 256, true, 2>(ma, mb, mo, args, bound, stream)
                            : run_mx<GEMM_FPROP, 256, false, 2>(ma, mb, mo, args, bound, stream);
            if (kind == GEMM_FPROP && act)
                return bf16 ? run_mx<GEMM_FPROP, 256, true, 1>(ma, mb, mo, args, bound, stream)
                            : run_mx<GEMM_FPROP, 256, false, 1>(ma, mb, mo, args, bound, stream);
            if (kind == GEMM_FPROP)
                return bf16 ? run_mx<GEMM_FPROP, 256, true>(ma, mb, mo, args, bound, stream)
                            : run_mx<GEMM_FPROP, 256, false>(ma, mb, mo, args, bound, stream);
            return bf16 ? run_mx<GEMM_DGRAD, 256, true>(ma, mb, mo, args, bound, stream)
                        : run_mx<GEMM_DGRAD, 256, false>(ma, mb, mo, args, bound, stream);
        }
        const int64_t bound = ((rows_cap + 127) / 128 + G) * (n_out / 128);
        if (kind == GEMM_FPROP)
            return out_dtype == GQ_DTYPE_BF16 ? run_mx<GEMM_FPROP, 128, true>(ma, mb, ma, args, bound, stream)
                                              : run_mx<GEMM_FPROP, 128, false>(ma, mb, ma, args, bound, stream);
        return out_dtype == GQ_DTYPE_BF16 ? run_mx<GEMM_DGRAD, 128, true>(ma, mb, ma, args, bound, stream)
                                          : run_mx<GEMM_DGRAD, 128, false>(ma, mb, ma, args, bound, stream);
    }
    case GEMM_WGRAD_MX: {
        if (!make_map_u8(&ma, a.data, a.rows, a.cols, 128) || !make_map_u8(&mb, b.data, b.rows, b.cols, 128))
            return GQ_ERR_CUDA;
        CUtensorMap mo;
        const bool wide = kWideTiles && k % 256 == 0;    // 32-row boxes per warp, else 128-row boxes
        const int64_t ntiles = wgrad_mx_tiles(G, n, k);
        if (workspace && ntiles < (int64_t(1) << 31)) {
            // run-time tile order: the claim counter starts at zero
            if (cudaMemsetAsync(workspace, 0, sizeof(unsigned long long), stream) != cudaSuccess)
                return GQ_ERR_CUDA;
            args.claim = static_cast<unsigned long long*>(workspace);
        }
        if (!make_tensor_map_2d(&mo, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, out, (int64_t)G * n, k, 32, wide ? 32 : 128))
            return GQ_ERR_CUDA;
        if (wide) {
            const int64_t bound = (int64_t)G * (n / 128) * (k / 256);
            return run_mx<GEMM_WGRAD_MX, 256, false>(ma, mb, mo, args, bound, stream);
        }
        const int64_t bound = (int64_t)G * (n / 128) * (k / 128);
        return run_mx<GEMM_WGRAD_MX, 128, false>(ma, mb, mo, args, bound, stream);
    }
    case GEMM_WGRAD_CHANNEL: {
        if (!make_map_u8(&ma, a.data, a.rows, a.cols, 128) || !make_map_u8(&mb, b.data, b.rows, b.cols, 128))
            return GQ_ERR_CUDA;
        if (prepare(k_gemm_wgrad_channel, ChShape::SMEM) != cudaSuccess)
            return GQ_ERR_CUDA;
        const int64_t bound = (int64_t)G * (n / 128) * (k / 128);
        const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(bound, device_info().sm_count));
        k_gemm_wgrad_channel<<<(unsigned)grid, 384, ChShape::SMEM, stream>>>(ma, mb, args);
        return cudaGetLastError() == cudaSuccess ? GQ_OK : GQ_ERR_CUDA;
    }
    }
    return GQ_ERR_UNSUPPORTED;
}

}  // namespace gq
