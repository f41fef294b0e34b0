// Device-side helpers shared by the quantizer and GEMM kernels: status
// flag handling and the in-CTA scan of the split sizes.
#pragma once

#include <cstdint>

#include "gq_internal.h"

namespace gq {

// Volatile read of the call's status word (the noop flag).
__device__ __forceinline__ int32_t load_status(const int32_t* status)
{
    return *reinterpret_cast<const volatile int32_t*>(status);
}

// Record the first device-side error of a stream-ordered sequence.
__device__ __forceinline__ void set_status(int32_t* status, int32_t code)
{
    atomicCAS(status, 0, code);
}

// Scan of the split sizes inside one CTA (every thread calls it).
//
// Fills s_off[0..G] with the group row offsets o_g (s_off[G] = L) and
// s_tp[0..G] with the prefix sums of the 128-row tile counts
// T_g = ceil(m_g / 128).  `splits == nullptr` selects the uniform split
// rows_cap / G.  Returns 0, or GQ_ERR_SPLITS when a split is negative or not
// a multiple of `align`, or the splits sum past rows_cap; every thread gets
// the same value.  blockDim.x must be a multiple of 32.
//
// OffT is int64_t, or int32_t where the caller has bounded rows_cap below
// 2^31 (offsets never pass rows_cap: a larger sum is a split error).
template <typename OffT>
__device__ __forceinline__ int block_scan_splits(const int32_t* __restrict__ splits, int G,
                                                 int64_t rows_cap, int align, OffT* s_off,
                                                 int32_t* s_tp, int64_t* s_w64, int32_t* s_w32)
{
    const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5;
    const int nw = nt >> 5;
    const int64_t uniform = splits ? 0 : rows_cap / G;
    int64_t carry_rows = 0;
    int32_t carry_tiles = 0;
    int bad = 0;
    for (int base = 0; base < G; base += nt) {
        const int g = base + tid;
        int64_t m = 0;
        if (g < G) {
            m = splits ? (int64_t)__ldg(splits + g) : uniform;
            if (m < 0 || (m % align) != 0)
                bad = 1;
            if (m < 0)
                m = 0;
        }
        const int32_t t = (int32_t)((m + 127) >> 7);
        int64_t xr = m;
        int32_t xt = t;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int64_t yr = __shfl_up_sync(0xffffffffu, xr, d);
            const int32_t yt = __shfl_up_sync(0xffffffffu, xt, d);
            if (lane >= d) {
                xr += yr;
                xt += yt;
            }
        }
        if (lane == 31) {
            s_w64[warp] = xr;
            s_w32[warp] = xt;
        }
        __syncthreads();
        if (warp == 0) {
            int64_t wr = lane < nw ? s_w64[lane] : 0;
            int32_t wt = lane < nw ? s_w32[lane] : 0;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int64_t yr = __shfl_up_sync(0xffffffffu, wr, d);
                const int32_t yt = __shfl_up_sync(0xffffffffu, wt, d);
                if (lane >= d) {
                    wr += yr;
                    wt += yt;
                }
            }
            s_w64[lane] = wr;
            s_w32[lane] = wt;
        }
        __syncthreads();
        if (g < G) {
            s_off[g] = (OffT)(carry_rows + (warp > 0 ? s_w64[warp - 1] : 0) + xr - m);
            s_tp[g] = carry_tiles + (warp > 0 ? s_w32[warp - 1] : 0) + xt - t;
        }
        carry_rows += s_w64[nw - 1];
        carry_tiles += s_w32[nw - 1];
        __syncthreads();
    }
    if (tid == 0) {
        s_off[G] = (OffT)carry_rows;
        s_tp[G] = carry_tiles;
    }
    bad = __syncthreads_or(bad || carry_rows > rows_cap);
    return bad ? GQ_ERR_SPLITS : 0;
}

// Largest g in [0, G) with s_tp[g] <= t: the group that owns 128-row tile t
// (empty groups before it share its prefix value and lose to it).
__device__ __forceinline__ int group_of_tile(const int32_t* s_tp, int G, int64_t t)
{
    int lo = 0, hi = G - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)s_tp[mid] <= t)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

}  // namespace gq
