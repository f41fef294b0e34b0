// Host-side helpers: per-device facts and the TMA tensor-map encoder (taken
// from the driver at run time, so that loading the library needs no GPU).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <map>
#include <mutex>

#include "gq_internal.h"

namespace gq {

const DeviceInfo& device_info()
{
    // one entry per device ordinal, filled on first use (node addresses stay
    // valid as the map grows)
    static std::mutex mu;
    static std::map<int, DeviceInfo> infos;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0)
        dev = 0;
    std::lock_guard<std::mutex> lock(mu);
    auto it = infos.find(dev);
    if (it != infos.end())
        return it->second;
    DeviceInfo d;
    cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
    int optin = 0;
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    d.smem_optin = (size_t)optin;
    if (d.sm_count <= 0)
        d.sm_count = 1;
    return infos.emplace(dev, d).first->second;
}

bool current_context_id(unsigned long long* id)
{
    using PfnCtxGetCurrent = CUresult (*)(CUcontext*);
    using PfnCtxGetId = CUresult (*)(CUcontext, unsigned long long*);
    static PfnCtxGetCurrent get_current = nullptr;
    static PfnCtxGetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PfnCtxGetCurrent>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PfnCtxGetId>(p);
    });
    if (!get_current || !get_id)
        return false;
    CUcontext ctx = nullptr;
    return get_current(&ctx) == CUDA_SUCCESS && ctx && get_id(ctx, id) == CUDA_SUCCESS;
}

cudaError_t prepare_kernel(const void* fn, int dyn_smem, int threads, int* blocks_per_sm)
{
    struct Entry {
        const void* fn;
        unsigned long long ctx;
        int dyn_smem, threads, per_sm;
    };
    static std::mutex mu;
    static Entry cache[256];
    static int used = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return cudaErrorInvalidDevice;
    // a runtime call that makes the device's primary context current when
    // no context is yet (the first call of a process)
    unsigned long long ctx = 0;
    if (!current_context_id(&ctx)) {
        if (cudaSetDevice(dev) != cudaSuccess || !current_context_id(&ctx))
            return cudaErrorInvalidDevice;
    }
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i) {
        const Entry& e = cache[i];
        if (e.fn == fn && e.ctx == ctx && e.dyn_smem == dyn_smem && e.threads == threads) {
            if (blocks_per_sm)
                *blocks_per_sm = e.per_sm;
            return cudaSuccess;
        }
    }
    if (dyn_smem > 48 * 1024) {
        const cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_smem);
        if (err != cudaSuccess)
            return err;
    }
    int n = 1;
    if (threads > 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, (size_t)dyn_smem) != cudaSuccess) {
            (void)cudaGetLastError();            // leave no error behind for the launch check
            n = 1;
        }
        if (n < 1)
            n = 1;
    }
    if (used < 256)
        cache[used++] = Entry{fn, ctx, dyn_smem, threads, n};
    if (blocks_per_sm)
        *blocks_per_sm = n;
    return cudaSuccess;
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

}  // namespace

namespace {

bool encode_2d(CUtensorMap* map, CUtensorMapDataType dtype, int elem_bytes, const void* base,
               int64_t rows, int64_t cols, int box_cols, int box_rows, CUtensorMapSwizzle swizzle)
{
    auto enc = tensor_map_encoder();
    if (!enc || rows <= 0 || cols <= 0)
        return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * (cuuint64_t)elem_bytes};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    const CUresult r = enc(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

bool make_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, int elem_bytes,
                        const void* base, int64_t rows, int64_t cols, int box_cols, int box_rows)
{
    return encode_2d(map, dtype, elem_bytes, base, rows, cols, box_cols, box_rows,
                     CU_TENSOR_MAP_SWIZZLE_128B);
}

bool make_tensor_map_2d_sw64(CUtensorMap* map, CUtensorMapDataType dtype, int elem_bytes,
                             const void* base, int64_t rows, int64_t cols, int box_cols,
                             int box_rows)
{
    return encode_2d(map, dtype, elem_bytes, base, rows, cols, box_cols, box_rows,
                     CU_TENSOR_MAP_SWIZZLE_64B);
}

bool make_tensor_map_2d_plain(CUtensorMap* map, CUtensorMapDataType dtype, int elem_bytes,
                              const void* base, int64_t rows, int64_t cols, int box_cols,
                              int box_rows)
{
    return encode_2d(map, dtype, elem_bytes, base, rows, cols, box_cols, box_rows,
                     CU_TENSOR_MAP_SWIZZLE_NONE);
}

}  // namespace gq
