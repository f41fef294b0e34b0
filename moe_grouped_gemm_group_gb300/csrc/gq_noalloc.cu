// gq_gemm_wgrad_noalloc: the k-grouped wgrad with its tile-claim workspace
// in library-owned device memory, for callers that cannot provide one.
//
// The workspace is a file-scope __device__ array of GQ_WGRAD_WORKSPACE_BYTES
// bytes.  Every device that loads the library holds one copy of it until the
// process exits.  Host code must not pass the array's name to a kernel (on
// the host it names a stand-in object, not device memory): the device address
// is looked up once per device with cudaGetSymbolAddress, with that device
// current, and handed to the regular entry point as its workspace.

#include <mutex>

#include <cuda_runtime.h>

#include "gq.h"

namespace {

// The claim counter of the run-time tile order lives in its first 8 bytes;
// every call clears them on its stream before the kernel runs.
static __device__ __align__(256) unsigned char g_wgrad_scratch[GQ_WGRAD_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up on
// the first call there), or nullptr with *err set.
void* scratch_address(gq_status* err)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *err = GQ_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_wgrad_scratch) != cudaSuccess || !p) {
            *err = GQ_ERR_CUDA;
            return nullptr;
        }
        g_addr[dev] = p;
    }
    return g_addr[dev];
}

}  // namespace

extern "C" gq_status gq_gemm_wgrad_noalloc(const gq_quantized* dy, const gq_quantized* x,
                                           const int32_t* d_split_sizes, int32_t num_groups,
                                           int64_t n, int64_t k, float* dw, int32_t accumulate,
                                           int32_t* d_status, gq_stream_t stream)
{
    // The claim counter counts tiles in 32-bit halves: larger problems are
    // refused rather than run in another order.
    if (num_groups >= 1 && n > 0 && k > 0 && n % 128 == 0 && k % 128 == 0) {
        const int64_t tiles = (int64_t)num_groups * (n / 128) * (k / (k % 256 == 0 ? 256 : 128));
        if (tiles >= (int64_t(1) << 31))
            return GQ_ERR_INVALID_ARG;
    }
    gq_status err = GQ_OK;
    void* ws = scratch_address(&err);
    if (!ws)
        return err;
    return gq_gemm_wgrad(dy, x, d_split_sizes, num_groups, n, k, dw, accumulate, ws,
                         GQ_WGRAD_WORKSPACE_BYTES, d_status, stream);
}
