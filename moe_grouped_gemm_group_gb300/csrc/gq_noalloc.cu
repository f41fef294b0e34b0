// gq_gemm_wgrad_noalloc: the k-grouped wgrad with its tile-claim workspace
// in library-owned device memory, for callers that cannot provide one.
//
// The workspace is a file-scope __device__ array of GQ_WGRAD_WORKSPACE_BYTES
// bytes.  Every device that loads the library holds one copy of it until the
// process exits.  Host code must not pass the array's name to a kernel (on
// the host it names a stand-in object, not device memory): the device address
// is looked up with cudaGetSymbolAddress once per CUDA context, on the first
// call made with that context current, and handed to the regular entry point
// as its workspace.

#include <cuda_runtime.h>

#include <mutex>
#include <vector>

#include "gq_internal.h"

namespace {

// The claim counter of the run-time tile order lives in its first 8 bytes;
// every call clears them on its stream before the kernel runs.
static __device__ __align__(256) unsigned char g_wgrad_scratch[GQ_WGRAD_WORKSPACE_BYTES];

// The address of the array is a property of the context it was looked up in:
// a device reset or a second context on the same device loads the module
// again, at another address.  Cached addresses are keyed by the driver's
// context ID, which is unique for the life of the process (a handle value can
// be reused after its context is destroyed; an ID cannot).
struct Entry {
    unsigned long long ctx_id;
    void* addr;
};
std::mutex g_mu;
std::vector<Entry> g_addr;

// Device address of the scratch array in the current context (looked up on
// the first call there), or nullptr with *err set.
void* scratch_address(gq_status* err)
{
    unsigned long long id = 0;
    const bool have_id = gq::current_context_id(&id);     // false while no context is current
    if (have_id) {
        std::lock_guard<std::mutex> lock(g_mu);
        for (const Entry& e : g_addr)
            if (e.ctx_id == id)
                return e.addr;
    }
    // set-up in this context (a runtime call: it makes the device's primary
    // context current when none was)
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_wgrad_scratch) != cudaSuccess || !p) {
        *err = GQ_ERR_CUDA;
        return nullptr;
    }
    if (!have_id && !gq::current_context_id(&id)) {
        *err = GQ_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    for (const Entry& e : g_addr)
        if (e.ctx_id == id)
            return e.addr;
    g_addr.push_back(Entry{id, p});
    return p;
}

}  // namespace

extern "C" gq_status gq_gemm_wgrad_noalloc(const gq_quantized* dy, const gq_quantized* x,
                                           const int32_t* d_split_sizes, int32_t num_groups,
                                           int64_t n, int64_t k, float* dw, int32_t accumulate,
                                           int32_t* d_status, gq_stream_t stream)
{
    // The claim counter counts tiles in 32-bit halves: larger problems are
    // refused rather than run in another order (the count is the launcher's).
    if (num_groups >= 1 && n > 0 && k > 0 && n % 128 == 0 && k % 128 == 0 &&
        gq::wgrad_mx_tiles(num_groups, n, k) >= (int64_t(1) << 31))
        return GQ_ERR_INVALID_ARG;
    gq_status err = GQ_OK;
    void* ws = scratch_address(&err);
    if (!ws)
        return err;
    return gq_gemm_wgrad(dy, x, d_split_sizes, num_groups, n, k, dw, accumulate, ws,
                         GQ_WGRAD_WORKSPACE_BYTES, d_status, stream);
}
