// gq_check_wait_limit: a self-check of the bounded wait that every kernel of
// the library takes on its mbarriers (ptx::mbar_wait / mbar_wait_warp).
//
// One CTA of two warps waits on an mbarrier that nothing ever arrives on.
// The first warp to pass the wait limit records GQ_ERR_TIMEOUT in the status
// word and raises the CTA's abort flag; the other warp, polling the flag,
// gives up too.  Both report how long they waited and whether the barrier's
// phase completed (it never does), and the kernel returns normally, so the
// CUDA context stays usable and the host reads the status as it reads any
// other device-side error.  Nothing is faulted, trapped or left running.

#include <cuda_runtime.h>

#include "gq.h"
#include "gq_ptx.cuh"

namespace {

__global__ void __launch_bounds__(64, 1) k_check_wait_limit(int32_t* status, uint64_t* report)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    // The noop flag: every thread reads it before anyone can write it.
    if (gq::load_status(status) != 0)
        return;
    if (threadIdx.x == 0) {
        gq::ptx::mbar_init(&bar, 1);
        gq::ptx::fence_barrier_init();
        abort_flag = 0;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5;
    const uint64_t t0 = gq::ptx::globaltimer();
    const bool done = gq::ptx::mbar_wait_warp(&bar, 0u, &abort_flag, status);
    const uint64_t t1 = gq::ptx::globaltimer();
    if ((threadIdx.x & 31) == 0 && report) {
        report[2 * warp] = t1 - t0;
        report[2 * warp + 1] = done ? 1u : 0u;
    }
}

}  // namespace

extern "C" gq_status gq_check_wait_limit(int32_t* d_status, uint64_t* d_report, gq_stream_t stream)
{
    if (!d_status)
        return GQ_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(d_status) % 4 != 0 || reinterpret_cast<uintptr_t>(d_report) % 8 != 0)
        return GQ_ERR_ALIGNMENT;
    k_check_wait_limit<<<1, 64, 0, (cudaStream_t)stream>>>(d_status, d_report);
    return cudaGetLastError() == cudaSuccess ? GQ_OK : GQ_ERR_CUDA;
}
