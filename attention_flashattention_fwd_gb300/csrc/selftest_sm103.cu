// selftest_sm103.cu -- a kernel whose barrier wait can never complete, to
// check the library's failure path on the GPU without faulting it.
//
// Every pipeline wait in the attention kernels is bounded (mbar_wait and the
// waits built on mbar_try_wait give up after kWaitLimitNs); a wait that runs
// out sets a bit in a device error word, the kernel leaves its loops, and
// attn_device_error reports ATTN_ERR_TIMEOUT.  This kernel initialises an
// mbarrier that nothing ever arrives on, waits on it with the same bounded
// wait, and reports through the same path, so a test can see the whole
// failure path run out, report, and leave the context usable.
#include "gbattn_internal.h"
#include "sm103_ptx.cuh"

namespace gbattn {

__device__ unsigned int g_selftest_error = 0;

__global__ void attn_selftest_timeout_kernel() {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    const uint32_t b = smem_addr(&bar);
    mbar_init(b, 1);
    fence_barrier_init();
    if (!mbar_wait(b, 0)) atomicOr(&g_selftest_error, kErrBitTimeout);  // nothing arrives
}

// The index check of the debug builds on an index one past the end of a
// one-element buffer: the check fails, sets kErrBitBounds and the kernel makes
// no access at all (in either build: the access is not written).
__global__ void attn_selftest_bounds_kernel(long long n) {
    if (threadIdx.x != 0) return;
    (void)gb_index_ok(&g_selftest_error, n, n, n);
}

int launch_selftest_bounds(cudaStream_t stream) {
#ifdef GBATTN_DEBUG
    attn_selftest_bounds_kernel<<<1, 32, 0, stream>>>(1);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
#else
    (void)stream;
    return ATTN_ERR_UNSUPPORTED;  // release builds carry no index checks
#endif
}

int launch_selftest_timeout(cudaStream_t stream) {
    attn_selftest_timeout_kernel<<<1, 32, 0, stream>>>();
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

unsigned read_and_clear_selftest_error() {
    unsigned v = 0, zero = 0;
    cudaMemcpyFromSymbol(&v, g_selftest_error, sizeof v);
    cudaMemcpyToSymbol(g_selftest_error, &zero, sizeof zero);
    return v;
}

}  // namespace gbattn
