// selftest.cu -- exercises the bounded wait every streaming kernel relies on,
// without a fault: one CTA in which a role waits on an mbarrier phase that
// nothing ever completes.  It gives up after the limit, records
// FFN_ERR_TIMEOUT in the device status word and raises the CTA's abort flag;
// a second role, waiting with a far longer limit on another such barrier, is
// released by that flag within about a millisecond (the suspend hint of the
// wait), exactly the path the GEMM and decode kernels take when a copy or a
// peer never arrives.  The kernel then returns normally: the context stays
// usable.
#include "ffn_internal.cuh"

namespace ffn {
namespace {

__global__ void __launch_bounds__(64) bounded_wait_probe_kernel(uint64_t limit_ns, unsigned *err) {
    __shared__ __align__(8) uint64_t bar_a, bar_b;
    __shared__ int s_abort;
    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_u32(&bar_a), 1);
        ptx::mbar_init(ptx::smem_u32(&bar_b), 1);
        s_abort = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();
    volatile int *abort_flag = &s_abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        // warp 0: gives up after limit_ns; warp 1: would wait 1000x longer
        const uint64_t limit = warp == 0 ? limit_ns : 1000 * limit_ns;
        const uint32_t bar = ptx::smem_u32(warp == 0 ? &bar_a : &bar_b);
        if (!ptx::mbar_wait(bar, 0, abort_flag, limit)) {
            atomicOr(err, DEVERR_TIMEOUT);
            *abort_flag = 1;
        }
    }
    __syncthreads();
}

}  // namespace

cudaError_t launch_bounded_wait_probe(uint64_t limit_ns, cudaStream_t s) {
    unsigned *err = device_status_word();
    if (!err) return cudaErrorUnknown;
    LaunchScope scope(K_SELFTEST, s);
    bounded_wait_probe_kernel<<<1, 64, 0, s>>>(limit_ns, err);
    return cudaGetLastError();
}

}  // namespace ffn
