// selftest.cu -- a diagnostic kernel for the library's failure detection: it
// waits, through the same bounded-wait helper as every ring stage of the
// projection kernels, on a shared-memory barrier that nothing ever arrives
// on.  The wait gives up after its cycle limit, records the timeout in the
// device status word and the kernel returns: the GPU context stays usable.
#include "dec_ptx.cuh"

namespace wl {

__global__ void selftest_wait_kernel(unsigned *status)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        // phase 0 never completes: no thread arrives
        (void)mbar_wait(&bar, 0, status, kWaitRingFull);
    }
}

}  // namespace wl

using namespace wl;

extern "C" wl_status wl_selftest_wait(void *stream)
{
    wl_status st = WL_OK;
    const DeviceInfo *di = device_info(&st);
    if (!di) return st;
    selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(di->status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
    return WL_OK;
}
