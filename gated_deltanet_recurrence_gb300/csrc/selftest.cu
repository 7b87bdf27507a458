// selftest.cu -- gdn_selftest_bounded_wait: shows that the library's bounded device wait gives up.
//
// Every tensor-core kernel waits on mbarriers (TMA arrivals, MMA commits, hand-offs between warp
// roles) through ptx::mbar_wait, which stops polling once its time bound has passed; the kernel
// then records GDN_ERR_TIMEOUT, stops issuing work and returns, so a lost arrival costs an error
// status instead of a hung GPU.  This entry point runs that same wait on a phase that nothing
// ever completes, with a short bound chosen by the caller, and writes what the wait reported:
// the expiry path is exercised without faulting, trapping or hanging anything.
#include "gdn_internal.cuh"
#include "sm100_ptx.cuh"

namespace {

using namespace gdn::ptx;

// One thread: an mbarrier expecting one arrival that never comes.  Waiting for its first phase
// (parity 0) cannot succeed, so mbar_wait returns false once limit_ns has passed.
__global__ void bounded_wait_kernel(uint64_t limit_ns, int* status) {
    __shared__ uint64_t bar;
    mbar_init(&bar, 1);
    fence_mbar_init();
    const bool completed = mbar_wait(&bar, 0, limit_ns);
    *status = completed ? GDN_OK : GDN_ERR_TIMEOUT;
}

}  // namespace

extern "C" int gdn_selftest_bounded_wait(unsigned long long limit_ns, int* device_status,
                                         void* stream) {
    if (!device_status || (reinterpret_cast<uintptr_t>(device_status) & 3u) != 0) return GDN_ERR_ARG;
    if (limit_ns < 1000ull || limit_ns > 1000000000ull) return GDN_ERR_ARG;
    bounded_wait_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(limit_ns, device_status);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}
