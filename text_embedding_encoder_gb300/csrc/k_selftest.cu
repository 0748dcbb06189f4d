// Failure-detection self-test of the bounded device waits.
//
// Every pipeline wait in the tensor-core kernels is an mbarrier wait with a
// cycle limit; when it expires the kernel raises its abort flag, drains, frees
// TMEM and sets the timeout bit of the context's status word.  This kernel
// exercises that path on purpose: one thread waits, with the same bounded
// wait, on a barrier that nothing ever completes, and records the expiry in
// the status word.  It returns once the limit expires; nothing faults.
#include "tee_internal.cuh"

#include "tc_ptx.cuh"

namespace {

__global__ void selftest_wait_kernel(long long limit, unsigned int* status) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    const uint32_t b = tc::smem_u32(&bar);
    tc::mbar_init(b, 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // phase 0 needs one arrival that never comes
    if (!tc::mbar_wait_limit(b, 0, &abort_flag, limit)) atomicOr(status, TEE_STATUS_TIMEOUT);
}

}  // namespace

cudaError_t launch_selftest_wait(long long limit_cycles, unsigned int* status, cudaStream_t s) {
    selftest_wait_kernel<<<1, 32, 0, s>>>(limit_cycles, status);
    return cudaGetLastError();
}
