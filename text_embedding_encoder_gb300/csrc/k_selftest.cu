// Self-tests of device-side pieces that cannot be reached alone through the
// pass: the bounded device waits (failure detection) and the GELU that the
// GeGLU epilogue of the tensor-core projection evaluates.
//
// Failure detection.
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

// y[i] = GELU(a[i]) exactly as the GeGLU epilogue of the tensor-core
// projection computes it (tc::gelu_as: erf by Abramowitz & Stegun 7.1.26).
__global__ void selftest_gelu_kernel(const float* __restrict__ a, float* __restrict__ y, long long n) {
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) y[i] = tc::gelu_as(a[i]);
}

}  // namespace

extern "C" int tee_selftest_gelu(const float* d_a, float* d_y, long long n, void* stream) {
    if (n < 0) return tee_set_global_error(TEE_EINVAL, "selftest_gelu: n must be >= 0");
    if (n == 0) return TEE_OK;
    if (!d_a || !d_y) return tee_set_global_error(TEE_EINVAL, "selftest_gelu: NULL pointer");
    if ((reinterpret_cast<uintptr_t>(d_a) | reinterpret_cast<uintptr_t>(d_y)) & 3)
        return tee_set_global_error(TEE_EINVAL, "selftest_gelu: buffers must be 4-byte aligned");
    long long blocks = (n + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    selftest_gelu_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(d_a, d_y, n);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return tee_set_global_error(TEE_ECUDA, cudaGetErrorString(e));
    return TEE_OK;
}

cudaError_t launch_selftest_wait(long long limit_cycles, unsigned int* status, cudaStream_t s) {
    selftest_wait_kernel<<<1, 32, 0, s>>>(limit_cycles, status);
    return cudaGetLastError();
}
