// selftest.cu -- exercises the bounded-wait path of the kernels without a
// fault: one thread waits on an mbarrier phase that nothing completes.
#include "internal.h"
#include "ptx.cuh"

namespace dsa {
namespace {

__global__ void wait_timeout_kernel(uint64_t limit_ns, int32_t* status) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_mbar_init();
        // nobody arrives: the wait gives up after limit_ns
        if (!mbar_wait_for(smem_u32(&bar), 0, limit_ns)) latch_status(status, DSA_ERR_TIMEOUT);
    }
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" dsa_status dsa_selftest_wait_timeout(void* ws, uint32_t limit_us, void* stream) {
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 15u)) return DSA_ERR_WORKSPACE;
    if (limit_us == 0 || limit_us > 1000000u) return DSA_ERR_INVALID_ARG;
    wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>((uint64_t)limit_us * 1000u,
                                                                         static_cast<int32_t*>(ws));
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return DSA_ERR_CUDA;
    count_launches(1);
    return DSA_OK;
}
