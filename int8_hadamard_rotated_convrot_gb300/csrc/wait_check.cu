// Failure detection without a fault: one CTA waits on an mbarrier through the
// bounded wait that the GEMM, LoRA and ring-pack kernels use. When nothing
// arrives the wait gives up after its limit and the kernel reports
// CONVROT_ERR_TIMEOUT through the caller's status word, exactly as those
// kernels do on a stalled copy or MMA; the context stays usable. The page has
// no counterpart (it describes no device-side waits).

#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/convrot.h"
#include "internal.h"
#include "tc_common.cuh"

namespace convrot {
namespace {

__global__ void wait_check_kernel(int32_t *dev_status, uint64_t limit_ns, int arrive)
{
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = static_cast<uint32_t>(__cvta_generic_to_shared(&bar));
    if (threadIdx.x == 0) {
        tc::mbar_init(b, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0 && arrive) tc::mbar_arrive(b);
    __syncthreads();
    // Every thread waits, as the epilogue warps of the GEMM do.
    const bool ok = tc::mbar_wait(b, 0, limit_ns);
    if (!ok && threadIdx.x == 0) atomicExch(dev_status, CONVROT_ERR_TIMEOUT);
}

}  // namespace

cudaError_t launch_wait_check(int32_t *dev_status, uint64_t limit_ns, int arrive, cudaStream_t stream)
{
    wait_check_kernel<<<1, 64, 0, stream>>>(dev_status, limit_ns, arrive);
    return cudaGetLastError();
}

}  // namespace convrot
