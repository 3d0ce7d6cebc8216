// situ_glu_selftest.cu — a check of the tensor-core kernels' failure path that faults nothing:
// one CTA waits, with the same bounded wait the pipelines use, on an mbarrier that nothing ever
// completes. The wait must give up after its time limit, write 1 to the status word and let the
// kernel return normally, leaving the context usable.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/situ_glu.h"
#include "situ_host.h"
#include "situ_tc.cuh"

namespace {

using namespace situ_tc;

__global__ void __launch_bounds__(32, 1) wait_timeout_kernel(int* status, unsigned long long* elapsed_ns) {
    __shared__ uint64_t never;
    __shared__ Barriers bars;
    if (threadIdx.x == 0) {
        mbar_init(&never, 1);                        // one arrival expected; none will come
        bars.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    if (threadIdx.x == 0) {
        const uint64_t t0 = global_ns();
        const bool done = mbar_wait(&never, 0, &bars, status);
        if (elapsed_ns) *elapsed_ns = global_ns() - t0;
        if (done && status) atomicExch(status, 2);   // the phase cannot have completed
    }
}

}  // namespace

extern "C" {

int situ_glu_selftest_wait_timeout(int* status, unsigned long long* elapsed_ns, cudaStream_t stream) {
    if (!status || !situ_host::aligned(status, 4) || (elapsed_ns && !situ_host::aligned(elapsed_ns, 8)))
        return SITU_GLU_INVALID_ARG;
    wait_timeout_kernel<<<1, 32, 0, stream>>>(status, elapsed_ns);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return situ_host::cuda_fail(e);
    return SITU_GLU_OK;
}

}  // extern "C"
