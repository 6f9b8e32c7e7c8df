// Self-test of the bounded waits every kernel of the library relies on: a
// single CTA waits on a shared-memory barrier that nothing completes, with
// the same helper (mbar_wait) and a caller-given time limit.  When the limit
// passes the wait gives up, the kernel raises HPC_FLAG_TIMEOUT and returns,
// so the context stays usable.  No fault, trap or unbounded wait is involved.
#include "internal.h"
#include "ptx.cuh"

namespace hpc {
namespace {

__global__ void selftest_wait_kernel(int32_t *flags, unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_word;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);  // one arrival expected; none ever comes
        abort_word = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        volatile int *abort = &abort_word;
        if (!mbar_wait(&bar, 0, abort, limit_ns)) atomicOr(flags, (int)HPC_FLAG_TIMEOUT);
    }
}

}  // namespace
}  // namespace hpc

using namespace hpc;

extern "C" hpc_status hpc_selftest_wait_timeout(int32_t *d_flags, int32_t limit_us,
                                                hpc_stream_t stream) {
    if (!d_flags || limit_us < 1 || limit_us > 1000000) return HPC_ERR_ARG;
    selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        d_flags, (unsigned long long)limit_us * 1000ull);
    return cudaGetLastError() == cudaSuccess ? HPC_OK : HPC_ERR_CUDA;
}
