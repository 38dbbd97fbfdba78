// Self-test of the bounded device waits that every tensor-core kernel uses.
//
// One CTA initialises an mbarrier that nothing ever arrives at and waits on
// it with the same bounded wait as the kernels (tc_ptx.cuh), under a limit
// the caller chooses.  No TMA copy, MMA or tensor-memory allocation is in
// flight, so giving up is the whole of what happens: the wait records the
// timeout in this translation unit's device error word and the kernel
// returns.  The host then sees ST_ERR_DEVICE_TIMEOUT from st_device_error,
// the same report a kernel whose wait ran out would give, and the context
// stays usable.
#include <cuda_runtime.h>

#include "common.h"
#include "tc_ptx.cuh"

namespace st {
namespace {

__global__ void __launch_bounds__(32, 1) wait_selftest_kernel(long long limit) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_word;
    const uint32_t b = tc::smem_u32(&bar);
    if (threadIdx.x == 0) {
        tc::mbar_init(b, 1);
        abort_word = 0;
        tc::fence_barrier_init();
    }
    __syncwarp();
    if (threadIdx.x == 0) tc::mbar_wait_limit(b, 0, &abort_word, limit);   // phase 0 never completes
    __syncwarp();
}

}  // namespace

int selftest_device_error(bool clear) {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, tc::g_device_error, sizeof(int)) != cudaSuccess) return -1;
    if (clear && v) {
        const int zero = 0;
        cudaMemcpyToSymbol(tc::g_device_error, &zero, sizeof(int));
    }
    return v;
}

}  // namespace st

extern "C" int st_selftest_bounded_wait(long long limit_cycles, void* stream) {
    // at least one polling round, at most the kernels' own limit (~2 s)
    if (limit_cycles < 1 || limit_cycles > st::tc::kWaitLimitCycles) return ST_ERR_INVALID_ARG;
    st::wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(limit_cycles);
    return st::record_cuda_error((int)cudaGetLastError());
}
