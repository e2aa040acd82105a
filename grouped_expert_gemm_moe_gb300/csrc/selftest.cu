// selftest.cu -- moe_selftest_bounded_wait: the library's bounded waits run
// on a condition that is, or is not, ever met, with a short caller-given
// limit, so that a test can watch the timeout path report MOE_ERR_TIMEOUT
// through dev_error and return, with the context still usable afterwards.
//
// The waits are the very device functions the kernels use (common.cuh):
// the decode layer's grid barrier, and the mbarrier waits of the tensor-core
// kernels (one thread, and the warp-uniform form that precedes tcgen05.ld /
// tcgen05.st).  No copy or MMA is in flight while they wait: nothing but the
// wait itself can be left behind when it gives up.
#include "common.cuh"

namespace moe {

constexpr int SELFTEST_BLOCKS = 2;
constexpr int SELFTEST_THREADS = 64;

// Every CTA arrives once at the barrier; its target is the grid size (met)
// or one more (never met).  `count` ends at gridDim.x either way.
__global__ void __launch_bounds__(SELFTEST_THREADS) selftest_grid_barrier_kernel(
    unsigned *count, unsigned extra, uint64_t limit_ns, unsigned *passed, int32_t *dev_error) {
    __shared__ int fail;
    if (threadIdx.x == 0) fail = 0;
    __syncthreads();
    const bool ok = grid_barrier(count, gridDim.x + extra, &fail, dev_error, limit_ns);
    if (ok && threadIdx.x == 0) atomicAdd(passed, 1u);
}

// One mbarrier expecting one arrival; thread 0 arrives (met) or nobody does
// (never met).  warp_wide: all 32 lanes of warp 0 wait with the warp-uniform
// wait; else thread 0 alone waits.
__global__ void __launch_bounds__(32) selftest_mbar_kernel(int arrive, int warp_wide,
                                                           uint64_t limit_ns, unsigned *passed,
                                                           int32_t *dev_error) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (arrive && threadIdx.x == 0) mbar_arrive(&bar);
    __syncwarp();
    if (warp_wide) {
        const bool ok = mbar_wait_warp(&bar, 0, dev_error, limit_ns);
        if (ok) atomicAdd(passed, 1u);                  // 32 on success
    } else if (threadIdx.x == 0) {
        if (mbar_wait(&bar, 0, dev_error, limit_ns)) atomicAdd(passed, 1u);
    }
}

}  // namespace moe

extern "C" moe_status moe_selftest_bounded_wait(int kind, int satisfiable, uint64_t limit_ns,
                                                unsigned *counters, int32_t *dev_error,
                                                cudaStream_t stream) {
    using namespace moe;
    if (!counters || !dev_error) return MOE_ERR_INVALID_ARG;
    if (kind < 0 || kind > 2 || limit_ns < 1000ull || limit_ns > 10000000000ull)
        return MOE_ERR_INVALID_ARG;
    if (cudaMemsetAsync(counters, 0, 2 * sizeof(unsigned), stream) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (kind == 0) {
        // cooperative: both CTAs resident, so a met target is reached
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(SELFTEST_BLOCKS);
        cfg.blockDim = dim3(SELFTEST_THREADS);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const unsigned extra = satisfiable ? 0u : 1u;
        if (cudaLaunchKernelEx(&cfg, selftest_grid_barrier_kernel, counters, extra, limit_ns,
                               counters + 1, dev_error) != cudaSuccess)
            return MOE_ERR_CUDA;
        return launch_status();
    }
    selftest_mbar_kernel<<<1, 32, 0, stream>>>(satisfiable ? 1 : 0, kind == 2 ? 1 : 0, limit_ns,
                                               counters + 1, dev_error);
    return launch_status();
}
