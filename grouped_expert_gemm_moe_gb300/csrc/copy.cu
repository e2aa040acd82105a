// copy.cu -- a copy done by the SMs, for moving a layer's inputs in and its
// output out of pinned host memory.
//
// Pinned host memory (cudaHostAlloc) is mapped into the device's address
// space; on GB300 the SMs read and write it over NVLink-C2C.  Many SMs with
// 16-byte loads in flight move a few MB this way faster than one copy-engine
// transfer, and a kernel node costs less latency in a CUDA graph than a
// memcpy node, which is what an end-to-end step of a decode batch pays.
#include <algorithm>

#include "common.cuh"

namespace moe {

constexpr int CP_THREADS = 256;
constexpr int CP_UNROLL = 4;          // 16-byte loads in flight per thread

__global__ void __launch_bounds__(CP_THREADS) copy_kernel(const uint4 *__restrict__ src,
                                                          uint4 *__restrict__ dst, int64_t n) {
    pdl_wait();
    pdl_trigger();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * CP_THREADS * CP_UNROLL;
    for (int64_t i0 = static_cast<int64_t>(blockIdx.x) * CP_THREADS * CP_UNROLL + threadIdx.x;
         i0 < n; i0 += stride) {
        uint4 v[CP_UNROLL];
#pragma unroll
        for (int u = 0; u < CP_UNROLL; ++u) {
            const int64_t i = i0 + static_cast<int64_t>(u) * CP_THREADS;
            if (i < n) v[u] = __ldcs(src + i);
        }
#pragma unroll
        for (int u = 0; u < CP_UNROLL; ++u) {
            const int64_t i = i0 + static_cast<int64_t>(u) * CP_THREADS;
            if (i < n) __stcs(dst + i, v[u]);
        }
    }
}

}  // namespace moe

using namespace moe;

extern "C" moe_status moe_copy(void *dst, const void *src, size_t bytes, cudaStream_t stream) {
    if (bytes == 0) return MOE_OK;
    if (!dst || !src) return MOE_ERR_INVALID_ARG;
    if (bytes % 16 != 0 || !aligned16(dst) || !aligned16(src)) return MOE_ERR_ALIGNMENT;
    const int64_t n = static_cast<int64_t>(bytes / 16);
    const int64_t per_block = static_cast<int64_t>(CP_THREADS) * CP_UNROLL;
    const int blocks =
        static_cast<int>(std::min<int64_t>((n + per_block - 1) / per_block, sm_count() * 8ll));
    launch(copy_kernel, blocks, CP_THREADS, 0, stream, static_cast<const uint4 *>(src),
           static_cast<uint4 *>(dst), n);
    return launch_status();
}
