// route.cu -- router logits and top-k routing (one warp per token, see
// route_token.cuh).
#include "route_token.cuh"

namespace moe {

template <int PER_LANE>
__global__ void __launch_bounds__(256) route_kernel(const float *__restrict__ logits, int T,
                                                    int E, int k, int renormalize,
                                                    int32_t *__restrict__ topk_ids,
                                                    float *__restrict__ topk_w,
                                                    int32_t *dev_error) {
    pdl_wait();
    pdl_trigger();
    const int lane = lane_id();
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (t >= T) return;
    int id;
    float w;
    if (!route_token<PER_LANE>(logits + static_cast<size_t>(t) * E, E, k, renormalize, id, w)) {
        if (lane == 0) report(dev_error, MOE_ERR_DEVICE_CHECK);
        return;
    }
    if (lane < k) {
        topk_ids[static_cast<size_t>(t) * k + lane] = id;
        topk_w[static_cast<size_t>(t) * k + lane] = w;
    }
}

// logits[t,e] = sum_c x[t,c] * w_r[e,c] (+ bias[e]).  A block computes a
// 16-token x 64-expert tile; x and w_r chunks of 64 columns are staged in
// shared memory as fp32; every output is summed over c in ascending order.
__global__ void __launch_bounds__(256) router_logits_kernel(const uint16_t *__restrict__ x,
                                                            const uint16_t *__restrict__ w_r,
                                                            const float *__restrict__ bias,
                                                            int T, int H, int E,
                                                            float *__restrict__ logits) {
    __shared__ float xs[16][65];
    __shared__ float ws[64][65];
    pdl_wait();
    pdl_trigger();
    const int t0 = blockIdx.x * 16, e0 = blockIdx.y * 64;
    const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int c0 = 0; c0 < H; c0 += 64) {
        for (int i = threadIdx.x; i < 16 * 64; i += 256) {
            const int r = i / 64, c = i % 64;
            const int t = t0 + r, cc = c0 + c;
            xs[r][c] = (t < T && cc < H) ? bf_lo(x[static_cast<size_t>(t) * H + cc]) : 0.f;
        }
        for (int i = threadIdx.x; i < 64 * 64; i += 256) {
            const int r = i / 64, c = i % 64;
            const int e = e0 + r, cc = c0 + c;
            ws[r][c] = (e < E && cc < H) ? bf_lo(w_r[static_cast<size_t>(e) * H + cc]) : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int c = 0; c < 64; ++c) {
            const float xv = xs[ty][c];
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[q] = fmaf(xv, ws[tx + 16 * q][c], acc[q]);
        }
        __syncthreads();
    }
    const int t = t0 + ty;
    if (t < T) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int e = e0 + tx + 16 * q;
            if (e < E) logits[static_cast<size_t>(t) * E + e] = acc[q] + (bias ? bias[e] : 0.f);
        }
    }
}

}  // namespace moe

using namespace moe;

extern "C" moe_status moe_route(const float *logits, int T, int E, int k, int renormalize,
                                int32_t *topk_ids, float *topk_w, int32_t *dev_error,
                                cudaStream_t stream) {
    if (!logits || !topk_ids || !topk_w || T < 1 || E < 1 || k < 1 || k > E || k > 32)
        return MOE_ERR_INVALID_ARG;
    if (E > 1024) return MOE_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(T) * E >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
    const int threads = 256, blocks = (T + 7) / 8;
    const int per_lane = (E + 31) / 32;
    if (per_lane <= 1)
        launch(route_kernel<1>, blocks, threads, 0, stream, logits, T, E, k, renormalize, topk_ids, topk_w, dev_error);
    else if (per_lane <= 2)
        launch(route_kernel<2>, blocks, threads, 0, stream, logits, T, E, k, renormalize, topk_ids, topk_w, dev_error);
    else if (per_lane <= 4)
        launch(route_kernel<4>, blocks, threads, 0, stream, logits, T, E, k, renormalize, topk_ids, topk_w, dev_error);
    else if (per_lane <= 8)
        launch(route_kernel<8>, blocks, threads, 0, stream, logits, T, E, k, renormalize, topk_ids, topk_w, dev_error);
    else if (per_lane <= 16)
        launch(route_kernel<16>, blocks, threads, 0, stream, logits, T, E, k, renormalize, topk_ids, topk_w, dev_error);
    else
        launch(route_kernel<32>, blocks, threads, 0, stream, logits, T, E, k, renormalize, topk_ids, topk_w, dev_error);
    return launch_status();
}

extern "C" moe_status moe_router_logits(const uint16_t *x, const uint16_t *w_r, const float *bias,
                                        int T, int H, int E, float *logits, cudaStream_t stream) {
    if (!x || !w_r || !logits || T < 1 || H < 1 || E < 1) return MOE_ERR_INVALID_ARG;
    if (static_cast<int64_t>(T) * H >= (1ll << 31) || static_cast<int64_t>(E) * H >= (1ll << 31))
        return MOE_ERR_UNSUPPORTED;
    dim3 grid((T + 15) / 16, (E + 63) / 64);
    launch(router_logits_kernel, grid, 256, 0, stream, x, w_r, bias, T, H, E, logits);
    return launch_status();
}
