// route.cu -- router logits and top-k routing.
//
// Routing is one warp per token with a warp-shuffle top-k ("switchyard"
// page, 02 Kernels and dispatch, "Route and sort": each token routed in one
// warp).  Each lane holds E/32 logits in registers; k rounds of a warp
// arg-max (larger logit wins, ties go to the lower expert index) pick the
// experts in descending order.  The softmax runs over all E logits; the
// difference L_e - max is corrected for its fp32 rounding (an error-free
// two-term difference) before expf, and the denominator is summed in fp64,
// so each weight is within a few fp32 ulps of the exact value.
#include <math.h>

#include "common.cuh"

namespace moe {

template <int PER_LANE>
__global__ void __launch_bounds__(256) route_kernel(const float *__restrict__ logits, int T,
                                                    int E, int k, int renormalize,
                                                    int32_t *__restrict__ topk_ids,
                                                    float *__restrict__ topk_w,
                                                    int32_t *dev_error) {
    const int lane = lane_id();
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (t >= T) return;
    const float *L = logits + static_cast<size_t>(t) * E;

    float v[PER_LANE];
    bool nan_seen = false;
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
        const int e = lane + 32 * i;
        v[i] = e < E ? __ldg(L + e) : -INFINITY;
        nan_seen |= isnan(v[i]);
    }
    if (__any_sync(FULL, nan_seen)) {
        if (lane == 0) report(dev_error, MOE_ERR_DEVICE_CHECK);
        return;
    }

    uint32_t taken = 0;          // bit i: expert lane + 32 i already chosen
    int my_id = 0;               // lane j < k keeps the j-th choice
    float my_val = 0.f, vmax = 0.f;
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i) {
            const int e = lane + 32 * i;
            if (e < E && !((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < bi))) {
                bv = v[i];
                bi = e;
            }
        }
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) {
            const float ov = __shfl_xor_sync(FULL, bv, d);
            const int oi = __shfl_xor_sync(FULL, bi, d);
            if (ov > bv || (ov == bv && oi < bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        if (lane == j) {
            my_id = bi;
            my_val = bv;
        }
        if (j == 0) vmax = bv;
    }

    // exp(L_e - max): s = fl(L_e - max) and its exact rounding error r from
    // Knuth's two-sum, so exp(L_e - max) = expf(s) * exp(r) ~= expf(s) * (1 + r).
    auto shifted_exp = [vmax](float x) {
        const float s = x - vmax;
        const float bb = s - x;
        float r = (x - (s - bb)) + (-vmax - bb);
        if (!isfinite(r)) r = 0.f;
        const float e = expf(s);
        return fmaf(e, r, e);
    };
    double den = 0.0;
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
        const int e = lane + 32 * i;
        if (e < E) den += static_cast<double>(shifted_exp(v[i]));
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) den += __shfl_xor_sync(FULL, den, d);

    const float ej = lane < k ? shifted_exp(my_val) : 0.f;
    double sel = static_cast<double>(ej);
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) sel += __shfl_xor_sync(FULL, sel, d);

    if (lane < k) {
        const double w = static_cast<double>(ej) / (renormalize ? sel : den);
        topk_ids[static_cast<size_t>(t) * k + lane] = my_id;
        topk_w[static_cast<size_t>(t) * k + lane] = static_cast<float>(w);
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
        route_kernel<1><<<blocks, threads, 0, stream>>>(logits, T, E, k, renormalize, topk_ids, topk_w, dev_error);
    else if (per_lane <= 2)
        route_kernel<2><<<blocks, threads, 0, stream>>>(logits, T, E, k, renormalize, topk_ids, topk_w, dev_error);
    else if (per_lane <= 4)
        route_kernel<4><<<blocks, threads, 0, stream>>>(logits, T, E, k, renormalize, topk_ids, topk_w, dev_error);
    else if (per_lane <= 8)
        route_kernel<8><<<blocks, threads, 0, stream>>>(logits, T, E, k, renormalize, topk_ids, topk_w, dev_error);
    else if (per_lane <= 16)
        route_kernel<16><<<blocks, threads, 0, stream>>>(logits, T, E, k, renormalize, topk_ids, topk_w, dev_error);
    else
        route_kernel<32><<<blocks, threads, 0, stream>>>(logits, T, E, k, renormalize, topk_ids, topk_w, dev_error);
    return launch_status();
}

extern "C" moe_status moe_router_logits(const uint16_t *x, const uint16_t *w_r, const float *bias,
                                        int T, int H, int E, float *logits, cudaStream_t stream) {
    if (!x || !w_r || !logits || T < 1 || H < 1 || E < 1) return MOE_ERR_INVALID_ARG;
    if (static_cast<int64_t>(T) * H >= (1ll << 31) || static_cast<int64_t>(E) * H >= (1ll << 31))
        return MOE_ERR_UNSUPPORTED;
    dim3 grid((T + 15) / 16, (E + 63) / 64);
    router_logits_kernel<<<grid, 256, 0, stream>>>(x, w_r, bias, T, H, E, logits);
    return launch_status();
}
