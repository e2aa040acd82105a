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

// logits[t,e] = sum_c x[t,c] * w_r[e,c] (+ bias[e]).  A block computes TOK
// tokens x 64 experts; its 8 warps split the hidden dimension into 8
// contiguous ranges of 16-byte chunks, and lane l of a warp owns experts
// e0+l and e0+l+32 for all TOK tokens.  Per chunk a lane reads its two
// w_r chunks and the TOK x chunks (the same address across the warp, one
// broadcast each).  Each warp's partial sums (columns ascending) are then
// added in warp order 0..7 through shared memory, so every logit has one
// fixed summation order.
constexpr int RL_WARPS = 8;

template <int TOK>
__global__ void __launch_bounds__(RL_WARPS * 32) router_logits_kernel(
    const uint16_t *__restrict__ x, const uint16_t *__restrict__ w_r,
    const float *__restrict__ bias, int T, int H, int E, float *__restrict__ logits) {
    __shared__ float part[RL_WARPS][TOK][64];
    pdl_wait();
    pdl_trigger();
    const int lane = lane_id(), warp = threadIdx.x >> 5;
    const int t0 = blockIdx.x * TOK, e0 = blockIdx.y * 64;
    const int chunks = H / 8;
    const int c_begin = warp * chunks / RL_WARPS, c_end = (warp + 1) * chunks / RL_WARPS;
    const int ea = e0 + lane, eb = e0 + lane + 32;
    const bool has_a = ea < E, has_b = eb < E;
    const uint16_t *wa = w_r + static_cast<int64_t>(has_a ? ea : 0) * H;
    const uint16_t *wb = w_r + static_cast<int64_t>(has_b ? eb : 0) * H;
    const uint16_t *xr[TOK];
#pragma unroll
    for (int i = 0; i < TOK; ++i)
        xr[i] = x + static_cast<int64_t>(t0 + i < T ? t0 + i : 0) * H;
    float acc[TOK][2];
#pragma unroll
    for (int i = 0; i < TOK; ++i) acc[i][0] = acc[i][1] = 0.f;
#pragma unroll 4
    for (int c = c_begin; c < c_end; ++c) {
        const uint4 va = ld_nc(wa + c * 8), vb = ld_nc(wb + c * 8);
        uint4 vx[TOK];
#pragma unroll
        for (int i = 0; i < TOK; ++i) vx[i] = ld_nc(xr[i] + c * 8);
        const uint32_t pa[4] = {va.x, va.y, va.z, va.w}, pb[4] = {vb.x, vb.y, vb.z, vb.w};
#pragma unroll
        for (int i = 0; i < TOK; ++i) {
            const uint32_t px[4] = {vx[i].x, vx[i].y, vx[i].z, vx[i].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float x0 = bf_lo(px[q]), x1 = bf_hi(px[q]);
                acc[i][0] = fmaf(x0, bf_lo(pa[q]), acc[i][0]);
                acc[i][0] = fmaf(x1, bf_hi(pa[q]), acc[i][0]);
                acc[i][1] = fmaf(x0, bf_lo(pb[q]), acc[i][1]);
                acc[i][1] = fmaf(x1, bf_hi(pb[q]), acc[i][1]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < TOK; ++i) {
        part[warp][i][lane] = acc[i][0];
        part[warp][i][lane + 32] = acc[i][1];
    }
    __syncthreads();
    for (int o = threadIdx.x; o < TOK * 64; o += blockDim.x) {
        const int i = o / 64, e = e0 + o % 64, t = t0 + i;
        if (t >= T || e >= E) continue;
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < RL_WARPS; ++w) v += part[w][i][o % 64];
        logits[static_cast<int64_t>(t) * E + e] = v + (bias ? bias[e] : 0.f);
    }
}

// Router logits and top-k in one launch.  A CTA takes TOK tokens: for each
// block of 64 experts its 8 warps form the logits exactly as
// router_logits_kernel does (the same per-logit summation order, so the
// same fp32 values), into shared memory; then warp i routes token i from
// those logits with route_token, so ids and weights equal those of
// moe_router_logits followed by moe_route bit for bit.
template <int TOK, int PER_LANE>
__global__ void __launch_bounds__(RL_WARPS * 32) router_route_kernel(
    const uint16_t *__restrict__ x, const uint16_t *__restrict__ w_r,
    const float *__restrict__ bias, int T, int H, int E, int k, int renormalize,
    float *__restrict__ logits, int32_t *__restrict__ topk_ids, float *__restrict__ topk_w,
    int32_t *dev_error) {
    __shared__ float part[RL_WARPS][TOK][64];
    extern __shared__ float s_logits[];              // [TOK][E]
    pdl_wait();
    pdl_trigger();
    const int lane = lane_id(), warp = threadIdx.x >> 5;
    const int t0 = blockIdx.x * TOK;
    const int chunks = H / 8;
    const int c_begin = warp * chunks / RL_WARPS, c_end = (warp + 1) * chunks / RL_WARPS;
    const uint16_t *xr[TOK];
#pragma unroll
    for (int i = 0; i < TOK; ++i)
        xr[i] = x + static_cast<int64_t>(t0 + i < T ? t0 + i : 0) * H;
    for (int e0 = 0; e0 < E; e0 += 64) {
        const int ea = e0 + lane, eb = e0 + lane + 32;
        const uint16_t *wa = w_r + static_cast<int64_t>(ea < E ? ea : 0) * H;
        const uint16_t *wb = w_r + static_cast<int64_t>(eb < E ? eb : 0) * H;
        float acc[TOK][2];
#pragma unroll
        for (int i = 0; i < TOK; ++i) acc[i][0] = acc[i][1] = 0.f;
#pragma unroll 4
        for (int c = c_begin; c < c_end; ++c) {
            const uint4 va = ld_nc(wa + c * 8), vb = ld_nc(wb + c * 8);
            uint4 vx[TOK];
#pragma unroll
            for (int i = 0; i < TOK; ++i) vx[i] = ld_nc(xr[i] + c * 8);
            const uint32_t pa[4] = {va.x, va.y, va.z, va.w}, pb[4] = {vb.x, vb.y, vb.z, vb.w};
#pragma unroll
            for (int i = 0; i < TOK; ++i) {
                const uint32_t px[4] = {vx[i].x, vx[i].y, vx[i].z, vx[i].w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float x0 = bf_lo(px[q]), x1 = bf_hi(px[q]);
                    acc[i][0] = fmaf(x0, bf_lo(pa[q]), acc[i][0]);
                    acc[i][0] = fmaf(x1, bf_hi(pa[q]), acc[i][0]);
                    acc[i][1] = fmaf(x0, bf_lo(pb[q]), acc[i][1]);
                    acc[i][1] = fmaf(x1, bf_hi(pb[q]), acc[i][1]);
                }
            }
        }
        __syncthreads();                             // part[] free from the last block
#pragma unroll
        for (int i = 0; i < TOK; ++i) {
            part[warp][i][lane] = acc[i][0];
            part[warp][i][lane + 32] = acc[i][1];
        }
        __syncthreads();
        for (int o = threadIdx.x; o < TOK * 64; o += blockDim.x) {
            const int i = o / 64, e = e0 + o % 64, t = t0 + i;
            if (e >= E) continue;
            float v = 0.f;
#pragma unroll
            for (int w = 0; w < RL_WARPS; ++w) v += part[w][i][o % 64];
            v += bias ? bias[e] : 0.f;
            s_logits[i * E + e] = v;
            if (logits && t < T) logits[static_cast<int64_t>(t) * E + e] = v;
        }
    }
    __syncthreads();
    if (warp < TOK && t0 + warp < T) {
        const int t = t0 + warp;
        int id;
        float w;
        if (!route_token<PER_LANE>(s_logits + warp * E, E, k, renormalize, id, w)) {
            if (lane == 0) report(dev_error, MOE_ERR_DEVICE_CHECK);
            return;
        }
        if (lane < k) {
            topk_ids[static_cast<int64_t>(t) * k + lane] = id;
            topk_w[static_cast<int64_t>(t) * k + lane] = w;
        }
    }
}

template <int TOK, int PER_LANE>
static void launch_router_route(int T, int E, size_t smem, cudaStream_t stream,
                                const uint16_t *x, const uint16_t *w_r, const float *bias, int H,
                                int k, int renormalize, float *logits, int32_t *ids, float *w,
                                int32_t *dev_error) {
    launch(router_route_kernel<TOK, PER_LANE>, (T + TOK - 1) / TOK, RL_WARPS * 32, smem, stream,
           x, w_r, bias, T, H, E, k, renormalize, logits, ids, w, dev_error);
}

template <int TOK>
static void router_route_dispatch(int per_lane, int T, int E, size_t smem, cudaStream_t stream,
                                  const uint16_t *x, const uint16_t *w_r, const float *bias,
                                  int H, int k, int renormalize, float *logits, int32_t *ids,
                                  float *w, int32_t *dev_error) {
#define MOE_RR(PL) launch_router_route<TOK, PL>(T, E, smem, stream, x, w_r, bias, H, k, \
                                                renormalize, logits, ids, w, dev_error)
    if (per_lane <= 1) MOE_RR(1);
    else if (per_lane <= 2) MOE_RR(2);
    else if (per_lane <= 4) MOE_RR(4);
    else if (per_lane <= 8) MOE_RR(8);
    else if (per_lane <= 16) MOE_RR(16);
    else MOE_RR(32);
#undef MOE_RR
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
    if (H % 8 != 0) return MOE_ERR_ALIGNMENT;
    if (!aligned16(x) || !aligned16(w_r)) return MOE_ERR_ALIGNMENT;
    // few tokens per block for small batches (more blocks), 8 for large ones
    if (T <= 512) {
        dim3 grid((T + 1) / 2, (E + 63) / 64);
        launch(router_logits_kernel<2>, grid, RL_WARPS * 32, 0, stream, x, w_r, bias, T, H, E,
               logits);
    } else {
        dim3 grid((T + 7) / 8, (E + 63) / 64);
        launch(router_logits_kernel<8>, grid, RL_WARPS * 32, 0, stream, x, w_r, bias, T, H, E,
               logits);
    }
    return launch_status();
}

extern "C" moe_status moe_router_route(const uint16_t *x, const uint16_t *w_r, const float *bias,
                                       int T, int H, int E, int k, int renormalize,
                                       float *logits, int32_t *topk_ids, float *topk_w,
                                       int32_t *dev_error, cudaStream_t stream) {
    if (!x || !w_r || !topk_ids || !topk_w || T < 1 || H < 1 || E < 1 || k < 1 || k > E ||
        k > 32)
        return MOE_ERR_INVALID_ARG;
    if (E > 1024) return MOE_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(T) * H >= (1ll << 31) || static_cast<int64_t>(E) * H >= (1ll << 31) ||
        static_cast<int64_t>(T) * E >= (1ll << 31))
        return MOE_ERR_UNSUPPORTED;
    if (H % 8 != 0 || !aligned16(x) || !aligned16(w_r)) return MOE_ERR_ALIGNMENT;
    const int per_lane = (E + 31) / 32;
    if (T <= 512 || E > 512) {               // 8-token CTAs only while [8][E] fits 16 KB
        const size_t smem = static_cast<size_t>(2) * E * sizeof(float);
        router_route_dispatch<2>(per_lane, T, E, smem, stream, x, w_r, bias, H, k, renormalize,
                                 logits, topk_ids, topk_w, dev_error);
    } else {
        const size_t smem = static_cast<size_t>(8) * E * sizeof(float);
        router_route_dispatch<8>(per_lane, T, E, smem, stream, x, w_r, bias, H, k, renormalize,
                                 logits, topk_ids, topk_w, dev_error);
    }
    return launch_status();
}
