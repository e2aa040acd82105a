// route_token.cuh -- per-token top-k routing by one warp, shared by the
// routing kernel and the fused small-batch route + permute kernel.
//
// Each lane holds E/32 logits in registers; k rounds of a warp arg-max
// (larger logit wins, ties go to the lower expert index) pick the experts in
// descending order ("switchyard" page, 02 Kernels and dispatch, "Route and
// sort": each token routed in one warp).  The softmax runs over all E
// logits; L_e - max is corrected for its fp32 rounding and the denominator is
// summed in fp32 with compensation, so each weight is within a few fp32 ulps
// of the exact value.
#pragma once

#include <math.h>

#include "common.cuh"

namespace moe {

// Routes one token with the calling warp.  Lane j < k receives the j-th
// chosen expert and its weight.  Returns false (on every lane) if a logit is
// not finite (NaN or +-inf: the softmax of such a row has no finite
// weights), leaving the outputs undefined.
template <int PER_LANE>
__device__ __forceinline__ bool route_token(const float *L, int E, int k,
                                            int renormalize, int &my_id, float &my_w) {
    const int lane = lane_id();
    float v[PER_LANE];
    bool nan_seen = false;
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
        const int e = lane + 32 * i;
        v[i] = e < E ? L[e] : -INFINITY;          // global or shared memory
        nan_seen |= e < E && !isfinite(v[i]);
    }
    if (__any_sync(FULL, nan_seen)) return false;

    uint32_t taken = 0;          // bit i: expert lane + 32 i already chosen
    float my_val = 0.f, vmax = 0.f;
    my_id = 0;
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
    // sums of positive terms in fp32 with their rounding errors carried
    // alongside (Knuth's two-sum), so each sum is within ~1 ulp of exact
    // without double-precision arithmetic (slow on this part)
    auto add2 = [](float &hi, float &lo, float x) {
        const float s = hi + x;
        const float bb = s - hi;
        lo += (hi - (s - bb)) + (x - bb);
        hi = s;
    };
    float den = 0.f, den_lo = 0.f;
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
        const int e = lane + 32 * i;
        if (e < E) add2(den, den_lo, shifted_exp(v[i]));
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
        const float oh = __shfl_xor_sync(FULL, den, d), ol = __shfl_xor_sync(FULL, den_lo, d);
        add2(den, den_lo, oh);
        den_lo += ol;
    }
    den += den_lo;

    const float ej = lane < k ? shifted_exp(my_val) : 0.f;
    float sel = ej, sel_lo = 0.f;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
        const float oh = __shfl_xor_sync(FULL, sel, d), ol = __shfl_xor_sync(FULL, sel_lo, d);
        add2(sel, sel_lo, oh);
        sel_lo += ol;
    }
    sel += sel_lo;
    my_w = __fdiv_rn(ej, renormalize ? sel : den);
    return true;
}

}  // namespace moe
