// combine.cu -- gather-based weighted combine back to token order.
//
// Each output chunk of 8 hidden elements gathers its token's k routed rows
// (and S shared rows) from y_perm and sums them in fp32 in a fixed order,
// so the result is the same bytes on every run.  The "dispatch" project's
// Phase 6 pull request (Summary) had to widen a repeatability check because
// its index_add_ (atomicAdd) combine is not bitwise deterministic; a gather
// has no such race.
#include "common.cuh"

namespace moe {

// 8-element chunks per thread.  One keeps a thread within 64 registers with
// its 8 row loads in flight, so an SM holds 1024 threads of them; two chunks
// per thread (139 registers, 3 blocks per SM) left the batch's tokens to run
// in ~5 waves and DRAM 43 % busy at T=2048.
constexpr int CB_CPT = 1;

__global__ void __launch_bounds__(256, 4) combine_kernel(
    const uint16_t *__restrict__ y_perm, const int32_t *__restrict__ row_of_slot,
    const float *__restrict__ topk_w, const int32_t *__restrict__ offsets, int E, int T, int k,
    int S, int H, const uint16_t *residual, uint16_t *out, int32_t *dev_error) {
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.y + blockIdx.z * gridDim.y;   // tokens over grid y and z
    const int c0 = (blockIdx.x * blockDim.x + threadIdx.x) * CB_CPT;   // first chunk
    const int chunks = H / 8;
    if (t >= T || c0 >= chunks) return;
    const int64_t n = static_cast<int64_t>(T) * k;
    // shared rows follow the routed rows: at n (dropless) or after the
    // served routed rows (capacity-limited permute: offsets[E])
    int64_t shared0 = offsets ? static_cast<int64_t>(offsets[E]) : n;
    if (shared0 < 0 || shared0 > n) {            // inconsistent offsets: skip the shared rows
        if (S > 0) report(dev_error, MOE_ERR_DEVICE_CHECK);
        shared0 = 0;
        S = 0;
    }
    float acc[CB_CPT][8];
#pragma unroll
    for (int q = 0; q < CB_CPT; ++q)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[q][i] = 0.f;
    auto accumulate = [&](int q, const uint4 &v, float w) {
        const uint32_t p[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc[q][2 * i] = fmaf(w, bf_lo(p[i]), acc[q][2 * i]);
            acc[q][2 * i + 1] = fmaf(w, bf_hi(p[i]), acc[q][2 * i + 1]);
        }
    };
    // up to 8 routed rows at a time: their indices and weights first, then
    // every row's chunks, so the gathers overlap; sums stay in j order
    constexpr int BATCH = 8;
    for (int j0 = 0; j0 < k; j0 += BATCH) {
        int32_t r[BATCH];
        float w[BATCH];
        bool ok[BATCH];
#pragma unroll
        for (int j = 0; j < BATCH; ++j) {
            ok[j] = false;
            if (j0 + j < k) {
                const int64_t slot = static_cast<int64_t>(t) * k + j0 + j;
                r[j] = row_of_slot[slot];
                w[j] = topk_w[slot];
                ok[j] = r[j] >= 0 && r[j] < n;
                // a slot dropped by the capacity limit adds nothing
                if (!ok[j] && r[j] != MOE_ROW_DROPPED) report(dev_error, MOE_ERR_DEVICE_CHECK);
            }
        }
        uint4 v[BATCH][CB_CPT];
#pragma unroll
        for (int j = 0; j < BATCH; ++j)
#pragma unroll
            for (int q = 0; q < CB_CPT; ++q)
                if (ok[j] && c0 + q < chunks)
                    v[j][q] = ld_nc(y_perm + static_cast<int64_t>(r[j]) * H + (c0 + q) * 8);
#pragma unroll
        for (int j = 0; j < BATCH; ++j)
#pragma unroll
            for (int q = 0; q < CB_CPT; ++q)
                if (ok[j] && c0 + q < chunks) accumulate(q, v[j][q], w[j]);
    }
    for (int s0 = 0; s0 < S; s0 += BATCH) {              // shared rows, s ascending
        uint4 v[BATCH][CB_CPT];
#pragma unroll
        for (int j = 0; j < BATCH; ++j)
#pragma unroll
            for (int q = 0; q < CB_CPT; ++q)
                if (s0 + j < S && c0 + q < chunks)
                    v[j][q] = ld_nc(y_perm + (shared0 + static_cast<int64_t>(s0 + j) * T + t) * H +
                                    (c0 + q) * 8);
#pragma unroll
        for (int j = 0; j < BATCH; ++j)
#pragma unroll
            for (int q = 0; q < CB_CPT; ++q)
                if (s0 + j < S && c0 + q < chunks) accumulate(q, v[j][q], 1.0f);
    }
#pragma unroll
    for (int q = 0; q < CB_CPT; ++q) {
        const int c = c0 + q;
        if (c >= chunks) break;
        if (residual) {
            const uint4 v = ld_nc(residual + static_cast<int64_t>(t) * H + c * 8);
            const uint32_t p[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[q][2 * i] += bf_lo(p[i]);
                acc[q][2 * i + 1] += bf_hi(p[i]);
            }
        }
        uint4 o;
        o.x = pack_bf16x2(acc[q][0], acc[q][1]);
        o.y = pack_bf16x2(acc[q][2], acc[q][3]);
        o.z = pack_bf16x2(acc[q][4], acc[q][5]);
        o.w = pack_bf16x2(acc[q][6], acc[q][7]);
        *reinterpret_cast<uint4 *>(out + static_cast<int64_t>(t) * H + c * 8) = o;
    }
}

}  // namespace moe

using namespace moe;

namespace moe {
static moe_status combine_impl(const uint16_t *y_perm, const int32_t *row_of_slot,
                               const float *topk_w, const int32_t *offsets, int E, int T, int k,
                               int S, int H, const uint16_t *residual, uint16_t *out,
                               int32_t *dev_error, cudaStream_t stream) {
    if (!y_perm || !row_of_slot || !topk_w || !out || T < 1 || k < 1 || k > 32 || S < 0 || H < 1)
        return MOE_ERR_INVALID_ARG;
    const int64_t M = static_cast<int64_t>(T) * k + static_cast<int64_t>(S) * T;
    if (M * H >= (1ll << 31) || T > 65535 * 64) return MOE_ERR_UNSUPPORTED;
    if (H % 8 != 0 || !aligned16(y_perm) || !aligned16(out) || (residual && !aligned16(residual)))
        return MOE_ERR_ALIGNMENT;
    const int chunks = H / 8;
    const int per_thread = (chunks + CB_CPT - 1) / CB_CPT;
    const int threads = per_thread >= 256 ? 256 : ((per_thread + 31) / 32) * 32;
    // tokens over grid y (at most 65535) and z
    const int ty = T < 65535 ? T : 65535;
    dim3 grid((per_thread + threads - 1) / threads, ty, (T + ty - 1) / ty);
    launch(combine_kernel, grid, threads, 0, stream, y_perm, row_of_slot, topk_w, offsets, E, T, k,
           S, H, residual, out, dev_error);
    return launch_status();
}
}  // namespace moe

extern "C" moe_status moe_combine(const uint16_t *y_perm, const int32_t *row_of_slot,
                                  const float *topk_w, int T, int k, int S, int H,
                                  const uint16_t *residual, uint16_t *out, int32_t *dev_error,
                                  cudaStream_t stream) {
    return combine_impl(y_perm, row_of_slot, topk_w, nullptr, 0, T, k, S, H, residual, out,
                        dev_error, stream);
}

extern "C" moe_status moe_combine_capped(const uint16_t *y_perm, const int32_t *row_of_slot,
                                         const float *topk_w, const int32_t *offsets, int E,
                                         int T, int k, int S, int H, const uint16_t *residual,
                                         uint16_t *out, int32_t *dev_error,
                                         cudaStream_t stream) {
    if (!offsets || E < 1) return MOE_ERR_INVALID_ARG;
    return combine_impl(y_perm, row_of_slot, topk_w, offsets, E, T, k, S, H, residual, out,
                        dev_error, stream);
}
