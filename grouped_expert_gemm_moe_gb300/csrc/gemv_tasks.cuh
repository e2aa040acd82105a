// gemv_tasks.cuh -- the per-warp work of the grouped GEMV (bf16 weights),
// shared by the standalone GEMV kernels (gemv.cu) and the single-launch
// decode layer (decode_layer.cu), so both compute every dot product in the
// same order and give the same bytes.
//
// Lane l covers the 16-byte chunks l, l+32, l+64, ... of K; all of a task's
// weight and activation loads are issued before the first multiply, so one
// memory latency covers the task.  The functions return per-lane partial
// sums; the caller reduces them across the warp (warp_sum) and stores.
#pragma once

#include "common.cuh"

namespace moe {

__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8]) {
    f[0] = bf_lo(v.x); f[1] = bf_hi(v.x);
    f[2] = bf_lo(v.y); f[3] = bf_hi(v.y);
    f[4] = bf_lo(v.z); f[5] = bf_hi(v.z);
    f[6] = bf_lo(v.w); f[7] = bf_hi(v.w);
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

// Gate/up task: the gate row wg and the up row wu (K = chunks * 8 bf16)
// against nrr <= NR activation rows xrow[r].  sg[r], su[r]: per-lane partial
// sums of gate . x_r and up . x_r.
template <int NCH, int NR>
__device__ __forceinline__ void gateup_partial_bf16(const uint16_t *const (&xrow)[NR], int nrr,
                                                    const uint16_t *wg, const uint16_t *wu,
                                                    int chunks, uint64_t pol, float (&sg)[NR],
                                                    float (&su)[NR]) {
    const int lane = lane_id();
#pragma unroll
    for (int r = 0; r < NR; ++r) sg[r] = su[r] = 0.f;
    for (int seg = 0; seg < chunks; seg += 32 * NCH) {
        uint4 vg[NCH], vu[NCH], vx[NR][NCH];
#pragma unroll
        for (int u = 0; u < NCH; ++u) {
            const int q = seg + lane + 32 * u;
            if (q < chunks) {
                vg[u] = ld_stream(wg + q * 8, pol);
                vu[u] = ld_stream(wu + q * 8, pol);
#pragma unroll
                for (int r = 0; r < NR; ++r)
                    if (r < nrr) vx[r][u] = ld_nc(xrow[r] + q * 8);
            }
        }
#pragma unroll
        for (int u = 0; u < NCH; ++u) {
            if (seg + lane + 32 * u >= chunks) continue;
            float fg[8], fu[8];
            unpack8(vg[u], fg);
            unpack8(vu[u], fu);
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                if (r >= nrr) break;
                float fx[8];
                unpack8(vx[r][u], fx);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    sg[r] = fmaf(fg[e], fx[e], sg[r]);
                    su[r] = fmaf(fu[e], fx[e], su[r]);
                }
            }
        }
    }
}

// Down task: weight rows n0 .. n0+RW-1 of wd (row stride I; rows >= H are
// skipped) against nrr <= NR hidden rows hr + r*I.  acc[r][w]: per-lane
// partial sums.  H_COHERENT: the hidden rows were written earlier in the
// same launch (read through L2, not the read-only path).
template <int NCH, int RW, int NR, bool H_COHERENT = false>
__device__ __forceinline__ void down_partial_bf16(const uint16_t *hr, int I, int nrr,
                                                  const uint16_t *wd, int n0, int H, int chunks,
                                                  uint64_t pol, float (&acc)[NR][RW]) {
    const int lane = lane_id();
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int w = 0; w < RW; ++w) acc[r][w] = 0.f;
    for (int seg = 0; seg < chunks; seg += 32 * NCH) {
        uint4 vw[RW][NCH], vx[NR][NCH];
#pragma unroll
        for (int u = 0; u < NCH; ++u) {
            const int q = seg + lane + 32 * u;
            if (q < chunks) {
#pragma unroll
                for (int w = 0; w < RW; ++w)
                    if (n0 + w < H) vw[w][u] = ld_stream(wd + static_cast<int64_t>(w) * I + q * 8, pol);
#pragma unroll
                for (int r = 0; r < NR; ++r)
                    if (r < nrr) {
                        const uint16_t *p = hr + static_cast<int64_t>(r) * I + q * 8;
                        vx[r][u] = H_COHERENT ? ld_cg(p) : ld_nc(p);
                    }
            }
        }
#pragma unroll
        for (int u = 0; u < NCH; ++u) {
            if (seg + lane + 32 * u >= chunks) continue;
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                if (r >= nrr) break;
                float fx[8];
                unpack8(vx[r][u], fx);
#pragma unroll
                for (int w = 0; w < RW; ++w) {
                    if (n0 + w >= H) break;
                    float fw[8];
                    unpack8(vw[w][u], fw);
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[r][w] = fmaf(fw[e], fx[e], acc[r][w]);
                }
            }
        }
    }
}

// The weights of the first 32 * NCH chunks of a down task (what
// down_partial_bf16 loads first), for a caller that issues them early.
template <int NCH, int RW>
__device__ __forceinline__ void down_load_first(const uint16_t *wd, int I, int n0, int H,
                                                int chunks, uint64_t pol, uint4 (&vw)[RW][NCH]) {
    const int lane = lane_id();
#pragma unroll
    for (int u = 0; u < NCH; ++u) {
        const int q = lane + 32 * u;
        if (q < chunks) {
#pragma unroll
            for (int w = 0; w < RW; ++w)
                if (n0 + w < H) vw[w][u] = ld_stream(wd + static_cast<int64_t>(w) * I + q * 8, pol);
        }
    }
}

// down_partial_bf16 for one hidden row whose first 32 * NCH weight chunks
// are already in `first` (from down_load_first): the same loads after
// those and the same sums in the same order.
template <int NCH, int RW, bool H_COHERENT>
__device__ __forceinline__ void down_partial_bf16_first(const uint16_t *hr, int I,
                                                        const uint16_t *wd, int n0, int H,
                                                        int chunks, uint64_t pol,
                                                        const uint4 (&first)[RW][NCH],
                                                        float (&acc)[1][RW]) {
    const int lane = lane_id();
#pragma unroll
    for (int w = 0; w < RW; ++w) acc[0][w] = 0.f;
    auto segment = [&](int seg, const uint4 (&vw)[RW][NCH], const uint4 (&vx)[NCH]) {
#pragma unroll
        for (int u = 0; u < NCH; ++u) {
            if (seg + lane + 32 * u >= chunks) continue;
            float fx[8];
            unpack8(vx[u], fx);
#pragma unroll
            for (int w = 0; w < RW; ++w) {
                if (n0 + w >= H) break;
                float fw[8];
                unpack8(vw[w][u], fw);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[0][w] = fmaf(fw[e], fx[e], acc[0][w]);
            }
        }
    };
    {                                            // chunks 0 .. 32 NCH - 1: weights in `first`
        uint4 vx[NCH];
#pragma unroll
        for (int u = 0; u < NCH; ++u) {
            const int q = lane + 32 * u;
            if (q < chunks) vx[u] = H_COHERENT ? ld_cg(hr + q * 8) : ld_nc(hr + q * 8);
        }
        segment(0, first, vx);
    }
    for (int seg = 32 * NCH; seg < chunks; seg += 32 * NCH) {
        uint4 vw[RW][NCH], vx[NCH];
#pragma unroll
        for (int u = 0; u < NCH; ++u) {
            const int q = seg + lane + 32 * u;
            if (q < chunks) {
#pragma unroll
                for (int w = 0; w < RW; ++w)
                    if (n0 + w < H) vw[w][u] = ld_stream(wd + static_cast<int64_t>(w) * I + q * 8, pol);
                vx[u] = H_COHERENT ? ld_cg(hr + q * 8) : ld_nc(hr + q * 8);
            }
        }
        segment(seg, vw, vx);
    }
}

}  // namespace moe
