// gemv.cu -- grouped GEMV for decode-sized batches (bf16 and int8 weights).
//
// The "switchyard" page (02 Kernels and dispatch, "One launch for all
// experts") serves decode with a grouped GEMV that it measured at 73 % of
// the T4's memory bandwidth.  With a few
// rows per expert the FFN is a weight stream: every expert weight row is
// read from HBM once, with coalesced 128-bit loads (a warp reads 512
// contiguous bytes per instruction), and dotted with the handful of
// activation rows of its expert, which stay in L1/L2.
//
// Work unit ("task") of a warp:
//   gate/up pass: (active group a, intermediate row i): the gate row i and
//                 the up row I+i of expert g against the group's rows,
//                 h[r,i] = bf16(silu(gate) * up);
//   down pass:    (active group a, RW consecutive output rows n): y[r,n].
// Lane l covers the 16-byte chunks l, l+32, l+64, ... of the K dimension;
// all of a task's weight loads are issued before any arithmetic, so each
// warp keeps 8 KB in flight.  A group with more rows than NR is processed
// in blocks of NR rows (the weight row is re-read from L2).
#include <algorithm>
#include <mutex>

#include "gemv_tasks.cuh"

namespace moe {

constexpr int GEMV_THREADS = 256;

// Active (non-empty) groups, compacted by warp 0; validates the offsets.
struct ActiveGroups {
    int group[1024];
    int row0[1024];
    int nrows[1024];
    int count;
};

__device__ __forceinline__ int load_active_groups(ActiveGroups &ag, const int32_t *offsets, int G,
                                                  int M, int32_t *dev_error) {
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int total = 0;
        bool bad = false;
        for (int base = 0; base < G; base += 32) {
            const int g = base + lane;
            int o0 = 0, o1 = 0;
            if (g < G) {
                o0 = offsets[g];
                o1 = offsets[g + 1];
                if (o0 < 0 || o1 < o0 || o1 > M) bad = true;
            }
            const bool has = g < G && o1 > o0;
            const unsigned b = __ballot_sync(FULL, has);
            if (has) {
                const int pos = total + __popc(b & ((1u << lane) - 1u));
                ag.group[pos] = g;
                ag.row0[pos] = o0;
                ag.nrows[pos] = o1 - o0;
            }
            total += __popc(b);
        }
        bad = __any_sync(FULL, bad);
        if (lane == 0) {
            ag.count = bad ? 0 : total;
            if (bad) report(dev_error, MOE_ERR_DEVICE_CHECK);
        }
    }
    __syncthreads();
    return ag.count;
}

// 16 int8 (biased) -> 16 fp32
__device__ __forceinline__ void unpack16_s8(const uint4 v, float (&f)[16]) {
    const uint32_t w[4] = {bias_s8x4(v.x), bias_s8x4(v.y), bias_s8x4(v.z), bias_s8x4(v.w)};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int b = 0; b < 4; ++b) f[4 * i + b] = s8_to_f32(w[i], b);
    }
}

// ------------------------------------------------------------------ bf16
//
// A task's loads -- the weight rows' chunks and the NR activation rows'
// chunks this lane needs -- are all issued before the first multiply, so
// one memory latency covers the whole task.  NR (1 or 2) is the number of
// a group's rows handled per pass, picked from the average rows per group.

template <int NCH, int NR>
__global__ void __launch_bounds__(GEMV_THREADS) gemv_gateup_bf16(
    const uint16_t *__restrict__ x_perm, const int32_t *__restrict__ offsets, int G, int M, int H,
    int I, const uint16_t *__restrict__ w_gu, uint16_t *__restrict__ h, int32_t *dev_error) {
    __shared__ ActiveGroups ag;
    pdl_wait();
    pdl_trigger();
    const int na = load_active_groups(ag, offsets, G, M, dev_error);
    const uint64_t pol = policy_evict_first();
    const int lane = lane_id(), wpb = blockDim.x >> 5;
    const int chunks = H / 8;
    const int64_t ntasks = static_cast<int64_t>(na) * I;
    for (int64_t task = static_cast<int64_t>(blockIdx.x) * wpb + (threadIdx.x >> 5); task < ntasks;
         task += static_cast<int64_t>(gridDim.x) * wpb) {
        const int a = static_cast<int>(task / I), i = static_cast<int>(task % I);
        const int g = ag.group[a], r0 = ag.row0[a], nr = ag.nrows[a];
        const uint16_t *wg = w_gu + (static_cast<int64_t>(g) * 2 * I + i) * H;
        const uint16_t *wu = wg + static_cast<int64_t>(I) * H;
        for (int rb = 0; rb < nr; rb += NR) {
            const int nrr = min(NR, nr - rb);
            const uint16_t *xr = x_perm + static_cast<int64_t>(r0 + rb) * H;
            const uint16_t *xrow[NR];
#pragma unroll
            for (int r = 0; r < NR; ++r) xrow[r] = xr + static_cast<int64_t>(r) * H;
            float sg[NR], su[NR];
            gateup_partial_bf16<NCH, NR>(xrow, nrr, wg, wu, chunks, pol, sg, su);
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                if (r >= nrr) break;
                const float gv = warp_sum(sg[r]), uv = warp_sum(su[r]);
                if (lane == 0) {
                    const __nv_bfloat16 hv = __float2bfloat16_rn(silu_f(gv) * uv);
                    h[static_cast<int64_t>(r0 + rb + r) * I + i] =
                        *reinterpret_cast<const uint16_t *>(&hv);
                }
            }
        }
    }
}

template <int NCH, int RW, int NR>
__global__ void __launch_bounds__(GEMV_THREADS) gemv_down_bf16(
    const uint16_t *__restrict__ h, const int32_t *__restrict__ offsets, int G, int M, int H,
    int I, const uint16_t *__restrict__ w_down, uint16_t *__restrict__ y_perm,
    int32_t *dev_error) {
    __shared__ ActiveGroups ag;
    pdl_wait();
    pdl_trigger();
    const int na = load_active_groups(ag, offsets, G, M, dev_error);
    const uint64_t pol = policy_evict_first();
    const int lane = lane_id(), wpb = blockDim.x >> 5;
    const int chunks = I / 8;
    const int nblk = (H + RW - 1) / RW;
    const int64_t ntasks = static_cast<int64_t>(na) * nblk;
    for (int64_t task = static_cast<int64_t>(blockIdx.x) * wpb + (threadIdx.x >> 5); task < ntasks;
         task += static_cast<int64_t>(gridDim.x) * wpb) {
        const int a = static_cast<int>(task / nblk), n0 = static_cast<int>(task % nblk) * RW;
        const int g = ag.group[a], r0 = ag.row0[a], nr = ag.nrows[a];
        const uint16_t *wd = w_down + (static_cast<int64_t>(g) * H + n0) * I;
        for (int rb = 0; rb < nr; rb += NR) {
            const int nrr = min(NR, nr - rb);
            const uint16_t *hr = h + static_cast<int64_t>(r0 + rb) * I;
            float acc[NR][RW];
            down_partial_bf16<NCH, RW, NR>(hr, I, nrr, wd, n0, H, chunks, pol, acc);
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                if (r >= nrr) break;
#pragma unroll
                for (int w = 0; w < RW; ++w) {
                    const float v = warp_sum(acc[r][w]);
                    if (lane == 0 && n0 + w < H) {
                        const __nv_bfloat16 b = __float2bfloat16_rn(v);
                        y_perm[static_cast<int64_t>(r0 + rb + r) * H + n0 + w] =
                            *reinterpret_cast<const uint16_t *>(&b);
                    }
                }
            }
        }
    }
}

// ------------------------------------------------------------------ int8

template <int NCH, int NR>
__global__ void __launch_bounds__(GEMV_THREADS) gemv_gateup_w8(
    const uint16_t *__restrict__ x_perm, const int32_t *__restrict__ offsets, int G, int M, int H,
    int I, const int8_t *__restrict__ q_gu, const float *__restrict__ s_gu,
    uint16_t *__restrict__ h, int32_t *dev_error) {
    __shared__ ActiveGroups ag;
    pdl_wait();
    pdl_trigger();
    const int na = load_active_groups(ag, offsets, G, M, dev_error);
    const uint64_t pol = policy_evict_first();
    const int lane = lane_id(), wpb = blockDim.x >> 5;
    const int chunks = H / 16;                   // 16 int8 per 16-byte chunk
    const int64_t ntasks = static_cast<int64_t>(na) * I;
    for (int64_t task = static_cast<int64_t>(blockIdx.x) * wpb + (threadIdx.x >> 5); task < ntasks;
         task += static_cast<int64_t>(gridDim.x) * wpb) {
        const int a = static_cast<int>(task / I), i = static_cast<int>(task % I);
        const int g = ag.group[a], r0 = ag.row0[a], nr = ag.nrows[a];
        const int8_t *wg = q_gu + (static_cast<int64_t>(g) * 2 * I + i) * H;
        const int8_t *wu = wg + static_cast<int64_t>(I) * H;
        const float scg = s_gu[static_cast<int64_t>(g) * 2 * I + i];
        const float scu = s_gu[static_cast<int64_t>(g) * 2 * I + I + i];
        for (int rb = 0; rb < nr; rb += NR) {
            const int nrr = min(NR, nr - rb);
            const uint16_t *xr = x_perm + static_cast<int64_t>(r0 + rb) * H;
            float sg[NR], su[NR];
#pragma unroll
            for (int r = 0; r < NR; ++r) sg[r] = su[r] = 0.f;
            for (int seg = 0; seg < chunks; seg += 32 * NCH) {
                uint4 vg[NCH], vu[NCH], vx[NR][NCH][2];
#pragma unroll
                for (int u = 0; u < NCH; ++u) {
                    const int q = seg + lane + 32 * u;
                    if (q < chunks) {
                        vg[u] = ld_stream(wg + q * 16, pol);
                        vu[u] = ld_stream(wu + q * 16, pol);
#pragma unroll
                        for (int r = 0; r < NR; ++r)
                            if (r < nrr) {
                                vx[r][u][0] = ld_nc(xr + static_cast<int64_t>(r) * H + q * 16);
                                vx[r][u][1] = ld_nc(xr + static_cast<int64_t>(r) * H + q * 16 + 8);
                            }
                    }
                }
#pragma unroll
                for (int u = 0; u < NCH; ++u) {
                    if (seg + lane + 32 * u >= chunks) continue;
                    float fg[16], fu[16];
                    unpack16_s8(vg[u], fg);
                    unpack16_s8(vu[u], fu);
#pragma unroll
                    for (int r = 0; r < NR; ++r) {
                        if (r >= nrr) break;
                        float fx0[8], fx1[8];
                        unpack8(vx[r][u][0], fx0);
                        unpack8(vx[r][u][1], fx1);
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            sg[r] = fmaf(fg[e], fx0[e], sg[r]);
                            su[r] = fmaf(fu[e], fx0[e], su[r]);
                        }
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            sg[r] = fmaf(fg[8 + e], fx1[e], sg[r]);
                            su[r] = fmaf(fu[8 + e], fx1[e], su[r]);
                        }
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                if (r >= nrr) break;
                const float gv = warp_sum(sg[r]) * scg, uv = warp_sum(su[r]) * scu;
                if (lane == 0) {
                    const __nv_bfloat16 hv = __float2bfloat16_rn(silu_f(gv) * uv);
                    h[static_cast<int64_t>(r0 + rb + r) * I + i] =
                        *reinterpret_cast<const uint16_t *>(&hv);
                }
            }
        }
    }
}

template <int NCH, int RW, int NR>
__global__ void __launch_bounds__(GEMV_THREADS) gemv_down_w8(
    const uint16_t *__restrict__ h, const int32_t *__restrict__ offsets, int G, int M, int H,
    int I, const int8_t *__restrict__ q_down, const float *__restrict__ s_down,
    uint16_t *__restrict__ y_perm, int32_t *dev_error) {
    __shared__ ActiveGroups ag;
    pdl_wait();
    pdl_trigger();
    const int na = load_active_groups(ag, offsets, G, M, dev_error);
    const uint64_t pol = policy_evict_first();
    const int lane = lane_id(), wpb = blockDim.x >> 5;
    const int chunks = I / 16;
    const int nblk = (H + RW - 1) / RW;
    const int64_t ntasks = static_cast<int64_t>(na) * nblk;
    for (int64_t task = static_cast<int64_t>(blockIdx.x) * wpb + (threadIdx.x >> 5); task < ntasks;
         task += static_cast<int64_t>(gridDim.x) * wpb) {
        const int a = static_cast<int>(task / nblk), n0 = static_cast<int>(task % nblk) * RW;
        const int g = ag.group[a], r0 = ag.row0[a], nr = ag.nrows[a];
        const int8_t *wd = q_down + (static_cast<int64_t>(g) * H + n0) * I;
        for (int rb = 0; rb < nr; rb += NR) {
            const int nrr = min(NR, nr - rb);
            const uint16_t *hr = h + static_cast<int64_t>(r0 + rb) * I;
            float acc[NR][RW];
#pragma unroll
            for (int r = 0; r < NR; ++r)
#pragma unroll
                for (int w = 0; w < RW; ++w) acc[r][w] = 0.f;
            for (int seg = 0; seg < chunks; seg += 32 * NCH) {
                uint4 vw[RW][NCH], vx[NR][NCH][2];
#pragma unroll
                for (int u = 0; u < NCH; ++u) {
                    const int q = seg + lane + 32 * u;
                    if (q < chunks) {
#pragma unroll
                        for (int w = 0; w < RW; ++w)
                            if (n0 + w < H) vw[w][u] = ld_stream(wd + static_cast<int64_t>(w) * I + q * 16, pol);
#pragma unroll
                        for (int r = 0; r < NR; ++r)
                            if (r < nrr) {
                                vx[r][u][0] = ld_nc(hr + static_cast<int64_t>(r) * I + q * 16);
                                vx[r][u][1] = ld_nc(hr + static_cast<int64_t>(r) * I + q * 16 + 8);
                            }
                    }
                }
#pragma unroll
                for (int u = 0; u < NCH; ++u) {
                    if (seg + lane + 32 * u >= chunks) continue;
#pragma unroll
                    for (int r = 0; r < NR; ++r) {
                        if (r >= nrr) break;
                        float fx0[8], fx1[8];
                        unpack8(vx[r][u][0], fx0);
                        unpack8(vx[r][u][1], fx1);
#pragma unroll
                        for (int w = 0; w < RW; ++w) {
                            if (n0 + w >= H) break;
                            float fw[16];
                            unpack16_s8(vw[w][u], fw);
#pragma unroll
                            for (int e = 0; e < 8; ++e) acc[r][w] = fmaf(fw[e], fx0[e], acc[r][w]);
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                acc[r][w] = fmaf(fw[8 + e], fx1[e], acc[r][w]);
                        }
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                if (r >= nrr) break;
#pragma unroll
                for (int w = 0; w < RW; ++w) {
                    const float v = warp_sum(acc[r][w]);
                    if (lane == 0 && n0 + w < H) {
                        const float sc = s_down[static_cast<int64_t>(g) * H + n0 + w];
                        const __nv_bfloat16 b = __float2bfloat16_rn(v * sc);
                        y_perm[static_cast<int64_t>(r0 + rb + r) * H + n0 + w] =
                            *reinterpret_cast<const uint16_t *>(&b);
                    }
                }
            }
        }
    }
}

// ------------------------------------------------------------------ host

static int pick_nch(int chunks) {            // chunks = 16-byte chunks per row
    const int per_lane = (chunks + 31) / 32;
    return per_lane <= 1 ? 1 : per_lane <= 2 ? 2 : per_lane <= 4 ? 4 : 8;
}

// rows per pass from the mean rows per group (M / G): 1, else 2 (groups
// with more rows take several passes over the weight row, from L2)
static int pick_nr(int M, int G) { return 2 * static_cast<int64_t>(M) <= 3ll * G ? 1 : 2; }

// All blocks of a GEMV launch are resident at once (grid = blocks per SM x
// SMs), so the grid-stride task loop never waits for a second wave.
template <typename Kernel>
static int resident_grid(Kernel kernel) {
    static int per_sm_of_device[64] = {0};     // one cache per kernel instantiation
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
    if (per_sm_of_device[dev] < 1) {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, GEMV_THREADS, 0) !=
                cudaSuccess || per_sm < 1)
            per_sm = 1;
        per_sm_of_device[dev] = per_sm;
    }
    return per_sm_of_device[dev] * sm_count();
}

template <typename Kernel, typename... A>
static void launch_resident(Kernel kernel, cudaStream_t s, A... a) {
    launch(kernel, resident_grid(kernel), GEMV_THREADS, 0, s, a...);
}

#define MOE_GEMV_NR(KERNEL, NR_, ...)                                     \
    switch (NR_) {                                                        \
        case 1: launch_resident(KERNEL<__VA_ARGS__, 1>, s, a...); break;  \
        default: launch_resident(KERNEL<__VA_ARGS__, 2>, s, a...); break; \
    }

template <typename... A>
static void launch_gateup_bf16(int nch, int nr, cudaStream_t s, A... a) {
    switch (nch) {
        case 1: MOE_GEMV_NR(gemv_gateup_bf16, nr, 1); break;
        case 2: MOE_GEMV_NR(gemv_gateup_bf16, nr, 2); break;
        case 4: MOE_GEMV_NR(gemv_gateup_bf16, nr, 4); break;
        default: MOE_GEMV_NR(gemv_gateup_bf16, nr, 8); break;
    }
}
template <typename... A>
static void launch_down_bf16(int nch, int nr, cudaStream_t s, A... a) {
    switch (nch) {
        case 1: MOE_GEMV_NR(gemv_down_bf16, nr, 1, 4); break;
        case 2: MOE_GEMV_NR(gemv_down_bf16, nr, 2, 4); break;
        case 4: MOE_GEMV_NR(gemv_down_bf16, nr, 4, 4); break;
        default: MOE_GEMV_NR(gemv_down_bf16, nr, 8, 2); break;
    }
}
template <typename... A>
static void launch_gateup_w8(int nch, int nr, cudaStream_t s, A... a) {
    switch (nch) {
        case 1: MOE_GEMV_NR(gemv_gateup_w8, nr, 1); break;
        case 2: MOE_GEMV_NR(gemv_gateup_w8, nr, 2); break;
        case 4: MOE_GEMV_NR(gemv_gateup_w8, nr, 4); break;
        default: MOE_GEMV_NR(gemv_gateup_w8, nr, 8); break;
    }
}
template <typename... A>
static void launch_down_w8(int nch, int nr, cudaStream_t s, A... a) {
    switch (nch) {
        case 1: MOE_GEMV_NR(gemv_down_w8, nr, 1, 4); break;
        case 2: MOE_GEMV_NR(gemv_down_w8, nr, 2, 4); break;
        case 4: MOE_GEMV_NR(gemv_down_w8, nr, 4, 4); break;
        default: MOE_GEMV_NR(gemv_down_w8, nr, 8, 2); break;
    }
}
#undef MOE_GEMV_NR
}  // namespace moe

using namespace moe;

extern "C" size_t moe_ffn_workspace_size(int M, int I) {
    if (M < 0 || I < 0) return 0;
    const size_t bytes = static_cast<size_t>(M) * static_cast<size_t>(I) * 2;
    return (bytes + 255) & ~static_cast<size_t>(255);
}

namespace moe {
// argument checks shared by every FFN entry point
moe_status check_ffn_args(const void *x_perm, const int32_t *offsets, int G, int M, int H, int I,
                          const void *w_gu, const void *w_down, const void *y_perm,
                          const void *workspace, size_t workspace_bytes, int k_align) {
    if (!x_perm || !offsets || !w_gu || !w_down || !y_perm || !workspace)
        return MOE_ERR_INVALID_ARG;
    if (G < 1 || M < 1 || H < 1 || I < 1) return MOE_ERR_INVALID_ARG;
    if (G > 1024) return MOE_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(M) * H >= (1ll << 31) || static_cast<int64_t>(M) * I >= (1ll << 31) ||
        static_cast<int64_t>(G) * 2 * I * H >= (1ll << 40))
        return MOE_ERR_UNSUPPORTED;
    if (H % k_align != 0 || I % k_align != 0) return MOE_ERR_ALIGNMENT;
    if (!aligned16(x_perm) || !aligned16(w_gu) || !aligned16(w_down) || !aligned16(y_perm) ||
        !aligned16(workspace))
        return MOE_ERR_ALIGNMENT;
    if (workspace_bytes < moe_ffn_workspace_size(M, I)) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}
}  // namespace moe

namespace moe {
static moe_status check_phase_args(const void *in, const int32_t *offsets, int G, int M, int H,
                                   int I, const void *w, const void *out, int k_align) {
    if (!in || !offsets || !w || !out || G < 1 || M < 1 || H < 1 || I < 1)
        return MOE_ERR_INVALID_ARG;
    if (G > 1024) return MOE_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(M) * H >= (1ll << 31) || static_cast<int64_t>(M) * I >= (1ll << 31))
        return MOE_ERR_UNSUPPORTED;
    if (H % k_align != 0 || I % k_align != 0) return MOE_ERR_ALIGNMENT;
    if (!aligned16(in) || !aligned16(w) || !aligned16(out)) return MOE_ERR_ALIGNMENT;
    return MOE_OK;
}
}  // namespace moe

extern "C" moe_status moe_grouped_gemv_gate_up(const uint16_t *x_perm, const int32_t *offsets,
                                               int G, int M, int H, int I, const uint16_t *w_gu,
                                               uint16_t *h, int32_t *dev_error,
                                               cudaStream_t stream) {
    moe_status st = check_phase_args(x_perm, offsets, G, M, H, I, w_gu, h, 8);
    if (st != MOE_OK) return st;
    launch_gateup_bf16(pick_nch(H / 8), pick_nr(M, G), stream, x_perm, offsets, G, M, H, I, w_gu, h, dev_error);
    return launch_status();
}

extern "C" moe_status moe_grouped_gemv_down(const uint16_t *h, const int32_t *offsets, int G,
                                            int M, int H, int I, const uint16_t *w_down,
                                            uint16_t *y_perm, int32_t *dev_error,
                                            cudaStream_t stream) {
    moe_status st = check_phase_args(h, offsets, G, M, H, I, w_down, y_perm, 8);
    if (st != MOE_OK) return st;
    launch_down_bf16(pick_nch(I / 8), pick_nr(M, G), stream, h, offsets, G, M, H, I, w_down, y_perm, dev_error);
    return launch_status();
}

extern "C" moe_status moe_grouped_gemv(const uint16_t *x_perm, const int32_t *offsets, int G,
                                       int M, int H, int I, const uint16_t *w_gu,
                                       const uint16_t *w_down, uint16_t *y_perm, void *workspace,
                                       size_t workspace_bytes, int32_t *dev_error,
                                       cudaStream_t stream) {
    moe_status st = check_ffn_args(x_perm, offsets, G, M, H, I, w_gu, w_down, y_perm, workspace,
                                   workspace_bytes, 8);
    if (st != MOE_OK) return st;
    uint16_t *h = static_cast<uint16_t *>(workspace);
    launch_gateup_bf16(pick_nch(H / 8), pick_nr(M, G), stream, x_perm, offsets, G, M, H, I, w_gu, h, dev_error);
    if ((st = launch_status()) != MOE_OK) return st;
    launch_down_bf16(pick_nch(I / 8), pick_nr(M, G), stream, static_cast<const uint16_t *>(h), offsets, G, M, H, I,
                     w_down, y_perm, dev_error);
    return launch_status();
}

extern "C" moe_status moe_grouped_gemv_w8(const uint16_t *x_perm, const int32_t *offsets, int G,
                                          int M, int H, int I, const int8_t *q_gu,
                                          const float *s_gu, const int8_t *q_down,
                                          const float *s_down, uint16_t *y_perm, void *workspace,
                                          size_t workspace_bytes, int32_t *dev_error,
                                          cudaStream_t stream) {
    moe_status st = check_ffn_args(x_perm, offsets, G, M, H, I, q_gu, q_down, y_perm, workspace,
                                   workspace_bytes, 16);
    if (st != MOE_OK) return st;
    if (!s_gu || !s_down) return MOE_ERR_INVALID_ARG;
    uint16_t *h = static_cast<uint16_t *>(workspace);
    launch_gateup_w8(pick_nch(H / 16), pick_nr(M, G), stream, x_perm, offsets, G, M, H, I, q_gu, s_gu, h,
                     dev_error);
    if ((st = launch_status()) != MOE_OK) return st;
    launch_down_w8(pick_nch(I / 16), pick_nr(M, G), stream, static_cast<const uint16_t *>(h), offsets, G, M, H, I,
                   q_down, s_down, y_perm, dev_error);
    return launch_status();
}

// ---------------------------------------------------------------------------
// moe_grouped_gemv_noalloc: the grouped GEMV for callers that cannot allocate
// device memory.  Its only scratch, the bf16 hidden rows h [M, I], lives in
// the file-scope array below instead of a caller workspace.  The array is
// part of this library's device image, so every GPU that loads the library
// holds these bytes until the process exits.

namespace moe {

constexpr size_t NOALLOC_SCRATCH_BYTES = size_t(8) << 20;   // 8 MiB: M * I <= 4,194,304

static __device__ __align__(256) uint8_t g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch on the current device.  In host code
// the array's name only stands for the symbol; the address a kernel can use
// is looked up once per device (with that device current) and cached.
static uint16_t *noalloc_scratch(moe_status *st) {
    static std::mutex mu;
    static void *addr[64] = {nullptr};
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        *st = MOE_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            *st = MOE_ERR_CUDA;
            return nullptr;
        }
        addr[dev] = p;
    }
    return static_cast<uint16_t *>(addr[dev]);
}

}  // namespace moe

extern "C" moe_status moe_grouped_gemv_noalloc(const uint16_t *x_perm, const int32_t *offsets,
                                               int G, int M, int H, int I, const uint16_t *w_gu,
                                               const uint16_t *w_down, uint16_t *y_perm,
                                               int32_t *dev_error, cudaStream_t stream) {
    moe_status st = MOE_OK;
    uint16_t *h = noalloc_scratch(&st);
    if (h == nullptr) return st;
    // The same argument checks as moe_grouped_gemv, with the built-in array
    // as the workspace: h = M x I bf16 must fit in it, else MOE_ERR_WORKSPACE.
    st = check_ffn_args(x_perm, offsets, G, M, H, I, w_gu, w_down, y_perm, h,
                        NOALLOC_SCRATCH_BYTES, 8);
    if (st != MOE_OK) return st;
    // Nothing in the scratch has to start at zero: the gate/up pass writes
    // every h row of every non-empty group before the down pass reads it.
    launch_gateup_bf16(pick_nch(H / 8), pick_nr(M, G), stream, x_perm, offsets, G, M, H, I, w_gu, h, dev_error);
    if ((st = launch_status()) != MOE_OK) return st;
    launch_down_bf16(pick_nch(I / 8), pick_nr(M, G), stream, static_cast<const uint16_t *>(h), offsets, G, M, H,
                     I, w_down, y_perm, dev_error);
    return launch_status();
}
