// decode_layer.cu -- a whole MoE layer for a decode-sized batch in one launch.
//
// The pages' Triton kernels lose most at one token ("dispatch" Phase 6 pull
// request, Summary: 2.4-4.1x behind vLLM's fused MoE there), where a layer is
// four short launches around a weight stream.  Here the layer is one
// cooperative launch of CTAs that all stay resident:
//
//   phase 0  every CTA routes the T <= 8 tokens itself (one warp per token,
//            route_token) and sorts the T*k <= 64 slots by expert (stable) in
//            shared memory: no grid-wide step and no gather of activation
//            rows, the GEMV reads x[token] directly;
//   phase 1  grouped GEMV gate/up + SwiGLU over (group, intermediate row)
//            tasks -> h;                                  grid barrier
//   phase 2  grouped GEMV down over (group, output rows) tasks -> y;
//                                                         grid barrier
//   phase 3  combine: out[t] = sum_j w[t,j] y[row(t,j)] + shared rows
//            (+ residual), fp32, fixed order.
//
// Phases 1-3 use the GEMV's own task code (gemv_tasks.cuh) and the combine's
// summation order, so the result is the bytes of moe_route + moe_permute +
// moe_grouped_gemv + moe_combine.  The grid barrier counts arrivals in a
// word of the caller's workspace, zeroed on the stream before the launch;
// its waits are bounded (1 s): on running out a CTA records MOE_ERR_TIMEOUT
// and returns.
#include "gemv_tasks.cuh"
#include "route_token.cuh"

namespace moe {

constexpr int DL_THREADS = 256;
constexpr int DL_MAX_SLOTS = 64;                  // T * k
constexpr int DL_MAX_ROWS = 128;                  // T * k + S * T
constexpr int DL_DOWN_RW = 4;                     // output rows per down task (8 KB of weights)

struct DecodePlan {
    int ids[DL_MAX_SLOTS];
    float w[DL_MAX_SLOTS];
    int row_of_slot[DL_MAX_SLOTS];
    int sorted_e[DL_MAX_SLOTS];
    int tok[DL_MAX_ROWS];                         // token of permuted row r
    int group[DL_MAX_ROWS + 1];                   // active groups in order
    int row0[DL_MAX_ROWS + 1];                    // their first rows (+ end)
    int na;
    int bad;
    int fail;
};

template <int PER_LANE>
__global__ void __launch_bounds__(DL_THREADS, 2) decode_layer_kernel(
    const float *__restrict__ logits, const uint16_t *__restrict__ x, int T, int E, int S, int k,
    int renormalize, int H, int I, const uint16_t *__restrict__ w_gu,
    const uint16_t *__restrict__ w_down, const uint16_t *residual, uint16_t *out,
    int32_t *__restrict__ topk_ids, float *__restrict__ topk_w, unsigned *barrier,
    uint16_t *__restrict__ h, uint16_t *__restrict__ y, int32_t *dev_error) {
    __shared__ DecodePlan pl;
    const int tid = threadIdx.x, lane = lane_id(), warp = tid >> 5;
    const int n = T * k, M = n + S * T;
    if (tid == 0) {
        pl.bad = 0;
        pl.fail = 0;
    }
    pdl_wait();
    __syncthreads();

    // ---------------------------------------------------------- phase 0
    if (warp < T) {
        int id;
        float wt;
        if (!route_token<PER_LANE>(logits + static_cast<int64_t>(warp) * E, E, k, renormalize,
                                   id, wt)) {
            if (lane == 0) pl.bad = 1;             // a NaN logit
        } else if (lane < k) {
            pl.ids[warp * k + lane] = id;
            pl.w[warp * k + lane] = wt;
            if (blockIdx.x == 0) {
                if (topk_ids) topk_ids[warp * k + lane] = id;
                if (topk_w) topk_w[warp * k + lane] = wt;
            }
        }
    }
    __syncthreads();
    if (pl.bad) {                                   // identical in every CTA
        if (blockIdx.x == 0 && tid == 0) report(dev_error, MOE_ERR_DEVICE_CHECK);
        return;
    }
    if (tid < n) {                                  // stable counting position
        const int e = pl.ids[tid];
        int pos = 0;
        for (int s = 0; s < n; ++s) {
            const int es = pl.ids[s];
            pos += (es < e) || (es == e && s < tid);
        }
        pl.row_of_slot[tid] = pos;
        pl.sorted_e[pos] = e;
        pl.tok[pos] = tid / k;
    }
    if (tid < S * T) pl.tok[n + tid] = tid % T;
    __syncthreads();
    if (warp == 0) {
        int base = 0;
        for (int r0 = 0; r0 < n; r0 += 32) {
            const int r = r0 + lane;
            const bool lead = r < n && (r == 0 || pl.sorted_e[r] != pl.sorted_e[r - 1]);
            const unsigned b = __ballot_sync(FULL, lead);
            if (lead) {
                const int a = base + __popc(b & ((1u << lane) - 1u));
                pl.group[a] = pl.sorted_e[r];
                pl.row0[a] = r;
            }
            base += __popc(b);
        }
        if (lane < S) {
            pl.group[base + lane] = E + lane;
            pl.row0[base + lane] = n + lane * T;
        }
        if (lane == 0) {
            pl.na = base + S;
            pl.row0[base + S] = M;
        }
    }
    __syncthreads();
    const int na = pl.na;
    const int wpb = blockDim.x >> 5;
    const int64_t gwarp = static_cast<int64_t>(blockIdx.x) * wpb + warp;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * wpb;
    const uint64_t pol = policy_evict_first();

    // ---------------------------------------------------------- phase 1
    {
        const int chunks = H / 8;
        const int64_t ntasks = static_cast<int64_t>(na) * I;
        for (int64_t task = gwarp; task < ntasks; task += nwarps) {
            const int a = static_cast<int>(task / I), i = static_cast<int>(task % I);
            const int g = pl.group[a], r0 = pl.row0[a], nr = pl.row0[a + 1] - r0;
            const uint16_t *wg = w_gu + (static_cast<int64_t>(g) * 2 * I + i) * H;
            const uint16_t *wu = wg + static_cast<int64_t>(I) * H;
            for (int r = 0; r < nr; ++r) {
                const uint16_t *xrow[1] = {x + static_cast<int64_t>(pl.tok[r0 + r]) * H};
                float sg[1], su[1];
                gateup_partial_bf16<4, 1>(xrow, 1, wg, wu, chunks, pol, sg, su);
                const float gv = warp_sum(sg[0]), uv = warp_sum(su[0]);
                if (lane == 0) {
                    const __nv_bfloat16 hv = __float2bfloat16_rn(silu_f(gv) * uv);
                    h[static_cast<int64_t>(r0 + r) * I + i] =
                        *reinterpret_cast<const uint16_t *>(&hv);
                }
            }
        }
    }
    // The down weights do not depend on h: each warp loads the first chunks
    // of its first phase-2 task now, so that they are in flight while the
    // other warps finish phase 1 and the grid meets at the barrier.
    const int chunks2 = I / 8;
    const int nblk2 = (H + DL_DOWN_RW - 1) / DL_DOWN_RW;
    const int64_t ntasks2 = static_cast<int64_t>(na) * nblk2;
    uint4 first[DL_DOWN_RW][4];
    if (gwarp < ntasks2) {
        const int a = static_cast<int>(gwarp / nblk2);
        const int n0 = static_cast<int>(gwarp % nblk2) * DL_DOWN_RW;
        down_load_first<4, DL_DOWN_RW>(w_down + (static_cast<int64_t>(pl.group[a]) * H + n0) * I,
                                       I, n0, H, chunks2, pol, first);
    }
    if (!grid_barrier(barrier, gridDim.x, &pl.fail, dev_error)) return;

    // ---------------------------------------------------------- phase 2
    {
        const int chunks = chunks2;
        const int nblk = nblk2;
        auto store_y = [&](const float (&acc)[1][DL_DOWN_RW], int row, int n0) {
#pragma unroll
            for (int w = 0; w < DL_DOWN_RW; ++w) {
                const float v = warp_sum(acc[0][w]);
                if (lane == 0 && n0 + w < H) {
                    const __nv_bfloat16 b = __float2bfloat16_rn(v);
                    y[static_cast<int64_t>(row) * H + n0 + w] =
                        *reinterpret_cast<const uint16_t *>(&b);
                }
            }
        };
        auto task_rows = [&](int64_t task, int rfirst) {
            const int a = static_cast<int>(task / nblk);
            const int n0 = static_cast<int>(task % nblk) * DL_DOWN_RW;
            const int g = pl.group[a], r0 = pl.row0[a], nr = pl.row0[a + 1] - r0;
            const uint16_t *wd = w_down + (static_cast<int64_t>(g) * H + n0) * I;
            for (int r = rfirst; r < nr; ++r) {
                float acc[1][DL_DOWN_RW];
                down_partial_bf16<4, DL_DOWN_RW, 1, true>(h + static_cast<int64_t>(r0 + r) * I,
                                                          I, 1, wd, n0, H, chunks, pol, acc);
                store_y(acc, r0 + r, n0);
            }
        };
        if (gwarp < ntasks2) {          // this warp's first task: its first chunks are loaded
            const int a = static_cast<int>(gwarp / nblk);
            const int n0 = static_cast<int>(gwarp % nblk) * DL_DOWN_RW;
            const int r0 = pl.row0[a];
            const uint16_t *wd = w_down + (static_cast<int64_t>(pl.group[a]) * H + n0) * I;
            float acc[1][DL_DOWN_RW];
            down_partial_bf16_first<4, DL_DOWN_RW, true>(h + static_cast<int64_t>(r0) * I, I, wd,
                                                         n0, H, chunks, pol, first, acc);
            store_y(acc, r0, n0);
            task_rows(gwarp, 1);        // its other hidden rows (T > 1)
        }
        for (int64_t task = gwarp + nwarps; task < ntasks2; task += nwarps) task_rows(task, 0);
    }
    if (!grid_barrier(barrier, 2u * gridDim.x, &pl.fail, dev_error)) return;
    pdl_trigger();

    // ---------------------------------------------------------- phase 3
    // the combine's order: routed j = 0..k-1, then shared s, then residual
    {
        const int chunks = H / 8;
        const int64_t items = static_cast<int64_t>(T) * chunks;
        for (int64_t it = static_cast<int64_t>(blockIdx.x) * blockDim.x + tid; it < items;
             it += static_cast<int64_t>(gridDim.x) * blockDim.x) {
            const int t = static_cast<int>(it / chunks), c = static_cast<int>(it % chunks);
            float acc[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = 0.f;
            for (int j = 0; j < k; ++j) {
                const int r = pl.row_of_slot[t * k + j];
                const float wj = pl.w[t * k + j];
                const uint4 v = ld_cg(y + static_cast<int64_t>(r) * H + c * 8);
                const uint32_t p[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    acc[2 * q] = fmaf(wj, bf_lo(p[q]), acc[2 * q]);
                    acc[2 * q + 1] = fmaf(wj, bf_hi(p[q]), acc[2 * q + 1]);
                }
            }
            for (int s = 0; s < S; ++s) {
                const uint4 v = ld_cg(y + (static_cast<int64_t>(n) + s * T + t) * H + c * 8);
                const uint32_t p[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    acc[2 * q] = fmaf(1.0f, bf_lo(p[q]), acc[2 * q]);
                    acc[2 * q + 1] = fmaf(1.0f, bf_hi(p[q]), acc[2 * q + 1]);
                }
            }
            if (residual) {
                const uint4 v = ld_nc(residual + static_cast<int64_t>(t) * H + c * 8);
                const uint32_t p[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    acc[2 * q] += bf_lo(p[q]);
                    acc[2 * q + 1] += bf_hi(p[q]);
                }
            }
            uint4 o;
            o.x = pack_bf16x2(acc[0], acc[1]);
            o.y = pack_bf16x2(acc[2], acc[3]);
            o.z = pack_bf16x2(acc[4], acc[5]);
            o.w = pack_bf16x2(acc[6], acc[7]);
            *reinterpret_cast<uint4 *>(out + static_cast<int64_t>(t) * H + c * 8) = o;
        }
    }
}

template <int PER_LANE>
static moe_status launch_decode_layer(size_t dummy, cudaStream_t stream, const float *logits,
                                      const uint16_t *x, int T, int E, int S, int k,
                                      int renormalize, int H, int I, const uint16_t *w_gu,
                                      const uint16_t *w_down, const uint16_t *residual,
                                      uint16_t *out, int32_t *topk_ids, float *topk_w,
                                      unsigned *barrier, uint16_t *h, uint16_t *y,
                                      int32_t *dev_error) {
    (void)dummy;
    // every CTA must be resident at once (grid barriers): the grid is the
    // occupancy-limited resident count and the launch is cooperative
    static int per_sm_of_device[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
    if (per_sm_of_device[dev] < 1) {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_layer_kernel<PER_LANE>,
                                                          DL_THREADS, 0) != cudaSuccess ||
            per_sm < 1)
            return MOE_ERR_CUDA;
        per_sm_of_device[dev] = per_sm;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(per_sm_of_device[dev] * sm_count());
    cfg.blockDim = dim3(DL_THREADS);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, decode_layer_kernel<PER_LANE>, logits, x, T, E, S, k,
                           renormalize, H, I, w_gu, w_down, residual, out, topk_ids, topk_w,
                           barrier, h, y, dev_error) != cudaSuccess)
        return MOE_ERR_CUDA;
    return launch_status();
}

static size_t round256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

}  // namespace moe

using namespace moe;

extern "C" size_t moe_decode_workspace_size(int T, int E, int S, int k, int H, int I) {
    if (T < 1 || E < 1 || S < 0 || k < 1 || H < 1 || I < 1) return 0;
    const size_t M = static_cast<size_t>(T) * k + static_cast<size_t>(S) * T;
    return 256 + round256(M * I * 2) + round256(M * H * 2);
}

extern "C" moe_status moe_decode_layer(const float *logits, const uint16_t *x, int T, int E,
                                       int S, int k, int renormalize, int H, int I,
                                       const uint16_t *w_gu, const uint16_t *w_down,
                                       const uint16_t *residual, uint16_t *out,
                                       int32_t *topk_ids, float *topk_w, void *workspace,
                                       size_t workspace_bytes, int32_t *dev_error,
                                       cudaStream_t stream) {
    if (!logits || !x || !w_gu || !w_down || !out || !workspace) return MOE_ERR_INVALID_ARG;
    if (T < 1 || E < 1 || S < 0 || k < 1 || k > E || k > 32 || H < 1 || I < 1)
        return MOE_ERR_INVALID_ARG;
    if (T > 8 || T * k > DL_MAX_SLOTS || S * T > DL_MAX_ROWS - DL_MAX_SLOTS || S > 32 ||
        E > 256)
        return MOE_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(E + S) * 2 * I * H >= (1ll << 40)) return MOE_ERR_UNSUPPORTED;
    if (H % 8 != 0 || I % 8 != 0) return MOE_ERR_ALIGNMENT;
    if (!aligned16(x) || !aligned16(w_gu) || !aligned16(w_down) || !aligned16(out) ||
        (residual && !aligned16(residual)) || !aligned16(workspace))
        return MOE_ERR_ALIGNMENT;
    if (workspace_bytes < moe_decode_workspace_size(T, E, S, k, H, I)) return MOE_ERR_WORKSPACE;
    const size_t M = static_cast<size_t>(T) * k + static_cast<size_t>(S) * T;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    unsigned *barrier = reinterpret_cast<unsigned *>(ws);
    uint16_t *h = reinterpret_cast<uint16_t *>(ws + 256);
    uint16_t *y = reinterpret_cast<uint16_t *>(ws + 256 + round256(M * I * 2));
    if (cudaMemsetAsync(barrier, 0, sizeof(unsigned), stream) != cudaSuccess) return MOE_ERR_CUDA;
    const int per_lane = (E + 31) / 32;
#define MOE_DL(PL)                                                                               \
    launch_decode_layer<PL>(0, stream, logits, x, T, E, S, k, renormalize, H, I, w_gu, w_down, \
                            residual, out, topk_ids, topk_w, barrier, h, y, dev_error)
    if (per_lane <= 1) return MOE_DL(1);
    if (per_lane <= 2) return MOE_DL(2);
    if (per_lane <= 4) return MOE_DL(4);
    return MOE_DL(8);
#undef MOE_DL
}
