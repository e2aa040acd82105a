// permute.cu -- stable sort of token slots by expert, and the row gather.
//
// The "switchyard" page (02 Kernels and dispatch, "Route and sort") orders
// the token rows by expert using a prefix scan over the whole block, with
// no atomic operations; this file does the same on sm_103a.
//
// The building block is a block-wide ranking of up to 1024 slots (one per
// thread, in slot order): each warp groups its 32 slots by expert with a
// match, the group leader stores the warp's count for that expert in its own
// shared-memory word (no two threads write the same word, so no atomics),
// the 32 per-warp counts of every expert are scanned across warps, and a
// slot's rank inside its expert is its warp's prefix plus its rank inside
// the warp.  Lanes and warps follow slot order, so the sort is stable.
//
//  * up to 1024 slots (decode): one kernel.  Every CTA ranks all slots
//    (identical results), CTA 0 writes the offsets and the permutation, and
//    all CTAs share the gather of activation rows into expert order;
//  * more slots: a counting kernel writes each 1024-slot chunk's per-expert
//    counts into the workspace; a placing kernel gives every chunk its base
//    per expert (the expert's offset plus the counts of earlier chunks),
//    ranks the chunk again and writes the permutation; a gather kernel
//    copies the rows.  Three launches, each spread over the GPU;
//  * moe_route_permute also routes, inside the small kernel.
#include <algorithm>
#include <climits>

#include "route_token.cuh"

namespace moe {

constexpr int CHUNK = 1024;          // slots ranked by one CTA (one per thread)

// Dynamic shared memory of a ranking CTA: per-warp counts [32][E] + totals [E+1].
inline size_t rank_smem_bytes(int E) { return (33 * static_cast<size_t>(E) + 1) * 4; }

// Rank the block's slots by expert.  e is this thread's expert (-1: no slot).
// s_cnt ([32][E]) must be zero on entry.  On return s_tot[g] is the block's
// count of expert g; the result is the thread's rank inside its expert
// within the block.
__device__ __forceinline__ int block_rank(int e, int E, int *s_cnt, int *s_tot) {
    const int lane = lane_id(), warp = threadIdx.x >> 5;
    const unsigned peers = __match_any_sync(FULL, e);
    const int wrank = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0 && wrank == 0) s_cnt[warp * E + e] = __popc(peers);
    __syncthreads();
    for (int g = threadIdx.x; g < E; g += blockDim.x) {
        int run = 0;
        for (int w = 0; w < 32; ++w) {
            const int c = s_cnt[w * E + g];
            s_cnt[w * E + g] = run;
            run += c;
        }
        s_tot[g] = run;
    }
    __syncthreads();
    return e >= 0 ? s_cnt[warp * E + e] + wrank : 0;
}

// Exclusive scan of v[0..E) in place by one whole warp.
__device__ __forceinline__ void warp_exclusive_scan_inplace(int *v, int E) {
    const int lane = lane_id();
    int carry = 0;
    for (int c0 = 0; c0 < E; c0 += 32) {
        const int g = c0 + lane;
        const int x = g < E ? v[g] : 0;
        const int inc = warp_inclusive_scan(x);
        if (g < E) v[g] = carry + inc - x;
        carry += __shfl_sync(FULL, inc, 31);
    }
}

// dst_row = x[t] (rounded to bf16 for fp32 activations); 16-byte copies by one warp.
template <bool X_F32>
__device__ __forceinline__ void copy_row(const void *__restrict__ x, int64_t t, int H,
                                         uint16_t *__restrict__ dst_row) {
    const int lane = lane_id(), chunks = H / 8;
    uint4 *dst = reinterpret_cast<uint4 *>(dst_row);
    if (X_F32) {
        const float4 *src = reinterpret_cast<const float4 *>(static_cast<const float *>(x) + t * H);
        for (int c = lane; c < chunks; c += 32) {
            const float4 a = __ldg(src + 2 * c), b = __ldg(src + 2 * c + 1);
            dst[c] = make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w),
                                pack_bf16x2(b.x, b.y), pack_bf16x2(b.z, b.w));
        }
    } else {
        // up to 8 chunks per lane loaded before any is stored, so a warp
        // keeps a whole 4 KB row in flight
        const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(x) + t * H);
        for (int c0 = 0; c0 < chunks; c0 += 32 * 8) {
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int c = c0 + lane + 32 * u;
                if (c < chunks) v[u] = __ldg(src + c);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int c = c0 + lane + 32 * u;
                if (c < chunks) dst[c] = v[u];
            }
        }
    }
}

// Invalid routing: every group empty, every slot unplaced, so no later
// kernel reads outside its buffers.
__device__ __forceinline__ void write_empty(int E, int S, int64_t n, int32_t *offsets,
                                            int32_t *row_of_slot) {
    for (int g = threadIdx.x; g <= E + S; g += blockDim.x) offsets[g] = 0;
    for (int64_t s = threadIdx.x; s < n; s += blockDim.x) row_of_slot[s] = -1;
}

// ------------------------------------------------------------ small batches

// Ranks all n <= 1024 slots (in every CTA), writes the permutation (CTA 0)
// and gathers the rows (all CTAs).  If ROUTE, the slots' experts come from
// routing the logits inside the kernel, one warp per token.
template <bool ROUTE, int PER_LANE, bool X_F32>
__global__ void __launch_bounds__(1024) permute_small_kernel(
    const int32_t *__restrict__ ids_in, const float *__restrict__ logits, int renormalize, int T,
    int E, int S, int k, const void *__restrict__ x, int H, int32_t *__restrict__ topk_ids,
    float *__restrict__ topk_w, int32_t *__restrict__ offsets, int32_t *__restrict__ sorted_slot,
    int32_t *__restrict__ row_of_slot, uint16_t *__restrict__ x_perm, int cap,
    int32_t *__restrict__ dropped, int32_t *dev_error) {
    extern __shared__ int smem[];
    int *s_cnt = smem;                          // [32][E]
    int *s_base = smem + 32 * E;                // [E+1]
    __shared__ int s_ids[CHUNK];
    __shared__ int s_sorted[CHUNK];
    const int tid = threadIdx.x, n = T * k;
    for (int i = tid; i < 32 * E; i += blockDim.x) s_cnt[i] = 0;
    pdl_wait();
    pdl_trigger();

    bool bad = false;
    if (ROUTE) {
        const int lane = lane_id(), warp = tid >> 5;
        for (int t = warp; t < T; t += blockDim.x >> 5) {
            int id;
            float w;
            if (!route_token<PER_LANE>(logits + static_cast<size_t>(t) * E, E, k, renormalize,
                                       id, w)) {
                bad = true;                      // a NaN logit
                continue;
            }
            if (lane < k) {
                s_ids[t * k + lane] = id;
                if (blockIdx.x == 0) {
                    topk_ids[t * k + lane] = id;
                    topk_w[t * k + lane] = w;
                }
            }
        }
        __syncthreads();
    }
    int e = -1;
    if (tid < n) {
        e = ROUTE ? s_ids[tid] : ids_in[tid];
        if (e < 0 || e >= E) {
            bad = true;
            e = -1;
        }
    }
    if (__syncthreads_or(bad)) {
        if (blockIdx.x == 0) {
            if (tid == 0) report(dev_error, MOE_ERR_DEVICE_CHECK);
            write_empty(E, S, n, offsets, row_of_slot);
        }
        return;
    }
    const int rank = block_rank(e, E, s_cnt, s_base);
    // an expert serves at most `cap` slots (all of them in the dropless call)
    for (int g = tid; g <= E; g += blockDim.x) s_base[g] = g < E ? min(s_base[g], cap) : 0;
    __syncthreads();
    if (tid < 32) warp_exclusive_scan_inplace(s_base, E + 1);
    __syncthreads();
    const int kept = s_base[E];                 // routed rows; shared rows follow
    if (blockIdx.x == 0) {
        for (int g = tid; g <= E + S; g += blockDim.x)
            offsets[g] = g <= E ? s_base[g] : kept + (g - E) * T;
        for (int r = kept + tid; r < n; r += blockDim.x) sorted_slot[r] = -1;
        if (tid == 0 && dropped) *dropped = n - kept;
    }
    if (e >= 0) {
        if (rank < cap) {
            const int pos = s_base[e] + rank;
            s_sorted[pos] = tid;
            if (blockIdx.x == 0) {
                sorted_slot[pos] = tid;
                row_of_slot[tid] = pos;
            }
        } else if (blockIdx.x == 0) {
            row_of_slot[tid] = MOE_ROW_DROPPED;
        }
    }
    __syncthreads();
    const int M = kept + S * T;
    const int warps = blockDim.x >> 5;
    for (int r = blockIdx.x * warps + (tid >> 5); r < M; r += gridDim.x * warps) {
        const int t = r < kept ? s_sorted[r] / k : (r - kept) % T;
        copy_row<X_F32>(x, t, H, x_perm + static_cast<int64_t>(r) * H);
    }
}

// ------------------------------------------------------------ large batches

// counts[c][0..E) = per-expert slot counts of chunk c; counts[c][E] = 1 if
// the chunk held an invalid expert id.
__global__ void __launch_bounds__(1024) permute_count_kernel(const int32_t *__restrict__ ids,
                                                             int64_t n, int E,
                                                             int32_t *__restrict__ counts,
                                                             int32_t *dev_error) {
    extern __shared__ int smem[];
    int *s_cnt = smem, *s_tot = smem + 32 * E;
    for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) s_cnt[i] = 0;
    pdl_wait();
    pdl_trigger();
    const int64_t s = static_cast<int64_t>(blockIdx.x) * CHUNK + threadIdx.x;
    int e = s < n ? ids[s] : -1;
    const bool bad = s < n && (e < 0 || e >= E);
    if (bad) e = -1;
    const int any_bad = __syncthreads_or(bad);
    block_rank(e, E, s_cnt, s_tot);
    int32_t *row = counts + static_cast<int64_t>(blockIdx.x) * (E + 1);
    for (int g = threadIdx.x; g < E; g += blockDim.x) row[g] = s_tot[g];
    if (threadIdx.x == 0) {
        row[E] = any_bad ? 1 : 0;
        if (any_bad) report(dev_error, MOE_ERR_DEVICE_CHECK);
    }
}

// Dynamic shared memory of the placing kernel: ranking area + bases [E].
inline size_t place_smem_bytes(int E) {
    return rank_smem_bytes(E) + static_cast<size_t>(2 * E + 1) * 4;
}

// Places chunk blockIdx.x.  The base of expert g in this chunk is g's offset
// (scan of all chunks' totals) plus g's count in earlier chunks; CTA 0 also
// writes the offsets table.
__global__ void __launch_bounds__(1024) permute_place_kernel(
    const int32_t *__restrict__ ids, int T, int E, int S, int k, const int32_t *__restrict__ counts,
    int nchunks, int32_t *__restrict__ offsets, int32_t *__restrict__ sorted_slot,
    int32_t *__restrict__ row_of_slot, int cap, int32_t *__restrict__ dropped) {
    extern __shared__ int smem[];
    int *s_cnt = smem;                           // [32][E], zero until the ranking
    int *s_tot = smem + 32 * E;                  // [E+1]
    int *s_base = s_tot + E + 1;                 // [E]
    int *s_off = s_base + E;                     // [E+1]
    __shared__ int s_bad;
    const int64_t n = static_cast<int64_t>(T) * k;
    const int c = blockIdx.x;
    for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) s_cnt[i] = 0;
    if (threadIdx.x == 0) s_bad = 0;
    pdl_wait();
    pdl_trigger();
    __syncthreads();
    for (int g = threadIdx.x; g < E; g += blockDim.x) {
        int total = 0, before = 0;
        // unrolled so that the chunks' counts are loaded together rather
        // than one L2 round trip after another
#pragma unroll 8
        for (int cc = 0; cc < nchunks; ++cc) {
            const int v = counts[static_cast<int64_t>(cc) * (E + 1) + g];
            total += v;
            if (cc < c) before += v;
        }
        s_tot[g] = total;
        s_base[g] = before;
    }
    for (int cc = threadIdx.x; cc < nchunks; cc += blockDim.x)
        if (counts[static_cast<int64_t>(cc) * (E + 1) + E]) s_bad = 1;
    __syncthreads();
    if (s_bad) {
        if (c == 0) write_empty(E, S, n, offsets, row_of_slot);
        return;
    }
    // offsets: exclusive scan of the served counts min(total, cap)
    for (int g = threadIdx.x; g <= E; g += blockDim.x) s_off[g] = g < E ? min(s_tot[g], cap) : 0;
    __syncthreads();
    if (threadIdx.x < 32) warp_exclusive_scan_inplace(s_off, E + 1);
    __syncthreads();
    const int64_t kept = s_off[E];               // routed rows; shared rows follow
    if (c == 0) {
        for (int g = threadIdx.x; g <= E + S; g += blockDim.x)
            offsets[g] = g <= E ? s_off[g]
                                : static_cast<int32_t>(kept + static_cast<int64_t>(g - E) * T);
        if (threadIdx.x == 0 && dropped) *dropped = static_cast<int32_t>(n - kept);
    }
    const int64_t s = static_cast<int64_t>(c) * CHUNK + threadIdx.x;
    if (s >= kept && s < n) sorted_slot[s] = -1;     // positions past the served rows
    const int e = s < n ? ids[s] : -1;
    const int rank = block_rank(e, E, s_cnt, s_tot);
    if (e >= 0) {
        const int grank = s_base[e] + rank;      // earlier chunks' slots of e + this chunk's
        if (grank < cap) {
            const int pos = s_off[e] + grank;
            sorted_slot[pos] = static_cast<int32_t>(s);
            row_of_slot[s] = pos;
        } else {
            row_of_slot[s] = MOE_ROW_DROPPED;
        }
    }
}

// x_perm[r] = x[token of row r]; one warp per row.
template <bool X_F32>
__global__ void __launch_bounds__(256) permute_gather_kernel(
    const void *__restrict__ x, int T, int E, int S, int k, int H,
    const int32_t *__restrict__ offsets, const int32_t *__restrict__ sorted_slot,
    uint16_t *__restrict__ x_perm) {
    pdl_wait();
    pdl_trigger();
    const int64_t n = static_cast<int64_t>(T) * k;
    const int64_t routed_rows = offsets[E];      // served routed rows
    const int64_t M = offsets[E + S];            // all rows; 0 after an invalid routing
    const int64_t wstride = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; r < M;
         r += wstride) {
        int64_t t;
        if (r < routed_rows) {
            const int64_t s = sorted_slot[r];
            if (s < 0 || s >= n) continue;
            t = s / k;
        } else {
            t = (r - routed_rows) % T;
        }
        copy_row<X_F32>(x, t, H, x_perm + r * H);
    }
}

// ------------------------------------------------------------------ host

// Raise a kernel's dynamic shared-memory limit once per device when needed.
template <typename Kernel>
static bool allow_smem(Kernel kernel, size_t bytes, int *done_per_device) {
    if (bytes <= 48 * 1024) return true;
    if (bytes + 16 * 1024 > static_cast<size_t>(max_smem_optin())) return false;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    if (!done_per_device[dev]) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 max_smem_optin() - 16 * 1024) != cudaSuccess)
            return false;
        done_per_device[dev] = 1;
    }
    return true;
}

template <bool ROUTE, int PER_LANE>
static moe_status launch_small(bool x_f32, const int32_t *ids, const float *logits,
                               int renormalize, int T, int E, int S, int k, const void *x, int H,
                               int32_t *topk_ids, float *topk_w, int32_t *offsets,
                               int32_t *sorted_slot, int32_t *row_of_slot, uint16_t *x_perm,
                               int cap, int32_t *dropped, int32_t *dev_error,
                               cudaStream_t stream) {
    const int64_t M = static_cast<int64_t>(T) * k + static_cast<int64_t>(S) * T;
    const int grid = static_cast<int>(std::min<int64_t>((M + 31) / 32, sm_count()));
    const size_t smem = rank_smem_bytes(E);
    static int done_f32[64] = {0}, done_bf16[64] = {0};
    if (x_f32) {
        auto kern = permute_small_kernel<ROUTE, PER_LANE, true>;
        if (!allow_smem(kern, smem, done_f32)) return MOE_ERR_UNSUPPORTED;
        launch(kern, grid, CHUNK, smem, stream, ids, logits, renormalize, T, E, S, k, x, H,
               topk_ids, topk_w, offsets, sorted_slot, row_of_slot, x_perm, cap, dropped,
               dev_error);
    } else {
        auto kern = permute_small_kernel<ROUTE, PER_LANE, false>;
        if (!allow_smem(kern, smem, done_bf16)) return MOE_ERR_UNSUPPORTED;
        launch(kern, grid, CHUNK, smem, stream, ids, logits, renormalize, T, E, S, k, x, H,
               topk_ids, topk_w, offsets, sorted_slot, row_of_slot, x_perm, cap, dropped,
               dev_error);
    }
    return launch_status();
}

static int64_t chunks_of(int T, int k) { return (static_cast<int64_t>(T) * k + CHUNK - 1) / CHUNK; }

}  // namespace moe

using namespace moe;

extern "C" size_t moe_permute_workspace_size(int T, int E, int S, int k) {
    (void)S;
    if (T < 1 || E < 1 || k < 1) return 0;
    if (static_cast<int64_t>(T) * k <= CHUNK) return 0;
    const size_t bytes = static_cast<size_t>(chunks_of(T, k)) * (E + 1) * 4;
    return (bytes + 255) & ~static_cast<size_t>(255);
}

namespace moe {
// moe_permute and moe_permute_capped: cap = slots an expert may serve
// (INT_MAX: all), dropped = device word for the dropped-slot count or NULL.
static moe_status permute_impl(const int32_t *topk_ids, int T, int E, int S, int k, int cap,
                               const void *x, int x_dtype, int H, int32_t *offsets,
                               int32_t *sorted_slot, int32_t *row_of_slot, uint16_t *x_perm,
                               int32_t *dropped, void *workspace, size_t workspace_bytes,
                               int32_t *dev_error, cudaStream_t stream) {
    if (!topk_ids || !x || !offsets || !sorted_slot || !row_of_slot || !x_perm)
        return MOE_ERR_INVALID_ARG;
    if (T < 1 || E < 1 || S < 0 || k < 1 || k > E || k > 32 || H < 1 || cap < 0)
        return MOE_ERR_INVALID_ARG;
    if (x_dtype != MOE_DTYPE_BF16 && x_dtype != MOE_DTYPE_F32) return MOE_ERR_INVALID_ARG;
    if (E + S > 1024) return MOE_ERR_UNSUPPORTED;
    const int64_t n = static_cast<int64_t>(T) * k, M = n + static_cast<int64_t>(S) * T;
    if (n >= (1ll << 31) || M * H >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
    if (H % 8 != 0 || !aligned16(x) || !aligned16(x_perm)) return MOE_ERR_ALIGNMENT;
    const bool f32 = x_dtype == MOE_DTYPE_F32;
    if (n <= CHUNK)
        return launch_small<false, 1>(f32, topk_ids, nullptr, 0, T, E, S, k, x, H, nullptr,
                                      nullptr, offsets, sorted_slot, row_of_slot, x_perm, cap,
                                      dropped, dev_error, stream);

    const size_t need = moe_permute_workspace_size(T, E, S, k);
    if (!workspace || workspace_bytes < need) return MOE_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 3u) != 0) return MOE_ERR_ALIGNMENT;
    int32_t *counts = static_cast<int32_t *>(workspace);
    const int nchunks = static_cast<int>(chunks_of(T, k));
    static int done_count[64] = {0}, done_place[64] = {0};
    if (!allow_smem(permute_count_kernel, rank_smem_bytes(E), done_count) ||
        !allow_smem(permute_place_kernel, place_smem_bytes(E), done_place))
        return MOE_ERR_UNSUPPORTED;
    launch(permute_count_kernel, nchunks, CHUNK, rank_smem_bytes(E), stream, topk_ids, n, E,
           counts, dev_error);
    moe_status st = launch_status();
    if (st != MOE_OK) return st;
    launch(permute_place_kernel, nchunks, CHUNK, place_smem_bytes(E), stream, topk_ids, T, E, S,
           k, static_cast<const int32_t *>(counts), nchunks, offsets, sorted_slot, row_of_slot,
           cap, dropped);
    if ((st = launch_status()) != MOE_OK) return st;
    const int blocks = static_cast<int>(std::min<int64_t>((M + 7) / 8, sm_count() * 8ll));
    if (f32)
        launch(permute_gather_kernel<true>, blocks, 256, 0, stream, x, T, E, S, k, H,
               static_cast<const int32_t *>(offsets), static_cast<const int32_t *>(sorted_slot),
               x_perm);
    else
        launch(permute_gather_kernel<false>, blocks, 256, 0, stream, x, T, E, S, k, H,
               static_cast<const int32_t *>(offsets), static_cast<const int32_t *>(sorted_slot),
               x_perm);
    return launch_status();
}
}  // namespace moe

extern "C" moe_status moe_permute(const int32_t *topk_ids, int T, int E, int S, int k,
                                  const void *x, int x_dtype, int H, int32_t *offsets,
                                  int32_t *sorted_slot, int32_t *row_of_slot, uint16_t *x_perm,
                                  void *workspace, size_t workspace_bytes, int32_t *dev_error,
                                  cudaStream_t stream) {
    return permute_impl(topk_ids, T, E, S, k, INT_MAX, x, x_dtype, H, offsets, sorted_slot,
                        row_of_slot, x_perm, nullptr, workspace, workspace_bytes, dev_error,
                        stream);
}

extern "C" moe_status moe_permute_capped(const int32_t *topk_ids, int T, int E, int S, int k,
                                         int capacity, const void *x, int x_dtype, int H,
                                         int32_t *offsets, int32_t *sorted_slot,
                                         int32_t *row_of_slot, uint16_t *x_perm,
                                         int32_t *dropped, void *workspace,
                                         size_t workspace_bytes, int32_t *dev_error,
                                         cudaStream_t stream) {
    if (!dropped) return MOE_ERR_INVALID_ARG;
    return permute_impl(topk_ids, T, E, S, k, capacity, x, x_dtype, H, offsets, sorted_slot,
                        row_of_slot, x_perm, dropped, workspace, workspace_bytes, dev_error,
                        stream);
}

extern "C" moe_status moe_route_permute(const float *logits, int T, int E, int S, int k,
                                        int renormalize, const void *x, int x_dtype, int H,
                                        int32_t *topk_ids, float *topk_w, int32_t *offsets,
                                        int32_t *sorted_slot, int32_t *row_of_slot,
                                        uint16_t *x_perm, int32_t *dev_error,
                                        cudaStream_t stream) {
    if (!logits || !x || !topk_ids || !topk_w || !offsets || !sorted_slot || !row_of_slot ||
        !x_perm)
        return MOE_ERR_INVALID_ARG;
    if (T < 1 || E < 1 || S < 0 || k < 1 || k > E || k > 32 || H < 1) return MOE_ERR_INVALID_ARG;
    if (x_dtype != MOE_DTYPE_BF16 && x_dtype != MOE_DTYPE_F32) return MOE_ERR_INVALID_ARG;
    if (static_cast<int64_t>(T) * k > CHUNK || E > 256 || E + S > 1024)
        return MOE_ERR_UNSUPPORTED;
    const int64_t M = static_cast<int64_t>(T) * k + static_cast<int64_t>(S) * T;
    if (M * H >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
    if (H % 8 != 0 || !aligned16(x) || !aligned16(x_perm)) return MOE_ERR_ALIGNMENT;
    const bool f32 = x_dtype == MOE_DTYPE_F32;
    const int per_lane = (E + 31) / 32;
    if (per_lane <= 1)
        return launch_small<true, 1>(f32, nullptr, logits, renormalize, T, E, S, k, x, H,
                                     topk_ids, topk_w, offsets, sorted_slot, row_of_slot, x_perm,
                                     INT_MAX, nullptr, dev_error, stream);
    if (per_lane <= 2)
        return launch_small<true, 2>(f32, nullptr, logits, renormalize, T, E, S, k, x, H,
                                     topk_ids, topk_w, offsets, sorted_slot, row_of_slot, x_perm,
                                     INT_MAX, nullptr, dev_error, stream);
    if (per_lane <= 4)
        return launch_small<true, 4>(f32, nullptr, logits, renormalize, T, E, S, k, x, H,
                                     topk_ids, topk_w, offsets, sorted_slot, row_of_slot, x_perm,
                                     INT_MAX, nullptr, dev_error, stream);
    return launch_small<true, 8>(f32, nullptr, logits, renormalize, T, E, S, k, x, H, topk_ids,
                                 topk_w, offsets, sorted_slot, row_of_slot, x_perm, INT_MAX,
                                 nullptr, dev_error, stream);
}
