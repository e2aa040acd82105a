// permute.cu -- stable sort of token slots by expert, and the row gather.
//
// "Rows sorted by expert with a block-wide prefix scan and no atomics"
// ("switchyard" page, 02 Kernels and dispatch, "Route and sort").  One CTA
// of NT threads sorts all T*k slots:
//   1. thread i owns the contiguous slot range [i*q, (i+1)*q) and counts its
//      slots per expert in its own shared-memory column cnt[e][i] (no two
//      threads ever write the same word, so no atomics);
//   2. each expert's row of counts is scanned across threads (a warp per
//      expert row), giving thread i's first position inside expert e;
//   3. one warp scans the E totals into the offsets table;
//   4. every thread walks its slots again and places each one at
//      offsets[e] + its running position in expert e.
// Thread order equals slot order, so the sort is stable.  A second kernel
// gathers the activation rows into expert order with 128-bit copies.
#include <algorithm>

#include "common.cuh"

namespace moe {

constexpr int PERM_SMEM_BUDGET = 160 * 1024;   // bytes for the count matrix

__global__ void __launch_bounds__(1024) permute_index_kernel(
    const int32_t *__restrict__ ids, int T, int E, int S, int k, int32_t *__restrict__ offsets,
    int32_t *__restrict__ sorted_slot, int32_t *__restrict__ row_of_slot, int32_t *dev_error) {
    extern __shared__ uint32_t cnt[];            // [E][NT]
    __shared__ uint32_t base[1024];              // expert start rows
    const int NT = blockDim.x, tid = threadIdx.x, lane = lane_id(), warp = tid >> 5;
    const int nwarps = NT >> 5;
    const int64_t n = static_cast<int64_t>(T) * k;
    const int64_t q = (n + NT - 1) / NT;
    const int64_t s0 = min(n, tid * q), s1 = min(n, s0 + q);

    for (int i = tid; i < E * NT; i += NT) cnt[i] = 0;
    __syncthreads();

    bool bad = false;
    for (int64_t s = s0; s < s1; ++s) {
        const int e = ids[s];
        if (e < 0 || e >= E) bad = true;
        else cnt[e * NT + tid] += 1;
    }
    if (__syncthreads_or(bad)) {
        // invalid routing: report it, leave every group empty and every slot
        // unplaced so that no later kernel reads outside its buffers
        if (tid == 0) report(dev_error, MOE_ERR_DEVICE_CHECK);
        for (int g = tid; g <= E + S; g += NT) offsets[g] = 0;
        for (int64_t s = tid; s < n; s += NT) row_of_slot[s] = -1;
        return;
    }

    // 2. exclusive scan of each expert's counts across threads
    for (int e = warp; e < E; e += nwarps) {
        uint32_t carry = 0;
        for (int c = 0; c < NT; c += 32) {
            const uint32_t v = cnt[e * NT + c + lane];
            const uint32_t inc = warp_inclusive_scan(v);
            cnt[e * NT + c + lane] = carry + inc - v;
            carry += __shfl_sync(FULL, inc, 31);
        }
        if (lane == 0) base[e] = carry;          // total of expert e (for now)
    }
    __syncthreads();

    // 3. exclusive scan of the totals -> offsets
    if (warp == 0) {
        uint32_t carry = 0;
        for (int c = 0; c < E; c += 32) {
            const int e = c + lane;
            const uint32_t v = e < E ? base[e] : 0u;
            const uint32_t inc = warp_inclusive_scan(v);
            if (e < E) {
                base[e] = carry + inc - v;
                offsets[e] = static_cast<int32_t>(carry + inc - v);
            }
            carry += __shfl_sync(FULL, inc, 31);
        }
        // shared experts: S groups of T rows each, tokens in order
        for (int s = lane; s <= S; s += 32)
            offsets[E + s] = static_cast<int32_t>(carry + static_cast<int64_t>(s) * T);
    }
    __syncthreads();

    // 4. stable placement
    for (int64_t s = s0; s < s1; ++s) {
        const int e = ids[s];
        const uint32_t pos = base[e] + cnt[e * NT + tid];
        cnt[e * NT + tid] += 1;
        sorted_slot[pos] = static_cast<int32_t>(s);
        row_of_slot[s] = static_cast<int32_t>(pos);
    }
}

// x_perm[r] = x[token of row r]; one warp per row, 16-byte (8 x bf16) chunks.
template <bool X_F32>
__global__ void __launch_bounds__(256) permute_gather_kernel(
    const void *__restrict__ x, int T, int E, int S, int k, int H,
    const int32_t *__restrict__ offsets, const int32_t *__restrict__ sorted_slot,
    uint16_t *__restrict__ x_perm) {
    const int lane = lane_id();
    const int64_t n = static_cast<int64_t>(T) * k;
    const int64_t M = n + static_cast<int64_t>(S) * T;
    const int64_t routed_rows = offsets[E];      // 0 after an invalid routing
    const int chunks = H / 8;
    const int64_t wstride = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; r < M;
         r += wstride) {
        int64_t t;
        if (r < n) {
            if (r >= routed_rows) continue;
            const int64_t s = sorted_slot[r];
            if (s < 0 || s >= n) continue;
            t = s / k;
        } else {
            if (routed_rows != n) continue;
            t = (r - n) % T;
        }
        uint4 *dst = reinterpret_cast<uint4 *>(x_perm + r * H);
        if (X_F32) {
            const float4 *src = reinterpret_cast<const float4 *>(static_cast<const float *>(x) + t * H);
            for (int c = lane; c < chunks; c += 32) {
                const float4 a = __ldg(src + 2 * c), b = __ldg(src + 2 * c + 1);
                uint4 o;
                o.x = pack_bf16x2(a.x, a.y);
                o.y = pack_bf16x2(a.z, a.w);
                o.z = pack_bf16x2(b.x, b.y);
                o.w = pack_bf16x2(b.z, b.w);
                dst[c] = o;
            }
        } else {
            const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(x) + t * H);
            for (int c = lane; c < chunks; c += 32) dst[c] = __ldg(src + c);
        }
    }
}

}  // namespace moe

using namespace moe;

extern "C" size_t moe_permute_workspace_size(int, int, int, int) { return 0; }

extern "C" moe_status moe_permute(const int32_t *topk_ids, int T, int E, int S, int k,
                                  const void *x, int x_dtype, int H, int32_t *offsets,
                                  int32_t *sorted_slot, int32_t *row_of_slot, uint16_t *x_perm,
                                  void *workspace, size_t workspace_bytes, int32_t *dev_error,
                                  cudaStream_t stream) {
    (void)workspace;
    (void)workspace_bytes;
    if (!topk_ids || !x || !offsets || !sorted_slot || !row_of_slot || !x_perm)
        return MOE_ERR_INVALID_ARG;
    if (T < 1 || E < 1 || S < 0 || k < 1 || k > E || k > 32 || H < 1) return MOE_ERR_INVALID_ARG;
    if (x_dtype != MOE_DTYPE_BF16 && x_dtype != MOE_DTYPE_F32) return MOE_ERR_INVALID_ARG;
    if (E + S > 1024) return MOE_ERR_UNSUPPORTED;
    const int64_t n = static_cast<int64_t>(T) * k, M = n + static_cast<int64_t>(S) * T;
    if (n >= (1ll << 31) || M * H >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
    if (H % 8 != 0 || !aligned16(x) || !aligned16(x_perm)) return MOE_ERR_ALIGNMENT;

    // threads: about 8 slots each, a power of two in [32, 1024] that keeps the
    // E x NT count matrix within the shared-memory budget
    int nt_max = 32;
    while (nt_max * 2 <= 1024 && static_cast<int64_t>(E) * nt_max * 2 * 4 <= PERM_SMEM_BUDGET)
        nt_max *= 2;
    if (static_cast<int64_t>(E) * nt_max * 4 > PERM_SMEM_BUDGET) return MOE_ERR_UNSUPPORTED;
    int nt = 32;
    while (nt < nt_max && static_cast<int64_t>(nt) * 8 < n) nt *= 2;
    const size_t smem = static_cast<size_t>(E) * nt * 4;
    if (smem > 48 * 1024) {
        // once per device, so that launches can be captured into CUDA graphs
        static bool attr_set[64] = {false};
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
        if (!attr_set[dev]) {
            if (cudaFuncSetAttribute(permute_index_kernel,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     PERM_SMEM_BUDGET) != cudaSuccess)
                return MOE_ERR_CUDA;
            attr_set[dev] = true;
        }
    }
    permute_index_kernel<<<1, nt, smem, stream>>>(topk_ids, T, E, S, k, offsets, sorted_slot,
                                                   row_of_slot, dev_error);
    moe_status st = launch_status();
    if (st != MOE_OK) return st;

    const int64_t warps_needed = M;
    const int64_t max_blocks = static_cast<int64_t>(sm_count()) * 8;
    const int blocks = static_cast<int>(std::min<int64_t>((warps_needed + 7) / 8, max_blocks));
    if (x_dtype == MOE_DTYPE_F32)
        permute_gather_kernel<true><<<blocks, 256, 0, stream>>>(x, T, E, S, k, H, offsets,
                                                                sorted_slot, x_perm);
    else
        permute_gather_kernel<false><<<blocks, 256, 0, stream>>>(x, T, E, S, k, H, offsets,
                                                                 sorted_slot, x_perm);
    return launch_status();
}
