// tc_common.cuh -- pieces shared by the tcgen05 grouped GEMM kernels:
// tile geometry, the per-expert tile scheduler and TMA tensor-map encoding.
#pragma once

#include <cudaTypedefs.h>

#include "common.cuh"

namespace moe {

constexpr int TC_BM = 128;        // token rows per tile (MMA M)
constexpr int TC_BK = 64;         // K per stage: one 128-byte swizzle row of bf16
constexpr int TC_THREADS = 192;   // 6 warps
constexpr int TC_ABOX = 16;       // rows per activation TMA box

struct TileInfo {
    int g, nt, m0, nrows;
};

// s_tile[g] = first linear tile of group g (s_tile[G] = total).
__device__ __forceinline__ TileInfo decode_tile(int t, const int *s_tile, const int *s_off, int G) {
    int lo = 0, hi = G - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_tile[mid] <= t) lo = mid;
        else hi = mid - 1;
    }
    TileInfo ti;
    ti.g = lo;
    const int u = t - s_tile[lo];
    const int rows = s_off[lo + 1] - s_off[lo];
    const int mt_count = (rows + TC_BM - 1) / TC_BM;
    ti.nt = u / mt_count;
    const int mt = u - ti.nt * mt_count;
    ti.m0 = s_off[lo] + mt * TC_BM;
    ti.nrows = min(TC_BM, rows - mt * TC_BM);
    return ti;
}

__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// The per-expert tile table, built by one warp at kernel start from the
// offsets table: group g owns n_tiles * ceil(rows_g / rows_per_tile) tiles starting at
// s_tile[g]; s_off mirrors the offsets.  Offsets that are negative, not
// monotone or beyond M make the whole launch a no-op with a device-check fault.
__device__ __forceinline__ void build_tile_table(const int32_t *offsets, int G, int M, int n_tiles,
                                                 int *s_off, int *s_tile, int *s_total,
                                                 int32_t *dev_error, int rows_per_tile = TC_BM) {
    const int lane = lane_id();
    int carry = 0;
    bool bad = false;
    for (int base = 0; base < G; base += 32) {
        const int g = base + lane;
        int tiles = 0;
        if (g < G) {
            const int o0 = offsets[g], o1 = offsets[g + 1];
            if (o0 < 0 || o1 < o0 || o1 > M) bad = true;
            else tiles = ((o1 - o0 + rows_per_tile - 1) / rows_per_tile) * n_tiles;
            s_off[g] = o0;
            if (g == G - 1) s_off[G] = o1;
        }
        const int inc = warp_inclusive_scan(tiles);
        if (g < G) s_tile[g] = carry + inc - tiles;
        carry += __shfl_sync(FULL, inc, 31);
    }
    bad = __any_sync(FULL, bad);
    if (lane == 0) {
        s_tile[G] = carry;
        *s_total = bad ? 0 : carry;
        if (bad) report(dev_error, MOE_ERR_DEVICE_CHECK);
    }
}

// ------------------------------------------------------------------ host

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2-D bf16 tensor [outer, inner] row-major, box [box_outer, 64], 128-byte swizzle.
inline bool encode_bf16_2d(CUtensorMap *map, const void *base, uint64_t inner, uint64_t outer,
                           uint32_t box_outer) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {inner * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(TC_BK), box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D uint8 tensor [outer, inner] row-major, box [box_outer, 64 bytes], no swizzle.
inline bool encode_u8_2d(CUtensorMap *map, const void *base, uint64_t inner, uint64_t outer,
                         uint32_t box_outer) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {inner};
    const cuuint32_t box[2] = {64u, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Raise a kernel's dynamic shared-memory limit to the device maximum once per
// device (not on every call, so that launches can be captured into graphs).
template <typename Kernel>
inline bool raise_smem_limit(Kernel kernel, int *done_per_device) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    if (!done_per_device[dev]) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 max_smem_optin()) != cudaSuccess)
            return false;
        done_per_device[dev] = 1;
    }
    return true;
}

moe_status check_ffn_args(const void *x_perm, const int32_t *offsets, int G, int M, int H, int I,
                          const void *w_gu, const void *w_down, const void *y_perm,
                          const void *workspace, size_t workspace_bytes, int k_align);

}  // namespace moe
