// tc_common.cuh -- pieces shared by the tcgen05 grouped GEMM kernels:
// tile geometry, the per-expert tile scheduler and TMA tensor-map encoding.
#pragma once

#include <cudaTypedefs.h>

#include "common.cuh"

namespace moe {

constexpr int TC_BM = 128;        // token rows per tile (MMA M)
constexpr int TC_BK = 64;         // K per stage: one 128-byte swizzle row of bf16
constexpr int TC_THREADS = 192;   // 6 warps

struct TileInfo {
    int g, nt, m0, nrows;
};

// s_tile[g] = first linear tile of group g (s_tile[G] = total); a group's
// rows are cut into blocks of rows_per_tile, the block index running fastest.
__device__ __forceinline__ TileInfo decode_tile(int t, const int *s_tile, const int *s_off, int G,
                                                int rows_per_tile = TC_BM) {
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
    const int mt_count = (rows + rows_per_tile - 1) / rows_per_tile;
    ti.nt = u / mt_count;
    const int mt = u - ti.nt * mt_count;
    ti.m0 = s_off[lo] + mt * rows_per_tile;
    ti.nrows = min(rows_per_tile, rows - mt * rows_per_tile);
    return ti;
}

__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// Two int8 in bits 0-7 and 16-23 of `spread` -> bf16x2, exactly.  With b
// the byte and m = b & 0x7F, the bf16 bit pattern 0x4300 | m is 128 + m and
// 0x4300 | (b & 0x80) is 128 (b >= 0) or 256 (b < 0), so their difference is
// the two's-complement value of b; it is an integer below 256 in magnitude,
// which bf16 holds exactly, so the rounded subtraction is exact.
__device__ __forceinline__ uint32_t s8x2_to_bf16x2(uint32_t spread) {
    const uint32_t val = (spread & 0x007F007Fu) | 0x43004300u;
    const uint32_t sub = (spread & 0x00800080u) | 0x43004300u;
    uint32_t r;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(val), "r"(sub));
    return r;
}

// 16 int8 -> 16 bf16 (two 16-byte chunks), exactly, in K order.
__device__ __forceinline__ void widen16(const uint4 v, uint4 &lo, uint4 &hi) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        o[2 * i] = s8x2_to_bf16x2(__byte_perm(w[i], 0u, 0x4140));       // bytes 0, 1
        o[2 * i + 1] = s8x2_to_bf16x2(__byte_perm(w[i], 0u, 0x4342));   // bytes 2, 3
    }
    lo = make_uint4(o[0], o[1], o[2], o[3]);
    hi = make_uint4(o[4], o[5], o[6], o[7]);
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// The int8 converters work in W8_GROUPS independent groups of
// W8_GROUP_THREADS threads (the token-row kernel of gemm_tc_w8.cu uses its
// own group count); group c widens the k-steps c, c + W8_GROUPS, ...
// of the CTA's sequence, so that several stages are converted at once and
// the conversion latency (shared-memory round trips, the proxy fence, the
// barrier hand-off) overlaps instead of adding up stage after stage.
constexpr int W8_GROUPS = 4;
constexpr int W8_GROUP_THREADS = 64;

// One raw int8 stage (ROWS rows x 64 bytes, row-major, as TMA left it) ->
// bf16 in the 128-byte-swizzled K-major layout (16-byte unit u of row r at
// unit u ^ (r & 7)).  gt: this thread's index in its converter group.
template <int ROWS>
__device__ __forceinline__ void widen_stage(const uint8_t *q, uint8_t *a, int gt) {
#pragma unroll 4
    for (int p = 0; p < (ROWS * 4) / W8_GROUP_THREADS; ++p) {
        const int chunk = gt + p * W8_GROUP_THREADS;              // 16 int8 each
        const int row = chunk >> 2, part = chunk & 3;
        const uint4 v = *reinterpret_cast<const uint4 *>(q + row * TC_BK + part * 16);
        uint4 lo, hi;
        widen16(v, lo, hi);
        uint8_t *arow = a + row * 128;
        const int sw = row & 7;
        *reinterpret_cast<uint4 *>(arow + (((2 * part) ^ sw) << 4)) = lo;
        *reinterpret_cast<uint4 *>(arow + (((2 * part + 1) ^ sw) << 4)) = hi;
    }
}

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

// The gate/up weights [G, 2, I, K] bf16 (rows 0..I-1 gate, I..2I-1 up of
// each group) as a 3-D tensor {K, I, 2G}: one box [2][rows][64] brings the
// gate rows and the matching up rows of a tile in a single copy, laid out
// as two 2-D boxes would be (gate rows, then up rows), 128-byte swizzle.
// int8 = true: the same for int8 weights (64-byte rows, no swizzle).
inline bool encode_gate_up_3d(CUtensorMap *map, const void *base, uint64_t K, uint64_t I,
                              uint64_t G, uint32_t rows, bool int8 = false) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const uint64_t esz = int8 ? 1 : 2;
    const cuuint64_t dims[3] = {K, I, 2 * G};
    const cuuint64_t strides[2] = {K * esz, I * K * esz};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(TC_BK), rows, 2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, int8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
               const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               int8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Two 64-element k-blocks per copy.  A bf16 matrix [rows, K] (K a multiple
// of 128) viewed as {64, rows, K/64}: the box {64, box_rows, 2} lands in
// shared memory as two 128-byte-swizzled [box_rows][64] tiles, k-block by
// k-block.  With gate_up: the [G, 2, I, K] gate/up weights viewed as {64, I,
// 2G, K/64}, box {64, box_rows, 2, 2}: per k-block the gate rows then the up
// rows.  (K % 128 != 0 would make the last k-block wrap into the next row.)
inline bool encode_kpair(CUtensorMap *map, const void *base, uint64_t K, uint64_t rows,
                         uint32_t box_rows) {
    auto enc = tensor_map_encoder();
    if (!enc || K % 128 != 0) return false;
    const cuuint64_t dims[3] = {64, rows, K / 64};
    const cuuint64_t strides[2] = {K * 2, 128};
    const cuuint32_t box[3] = {64, box_rows, 2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
inline bool encode_gate_up_kpair(CUtensorMap *map, const void *base, uint64_t K, uint64_t I,
                                 uint64_t G, uint32_t box_rows) {
    auto enc = tensor_map_encoder();
    if (!enc || K % 128 != 0) return false;
    const cuuint64_t dims[4] = {64, I, 2 * G, K / 64};
    const cuuint64_t strides[3] = {K * 2, I * K * 2, 128};
    const cuuint32_t box[4] = {64, box_rows, 2, 2};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides,
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

// Tile shape of each grouped GEMM call (gemm_tc.cu picks one; the values
// are moe_tile's, include/moe.h).
int pick_tile(int M, int G);
int pick_tile_w8(int M, int G);

// int8 weights, 256 weight rows x TN (16, 32 or 64) token rows (gemm_tc_dec_w8.cu).
template <bool SWIGLU>
moe_status launch_dec_w8(int tn, const void *tok, const void *q, const float *scales,
                         const int32_t *offsets, int G, int M, int K, int R, int NOUT, int UP_OFF,
                         uint16_t *out, int32_t *dev_error, cudaStream_t stream);

// int8 weights on CTA pairs: 256 weight rows (widened into TMEM) x up to
// 192 tokens (gemm_tc_pair_w8.cu).  K % 64 == 0, else MOE_ERR_UNSUPPORTED.
template <bool SWIGLU>
moe_status launch_tc_pair_w8(const void *act, const int8_t *q, const float *scales,
                             const int32_t *offsets, int G, int M, int K, int R, int NOUT,
                             int UP_OFF, uint16_t *out, int32_t *dev_error, cudaStream_t stream);

// 256 weight rows x up to 256 tokens on CTA pairs (gemm_tc_pair.cu).
template <bool SWIGLU>
moe_status launch_tc_pair(const void *act, const void *w, const int32_t *offsets, int G, int M,
                          int K, int R, int NOUT, int UP_OFF, uint16_t *out, int32_t *dev_error,
                          cudaStream_t stream);

moe_status check_ffn_args(const void *x_perm, const int32_t *offsets, int G, int M, int H, int I,
                          const void *w_gu, const void *w_down, const void *y_perm,
                          const void *workspace, size_t workspace_bytes, int k_align);

}  // namespace moe
