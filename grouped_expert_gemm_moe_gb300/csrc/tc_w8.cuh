// tc_w8.cuh -- pieces shared by the int8 weight-only tcgen05 kernels that
// read their raw weight rows one thread per row: the 64-byte-swizzled TMA
// layout of a raw tile and the widening of one row into the 128-byte-
// swizzled K-major bf16 layout the MMA reads from shared memory.
#pragma once

#include "tc_common.cuh"

namespace moe {

// int8 tensor maps with the 64-byte swizzle (box rows of 64 bytes: the
// 16-byte unit u of box row r lands at unit u ^ ((r >> 1) & 3), so 8 threads
// reading unit u of 8 consecutive rows hit 8 distinct bank groups).
// three_d: the gate/up weights [G, 2, I, K] as {K, I, G2 = 2G}, box
// {64, box_rows, 2} (box_rows gate rows, then the matching up rows);
// else [I rows, K] as {K, I}, box {64, box_rows}.
inline bool encode_u8_sw64(CUtensorMap *map, const void *base, uint64_t K, uint64_t I,
                           uint64_t G2, bool three_d, uint32_t box_rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {K, I, G2};
    const cuuint64_t strides[2] = {K, I * K};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(TC_BK), box_rows, 2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, three_d ? 3 : 2, const_cast<void *>(base), dims,
               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row `row` (64 int8, k order) of a raw tile written by a 64-byte-swizzled
// TMA box; `tile` 512-byte aligned.
__device__ __forceinline__ void load_raw_row_sw64(const uint8_t *tile, int row, uint4 (&v)[4]) {
    const uint8_t *r = tile + row * TC_BK;
    const int sw = (row >> 1) & 3;
#pragma unroll
    for (int p = 0; p < 4; ++p) v[p] = *reinterpret_cast<const uint4 *>(r + ((p ^ sw) << 4));
}

// 0, computed from every loaded value: a shared-memory load is only known to
// have read its bytes once an instruction has used the result, so a thread
// that releases a raw stage right after loading it first makes the release
// depend on this (e.g. as an offset of the barrier address).  Without it the
// stage may be overwritten by the next copy while the loads are still queued.
template <int N>
__device__ __forceinline__ uint32_t loads_done(const uint4 (&v)[N]) {
    uint32_t d = 0;
#pragma unroll
    for (int p = 0; p < N; ++p) d ^= v[p].x ^ v[p].y ^ v[p].z ^ v[p].w;
    asm volatile("and.b32 %0, %0, 0;" : "+r"(d)::"memory");
    return d;
}

// Widen one row of 64 int8 to bf16 (exact) into the 128-byte-swizzled
// K-major layout: 16-byte unit u of row r at unit u ^ (r & 7); `a` 1024-byte
// aligned.
__device__ __forceinline__ void store_row_sw128(uint8_t *a, int row, const uint4 (&v)[4]) {
    uint8_t *r = a + row * 128;
    const int sw = row & 7;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        uint4 lo, hi;
        widen16(v[p], lo, hi);
        *reinterpret_cast<uint4 *>(r + (((2 * p) ^ sw) << 4)) = lo;
        *reinterpret_cast<uint4 *>(r + (((2 * p + 1) ^ sw) << 4)) = hi;
    }
}

}  // namespace moe
