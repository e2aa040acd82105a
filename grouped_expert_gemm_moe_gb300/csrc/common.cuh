// common.cuh -- shared device helpers of libmoe.so (sm_103a only).
//
// Small wrappers over the PTX this library issues directly (mbarrier, TMA
// bulk tensor copies, tcgen05 MMA / TMEM), bf16 packing, warp scans and the
// host-side argument checks every entry point uses.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "moe.h"

namespace moe {

// ------------------------------------------------------------------ host side

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// number of SMs of the current device (cached per device id)
int sm_count();

// max dynamic shared memory per block (opt-in) of the current device
int max_smem_optin();

inline moe_status launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Launch with programmatic dependent launch (PDL) allowed: the kernel may
// be scheduled while the previous kernel on the stream is finishing; every
// kernel of this library calls pdl_wait() before it touches global memory,
// so the overlap only hides launch latency and prologues.  Setting the
// environment variable MOE_DISABLE_PDL=1 launches without the attribute.
bool pdl_enabled();

template <typename... KArgs, typename... Args>
inline cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(std::forward<Args>(args))...);
}

// ---------------------------------------------------------------- device side

// Wait until the grids this one depends on have completed and their writes
// are visible (a no-op when launched without PDL).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next kernel on the stream to be scheduled (it still waits for
// this grid's completion in its own pdl_wait()).
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

constexpr unsigned FULL = 0xffffffffu;

// A bounded wait gives up after this long (ns of %globaltimer) or this many
// polls, whichever comes first, and reports MOE_ERR_TIMEOUT.
constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;   // 1 s
constexpr uint32_t WAIT_LIMIT_POLLS = 1u << 28;

__device__ __forceinline__ void report(int32_t *dev_error, int code) {
    if (dev_error) *reinterpret_cast<volatile int32_t *>(dev_error) = code;
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ int lane_id() { return threadIdx.x & 31; }

template <typename T>
__device__ __forceinline__ T warp_inclusive_scan(T v) {
    const int lane = lane_id();
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        T o = __shfl_up_sync(FULL, v, d);
        if (lane >= d) v += o;
    }
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(FULL, v, d);
    return v;
}

// ---- bf16 <-> fp32 (a bf16 is the top half of an fp32, so widening is a shift)
__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 r = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&r);
}

// ---- int8 -> fp32, exact: place the biased byte in the mantissa of 2^23
// (0x4B000000 | (b + 128)) and subtract 2^23 + 128.
__device__ __forceinline__ float s8_to_f32(uint32_t word_biased, int byte_idx) {
    uint32_t bits = __byte_perm(word_biased, 0x4B000000u, 0x7540u + byte_idx);
    return __uint_as_float(bits) - 8388736.0f;
}
__device__ __forceinline__ uint32_t bias_s8x4(uint32_t w) { return w ^ 0x80808080u; }

// ---- loads
// read-once data: no L1 allocation, L2 line marked by `policy` (evict-first
// for weight streams, so they do not push out what is wanted again)
__device__ __forceinline__ uint4 ld_stream(const void *p, uint64_t policy) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p), "l"(policy));
    return r;
}
// coherent at GPU scope (L2, not L1): for data other CTAs of the same
// launch wrote before a grid-wide barrier
__device__ __forceinline__ uint4 ld_cg(const void *p) {
    uint4 r;
    asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}
__device__ __forceinline__ uint4 ld_nc(const void *p) {       // read-only, cached
    return __ldg(reinterpret_cast<const uint4 *>(p));
}

// ------------------------------------------------------------- mbarrier / TMA

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait until the phase of `bar` with the given parity has completed.  The
// wait is bounded: on running out it reports MOE_ERR_TIMEOUT and returns false.
// (The limit is an argument only so that moe_selftest_bounded_wait can run
// this very code with a short one; kernels use the default.)
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, int32_t *dev_error,
                                          uint64_t limit_ns = WAIT_LIMIT_NS) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t polls = 1;; ++polls) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((polls & 255u) == 0 &&
            (globaltimer() - t0 > limit_ns || polls >= WAIT_LIMIT_POLLS)) {
            report(dev_error, MOE_ERR_TIMEOUT);
            return false;
        }
    }
}

// The same wait with one outcome for the whole warp (every lane calls it):
// the warp-collective tcgen05.ld / tcgen05.st after it need every lane, even
// when the time limit runs out in some lanes only.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t *bar, uint32_t parity,
                                               int32_t *dev_error,
                                               uint64_t limit_ns = WAIT_LIMIT_NS) {
    return __all_sync(FULL, mbar_wait(bar, parity, dev_error, limit_ns));
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Grid-wide barrier of a launch whose CTAs are all resident (a cooperative
// launch): every CTA adds one to *count and waits until it reaches `target`
// (the caller zeroes the word before the launch and raises the target by
// gridDim.x per barrier).  Writes before the barrier are visible to every CTA
// after it.  The wait is bounded: on running out thread 0 reports
// MOE_ERR_TIMEOUT and sets *fail (a shared word the CTA initialised to 0),
// and every thread of the CTA gets false.
__device__ __forceinline__ bool grid_barrier(unsigned *count, unsigned target, int *fail,
                                             int32_t *dev_error,
                                             uint64_t limit_ns = WAIT_LIMIT_NS) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(count, 1u);
        const uint64_t t0 = globaltimer();
        for (uint32_t polls = 0;; ++polls) {
            if (ld_acquire_gpu(count) >= target) break;
            if ((polls & 63u) == 63u && globaltimer() - t0 > limit_ns) {
                report(dev_error, MOE_ERR_TIMEOUT);
                *reinterpret_cast<volatile int *>(fail) = 1;
                break;
            }
        }
        __threadfence();
    }
    __syncthreads();
    return *reinterpret_cast<volatile int *>(fail) == 0;
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 3-D tiled TMA load global -> shared (box [z][y][x], x innermost).
__device__ __forceinline__ void tma_load_3d(void *smem_dst, const CUtensorMap *map, uint64_t *bar,
                                            int x, int y, int z, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)),
        "l"(policy)
        : "memory");
}

// 4-D tiled TMA load global -> shared (box [w][z][y][x], x innermost).
__device__ __forceinline__ void tma_load_4d(void *smem_dst, const CUtensorMap *map, uint64_t *bar,
                                            int x, int y, int z, int w, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w),
        "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// 2-D tiled TMA load global -> shared, completion counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int x, int y, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// ---------------------------------------------------------------- tcgen05

template <uint32_t NCOLS>
__device__ __forceinline__ void tmem_alloc(uint32_t *slot) {   // whole warp
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(slot)),
                 "n"(NCOLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

template <uint32_t NCOLS>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr) {   // whole warp
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "n"(NCOLS)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every MMA this thread issued so far has completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns: thread i gets lane (base + i).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major bf16 tile stored with the
// 128-byte swizzle: rows of 64 elements (128 B), 8-row groups 1024 B apart.
// `addr` is the shared address of the first element of the slice; the tile
// base must be 1024-byte aligned.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t addr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);     // start address
    d |= static_cast<uint64_t>(1) << 16;                    // leading byte offset (unused)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;            // stride byte offset
    d |= static_cast<uint64_t>(1) << 46;                    // descriptor version
    d |= static_cast<uint64_t>(2) << 61;                    // 128-byte swizzle
    return d;
}

// Instruction descriptor: bf16 x bf16 -> fp32, both operands K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4)                                        // D fp32
           | (1u << 7)                                      // A bf16
           | (1u << 10)                                     // B bf16
           | (static_cast<uint32_t>(N >> 3) << 17)          // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);         // M / 16
}

}  // namespace moe
