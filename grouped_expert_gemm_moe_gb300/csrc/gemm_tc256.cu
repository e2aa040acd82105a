// gemm_tc256.cu -- prefill form of the tcgen05 grouped GEMM: 256-row token blocks.
//
// Same layer, same per-expert scheduling idea as gemm_tc.cu, shaped for
// batches with hundreds of rows per expert.  A tile is a block of up to 256
// token rows of one group times 256 weight rows: per K step the MMA warp
// issues two M=128, N=256 MMAs, one per 128-row half of the block, that
// share the weight tile in shared memory.  Operand bytes per FLOP drop by a
// third against 128 x 256 tiles (64 KB staged per 2 x 128 x 256 x 64 MMA
// work instead of 48 KB per half of it), which is what limits the single-
// tile kernel at prefill sizes.  The two accumulators take all 512 TMEM
// columns, so a tile's epilogue is not overlapped with the next tile's MMAs;
// eight epilogue warps (two per TMEM lane quarter, one per half) keep that
// gap short.
//
// Scheduling: tiles are (group, n-tile, 256-row block), block fastest,
// dealt round robin to the persistent CTAs, so CTAs running at the same
// time work on neighbouring tiles and share weight and activation tiles
// through L2.  A block with at most 128 rows (a group's tail) issues one MMA
// per K step.
#include <stdlib.h>

#include "tc_common.cuh"

namespace moe {

constexpr int P_BN = 256;
constexpr int P_STAGES = 3;
constexpr int P_EPI_WARPS = 8;
constexpr int P_THREADS = (2 + P_EPI_WARPS) * 32;

struct PCfg {
    static constexpr int A_BYTES = TC_BM * TC_BK * 2;           // one 128-row half
    static constexpr int B_BYTES = P_BN * TC_BK * 2;
    static constexpr int STAGE_BYTES = 2 * A_BYTES + B_BYTES;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr int BAR_BYTES = 256;
    static size_t smem_bytes(int G) {
        return 1024 + static_cast<size_t>(P_STAGES) * STAGE_BYTES + BAR_BYTES +
               2 * static_cast<size_t>(G + 1) * sizeof(int);
    }
};

struct PTile {
    int g, nt, m0, rows;
    bool two;                   // second 128-row half present
};

// s_tile[g] = first tile of group g; group g has n_tiles * ceil(rows_g / 256) tiles.
__device__ __forceinline__ PTile p_decode(int t, const int *s_tile, const int *s_off, int G) {
    int lo = 0, hi = G - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_tile[mid] <= t) lo = mid;
        else hi = mid - 1;
    }
    PTile ti;
    ti.g = lo;
    const int u = t - s_tile[lo];
    const int rows = s_off[lo + 1] - s_off[lo];
    const int nb = (rows + 255) / 256;
    ti.nt = u / nb;
    const int b = u - ti.nt * nb;
    ti.m0 = s_off[lo] + b * 256;
    ti.rows = min(256, rows - b * 256);
    ti.two = ti.rows > TC_BM;
    return ti;
}

// SWIGLU: out = h [M, NOUT=I], weights [G*2I, K=H], up rows at +UP_OFF = I.
// PLAIN : out = y [M, NOUT=H], weights [G*H,  K=I].
template <bool SWIGLU>
__global__ void __launch_bounds__(P_THREADS, 1)
    tc_grouped_gemm_256(const __grid_constant__ CUtensorMap tm_act,
                        const __grid_constant__ CUtensorMap tm_act128,
                        const __grid_constant__ CUtensorMap tm_w,
                        const __grid_constant__ CUtensorMap tm_act32,
                        const __grid_constant__ CUtensorMap tm_act64,
                        const __grid_constant__ CUtensorMap tm_act256,
                        const int32_t *__restrict__ offsets, int G, int M, int K, int R,
                        int NOUT, int UP_OFF, uint16_t *__restrict__ out, int32_t *dev_error) {
    using C = PCfg;
    constexpr int S = P_STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *stage0 = smem;                                  // [S][A1 | A2 | B]
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + S * C::STAGE_BYTES);
    uint64_t *empty = full + S;
    uint64_t *accf = empty + S;
    uint64_t *acce = accf + 1;
    uint64_t *drain = acce + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    int *s_total = reinterpret_cast<int *>(tmem_slot + 1);
    int *s_off = reinterpret_cast<int *>(reinterpret_cast<uint8_t *>(full) + C::BAR_BYTES);
    int *s_tile = s_off + (G + 1);

    const int warp = threadIdx.x >> 5, lane = lane_id();
    const int n_per_tile = SWIGLU ? P_BN / 2 : P_BN;
    const int n_tiles = (NOUT + n_per_tile - 1) / n_per_tile;
    const int KB = (K + TC_BK - 1) / TC_BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(accf, 1);
        mbar_init(acce, P_EPI_WARPS * 32);
        mbar_init(drain, 1);
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tm_act);
        prefetch_tmap(&tm_act32);
        prefetch_tmap(&tm_act64);
        prefetch_tmap(&tm_act128);
        prefetch_tmap(&tm_act256);
        prefetch_tmap(&tm_w);
    }
    if (warp == 1) tmem_alloc<C::TMEM_COLS>(tmem_slot);
    pdl_wait();
    pdl_trigger();
    if (warp == 2) build_tile_table(offsets, G, M, n_tiles, s_off, s_tile, s_total, dev_error, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int total = *s_total;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_a = policy_evict_last();
            int stage = 0;
            uint32_t phase = 0, filled = 0, fill_parity = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const PTile ti = p_decode(t, s_tile, s_off, G);
                // the block's token rows as one box of 16 .. 256 rows (the two
                // 128-row halves are contiguous in the stage), the smallest
                // that holds them; rows past the group are loaded, never stored
                const int abox = ti.rows <= 16 ? 16 : ti.rows <= 32 ? 32 : ti.rows <= 64 ? 64
                                 : ti.rows <= 128 ? 128 : 256;
                const CUtensorMap *tm_a = abox == 16 ? &tm_act : abox == 32 ? &tm_act32
                                        : abox == 64 ? &tm_act64 : abox == 128 ? &tm_act128
                                                                              : &tm_act256;
                const uint32_t bytes = abox * 128 + C::B_BYTES;
                const int wrow = ti.g * R + ti.nt * n_per_tile;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, dev_error)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[stage], bytes);
                    uint8_t *a1 = stage0 + stage * C::STAGE_BYTES;
                    uint8_t *a2 = a1 + C::A_BYTES;
                    uint8_t *b = a2 + C::A_BYTES;
                    const int kx = kb * TC_BK;
                    (void)a2;
                    tma_load_2d(a1, tm_a, &full[stage], kx, ti.m0, pol_a);
                    if (SWIGLU) {          // gate rows and up rows in one 3-D copy
                        tma_load_3d(b, &tm_w, &full[stage], kx, ti.nt * n_per_tile, 2 * ti.g,
                                    pol_w);
                    } else {
                        tma_load_2d(b, &tm_w, &full[stage], kx, wrow, pol_w);
                    }
                    filled |= 1u << stage;
                    fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            for (int s = 0; s < S; ++s)
                if ((filled >> s) & 1u) mbar_wait(&full[s], (fill_parity >> s) & 1u, dev_error);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(TC_BM, P_BN);
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const PTile ti = p_decode(t, s_tile, s_off, G);
                if (!mbar_wait(acce, acc_phase ^ 1u, dev_error)) break;
                tc_fence_after();
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&full[stage], phase, dev_error)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a1 = smem_u32(stage0 + stage * C::STAGE_BYTES);
                    const uint32_t a2 = a1 + C::A_BYTES;
                    const uint32_t b = a2 + C::A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < TC_BK / 16; ++kk) {
                        const uint64_t bd = sw128_kmajor_desc(b + kk * 32);
                        const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
                        tc_mma_bf16(tmem_base, sw128_kmajor_desc(a1 + kk * 32), bd, idesc, acc);
                        if (ti.two)
                            tc_mma_bf16(tmem_base + P_BN, sw128_kmajor_desc(a2 + kk * 32), bd,
                                        idesc, acc);
                    }
                    tc_commit(&empty[stage]);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit(accf);
                acc_phase ^= 1u;
            }
            tc_commit(drain);
            mbar_wait(drain, 0, dev_error);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue (warps 2..9)
        const int e = warp - 2;
        const int half = e >> 2;                // which 128-row half (accumulator)
        const int quarter = warp & 3;           // TMEM lanes this warp may access
        const int row_in_tile = half * TC_BM + quarter * 32 + lane;
        uint32_t acc_phase = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x) {
            const PTile ti = p_decode(t, s_tile, s_off, G);
            if (!mbar_wait_warp(accf, acc_phase, dev_error)) break;
            tc_fence_after();
            if (half == 0 || ti.two) {
                const bool valid = row_in_tile < ti.rows;
                uint16_t *orow = out + static_cast<int64_t>(ti.m0 + row_in_tile) * NOUT;
                const uint32_t tbase =
                    tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + half * P_BN;
                const int n0 = ti.nt * n_per_tile;
                if (SWIGLU) {
#pragma unroll 1
                    for (int c = 0; c < P_BN / 2; c += 16) {
                        uint32_t g[16], u[16];
                        tmem_ld16(tbase + c, g);
                        tmem_ld16(tbase + P_BN / 2 + c, u);
                        tmem_ld_wait();
                        if (valid && n0 + c < NOUT) {
                            uint32_t p[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const float h0 = silu_fast(__uint_as_float(g[2 * i])) *
                                                 __uint_as_float(u[2 * i]);
                                const float h1 = silu_fast(__uint_as_float(g[2 * i + 1])) *
                                                 __uint_as_float(u[2 * i + 1]);
                                p[i] = pack_bf16x2(h0, h1);
                            }
                            uint4 *dst = reinterpret_cast<uint4 *>(orow + n0 + c);
                            dst[0] = make_uint4(p[0], p[1], p[2], p[3]);
                            if (n0 + c + 8 < NOUT) dst[1] = make_uint4(p[4], p[5], p[6], p[7]);
                        }
                    }
                } else {
#pragma unroll 1
                    for (int c = 0; c < P_BN; c += 16) {
                        uint32_t v[16];
                        tmem_ld16(tbase + c, v);
                        tmem_ld_wait();
                        if (valid && n0 + c < NOUT) {
                            uint32_t p[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                p[i] = pack_bf16x2(__uint_as_float(v[2 * i]),
                                                   __uint_as_float(v[2 * i + 1]));
                            uint4 *dst = reinterpret_cast<uint4 *>(orow + n0 + c);
                            dst[0] = make_uint4(p[0], p[1], p[2], p[3]);
                            if (n0 + c + 8 < NOUT) dst[1] = make_uint4(p[4], p[5], p[6], p[7]);
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(acce);
            acc_phase ^= 1u;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<C::TMEM_COLS>(tmem_base);
    }
}

template <bool SWIGLU>
moe_status launch_tc256(const void *act, const void *w, const int32_t *offsets, int G, int M,
                        int K, int R, int NOUT, int UP_OFF, uint16_t *out, int32_t *dev_error,
                        cudaStream_t stream) {
    CUtensorMap tm_act, tm_act32, tm_act64, tm_act128, tm_act256, tm_w;
    if (!encode_bf16_2d(&tm_act, act, K, M, 16) || !encode_bf16_2d(&tm_act32, act, K, M, 32) ||
        !encode_bf16_2d(&tm_act64, act, K, M, 64) || !encode_bf16_2d(&tm_act128, act, K, M, 128) ||
        !encode_bf16_2d(&tm_act256, act, K, M, 256))
        return MOE_ERR_CUDA;
    if (SWIGLU ? !encode_gate_up_3d(&tm_w, w, K, UP_OFF, G, P_BN / 2)
               : !encode_bf16_2d(&tm_w, w, K, static_cast<uint64_t>(G) * R, P_BN))
        return MOE_ERR_CUDA;
    const size_t smem = PCfg::smem_bytes(G);
    if (smem > static_cast<size_t>(max_smem_optin())) return MOE_ERR_UNSUPPORTED;
    static int attr_done[64] = {0};
    if (!raise_smem_limit(tc_grouped_gemm_256<SWIGLU>, attr_done)) return MOE_ERR_CUDA;
    launch(tc_grouped_gemm_256<SWIGLU>, sm_count(), P_THREADS, smem, stream, tm_act, tm_act128,
           tm_w, tm_act32, tm_act64, tm_act256, offsets, G, M, K, R, NOUT, UP_OFF, out, dev_error);
    return launch_status();
}

template moe_status launch_tc256<true>(const void *, const void *, const int32_t *, int, int, int,
                                       int, int, int, uint16_t *, int32_t *, cudaStream_t);
template moe_status launch_tc256<false>(const void *, const void *, const int32_t *, int, int, int,
                                        int, int, int, uint16_t *, int32_t *, cudaStream_t);

}  // namespace moe
