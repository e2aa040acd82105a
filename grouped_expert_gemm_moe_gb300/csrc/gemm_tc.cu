// gemm_tc.cu -- all-experts grouped GEMM on the 5th-generation tensor cores.
//
// One launch covers every expert, with the SwiGLU activation applied in the
// GEMM's epilogue, as the "switchyard" page (02 Kernels and dispatch, "One
// launch for all experts") describes for its tensor-core kernel.  Written
// for sm_103a:
//
//  * persistent grid, one CTA per SM; a per-expert tile scheduler walks the
//    linear tile index over (group g, n-tile, m-tile) with the m-tile
//    fastest, so CTAs that run at the same time read the same weight tile
//    (one HBM read, the rest L2 hits).  The tile table is built on the
//    device from the offsets table: the host never learns the group sizes;
//  * warp 0: TMA producer (one thread) filling a ring of STAGES shared
//    memory stages with two copies each: the activation tile (token rows,
//    K-major, 128-byte swizzle, one box of 16/32/64/128 rows, the smallest
//    that holds the tile's rows) and the weight tile (SwiGLU: the gate rows
//    and the matching up rows in one 3-D box).  Copies per stage are the
//    ring's cost here, not bytes: on GB300 a third copy per stage cost 4-6 %;
//  * warp 1: TMEM allocator and MMA issuer (one thread): tcgen05.mma
//    kind::f16, M = 128 token rows, N = BN weight rows, K = 16 per
//    instruction, fp32 accumulators in TMEM, double-buffered (2 x BN
//    columns) so the epilogue of one tile overlaps the main loop of the next;
//  * warps 2-5: epilogue.  tcgen05.ld moves a thread's accumulator row into
//    registers; SWIGLU mode holds gate rows n0..n0+BN/2-1 in accumulator
//    columns [0, BN/2) and the matching up rows in [BN/2, BN), so
//    h = silu(gate) * up is formed in registers and stored as bf16; PLAIN
//    mode stores the accumulator as bf16.
// Every mbarrier wait is bounded (1 s); on running out the kernel records
// MOE_ERR_TIMEOUT, drains its own copies and MMAs, frees TMEM and returns.
#include <stdlib.h>
#include <string.h>

#include <algorithm>

#include <atomic>

#include "tc_common.cuh"

namespace moe {

template <int BN>
struct TcCfg {
    static constexpr int A_BYTES = TC_BM * TC_BK * 2;
    static constexpr int B_BYTES = BN * TC_BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = (192 * 1024) / STAGE_BYTES;
    static constexpr uint32_t TMEM_COLS = 2 * BN;
    static constexpr int BAR_BYTES = 256;
    static size_t smem_bytes(int G) {
        return 1024 + static_cast<size_t>(STAGES) * STAGE_BYTES + BAR_BYTES +
               2 * static_cast<size_t>(G + 1) * sizeof(int);
    }
};

// SWIGLU: out = h [M, NOUT=I], weights [G*2I, K=H], up rows at +UP_OFF = I.
// PLAIN : out = y [M, NOUT=H], weights [G*H,  K=I].
template <bool SWIGLU, int BN>
__global__ void __launch_bounds__(TC_THREADS, 1)
    tc_grouped_gemm(const __grid_constant__ CUtensorMap tm_act16,
                    const __grid_constant__ CUtensorMap tm_act32,
                    const __grid_constant__ CUtensorMap tm_act64,
                    const __grid_constant__ CUtensorMap tm_act128,
                    const __grid_constant__ CUtensorMap tm_w, const int32_t *__restrict__ offsets,
                    int G, int M, int K, int R, int NOUT, int UP_OFF, uint16_t *__restrict__ out,
                    int32_t *dev_error) {
    using C = TcCfg<BN>;
    constexpr int STAGES = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * C::A_BYTES;
    uint64_t *full = reinterpret_cast<uint64_t *>(sB + STAGES * C::B_BYTES);
    uint64_t *empty = full + STAGES;
    uint64_t *accf = empty + STAGES;
    uint64_t *acce = accf + 2;
    uint64_t *drain = acce + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    int *s_total = reinterpret_cast<int *>(tmem_slot + 1);
    int *s_off = reinterpret_cast<int *>(reinterpret_cast<uint8_t *>(full) + C::BAR_BYTES);
    int *s_tile = s_off + (G + 1);

    const int warp = threadIdx.x >> 5, lane = lane_id();
    const int n_per_tile = SWIGLU ? BN / 2 : BN;
    const int n_tiles = (NOUT + n_per_tile - 1) / n_per_tile;
    const int KB = (K + TC_BK - 1) / TC_BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accf[b], 1);
            mbar_init(&acce[b], 128);
        }
        mbar_init(drain, 1);
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tm_act16);
        prefetch_tmap(&tm_act32);
        prefetch_tmap(&tm_act64);
        prefetch_tmap(&tm_act128);
        prefetch_tmap(&tm_w);
    }
    if (warp == 1) tmem_alloc<C::TMEM_COLS>(tmem_slot);
    pdl_wait();       // predecessors' writes (offsets, activations) are visible after this
    pdl_trigger();
    if (warp == 2) build_tile_table(offsets, G, M, n_tiles, s_off, s_tile, s_total, dev_error);
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
            uint32_t phase = 0;
            uint32_t filled = 0, fill_parity = 0;     // per stage: ever filled / parity of last fill
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const TileInfo ti = decode_tile(t, s_tile, s_off, G);
                // the token rows as one box of 16, 32, 64 or 128 rows, the
                // smallest that holds the tile's rows (one copy per stage; rows
                // past the group are loaded but never stored)
                const int abox = ti.nrows <= 16 ? 16 : ti.nrows <= 32 ? 32
                                                     : ti.nrows <= 64 ? 64 : 128;
                const CUtensorMap *tm_a = abox == 16 ? &tm_act16 : abox == 32 ? &tm_act32
                                        : abox == 64 ? &tm_act64 : &tm_act128;
                const uint32_t bytes = abox * TC_BK * 2 + C::B_BYTES;
                const int wrow = ti.g * R + ti.nt * n_per_tile;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, dev_error)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[stage], bytes);
                    uint8_t *a = sA + stage * C::A_BYTES;
                    uint8_t *b = sB + stage * C::B_BYTES;
                    const int kx = kb * TC_BK;
                    tma_load_2d(a, tm_a, &full[stage], kx, ti.m0, pol_a);
                    if (SWIGLU) {          // gate rows and up rows in one 3-D copy
                        tma_load_3d(b, &tm_w, &full[stage], kx, ti.nt * n_per_tile, 2 * ti.g,
                                    pol_w);
                    } else {
                        tma_load_2d(b, &tm_w, &full[stage], kx, wrow, pol_w);
                    }
                    filled |= 1u << stage;
                    fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // drain: every copy this thread issued has landed before exit
            for (int s = 0; s < STAGES; ++s)
                if ((filled >> s) & 1u) mbar_wait(&full[s], (fill_parity >> s) & 1u, dev_error);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(TC_BM, BN);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                if (!mbar_wait(&acce[acc], acc_phase ^ 1u, dev_error)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&full[stage], phase, dev_error)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(sA + stage * C::A_BYTES);
                    const uint32_t b_addr = smem_u32(sB + stage * C::B_BYTES);
#pragma unroll
                    for (int kk = 0; kk < TC_BK / 16; ++kk)
                        tc_mma_bf16(d_tmem, sw128_kmajor_desc(a_addr + kk * 32),
                                    sw128_kmajor_desc(b_addr + kk * 32), idesc,
                                    (kb > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(&empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit(&accf[acc]);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            // drain: every MMA this thread issued has completed before exit
            tc_commit(drain);
            mbar_wait(drain, 0, dev_error);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue (warps 2..5)
        const int quarter = warp & 3;       // TMEM lanes this warp may access
        const int row_in_tile = quarter * 32 + lane;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x) {
            const TileInfo ti = decode_tile(t, s_tile, s_off, G);
            if (!mbar_wait_warp(&accf[acc], acc_phase, dev_error)) break;
            tc_fence_after();
            const bool valid = row_in_tile < ti.nrows;
            uint16_t *orow = out + static_cast<int64_t>(ti.m0 + row_in_tile) * NOUT;
            const uint32_t tbase =
                tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * BN;
            const int n0 = ti.nt * n_per_tile;
            if (SWIGLU) {
#pragma unroll 1
                for (int c = 0; c < BN / 2; c += 16) {
                    uint32_t g[16], u[16];
                    tmem_ld16(tbase + c, g);
                    tmem_ld16(tbase + BN / 2 + c, u);
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
                for (int c = 0; c < BN; c += 16) {
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
            tc_fence_before();
            mbar_arrive(&acce[acc]);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<C::TMEM_COLS>(tmem_base);
    }
}

// ------------------------------------------------------------------ host

template <bool SWIGLU, int BN>
static moe_status launch_tc(const void *act, const void *w, const int32_t *offsets, int G, int M,
                            int K, int R, int NOUT, int UP_OFF, uint16_t *out, int32_t *dev_error,
                            cudaStream_t stream) {
    CUtensorMap tm_act16, tm_act32, tm_act64, tm_act128, tm_w;
    if (!encode_bf16_2d(&tm_act16, act, K, M, 16) || !encode_bf16_2d(&tm_act32, act, K, M, 32) ||
        !encode_bf16_2d(&tm_act64, act, K, M, 64) || !encode_bf16_2d(&tm_act128, act, K, M, TC_BM))
        return MOE_ERR_CUDA;
    if (SWIGLU ? !encode_gate_up_3d(&tm_w, w, K, UP_OFF, G, BN / 2)
               : !encode_bf16_2d(&tm_w, w, K, static_cast<uint64_t>(G) * R, BN))
        return MOE_ERR_CUDA;
    const size_t smem = TcCfg<BN>::smem_bytes(G);
    if (smem > static_cast<size_t>(max_smem_optin())) return MOE_ERR_UNSUPPORTED;
    static int attr_done[64] = {0};
    if (!raise_smem_limit(tc_grouped_gemm<SWIGLU, BN>, attr_done)) return MOE_ERR_CUDA;
    launch(tc_grouped_gemm<SWIGLU, BN>, sm_count(), TC_THREADS, smem, stream, tm_act16, tm_act32,
           tm_act64, tm_act128, tm_w, offsets, G, M, K, R, NOUT, UP_OFF, out, dev_error);
    return launch_status();
}

}  // namespace moe

using namespace moe;

namespace moe {

// Tile override set by moe_set_gemm_tile (MOE_TILE_AUTO: none).
static std::atomic<int> g_forced_tile{MOE_TILE_AUTO};

// Tile shape per call, from the mean rows per group (M / G), chosen from
// GB300 measurements of the OLMoE- and DeepSeek-shaped layers:
//   <= 64 rows : 128 x 128 tiles.
//   <= 128 rows: 128 x 256 tiles.
//   more       : CTA-pair tiles of 256 weight rows x up to 256 tokens
//                (gemm_tc_pair.cu), when K is a multiple of 64 (else 128 x
//                256).
// Two other bf16 tile kernels were measured and are not in the library:
// weight-row tiles (the MMA's M over weight rows, N over a group's tokens),
// equal or slower once every ring stage took one copy per operand, and
// 256-row token blocks, 5-16 % slower than 128 x 256 at 32-1024 rows per
// group (their 512 TMEM columns leave no second accumulator buffer).
int pick_tile(int M, int G) {
    const int f = g_forced_tile.load(std::memory_order_relaxed);
    if (f == MOE_TILE_128x128 || f == MOE_TILE_128x256 || f == MOE_TILE_PAIR) return f;
    const int64_t m = M, g = G;
    return m <= 64 * g ? MOE_TILE_128x128 : m <= 128 * g ? MOE_TILE_128x256 : MOE_TILE_PAIR;
}

// int8 weights, from the mean rows per group (int8 layers on GB300, us per
// layer; 256-row weight tiles of gemm_tc_dec_w8.cu with 16/32/64 tokens, the
// 128-token-row tiles of gemm_tc_w8.cu, the CTA-pair tiles of
// gemm_tc_pair_w8.cu):
//     OLMoE rows/group      1      2      8     16     24     32     64    128    256
//     w8d16              99.3  119.8  123.4  162.7  188.9
//     w8d32             105.0  125.4  127.5  127.9  132.0  173.3
//     w8d64                                                138.4  185.5
//     rows              139.8  170.9  174.6  175.3  179.1  181.4  191.6  241.3  403.1
//     pair                                                 144.5  149.6  163.0  281.7
//     DeepSeek (2 shared experts of T rows each) at 31 / 62 / 124 / 252 rows per
//     group: w8d64 179.3 / 193.7, pair 195.7 / 207.0 / 222.3 / 330.8, rows
//     222.3 / 249.0 / 285.8 / 521.3.
// The pair tile takes over at 64 rows per group on average.
int pick_tile_w8(int M, int G) {
    const int f = g_forced_tile.load(std::memory_order_relaxed);
    if (f == MOE_TILE_W8_D16 || f == MOE_TILE_W8_D32 || f == MOE_TILE_W8_D64 ||
        f == MOE_TILE_W8_ROWS || f == MOE_TILE_W8_PAIR)
        return f;
    const int64_t m = M, g = G;
    if (m <= 10 * g) return MOE_TILE_W8_D16;
    if (m <= 24 * g) return MOE_TILE_W8_D32;
    if (m < 64 * g) return MOE_TILE_W8_D64;
    return MOE_TILE_W8_PAIR;
}
}  // namespace moe

extern "C" moe_status moe_set_gemm_tile(int tile) {
    if (tile < MOE_TILE_AUTO || tile > MOE_TILE_W8_PAIR) return MOE_ERR_INVALID_ARG;
    moe::g_forced_tile.store(tile, std::memory_order_relaxed);
    return MOE_OK;
}

template <bool SWIGLU>
static moe_status launch_tc_bn(const void *act, const void *w, const int32_t *offsets, int G,
                               int M, int K, int R, int NOUT, int UP_OFF, uint16_t *out,
                               int32_t *dev_error, cudaStream_t stream) {
    switch (pick_tile(M, G)) {
        case MOE_TILE_128x128:
            return launch_tc<SWIGLU, 128>(act, w, offsets, G, M, K, R, NOUT, UP_OFF, out,
                                          dev_error, stream);
        case MOE_TILE_128x256:
            return launch_tc<SWIGLU, 256>(act, w, offsets, G, M, K, R, NOUT, UP_OFF, out,
                                          dev_error, stream);
        default:
            // the pair kernel reads whole 64-deep k-blocks; other K take 128 x 256
            if (K % TC_BK == 0)
                return launch_tc_pair<SWIGLU>(act, w, offsets, G, M, K, R, NOUT, UP_OFF, out,
                                              dev_error, stream);
            return launch_tc<SWIGLU, 256>(act, w, offsets, G, M, K, R, NOUT, UP_OFF, out,
                                          dev_error, stream);
    }
}

extern "C" moe_status moe_grouped_gemm_gate_up(const uint16_t *x_perm, const int32_t *offsets,
                                               int G, int M, int H, int I, const uint16_t *w_gu,
                                               uint16_t *h, int32_t *dev_error,
                                               cudaStream_t stream) {
    moe_status st = check_ffn_args(x_perm, offsets, G, M, H, I, w_gu, w_gu, h, h,
                                   moe_ffn_workspace_size(M, I), 8);
    if (st != MOE_OK) return st;
    return launch_tc_bn<true>(x_perm, w_gu, offsets, G, M, H, 2 * I, I, I, h, dev_error, stream);
}

extern "C" moe_status moe_grouped_gemm_down(const uint16_t *h, const int32_t *offsets, int G,
                                            int M, int H, int I, const uint16_t *w_down,
                                            uint16_t *y_perm, int32_t *dev_error,
                                            cudaStream_t stream) {
    moe_status st = check_ffn_args(h, offsets, G, M, H, I, w_down, w_down, y_perm, y_perm,
                                   moe_ffn_workspace_size(M, I), 8);
    if (st != MOE_OK) return st;
    return launch_tc_bn<false>(h, w_down, offsets, G, M, I, H, H, 0, y_perm, dev_error, stream);
}

extern "C" moe_status moe_grouped_gemm_swiglu(const uint16_t *x_perm, const int32_t *offsets,
                                              int G, int M, int H, int I, const uint16_t *w_gu,
                                              const uint16_t *w_down, uint16_t *y_perm,
                                              void *workspace, size_t workspace_bytes,
                                              int32_t *dev_error, cudaStream_t stream) {
    moe_status st = check_ffn_args(x_perm, offsets, G, M, H, I, w_gu, w_down, y_perm, workspace,
                                   workspace_bytes, 8);
    if (st != MOE_OK) return st;
    uint16_t *h = static_cast<uint16_t *>(workspace);
    st = launch_tc_bn<true>(x_perm, w_gu, offsets, G, M, H, 2 * I, I, I, h, dev_error, stream);
    if (st != MOE_OK) return st;
    return launch_tc_bn<false>(h, w_down, offsets, G, M, I, H, H, 0, y_perm, dev_error, stream);
}
