// gemm_tc_w8.cu -- grouped GEMM with int8 weight-only experts on tcgen05.
//
// The "dispatch" README's phase 5a describes per-channel int8 weight-only
// experts: weights stored as int8 with one fp32 scale per output channel,
// activations kept in bf16.  The tensor cores' kind::f16 MMA needs both
// operands in bf16, so each weight tile is widened in shared memory:
//
//   warp 0      TMA producer of the activation tiles (bf16, 128-byte swizzle)
//   warp 6      TMA producer of the raw int8 weight tiles (own 4-deep ring)
//   warps 7-14  converters, four groups taking turns by k-step: int8 -> bf16
//               (exact: |q| <= 127 has 8 significant bits) into the
//               128-byte-swizzled K-major layout the MMA reads
//   warp 1      TMEM allocator + MMA issuer (M = 128 tokens, N = 256 weights)
//
//   warps 2-5   epilogue: accumulator * per-row scale (= sum x*q*scale, the
//               dequantised product), then SwiGLU or a plain bf16 store.
//
// Groups of fewer than 64 rows on average go to the 256-row weight tiles of
// gemm_tc_dec_w8.cu, larger ones to the CTA-pair tiles of gemm_tc_pair_w8.cu
// (both with the weights as the MMA's M, widened into tensor memory); these
// token-row tiles run when K is not a multiple of 64 (the other kernels copy
// whole 64-deep k-blocks) or when forced with moe_set_gemm_tile.
//
// The tile scheduler, tile order and failure handling (bounded waits, drains,
// TMEM freed on every path) are those of the bf16 kernel in gemm_tc.cu.
#include "tc_common.cuh"

namespace moe {

constexpr int W8_BN = 256;
constexpr int W8_STAGES = 3;        // activation + converted weight stages
constexpr int W8_RAW = 4;           // raw int8 weight stages (the HBM stream)
// Converter groups take the k-steps in turn (group = k-step mod
// W8_CONV_GROUPS) and wait on barriers by phase parity, which cannot tell a
// phase from the one two uses back: every barrier a converter waits on must
// be waited on by one group only, in order.  The raw ring's depth is a
// multiple of the group count for that; the stage-free signal of k-step q
// goes to barrier q mod W8_FREE, W8_FREE a common multiple of the stage and
// group counts, so the k-steps that wait on one barrier belong to one group.
constexpr int W8_CONV_GROUPS = W8_GROUPS;
constexpr int W8_FREE = 12;
constexpr int W8_CONV_THREADS = W8_CONV_GROUPS * W8_GROUP_THREADS;
static_assert(W8_RAW % W8_CONV_GROUPS == 0, "each raw stage must belong to one converter group");
static_assert(W8_FREE % W8_STAGES == 0 && W8_FREE % W8_CONV_GROUPS == 0,
              "stage-free barriers: a common multiple of stages and groups");
static_assert((2 * W8_STAGES + W8_FREE + 2 * W8_RAW + 5) * 8 + 8 <= 512, "barrier block");
constexpr int W8_THREADS = 7 * 32 + W8_CONV_THREADS;

struct W8Cfg {
    static constexpr int A_BYTES = TC_BM * TC_BK * 2;
    static constexpr int B_BYTES = W8_BN * TC_BK * 2;
    static constexpr int RAW_BYTES = W8_BN * TC_BK;
    static constexpr uint32_t TMEM_COLS = 2 * W8_BN;
    static constexpr int BAR_BYTES = 512;
    static size_t smem_bytes(int G) {
        return 1024 + static_cast<size_t>(W8_STAGES) * (A_BYTES + B_BYTES) +
               static_cast<size_t>(W8_RAW) * RAW_BYTES + BAR_BYTES +
               2 * static_cast<size_t>(G + 1) * sizeof(int);
    }
};

// Wait until the stage k-step `seq` will use is free: k-step seq - S, the
// stage's previous user, has been consumed by the MMA.
__device__ __forceinline__ bool stage_free(uint64_t *ab_free, int seq, int32_t *dev_error) {
    if (seq < W8_STAGES) return true;
    const int q = seq - W8_STAGES;
    return mbar_wait(&ab_free[q % W8_FREE], static_cast<uint32_t>((q / W8_FREE) & 1),
                     dev_error);
}

// SWIGLU: out = h [M, NOUT=I], int8 weights [G*2I, K=H], scales [G*2I].
// PLAIN : out = y [M, NOUT=H], int8 weights [G*H,  K=I], scales [G*H].
template <bool SWIGLU>
__global__ void __launch_bounds__(W8_THREADS, 1)
    tc_grouped_gemm_w8(const __grid_constant__ CUtensorMap tm_act,
                    const __grid_constant__ CUtensorMap tm_act128,
                       const __grid_constant__ CUtensorMap tm_act32,
                       const __grid_constant__ CUtensorMap tm_act64,
                       const __grid_constant__ CUtensorMap tm_q, const float *__restrict__ scales,
                       const int32_t *__restrict__ offsets, int G, int M, int K, int R, int NOUT,
                       int UP_OFF, uint16_t *__restrict__ out, int32_t *dev_error) {
    using C = W8Cfg;
    constexpr int BN = W8_BN;
    constexpr int S = W8_STAGES;
    constexpr int RS = W8_RAW;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sA = smem;
    uint8_t *sB = sA + S * C::A_BYTES;
    uint8_t *sQ = sB + S * C::B_BYTES;
    uint64_t *a_full = reinterpret_cast<uint64_t *>(sQ + RS * C::RAW_BYTES);
    uint64_t *b_full = a_full + S;
    uint64_t *ab_empty = b_full + S;              // [W8_FREE], by k-step number
    uint64_t *q_full = ab_empty + W8_FREE;
    uint64_t *q_empty = q_full + RS;
    uint64_t *accf = q_empty + RS;
    uint64_t *acce = accf + 2;
    uint64_t *drain = acce + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    int *s_total = reinterpret_cast<int *>(tmem_slot + 1);
    int *s_off = reinterpret_cast<int *>(reinterpret_cast<uint8_t *>(a_full) + C::BAR_BYTES);
    int *s_tile = s_off + (G + 1);

    const int warp = threadIdx.x >> 5, lane = lane_id();
    const int n_per_tile = SWIGLU ? BN / 2 : BN;
    const int n_tiles = (NOUT + n_per_tile - 1) / n_per_tile;
    const int KB = (K + TC_BK - 1) / TC_BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&a_full[s], 1);
            mbar_init(&b_full[s], W8_GROUP_THREADS);
        }
        for (int i = 0; i < W8_FREE; ++i) mbar_init(&ab_empty[i], 1);
        for (int r = 0; r < RS; ++r) {
            mbar_init(&q_full[r], 1);
            mbar_init(&q_empty[r], W8_GROUP_THREADS);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accf[b], 1);
            mbar_init(&acce[b], 128);
        }
        mbar_init(drain, 1);
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tm_act);
        prefetch_tmap(&tm_act32);
        prefetch_tmap(&tm_act64);
        prefetch_tmap(&tm_act128);
        prefetch_tmap(&tm_q);
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
        // ------------------------------------------- activation producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_last();
            int s = 0, seq = 0;
            uint32_t ph = 0, filled = 0, fill_par = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const TileInfo ti = decode_tile(t, s_tile, s_off, G);
                // a tile with more than 64 rows takes one 128-row box; a smaller
                // one only the 16-row boxes it needs (rows past the group are
                // loaded but never stored)
                const int abox = ti.nrows <= 16 ? 16 : ti.nrows <= 32 ? 32
                                                     : ti.nrows <= 64 ? 64 : 128;
                const CUtensorMap *tm_a = abox == 16 ? &tm_act : abox == 32 ? &tm_act32
                                        : abox == 64 ? &tm_act64 : &tm_act128;
                const uint32_t bytes = abox * TC_BK * 2;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!stage_free(ab_empty, seq, dev_error)) { ok = false; break; }
                    ++seq;
                    mbar_arrive_expect_tx(&a_full[s], bytes);
                    uint8_t *a = sA + s * C::A_BYTES;
                    tma_load_2d(a, tm_a, &a_full[s], kb * TC_BK, ti.m0, pol);
                    filled |= 1u << s;
                    fill_par = (fill_par & ~(1u << s)) | (ph << s);
                    if (++s == S) { s = 0; ph ^= 1u; }
                }
            }
            for (int i = 0; i < S; ++i)
                if ((filled >> i) & 1u) mbar_wait(&a_full[i], (fill_par >> i) & 1u, dev_error);
        }
        __syncwarp();
    } else if (warp == 6) {
        // ------------------------------------------- int8 weight producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            int r = 0;
            uint32_t ph = 0, filled = 0, fill_par = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const TileInfo ti = decode_tile(t, s_tile, s_off, G);
                const int wrow = ti.g * R + ti.nt * n_per_tile;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&q_empty[r], ph ^ 1u, dev_error)) { ok = false; break; }
                    mbar_arrive_expect_tx(&q_full[r], C::RAW_BYTES);
                    uint8_t *q = sQ + r * C::RAW_BYTES;
                    if (SWIGLU) {      // gate rows and up rows in one 3-D copy
                        tma_load_3d(q, &tm_q, &q_full[r], kb * TC_BK, ti.nt * n_per_tile,
                                    2 * ti.g, pol);
                    } else {
                        tma_load_2d(q, &tm_q, &q_full[r], kb * TC_BK, wrow, pol);
                    }
                    filled |= 1u << r;
                    fill_par = (fill_par & ~(1u << r)) | (ph << r);
                    if (++r == RS) { r = 0; ph ^= 1u; }
                }
            }
            for (int i = 0; i < RS; ++i)
                if ((filled >> i) & 1u) mbar_wait(&q_full[i], (fill_par >> i) & 1u, dev_error);
        }
        __syncwarp();
    } else if (warp >= 7) {
        // ------------------------------------------- converters int8 -> bf16
        const int ct = threadIdx.x - 7 * 32;
        const int grp = ct / W8_GROUP_THREADS, gt = ct % W8_GROUP_THREADS;
        int seq = 0;                                   // this CTA's k-step counter
        bool ok = true;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
            for (int kb = 0; kb < KB; ++kb, ++seq) {
                if (seq % W8_CONV_GROUPS != grp) continue;
                const int s = seq % S, r = seq % RS;
                const uint32_t rph = (seq / RS) & 1;
                if (!mbar_wait(&q_full[r], rph, dev_error) ||
                    !stage_free(ab_empty, seq, dev_error)) {
                    ok = false;
                    break;
                }
                // the stage's last reader was the tensor core (async proxy):
                // order its reads before these generic writes
                fence_proxy_async_smem();
                widen_stage<BN>(sQ + r * C::RAW_BYTES, sB + s * C::B_BYTES, gt);
                fence_proxy_async_smem();     // generic-proxy writes -> visible to the MMA
                mbar_arrive(&b_full[s]);
                mbar_arrive(&q_empty[r]);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(TC_BM, BN);
            int s = 0, acc = 0, seq = 0;
            uint32_t ph = 0, acc_ph = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                if (!mbar_wait(&acce[acc], acc_ph ^ 1u, dev_error)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&a_full[s], ph, dev_error) ||
                        !mbar_wait(&b_full[s], ph, dev_error)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(sA + s * C::A_BYTES);
                    const uint32_t b_addr = smem_u32(sB + s * C::B_BYTES);
#pragma unroll
                    for (int kk = 0; kk < TC_BK / 16; ++kk)
                        tc_mma_bf16(d_tmem, sw128_kmajor_desc(a_addr + kk * 32),
                                    sw128_kmajor_desc(b_addr + kk * 32), idesc,
                                    (kb > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(&ab_empty[seq % W8_FREE]);   // stage s is free after k-step seq
                    ++seq;
                    if (++s == S) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                tc_commit(&accf[acc]);
                acc ^= 1;
                if (acc == 0) acc_ph ^= 1u;
            }
            tc_commit(drain);
            mbar_wait(drain, 0, dev_error);
        }
        __syncwarp();
    } else {
        // ------------------------------------------- epilogue (warps 2..5)
        const int quarter = warp & 3;
        const int row_in_tile = quarter * 32 + lane;
        int acc = 0;
        uint32_t acc_ph = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x) {
            const TileInfo ti = decode_tile(t, s_tile, s_off, G);
            if (!mbar_wait_warp(&accf[acc], acc_ph, dev_error)) break;
            tc_fence_after();
            const bool valid = row_in_tile < ti.nrows;
            uint16_t *orow = out + static_cast<int64_t>(ti.m0 + row_in_tile) * NOUT;
            const uint32_t tbase =
                tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * BN;
            const int n0 = ti.nt * n_per_tile;
            const float *srow = scales + static_cast<int64_t>(ti.g) * R + n0;
            if (SWIGLU) {
#pragma unroll 1
                for (int c = 0; c < BN / 2; c += 16) {
                    uint32_t g[16], u[16];
                    tmem_ld16(tbase + c, g);
                    tmem_ld16(tbase + BN / 2 + c, u);
                    tmem_ld_wait();
                    if (valid && n0 + c < NOUT) {
                        const int nv = min(16, NOUT - n0 - c);     // 8 or 16
                        float sg[16], su[16];
#pragma unroll
                        for (int i = 0; i < 16; i += 4) {
                            const float4 a = i < nv ? __ldg(reinterpret_cast<const float4 *>(srow + c + i))
                                                    : make_float4(0.f, 0.f, 0.f, 0.f);
                            const float4 b = i < nv ? __ldg(reinterpret_cast<const float4 *>(srow + UP_OFF + c + i))
                                                    : make_float4(0.f, 0.f, 0.f, 0.f);
                            sg[i] = a.x; sg[i + 1] = a.y; sg[i + 2] = a.z; sg[i + 3] = a.w;
                            su[i] = b.x; su[i + 1] = b.y; su[i + 2] = b.z; su[i + 3] = b.w;
                        }
                        uint32_t p[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float g0 = __uint_as_float(g[2 * i]) * sg[2 * i];
                            const float g1 = __uint_as_float(g[2 * i + 1]) * sg[2 * i + 1];
                            const float u0 = __uint_as_float(u[2 * i]) * su[2 * i];
                            const float u1 = __uint_as_float(u[2 * i + 1]) * su[2 * i + 1];
                            p[i] = pack_bf16x2(silu_fast(g0) * u0, silu_fast(g1) * u1);
                        }
                        uint4 *dst = reinterpret_cast<uint4 *>(orow + n0 + c);
                        dst[0] = make_uint4(p[0], p[1], p[2], p[3]);
                        if (nv > 8) dst[1] = make_uint4(p[4], p[5], p[6], p[7]);
                    }
                }
            } else {
#pragma unroll 1
                for (int c = 0; c < BN; c += 16) {
                    uint32_t v[16];
                    tmem_ld16(tbase + c, v);
                    tmem_ld_wait();
                    if (valid && n0 + c < NOUT) {
                        const int nv = min(16, NOUT - n0 - c);
                        float sc[16];
#pragma unroll
                        for (int i = 0; i < 16; i += 4) {
                            const float4 a = i < nv ? __ldg(reinterpret_cast<const float4 *>(srow + c + i))
                                                    : make_float4(0.f, 0.f, 0.f, 0.f);
                            sc[i] = a.x; sc[i + 1] = a.y; sc[i + 2] = a.z; sc[i + 3] = a.w;
                        }
                        uint32_t p[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            p[i] = pack_bf16x2(__uint_as_float(v[2 * i]) * sc[2 * i],
                                               __uint_as_float(v[2 * i + 1]) * sc[2 * i + 1]);
                        uint4 *dst = reinterpret_cast<uint4 *>(orow + n0 + c);
                        dst[0] = make_uint4(p[0], p[1], p[2], p[3]);
                        if (nv > 8) dst[1] = make_uint4(p[4], p[5], p[6], p[7]);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&acce[acc]);
            acc ^= 1;
            if (acc == 0) acc_ph ^= 1u;
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
static moe_status launch_tc_w8(const void *act, const int8_t *q, const float *scales,
                               const int32_t *offsets, int G, int M, int K, int R, int NOUT,
                               int UP_OFF, uint16_t *out, int32_t *dev_error, cudaStream_t stream) {
    const int tile = pick_tile_w8(M, G);
    // CTA pairs read whole 64-deep k-blocks; other K take the token-row tiles
    if (tile == MOE_TILE_W8_PAIR && K % TC_BK == 0)
        return launch_tc_pair_w8<SWIGLU>(act, q, scales, offsets, G, M, K, R, NOUT, UP_OFF, out,
                                         dev_error, stream);
    if (tile == MOE_TILE_W8_D16 || tile == MOE_TILE_W8_D32 || tile == MOE_TILE_W8_D64)
        return launch_dec_w8<SWIGLU>(tile == MOE_TILE_W8_D16   ? 16
                                     : tile == MOE_TILE_W8_D32 ? 32
                                                               : 64,
                                     act, q, scales, offsets, G, M, K, R, NOUT, UP_OFF, out,
                                     dev_error, stream);
    CUtensorMap tm_act, tm_act32, tm_act64, tm_act128, tm_q;
    if (!encode_bf16_2d(&tm_act, act, K, M, 16) || !encode_bf16_2d(&tm_act32, act, K, M, 32) ||
        !encode_bf16_2d(&tm_act64, act, K, M, 64) || !encode_bf16_2d(&tm_act128, act, K, M, TC_BM))
        return MOE_ERR_CUDA;
    if (SWIGLU ? !encode_gate_up_3d(&tm_q, q, K, UP_OFF, G, W8_BN / 2, true)
               : !encode_u8_2d(&tm_q, q, K, static_cast<uint64_t>(G) * R, W8_BN))
        return MOE_ERR_CUDA;
    const size_t smem = W8Cfg::smem_bytes(G);
    if (smem > static_cast<size_t>(max_smem_optin())) return MOE_ERR_UNSUPPORTED;
    static int attr_done[64] = {0};
    if (!raise_smem_limit(tc_grouped_gemm_w8<SWIGLU>, attr_done)) return MOE_ERR_CUDA;
    launch(tc_grouped_gemm_w8<SWIGLU>, sm_count(), W8_THREADS, smem, stream, 
        tm_act, tm_act128, tm_act32, tm_act64, tm_q, scales, offsets, G, M, K, R, NOUT, UP_OFF, out,
        dev_error);
    return launch_status();
}

}  // namespace moe

using namespace moe;

extern "C" moe_status moe_grouped_gemm_swiglu_w8(const uint16_t *x_perm, const int32_t *offsets,
                                                 int G, int M, int H, int I, const int8_t *q_gu,
                                                 const float *s_gu, const int8_t *q_down,
                                                 const float *s_down, uint16_t *y_perm,
                                                 void *workspace, size_t workspace_bytes,
                                                 int32_t *dev_error, cudaStream_t stream) {
    moe_status st = check_ffn_args(x_perm, offsets, G, M, H, I, q_gu, q_down, y_perm, workspace,
                                   workspace_bytes, 16);
    if (st != MOE_OK) return st;
    if (!s_gu || !s_down) return MOE_ERR_INVALID_ARG;
    if (!aligned16(s_gu) || !aligned16(s_down)) return MOE_ERR_ALIGNMENT;
    uint16_t *h = static_cast<uint16_t *>(workspace);
    st = launch_tc_w8<true>(x_perm, q_gu, s_gu, offsets, G, M, H, 2 * I, I, I, h, dev_error,
                            stream);
    if (st != MOE_OK) return st;
    return launch_tc_w8<false>(h, q_down, s_down, offsets, G, M, I, H, H, 0, y_perm, dev_error,
                               stream);
}
