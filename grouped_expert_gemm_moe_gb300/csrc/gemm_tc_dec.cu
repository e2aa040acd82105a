// gemm_tc_dec.cu -- grouped GEMM for decode-sized expert groups, with the
// weights as the MMA's 128-row operand.
//
// With a handful of token rows per expert, a tile of 128 token rows is
// mostly empty, yet each k-step still costs the tensor core the full
// 128-row product and the shared memory the reads of 128 rows.  Here the
// product is turned around ("switchyard" page, 02 Kernels and dispatch: the
// grouped FFN over all experts in one launch, unchanged in what it computes):
//
//     D[f, j] = sum_k W_g[f, k] * X[j, k]       f: weight row, j: token row
//
// so the MMA's M = 128 runs over weight rows (output features) and its
// N = TN (16, 32 or 64) over the group's token rows.  A tile is (group g,
// 128 weight rows, a block of TN token rows); the blocks of one weight tile
// are consecutive tile indices, so CTAs running side by side share the
// weight tile through L2 and HBM sees it once.
//
//  * warp 0: TMA producer of the TNx64 token tiles, in a ring of their own
//    (they come from L2 for every k-step);
//  * warp 6: TMA producer of the 128x64 weight tiles (gate rows then up rows
//    in SWIGLU mode), the HBM stream.  bf16 tiles go straight to the MMA's
//    ring; int8 tiles (128 rows x 64 B) to a raw ring, from which warps
//    7-14, in four groups that take turns by k-step, widen them to bf16
//    (exact) in the 128-byte-swizzled K-major layout the MMA reads;
//  * warp 1: TMEM allocator and MMA issuer (kind::f16, M = 128, N = TN),
//    accumulators double-buffered in TMEM (2 x TN columns);
//  * warps 2-5: epilogue.  A thread owns TMEM lane f (one weight row) and
//    reads its TN token columns.  SWIGLU: lanes 0-63 hold gate rows i,
//    lanes 64-127 the matching up rows; the up values pass through shared
//    memory to the gate threads, which store h[j, i] = silu(g) * u.  PLAIN:
//    y[j, f] is stored directly.  int8 scales multiply the accumulator
//    (sum_k x q s = s * sum_k x q).
// Every wait is bounded (1 s); a wait that runs out records MOE_ERR_TIMEOUT,
// the kernel drains its own copies and MMAs, frees TMEM and returns.
#include "tc_common.cuh"

namespace moe {

constexpr int DEC_BM = 128;          // weight rows per tile (MMA M)

// KP: 64-element k-blocks per stage (2 for bf16 weights when K % 128 == 0:
// one copy per operand then moves twice the bytes; the ring's pace is set
// by copies and hand-offs per stage more than by bytes).
template <bool W8, int TN, int KP = 1>
struct DecCfg {
    static_assert(KP == 1 || (KP == 2 && !W8), "int8 stages hold one k-block");
    static constexpr int A_BYTES = DEC_BM * TC_BK * 2 * KP;     // bf16 weight tile
    static constexpr int B_BYTES = TN * TC_BK * 2 * KP;         // token tile
    static constexpr int RAW_BYTES = DEC_BM * TC_BK;            // int8 weight tile
    // Rings (sized to fit 227 KB of shared memory with G = 1024 groups):
    // token tiles TOK_STAGES deep, weight tiles STAGES deep, raw int8 tiles
    // RAW_STAGES deep.  The token ring is separate and deep because token
    // tiles come from L2 for every k-step: a short shared ring would put
    // that L2 round trip into every k-step's hand-off.
    static constexpr int TOK_STAGES = KP == 2 ? (TN <= 32 ? 8 : 4) : (TN <= 32 ? 16 : 8);
    static constexpr int STAGES = W8 ? 4 : KP == 2 ? (TN <= 16 ? 5 : 4) : (TN <= 16 ? 10 : 8);
    static constexpr int RAW_STAGES = W8 ? (TN <= 16 ? 12 : 8) : 0;
    // int8: converter groups take the k-steps in turn and wait by phase
    // parity, so each stage of both rings must always fall to the same group
    static_assert(!W8 || (STAGES % W8_GROUPS == 0 && RAW_STAGES % W8_GROUPS == 0),
                  "each ring stage must belong to one converter group");
    static constexpr int XBUF_BYTES = 64 * TN * 4;              // up values, fp32
    static constexpr uint32_t TMEM_COLS = 2 * TN < 32 ? 32 : 2 * TN;
    static constexpr int BAR_BYTES = 1024;
    static constexpr int THREADS = W8 ? 7 * 32 + 256 : 7 * 32;
    static constexpr size_t smem_bytes(int G) {
        return 1024 + static_cast<size_t>(STAGES) * A_BYTES +
               static_cast<size_t>(TOK_STAGES) * B_BYTES +
               static_cast<size_t>(RAW_STAGES) * RAW_BYTES + XBUF_BYTES + BAR_BYTES +
               2 * static_cast<size_t>(G + 1) * sizeof(int);
    }
    static_assert(smem_bytes(1024) <= 232448, "decode tile rings exceed shared memory");
    static_assert(2 * (TOK_STAGES + STAGES + RAW_STAGES) + 7 <= BAR_BYTES / 8 - 2,
                  "barrier area too small");
};

// SWIGLU: out = h [M, NOUT=I], weights [G*2I, K=H] (up rows at +UP_OFF = I).
// PLAIN : out = y [M, NOUT=H], weights [G*H,  K=I].
// R = weight rows per group.  scales: int8 only, [G*R] fp32.
template <bool SWIGLU, bool W8, int TN, int KP>
__global__ void __launch_bounds__(DecCfg<W8, TN, KP>::THREADS, 1)
    tc_grouped_gemm_dec(const __grid_constant__ CUtensorMap tm_tok,
                        const __grid_constant__ CUtensorMap tm_w, const float *__restrict__ scales,
                        const int32_t *__restrict__ offsets, int G, int M, int K, int R,
                        int NOUT, int UP_OFF, uint16_t *__restrict__ out, int32_t *dev_error) {
    using C = DecCfg<W8, TN, KP>;
    constexpr int S = C::STAGES;
    constexpr int TS = C::TOK_STAGES;
    constexpr int RS = C::RAW_STAGES > 0 ? C::RAW_STAGES : 1;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sA = smem;                                   // S x A_BYTES (1024-aligned)
    uint8_t *sB = sA + S * C::A_BYTES;                    // TS x B_BYTES (multiples of 1024)
    uint8_t *sQ = sB + TS * C::B_BYTES;                   // RAW_STAGES x RAW_BYTES
    float *xbuf = reinterpret_cast<float *>(sQ + C::RAW_STAGES * C::RAW_BYTES);
    uint64_t *bars = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(xbuf) +
                                                  C::XBUF_BYTES);
    uint64_t *b_full = bars;                // token tile landed
    uint64_t *b_empty = b_full + TS;        // token tile consumed by the MMA
    uint64_t *a_full = b_empty + TS;        // weight tile ready (TMA bytes, or converters)
    uint64_t *a_empty = a_full + S;         // weight tile consumed by the MMA
    uint64_t *q_full = a_empty + S;         // int8: raw tile landed
    uint64_t *q_empty = q_full + RS;        // int8: raw tile widened
    uint64_t *accf = q_empty + RS;
    uint64_t *acce = accf + 2;
    uint64_t *x_full = acce + 2;            // up values written (64 arrivals)
    uint64_t *x_empty = x_full + 1;         // up values read (64 arrivals)
    uint64_t *drain = x_empty + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    int *s_total = reinterpret_cast<int *>(tmem_slot + 1);
    int *s_off = reinterpret_cast<int *>(reinterpret_cast<uint8_t *>(bars) + C::BAR_BYTES);
    int *s_tile = s_off + (G + 1);

    const int warp = threadIdx.x >> 5, lane = lane_id();
    const int n_per_tile = SWIGLU ? DEC_BM / 2 : DEC_BM;
    const int n_tiles = (NOUT + n_per_tile - 1) / n_per_tile;
    const int KB = (K + TC_BK * KP - 1) / (TC_BK * KP);     // stages per tile

    if (threadIdx.x == 0) {
        for (int i = 0; i < TS; ++i) {
            mbar_init(&b_full[i], 1);
            mbar_init(&b_empty[i], 1);
        }
        for (int i = 0; i < S; ++i) {
            mbar_init(&a_full[i], W8 ? W8_GROUP_THREADS : 1);
            mbar_init(&a_empty[i], 1);
        }
        for (int i = 0; i < RS; ++i) {
            mbar_init(&q_full[i], 1);
            mbar_init(&q_empty[i], W8_GROUP_THREADS);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&accf[i], 1);
            mbar_init(&acce[i], 128);
        }
        mbar_init(x_full, 64);
        mbar_init(x_empty, 64);
        mbar_init(drain, 1);
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tm_tok);
        prefetch_tmap(&tm_w);
    }
    if (warp == 1) tmem_alloc<C::TMEM_COLS>(tmem_slot);
    pdl_wait();       // predecessors' writes (offsets, token rows) are visible after this
    pdl_trigger();
    if (warp == 2) build_tile_table(offsets, G, M, n_tiles, s_off, s_tile, s_total, dev_error, TN);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int total = *s_total;

    if (warp == 0) {
        // ------------------------------------------------ token tiles (from L2)
        if (lane == 0) {
            const uint64_t pol = policy_evict_last();
            int i = 0;
            uint32_t ph = 0, filled = 0, fill_par = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const TileInfo ti = decode_tile(t, s_tile, s_off, G, TN);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&b_empty[i], ph ^ 1u, dev_error)) { ok = false; break; }
                    mbar_arrive_expect_tx(&b_full[i], C::B_BYTES);
                    if (KP == 2)
                        tma_load_3d(sB + i * C::B_BYTES, &tm_tok, &b_full[i], 0, ti.m0, 2 * kb,
                                    pol);
                    else
                        tma_load_2d(sB + i * C::B_BYTES, &tm_tok, &b_full[i], kb * TC_BK, ti.m0,
                                    pol);
                    filled |= 1u << i;
                    fill_par = (fill_par & ~(1u << i)) | (ph << i);
                    if (++i == TS) { i = 0; ph ^= 1u; }
                }
            }
            for (int j = 0; j < TS; ++j)
                if ((filled >> j) & 1u) mbar_wait(&b_full[j], (fill_par >> j) & 1u, dev_error);
        }
        __syncwarp();
    } else if (warp == 6) {
        // ------------------------------------------------ weight tiles (the HBM stream)
        // bf16: straight into the MMA's weight ring; int8: into the raw ring
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            constexpr int NS = W8 ? RS : S;
            uint64_t *full = W8 ? q_full : a_full;
            uint64_t *empty = W8 ? q_empty : a_empty;
            uint8_t *ring = W8 ? sQ : sA;
            constexpr int STAGE = W8 ? C::RAW_BYTES : C::A_BYTES;
            int i = 0;
            uint32_t ph = 0, filled = 0, fill_par = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const TileInfo ti = decode_tile(t, s_tile, s_off, G, TN);
                const int wrow = ti.g * R + ti.nt * n_per_tile;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&empty[i], ph ^ 1u, dev_error)) { ok = false; break; }
                    mbar_arrive_expect_tx(&full[i], STAGE);
                    uint8_t *dst = ring + i * STAGE;
                    if (KP == 2) {     // two k-blocks (and gate + up rows) in one copy
                        if (SWIGLU)
                            tma_load_4d(dst, &tm_w, &full[i], 0, ti.nt * n_per_tile, 2 * ti.g,
                                        2 * kb, pol);
                        else
                            tma_load_3d(dst, &tm_w, &full[i], 0, wrow, 2 * kb, pol);
                    } else if (SWIGLU) {   // gate rows and up rows in one 3-D copy
                        tma_load_3d(dst, &tm_w, &full[i], kb * TC_BK, ti.nt * n_per_tile,
                                    2 * ti.g, pol);
                    } else {
                        tma_load_2d(dst, &tm_w, &full[i], kb * TC_BK, wrow, pol);
                    }
                    filled |= 1u << i;
                    fill_par = (fill_par & ~(1u << i)) | (ph << i);
                    if (++i == NS) { i = 0; ph ^= 1u; }
                }
            }
            for (int j = 0; j < NS; ++j)
                if ((filled >> j) & 1u) mbar_wait(&full[j], (fill_par >> j) & 1u, dev_error);
        }
        __syncwarp();
    } else if (W8 && warp >= 7) {
        // ------------------------------------------------ converters int8 -> bf16
        const int ct = threadIdx.x - 7 * 32;
        const int grp = ct / W8_GROUP_THREADS, gt = ct % W8_GROUP_THREADS;
        int seq = 0;                                   // this CTA's k-step counter
        bool ok = true;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
            for (int kb = 0; kb < KB; ++kb, ++seq) {
                if (seq % W8_GROUPS != grp) continue;
                const int s = seq % S, r = seq % RS;
                const uint32_t sph = (seq / S) & 1, rph = (seq / RS) & 1;
                if (!mbar_wait(&q_full[r], rph, dev_error) ||
                    !mbar_wait(&a_empty[s], sph ^ 1u, dev_error)) {
                    ok = false;
                    break;
                }
                // the stage's last reader was the tensor core (async proxy):
                // order its reads before these generic writes
                fence_proxy_async_smem();
                widen_stage<DEC_BM>(sQ + r * C::RAW_BYTES, sA + s * C::A_BYTES, gt);
                fence_proxy_async_smem();     // generic-proxy writes -> visible to the MMA
                mbar_arrive(&a_full[s]);
                mbar_arrive(&q_empty[r]);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(DEC_BM, TN);
            int s = 0, tb = 0, acc = 0;
            uint32_t ph = 0, tph = 0, acc_ph = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                if (!mbar_wait(&acce[acc], acc_ph ^ 1u, dev_error)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * TN);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&a_full[s], ph, dev_error) ||
                        !mbar_wait(&b_full[tb], tph, dev_error)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(sA + s * C::A_BYTES);
                    const uint32_t b_addr = smem_u32(sB + tb * C::B_BYTES);
#pragma unroll
                    for (int kq = 0; kq < KP; ++kq)
#pragma unroll
                        for (int kk = 0; kk < TC_BK / 16; ++kk)
                            tc_mma_bf16(d_tmem,
                                        sw128_kmajor_desc(a_addr + kq * DEC_BM * 128 + kk * 32),
                                        sw128_kmajor_desc(b_addr + kq * TN * 128 + kk * 32), idesc,
                                        (kb > 0 || kq > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(&a_empty[s]);
                    tc_commit(&b_empty[tb]);
                    if (++s == S) { s = 0; ph ^= 1u; }
                    if (++tb == TS) { tb = 0; tph ^= 1u; }
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
    } else if (warp >= 2 && warp <= 5) {
        // ------------------------------------------------ epilogue
        const int quarter = warp & 3;                 // TMEM lanes this warp may access
        const int f = quarter * 32 + lane;            // weight row within the tile
        int acc = 0;
        uint32_t acc_ph = 0, x_ph = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x) {
            const TileInfo ti = decode_tile(t, s_tile, s_off, G, TN);
            if (!mbar_wait_warp(&accf[acc], acc_ph, dev_error)) break;
            tc_fence_after();
            float d[TN];
            {
                const uint32_t taddr =
                    tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * TN;
                uint32_t v[16];
#pragma unroll
                for (int c = 0; c < TN; c += 16) {
                    tmem_ld16(taddr + c, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) d[c + i] = __uint_as_float(v[i]);
                }
            }
            tc_fence_before();
            mbar_arrive(&acce[acc]);                   // accumulator free for the next tile
            acc ^= 1;
            if (acc == 0) acc_ph ^= 1u;
            const int nrows = ti.nrows;
            if (SWIGLU) {
                const int i = ti.nt * 64 + (f & 63);            // intermediate index
                const bool up = f >= 64;
                float sc = 1.0f;
                if (W8 && i < NOUT)
                    sc = scales[static_cast<int64_t>(ti.g) * R + (up ? UP_OFF : 0) + i];
                if (up) {
                    if (!mbar_wait_warp(x_empty, x_ph ^ 1u, dev_error)) break;
#pragma unroll
                    for (int j = 0; j < TN; ++j) xbuf[j * 64 + (f - 64)] = d[j] * sc;
                    mbar_arrive(x_full);
                } else {
                    if (!mbar_wait_warp(x_full, x_ph, dev_error)) break;
                    if (i < NOUT) {
                        uint16_t *col = out + static_cast<int64_t>(ti.m0) * NOUT + i;
#pragma unroll
                        for (int j = 0; j < TN; ++j) {
                            if (j < nrows) {
                                const float hv = silu_fast(d[j] * sc) * xbuf[j * 64 + f];
                                const __nv_bfloat16 b = __float2bfloat16_rn(hv);
                                col[static_cast<int64_t>(j) * NOUT] =
                                    *reinterpret_cast<const uint16_t *>(&b);
                            }
                        }
                    }
                    mbar_arrive(x_empty);
                }
                x_ph ^= 1u;
            } else {
                const int n = ti.nt * DEC_BM + f;
                if (n < NOUT) {
                    const float sc = W8 ? scales[static_cast<int64_t>(ti.g) * R + n] : 1.0f;
                    uint16_t *col = out + static_cast<int64_t>(ti.m0) * NOUT + n;
#pragma unroll
                    for (int j = 0; j < TN; ++j) {
                        if (j < nrows) {
                            const __nv_bfloat16 b = __float2bfloat16_rn(d[j] * sc);
                            col[static_cast<int64_t>(j) * NOUT] =
                                *reinterpret_cast<const uint16_t *>(&b);
                        }
                    }
                }
            }
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

template <bool SWIGLU, bool W8, int TN, int KP>
static moe_status launch_dec_tn(const void *tok, const void *w, const float *scales,
                                const int32_t *offsets, int G, int M, int K, int R, int NOUT,
                                int UP_OFF, uint16_t *out, int32_t *dev_error,
                                cudaStream_t stream) {
    using C = DecCfg<W8, TN, KP>;
    CUtensorMap tm_tok, tm_w;
    if (KP == 2) {
        if (!encode_kpair(&tm_tok, tok, K, M, TN)) return MOE_ERR_CUDA;
        if (SWIGLU ? !encode_gate_up_kpair(&tm_w, w, K, UP_OFF, G, DEC_BM / 2)
                   : !encode_kpair(&tm_w, w, K, static_cast<uint64_t>(G) * R, DEC_BM))
            return MOE_ERR_CUDA;
    } else {
        if (!encode_bf16_2d(&tm_tok, tok, K, M, TN)) return MOE_ERR_CUDA;
        if (SWIGLU) {
            if (!encode_gate_up_3d(&tm_w, w, K, UP_OFF, G, DEC_BM / 2, W8)) return MOE_ERR_CUDA;
        } else if (W8) {
            if (!encode_u8_2d(&tm_w, w, K, static_cast<uint64_t>(G) * R, DEC_BM))
                return MOE_ERR_CUDA;
        } else {
            if (!encode_bf16_2d(&tm_w, w, K, static_cast<uint64_t>(G) * R, DEC_BM))
                return MOE_ERR_CUDA;
        }
    }
    const size_t smem = C::smem_bytes(G);
    if (smem > static_cast<size_t>(max_smem_optin())) return MOE_ERR_UNSUPPORTED;
    static int attr_done[64] = {0};
    if (!raise_smem_limit(tc_grouped_gemm_dec<SWIGLU, W8, TN, KP>, attr_done))
        return MOE_ERR_CUDA;
    launch(tc_grouped_gemm_dec<SWIGLU, W8, TN, KP>, sm_count(), C::THREADS, smem, stream, tm_tok,
           tm_w, scales, offsets, G, M, K, R, NOUT, UP_OFF, out, dev_error);
    return launch_status();
}

template <bool SWIGLU, bool W8, int TN>
static moe_status launch_dec_kp(const void *tok, const void *w, const float *scales,
                                const int32_t *offsets, int G, int M, int K, int R, int NOUT,
                                int UP_OFF, uint16_t *out, int32_t *dev_error,
                                cudaStream_t stream) {
    if (!W8 && K % 128 == 0)
        return launch_dec_tn<SWIGLU, W8, TN, W8 ? 1 : 2>(tok, w, scales, offsets, G, M, K, R,
                                                          NOUT, UP_OFF, out, dev_error, stream);
    return launch_dec_tn<SWIGLU, W8, TN, 1>(tok, w, scales, offsets, G, M, K, R, NOUT, UP_OFF,
                                            out, dev_error, stream);
}

// Token-block height TN for the decode kernel (16, 32 or 64).
template <bool SWIGLU, bool W8>
moe_status launch_dec(int tn, const void *tok, const void *w, const float *scales,
                      const int32_t *offsets, int G, int M, int K, int R, int NOUT, int UP_OFF,
                      uint16_t *out, int32_t *dev_error, cudaStream_t stream) {
    switch (tn) {
        case 16:
            return launch_dec_kp<SWIGLU, W8, 16>(tok, w, scales, offsets, G, M, K, R, NOUT, UP_OFF,
                                                 out, dev_error, stream);
        case 32:
            return launch_dec_kp<SWIGLU, W8, 32>(tok, w, scales, offsets, G, M, K, R, NOUT, UP_OFF,
                                                 out, dev_error, stream);
        default:
            return launch_dec_kp<SWIGLU, W8, 64>(tok, w, scales, offsets, G, M, K, R, NOUT, UP_OFF,
                                                 out, dev_error, stream);
    }
}

template moe_status launch_dec<true, false>(int, const void *, const void *, const float *,
                                            const int32_t *, int, int, int, int, int, int,
                                            uint16_t *, int32_t *, cudaStream_t);
template moe_status launch_dec<false, false>(int, const void *, const void *, const float *,
                                             const int32_t *, int, int, int, int, int, int,
                                             uint16_t *, int32_t *, cudaStream_t);
template moe_status launch_dec<true, true>(int, const void *, const void *, const float *,
                                           const int32_t *, int, int, int, int, int, int,
                                           uint16_t *, int32_t *, cudaStream_t);
template moe_status launch_dec<false, true>(int, const void *, const void *, const float *,
                                            const int32_t *, int, int, int, int, int, int,
                                            uint16_t *, int32_t *, cudaStream_t);

}  // namespace moe
