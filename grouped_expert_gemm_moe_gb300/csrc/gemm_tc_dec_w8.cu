// gemm_tc_dec_w8.cu -- int8 weight-only grouped GEMM for decode-sized expert
// groups: 256 weight rows per tile, the widened weights in tensor memory.
//
// Per-channel int8 weights with fp32 scales and bf16 activations ("dispatch"
// README, phase 5a), all experts in one launch ("switchyard" page, 02
// Kernels and dispatch): D[f, j] = sum_k W_g[f, k] * X[j, k] with the weight
// rows as the MMA's M and a block of TN token rows as its N, so no MMA rows
// go to the empty token rows of a small group.
//
// Why this shape: with 128 weight rows per tile and 64-deep k-steps, each
// 8 KB of int8 weights cost the MMA-issuing thread ~0.44 us (two barrier
// waits, four M = 128 MMAs, two commits; %globaltimer stamps at every
// hand-off), which held the weight stream near 3 TB/s.  Back to back on one
// SM an M = 128, N = 16 or 32 tcgen05.mma takes ~22.5 ns and a
// tcgen05.commit ~23 ns (measured), so at decode-sized N the per-k-step
// hand-offs, not the tensor core, set the pace.  Here a tile holds 256 weight
// rows (in SwiGLU mode the gate rows of 128 features and the matching up
// rows) and a k-step is KP = 2 k-blocks deep: 16 MMAs per hand-off for 32 KB
// of int8.  The widened bf16 weights go to tensor memory (tcgen05.mma takes
// its A operand from there) instead of shared memory, which leaves the
// shared memory to a raw ring of 4 x 32 KB.
//
//  * warp 0: TMA producer of the token tiles (TN rows x 64 KP, from L2);
//  * warp 6: TMA producer of the raw int8 weight tiles, KP boxes of 256 rows x
//    64 B per k-step, with the 64-byte swizzle (16-byte unit u of row r at
//    u ^ ((r >> 1) & 3)), so that threads reading one row each hit distinct
//    banks; in SwiGLU mode one 3-D box holds the 128 gate rows and the
//    matching 128 up rows;
//  * warps 7..: converters, NG groups of GW warps taking k-steps in turn.  In
//    a group, thread (warp w, lane l) owns weight row h * 128 + 32 (w % 4) + l
//    (h = bit 2 of the warp's index in the group) and KP * 8 / GW k-blocks:
//    it reads the row's int8 into registers, releases the raw stage, widens
//    them to bf16 (exact: |q| <= 127) and stores them, two per 32-bit column,
//    to TMEM lane 32 (w % 4) + l of the group's A stage -- a warp may only
//    reach the lane quarter w % 4, which this mapping respects;
//  * warp 1: TMEM allocator (512 columns) and MMA issuer: per 16-deep slice,
//    D1 += A_half0 * B and D2 += A_half1 * B with A from TMEM and the token
//    tile B from shared memory (M = 128, N = TN); accumulators
//    double-buffered in columns 0 .. 4 TN, the A stages after them;
//  * warps 2-5: epilogue, thread = TMEM lane f.  SwiGLU: the gate value of
//    feature f in D1 and its up value in D2, in the same lane, give
//    h[j, f] = silu(g s_g) * (u s_u) without an exchange; PLAIN: rows f and
//    128 + f.
// Every barrier a converter group waits on is waited on by that group alone,
// in order (ring depths multiples of NG): a parity wait cannot tell a phase
// from the one two uses back.  Every wait is bounded (1 s); a wait that runs
// out records MOE_ERR_TIMEOUT, the kernel drains its own copies and MMAs,
// frees TMEM and returns; waits followed by warp-collective tcgen05
// instructions take the same outcome in every lane.
#include "tc_common.cuh"
#include "tc_w8.cuh"

namespace moe {

namespace {

constexpr int DW_ROWS = 256;                          // weight rows per tile
constexpr int DW_KBLK_BYTES = DW_ROWS * TC_BK;        // int8 k-block of a tile: 16 KB
constexpr int DW_BAR_BYTES = 1024;
constexpr uint32_t DW_TMEM_COLS = 512;
// The configuration launched: two converter groups of 8 warps, 128-deep
// k-steps (two TMEM A stages of 128 columns, one per group; 4 raw stages of
// 32 KB).  Measured on the OLMoE int8 layer at T = 64 against the other
// shapes this template takes: one group of 16 warps (a thread per row and
// k-block) and 3 A stages: 137 us; one group of 8 warps, 3 stages: 134 us;
// 64-deep k-steps with 2 or 4 groups: 144 us; this one: 123 us.
constexpr int DW_NG = 2, DW_KP = 2, DW_GW = 8;

// KP 64-deep k-blocks per stage (a k-step); NG converter groups of GW warps
// (a thread per weight row and KP * 8 / GW k-blocks); accumulators in TMEM
// columns 0 .. 4 TN, then A stages of 64 KP columns (2 halves x 32 KP) as
// many as fit (a multiple of NG); as many raw stages (a multiple of NG, at
// most 32) as shared memory holds with G = 1024 groups.
template <int TN, int NG, int KP, int GW>
struct DwCfg {
    static constexpr int THREADS = 7 * 32 + NG * GW * 32;
    static constexpr int KPT = KP * 8 / GW;                  // k-blocks per converter thread
    static_assert(GW % 8 == 0 && KPT >= 1 && KPT * GW == KP * 8, "converter split");
    static constexpr int B_BYTES = TN * TC_BK * 2 * KP;      // token tile
    static constexpr int RAW_BYTES = DW_KBLK_BYTES * KP;     // raw int8 tile
    static constexpr uint32_t A_COL0 = 4 * TN < 32 ? 32 : 4 * TN;
    static constexpr uint32_t A_STAGE_COLS = 64 * KP;
    static constexpr int A_FIT = (DW_TMEM_COLS - A_COL0) / A_STAGE_COLS;
    static constexpr int STAGES = (A_FIT > 4 ? 4 : A_FIT) / NG * NG;    // A stages in TMEM
    static constexpr int TOK_STAGES = (TN <= 16 ? 16 : 8) / KP;
    static constexpr int RAW_FIT = (232448 - 1024 - TOK_STAGES * B_BYTES - DW_BAR_BYTES -
                                    2 * 1025 * 4) / RAW_BYTES;
    static constexpr int RAW_STAGES = (RAW_FIT > 32 ? 32 : RAW_FIT) / NG * NG;
    static_assert(RAW_STAGES >= 2 * NG && STAGES >= 2, "rings");
    static_assert(STAGES % NG == 0 && RAW_STAGES % NG == 0,
                  "each ring stage must belong to one converter group");
    static_assert(THREADS <= 1024, "block size");
    static_assert(A_COL0 + STAGES * A_STAGE_COLS <= DW_TMEM_COLS, "tensor-memory columns");
    static_assert((2 * (TOK_STAGES + STAGES + RAW_STAGES) + 5) * 8 + 8 <= DW_BAR_BYTES,
                  "barrier block");
    static constexpr size_t smem_bytes(int G) {
        return 1024 + static_cast<size_t>(TOK_STAGES) * B_BYTES +
               static_cast<size_t>(RAW_STAGES) * RAW_BYTES + DW_BAR_BYTES +
               2 * static_cast<size_t>(G + 1) * sizeof(int);
    }
    static_assert(smem_bytes(1024) <= 232448, "rings exceed shared memory");
};

// D[tmem] (+)= A[tmem] * B[smem]^T, bf16 inputs, fp32 accumulators.  A: M = 128
// rows in lanes 0-127, K along the columns, two bf16 per 32-bit column (the
// lower k in the low half).
__device__ __forceinline__ void tc_mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i writes lane (base + i).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

}  // namespace

// SWIGLU: out = h [M, NOUT=I], int8 weights [G*2I, K=H] (up rows at +UP_OFF = I).
// PLAIN : out = y [M, NOUT=H], int8 weights [G*H,  K=I].  scales: [G*R] fp32.
template <bool SWIGLU, int TN, int NG, int KP, int GW>
__global__ void __launch_bounds__(DwCfg<TN, NG, KP, GW>::THREADS, 1)
    tc_grouped_gemm_dec_w8(const __grid_constant__ CUtensorMap tm_tok,
                           const __grid_constant__ CUtensorMap tm_w,
                           const float *__restrict__ scales, const int32_t *__restrict__ offsets,
                           int G, int M, int K, int R, int NOUT, int UP_OFF,
                           uint16_t *__restrict__ out, int32_t *dev_error) {
    using C = DwCfg<TN, NG, KP, GW>;
    constexpr int S = C::STAGES;
    constexpr int TS = C::TOK_STAGES;
    constexpr int RS = C::RAW_STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sQ = smem;                                   // RS x RAW_BYTES (1024-aligned)
    uint8_t *sB = sQ + RS * C::RAW_BYTES;                 // TS x B_BYTES (multiples of 1024)
    uint64_t *bars = reinterpret_cast<uint64_t *>(sB + TS * C::B_BYTES);
    uint64_t *b_full = bars;                // token tile landed
    uint64_t *b_empty = b_full + TS;        // token tile consumed by the MMA
    uint64_t *a_full = b_empty + TS;        // A stage written to TMEM (one arrival per warp)
    uint64_t *a_empty = a_full + S;         // A stage consumed by the MMA
    uint64_t *q_full = a_empty + S;         // raw tile landed
    uint64_t *q_empty = q_full + RS;        // raw tile read (one arrival per warp)
    uint64_t *accf = q_empty + RS;
    uint64_t *acce = accf + 2;
    uint64_t *drain = acce + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    int *s_total = reinterpret_cast<int *>(tmem_slot + 1);
    int *s_off = reinterpret_cast<int *>(reinterpret_cast<uint8_t *>(bars) + DW_BAR_BYTES);
    int *s_tile = s_off + (G + 1);

    const int warp = threadIdx.x >> 5, lane = lane_id();
    const int n_per_tile = SWIGLU ? DW_ROWS / 2 : DW_ROWS;   // output features per tile
    const int n_tiles = (NOUT + n_per_tile - 1) / n_per_tile;
    const int KB = (K + TC_BK * KP - 1) / (TC_BK * KP);       // k-steps per tile

    if (threadIdx.x == 0) {
        for (int i = 0; i < TS; ++i) {
            mbar_init(&b_full[i], 1);
            mbar_init(&b_empty[i], 1);
        }
        for (int i = 0; i < S; ++i) {
            mbar_init(&a_full[i], GW);
            mbar_init(&a_empty[i], 1);
        }
        for (int i = 0; i < RS; ++i) {
            mbar_init(&q_full[i], 1);
            mbar_init(&q_empty[i], GW);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&accf[i], 1);
            mbar_init(&acce[i], 128);
        }
        mbar_init(drain, 1);
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tm_tok);
        prefetch_tmap(&tm_w);
    }
    if (warp == 1) tmem_alloc<DW_TMEM_COLS>(tmem_slot);
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
#pragma unroll
                    for (int kq = 0; kq < KP; ++kq)
                        tma_load_2d(sB + i * C::B_BYTES + kq * TN * 128, &tm_tok, &b_full[i],
                                    (kb * KP + kq) * TC_BK, ti.m0, pol);
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
        // ------------------------------------------------ raw int8 weight tiles (the HBM stream)
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            int i = 0;
            uint32_t ph = 0, filled = 0, fill_par = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const TileInfo ti = decode_tile(t, s_tile, s_off, G, TN);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&q_empty[i], ph ^ 1u, dev_error)) { ok = false; break; }
                    mbar_arrive_expect_tx(&q_full[i], C::RAW_BYTES);
#pragma unroll
                    for (int kq = 0; kq < KP; ++kq) {
                        uint8_t *dst = sQ + i * C::RAW_BYTES + kq * DW_KBLK_BYTES;
                        const int kx = (kb * KP + kq) * TC_BK;
                        if (SWIGLU)  // 128 gate rows then the 128 matching up rows, one copy
                            tma_load_3d(dst, &tm_w, &q_full[i], kx, ti.nt * n_per_tile, 2 * ti.g,
                                        pol);
                        else
                            tma_load_2d(dst, &tm_w, &q_full[i], kx, ti.g * R + ti.nt * n_per_tile,
                                        pol);
                    }
                    filled |= 1u << i;
                    fill_par = (fill_par & ~(1u << i)) | (ph << i);
                    if (++i == RS) { i = 0; ph ^= 1u; }
                }
            }
            for (int j = 0; j < RS; ++j)
                if ((filled >> j) & 1u) mbar_wait(&q_full[j], (fill_par >> j) & 1u, dev_error);
        }
        __syncwarp();
    } else if (warp >= 7) {
        // ------------------------------------------------ converters int8 -> bf16 in TMEM
        // seq % NG picks the group; with both ring depths multiples of NG,
        // group c always owns the stages congruent to c.
        constexpr int KPT = C::KPT;
        const int grp = (warp - 7) / GW, wi = (warp - 7) % GW;
        const int quarter = warp & 3;                  // the TMEM lanes this warp may reach
        const int half = (wi >> 2) & 1;                // weight rows 0-127 or 128-255
        const int kq0 = (wi >> 3) * KPT;               // this thread's first k-block
        const int rho = half * 128 + quarter * 32 + lane;    // row within the raw tile
        const int rsw = (rho >> 1) & 3;                // its 64-byte swizzle
        const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                               C::A_COL0 + static_cast<uint32_t>(half * 32 * KP);
        int seq = 0;                                   // this CTA's k-step counter
        bool ok = true;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
            for (int kb = 0; kb < KB; ++kb, ++seq) {
                if (seq % NG != grp) continue;
                const int s = seq % S, r = seq % RS;
                const uint32_t sph = (seq / S) & 1, rph = (seq / RS) & 1;
                if (!mbar_wait_warp(&q_full[r], rph, dev_error)) { ok = false; break; }
                const uint8_t *row = sQ + r * C::RAW_BYTES + kq0 * DW_KBLK_BYTES + rho * TC_BK;
                uint4 v[4 * KPT];
#pragma unroll
                for (int p = 0; p < 4 * KPT; ++p)
                    v[p] = *reinterpret_cast<const uint4 *>(row + (p >> 2) * DW_KBLK_BYTES +
                                                            (((p & 3) ^ rsw) << 4));
                const uint32_t done = loads_done(v);   // 0, once the loads have landed
                __syncwarp();
                if (lane == 0) mbar_arrive(&q_empty[r + done]);   // the warp's rows are in registers
                if (!mbar_wait_warp(&a_empty[s], sph ^ 1u, dev_error)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int kq = 0; kq < KPT; ++kq) {
                    uint32_t a[32];
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        uint4 lo, hi;
                        widen16(v[4 * kq + p], lo, hi);
                        a[8 * p + 0] = lo.x; a[8 * p + 1] = lo.y; a[8 * p + 2] = lo.z;
                        a[8 * p + 3] = lo.w; a[8 * p + 4] = hi.x; a[8 * p + 5] = hi.y;
                        a[8 * p + 6] = hi.z; a[8 * p + 7] = hi.w;
                    }
                    tmem_st32(t_row + static_cast<uint32_t>(s) * C::A_STAGE_COLS +
                                  static_cast<uint32_t>((kq0 + kq) * 32), a);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&a_full[s]);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        // D1 = rows 0-127 of the weight tile, D2 = rows 128-255, both against
        // the same token tile; A from TMEM, 8 columns per 16-deep slice.
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, TN);
            int s = 0, tb = 0, acc = 0;
            uint32_t ph = 0, tph = 0, acc_ph = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                if (!mbar_wait(&acce[acc], acc_ph ^ 1u, dev_error)) break;
                tc_fence_after();
                const uint32_t d1 = tmem_base + static_cast<uint32_t>(acc * 2 * TN);
                const uint32_t d2 = d1 + TN;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&a_full[s], ph, dev_error) ||
                        !mbar_wait(&b_full[tb], tph, dev_error)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a1 =
                        tmem_base + C::A_COL0 + static_cast<uint32_t>(s) * C::A_STAGE_COLS;
                    const uint32_t b_addr = smem_u32(sB + tb * C::B_BYTES);
#pragma unroll
                    for (int kq = 0; kq < KP; ++kq)
#pragma unroll
                        for (int kk = 0; kk < TC_BK / 16; ++kk) {
                            const uint64_t bd = sw128_kmajor_desc(b_addr + kq * TN * 128 + kk * 32);
                            const uint32_t accum = (kb > 0 || kq > 0 || kk > 0) ? 1u : 0u;
                            const uint32_t ak = a1 + static_cast<uint32_t>(kq * 32 + kk * 8);
                            tc_mma_bf16_ts(d1, ak, bd, idesc, accum);
                            tc_mma_bf16_ts(d2, ak + 32 * KP, bd, idesc, accum);
                        }
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
        const int f = quarter * 32 + lane;            // row within each 128-row half
        int acc = 0;
        uint32_t acc_ph = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x) {
            const TileInfo ti = decode_tile(t, s_tile, s_off, G, TN);
            if (!mbar_wait_warp(&accf[acc], acc_ph, dev_error)) break;
            tc_fence_after();
            const uint32_t taddr =
                tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * 2 * TN;
            const int nrows = ti.nrows;
            const int64_t srow = static_cast<int64_t>(ti.g) * R;
            const int i = ti.nt * 128 + f;             // SwiGLU: intermediate index
            float sg = 0.0f, su = 0.0f;
            if (SWIGLU && i < NOUT) {
                sg = scales[srow + i];
                su = scales[srow + UP_OFF + i];
            }
            // 16 token columns at a time; the accumulators are released
            // after the last TMEM load, before the last stores
#pragma unroll
            for (int c = 0; c < TN; c += 16) {
                uint32_t v[16], w[16];
                tmem_ld16(taddr + c, v);
                tmem_ld16(taddr + TN + c, w);
                tmem_ld_wait();
                if (c + 16 == TN) {
                    tc_fence_before();
                    mbar_arrive(&acce[acc]);           // accumulators free for the next tile
                }
                if (SWIGLU) {
                    if (i < NOUT) {
                        uint16_t *col = out + static_cast<int64_t>(ti.m0 + c) * NOUT + i;
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            if (c + j < nrows) {
                                const float hv = silu_fast(__uint_as_float(v[j]) * sg) *
                                                 (__uint_as_float(w[j]) * su);
                                const __nv_bfloat16 b = __float2bfloat16_rn(hv);
                                col[static_cast<int64_t>(j) * NOUT] =
                                    *reinterpret_cast<const uint16_t *>(&b);
                            }
                        }
                    }
                } else {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int n = ti.nt * DW_ROWS + h * 128 + f;
                        if (n < NOUT) {
                            const float sc = scales[srow + n];
                            uint16_t *col = out + static_cast<int64_t>(ti.m0 + c) * NOUT + n;
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                if (c + j < nrows) {
                                    const float d = __uint_as_float(h ? w[j] : v[j]);
                                    const __nv_bfloat16 b = __float2bfloat16_rn(d * sc);
                                    col[static_cast<int64_t>(j) * NOUT] =
                                        *reinterpret_cast<const uint16_t *>(&b);
                                }
                            }
                        }
                    }
                }
            }
            acc ^= 1;
            if (acc == 0) acc_ph ^= 1u;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<DW_TMEM_COLS>(tmem_base);
    }
}

// ------------------------------------------------------------------ host


template <bool SWIGLU, int TN, int NG, int KP, int GW>
static moe_status launch_dw(const void *tok, const void *q, const float *scales,
                            const int32_t *offsets, int G, int M, int K, int R, int NOUT,
                            int UP_OFF, uint16_t *out, int32_t *dev_error, cudaStream_t stream) {
    using C = DwCfg<TN, NG, KP, GW>;
    CUtensorMap tm_tok, tm_w;
    if (!encode_bf16_2d(&tm_tok, tok, K, M, TN)) return MOE_ERR_CUDA;
    if (SWIGLU ? !encode_u8_sw64(&tm_w, q, K, UP_OFF, 2 * static_cast<uint64_t>(G), true,
                                 DW_ROWS / 2)
               : !encode_u8_sw64(&tm_w, q, K, static_cast<uint64_t>(G) * R, 1, false, DW_ROWS))
        return MOE_ERR_CUDA;
    const size_t smem = C::smem_bytes(G);
    if (smem > static_cast<size_t>(max_smem_optin())) return MOE_ERR_UNSUPPORTED;
    static int attr_done[64] = {0};
    if (!raise_smem_limit(tc_grouped_gemm_dec_w8<SWIGLU, TN, NG, KP, GW>, attr_done))
        return MOE_ERR_CUDA;
    launch(tc_grouped_gemm_dec_w8<SWIGLU, TN, NG, KP, GW>, sm_count(), C::THREADS, smem, stream,
           tm_tok, tm_w, scales, offsets, G, M, K, R, NOUT, UP_OFF, out, dev_error);
    return launch_status();
}

// Token-block height TN (16, 32 or 64) for the 256-row int8 weight tiles.
template <bool SWIGLU>
moe_status launch_dec_w8(int tn, const void *tok, const void *q, const float *scales,
                         const int32_t *offsets, int G, int M, int K, int R, int NOUT, int UP_OFF,
                         uint16_t *out, int32_t *dev_error, cudaStream_t stream) {
    if (tn == 16)
        return launch_dw<SWIGLU, 16, DW_NG, DW_KP, DW_GW>(tok, q, scales, offsets, G, M, K, R, NOUT,
                                                          UP_OFF, out, dev_error, stream);
    if (tn == 32)
        return launch_dw<SWIGLU, 32, DW_NG, DW_KP, DW_GW>(tok, q, scales, offsets, G, M, K, R,
                                                          NOUT, UP_OFF, out, dev_error, stream);
    return launch_dw<SWIGLU, 64, DW_NG, DW_KP, DW_GW>(tok, q, scales, offsets, G, M, K, R, NOUT,
                                                      UP_OFF, out, dev_error, stream);
}

template moe_status launch_dec_w8<true>(int, const void *, const void *, const float *,
                                        const int32_t *, int, int, int, int, int, int, uint16_t *,
                                        int32_t *, cudaStream_t);
template moe_status launch_dec_w8<false>(int, const void *, const void *, const float *,
                                         const int32_t *, int, int, int, int, int, int, uint16_t *,
                                         int32_t *, cudaStream_t);

}  // namespace moe
