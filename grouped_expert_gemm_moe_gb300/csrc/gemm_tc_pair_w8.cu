// gemm_tc_pair_w8.cu -- int8 weight-only grouped GEMM on CTA pairs, for
// prefill-sized expert groups.
//
// Per-channel int8 weights with fp32 scales and bf16 activations ("dispatch"
// README, phase 5a), all experts in one launch with SwiGLU in the gate/up
// epilogue ("switchyard" page, 02 Kernels and dispatch, "One launch for all
// experts").  The tile shape is that of the bf16 pair kernel
// (gemm_tc_pair.cu): the MMA's M is 256 weight rows (128 per SM of the
// cluster pair), its N a block of at most 192 of the group's tokens (rounded
// up to 16), a k-step two 64-deep k-blocks.  The weights reach the tensor
// core as its A operand from tensor memory:
//
//  * warp 6 (each CTA) streams the CTA's 128 raw int8 weight rows, two
//    k-blocks per copy (64-byte swizzle), into a ring of its own shared
//    memory, completing on its own barrier;
//  * warps 7-14 (each CTA): two converter groups of 4 warps take k-steps in
//    turn; thread = TMEM lane = one weight row: it reads the row's 128 int8,
//    releases the raw stage, widens them to bf16 (exact) in registers, and
//    only then waits for its group's A stage and writes them there with
//    tcgen05.st, so that between the tensor core's release of a stage and
//    its refill lie two stores; CTA 0's converters also wait for
//    the k-step's token stage, so the MMA thread waits on one barrier per 8
//    MMAs; CTA 1's converters signal CTA 0's barrier across the cluster;
//  * warp 0 (each CTA) brings the CTA's half of the tokens (two k-blocks per
//    copy), completing on CTA 0's stage barrier, as in the bf16 pair kernel;
//  * warp 1 (CTA 0) issues tcgen05.mma.cta_group::2 with A from each CTA's
//    tensor memory and B from shared memory; the tensor cores of both SMs
//    run it, each CTA's TMEM receiving its 128 weight rows by N tokens;
//  * warps 2-5 (each CTA): epilogue, lane = weight row: the accumulator
//    times the row's scale, SwiGLU between lanes 8 apart (a CTA's 128 rows
//    are 64 features as 8 slices of 8 gate rows then their 8 up rows, the
//    converters choosing which raw row each lane takes), transposed through
//    1 KB of shared memory per warp into whole row segments of the output.
//
// Only the tokens are read by both SMs' tensor cores (TMA, async proxy);
// each SM's A operand is its own tensor memory, written by its own threads.
// Tensor memory per CTA: two accumulators of 192 columns, two A stages of
// 64 columns (one per converter group).  Every barrier a converter group
// waits on is waited on by that group alone, in order (the raw ring's depth
// is a multiple of the group count).  Every wait is bounded (1 s): on
// running out the kernel records MOE_ERR_TIMEOUT, stops issuing, drains what
// it can observe and meets its peer at the closing cluster barrier before
// freeing TMEM.
#include <algorithm>

#include "tc_common.cuh"
#include "tc_pair.cuh"
#include "tc_w8.cuh"

namespace moe {

namespace {

constexpr int PW_MAX_N = 192;                   // tokens per tile (MMA N)
constexpr int PW_W_ROWS = 256;                  // weight rows per tile (MMA M)
constexpr int PW_KB = 2;                        // 64-deep k-blocks per k-step
constexpr int PW_RAW_BYTES = PW_KB * 128 * TC_BK;            // 128 rows x 128 int8: 16 KB
constexpr int PW_TOK_BYTES = PW_KB * (PW_MAX_N / 2) * TC_BK * 2;   // 96 rows: 24 KB
constexpr int PW_RAW_STAGES = 6;                // a multiple of PW_NG
constexpr int PW_TOK_STAGES = 4;                // a multiple of PW_NG
constexpr int PW_NG = 2;                        // converter groups
constexpr int PW_A_STAGES = 2;                  // A stages, a multiple of PW_NG
constexpr uint32_t PW_A_COL0 = 2 * PW_MAX_N;   // A stages after the two accumulators
constexpr uint32_t PW_A_COLS = 32 * PW_KB;      // 128 bf16 per lane = 64 columns
constexpr uint32_t PW_TMEM_COLS = 512;
constexpr int PW_BAR_BYTES = 512;
constexpr int PW_EPI_WARPS = 4;
constexpr int PW_STAGING_BYTES = 1024;
constexpr int PW_XMAPS = PW_MAX_N / 32;          // token boxes of 16 .. 96 rows
constexpr int PW_MY_MAX = 128;
constexpr int PW_THREADS = (7 + 4 * PW_NG) * 32;   // 15 warps

static_assert(PW_RAW_STAGES % PW_NG == 0 && PW_TOK_STAGES % PW_NG == 0 &&
                  PW_A_STAGES % PW_NG == 0,
              "each ring stage must belong to one converter group");
static_assert(PW_A_COL0 + PW_A_STAGES * PW_A_COLS <= PW_TMEM_COLS, "tensor-memory columns");
static_assert((2 * (PW_RAW_STAGES + PW_TOK_STAGES + PW_A_STAGES) + 5) * 8 + 8 <= PW_BAR_BYTES,
              "barrier block");

// D (+)= A[tmem] * B[smem]^T on the CTA pair (A: each CTA's 128 rows at the
// same tensor-memory address).
__device__ __forceinline__ void tc_mma_pair_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tmem_st32_pw(uint32_t taddr, const uint32_t (&r)[32]) {
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

__device__ __forceinline__ void tmem_st_wait_pw() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// A group of `rows` tokens in balanced m-blocks of at most PW_MAX_N (sizes a
// multiple of 16, none empty).
__device__ __forceinline__ int pw_mblocks(int rows, int &bs) {
    const int nmb0 = (rows + PW_MAX_N - 1) / PW_MAX_N;
    bs = nmb0 > 0 ? (((rows + nmb0 - 1) / nmb0 + 15) & ~15) : PW_MAX_N;
    if (bs > PW_MAX_N) bs = PW_MAX_N;
    return nmb0 > 0 ? (rows + bs - 1) / bs : 0;
}

__device__ __forceinline__ void build_pw_table(const int32_t *offsets, int G, int M, int n_tiles,
                                               int *s_off, int *s_tile, int *s_total,
                                               int32_t *dev_error) {
    const int lane = lane_id();
    int carry = 0;
    bool bad = false;
    for (int base = 0; base < G; base += 32) {
        const int g = base + lane;
        int tiles = 0;
        if (g < G) {
            const int o0 = offsets[g], o1 = offsets[g + 1];
            if (o0 < 0 || o1 < o0 || o1 > M) {
                bad = true;
            } else {
                int bs;
                tiles = pw_mblocks(o1 - o0, bs) * n_tiles;
            }
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

__device__ __forceinline__ TileInfo decode_pw_tile(int t, const int *s_tile, const int *s_off,
                                                   int G) {
    int lo = 0, hi = G - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_tile[mid] <= t) lo = mid;
        else hi = mid - 1;
    }
    TileInfo ti;
    ti.g = lo;
    const int rows = s_off[lo + 1] - s_off[lo];
    int bs;
    const int nmb = pw_mblocks(rows, bs);
    const int u = t - s_tile[lo];
    ti.nt = u / nmb;
    const int mb = u - ti.nt * nmb;
    ti.m0 = s_off[lo] + mb * bs;
    ti.nrows = min(bs, rows - mb * bs);
    return ti;
}

}  // namespace

struct PairW8TokenMaps {
    CUtensorMap m[PW_XMAPS];
};

// SWIGLU: out = h [M, NOUT = I]; q [G, 2, I, K] int8 through a 4-D map
//         (k in block, row, gate/up plane 2g + s, k-block); scales [G * 2I].
// PLAIN : out = y [M, NOUT = H]; q [G * H, K] int8 through a 3-D map
//         (k in block, row, k-block); scales [G * H].
template <bool SWIGLU>
__global__ void __launch_bounds__(PW_THREADS, 1)
    tc_grouped_gemm_pair_w8(const __grid_constant__ PairW8TokenMaps tm_x,
                            const __grid_constant__ CUtensorMap tm_q,
                            const float *__restrict__ scales, const int32_t *__restrict__ offsets,
                            int G, int M, int K, int R, int NOUT, int UP_OFF,
                            uint16_t *__restrict__ out, int32_t *dev_error) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sQ = smem;                                        // raw int8 ring (own CTA)
    uint8_t *sX = sQ + PW_RAW_STAGES * PW_RAW_BYTES;           // token ring (B operand)
    uint8_t *staging = sX + PW_TOK_STAGES * PW_TOK_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(staging + PW_EPI_WARPS * PW_STAGING_BYTES);
    uint64_t *b_full = bars;                     // CTA 0: both CTAs' token copies
    uint64_t *b_empty = b_full + PW_TOK_STAGES;  // both CTAs: MMA commit (multicast)
    uint64_t *q_full = b_empty + PW_TOK_STAGES;  // own raw copy landed
    uint64_t *q_empty = q_full + PW_RAW_STAGES;  // own raw stage read (one arrival per warp)
    uint64_t *a_full = q_empty + PW_RAW_STAGES;  // CTA 0: A stage written in both CTAs
    uint64_t *a_empty = a_full + PW_A_STAGES;    // both CTAs: MMA commit (multicast)
    uint64_t *accf = a_empty + PW_A_STAGES;
    uint64_t *acce = accf + 2;
    uint64_t *drain = acce + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    int *s_total = reinterpret_cast<int *>(tmem_slot + 1);
    int4 *s_my = reinterpret_cast<int4 *>(reinterpret_cast<uint8_t *>(bars) + PW_BAR_BYTES);
    int *s_off = reinterpret_cast<int *>(s_my + PW_MY_MAX);
    int *s_tile = s_off + (G + 1);

    const int warp = threadIdx.x >> 5, lane = lane_id();
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    const int n_per_tile = SWIGLU ? PW_W_ROWS / 2 : PW_W_ROWS;
    const int n_tiles = (NOUT + n_per_tile - 1) / n_per_tile;
    const int KB = K / TC_BK;
    const int KS = (KB + PW_KB - 1) / PW_KB;

    if (threadIdx.x == 0) {
        for (int i = 0; i < PW_TOK_STAGES; ++i) {
            mbar_init(&b_full[i], 1);
            mbar_init(&b_empty[i], 1);
        }
        for (int i = 0; i < PW_RAW_STAGES; ++i) {
            mbar_init(&q_full[i], 1);
            mbar_init(&q_empty[i], 4);               // the group's 4 warps
        }
        for (int i = 0; i < PW_A_STAGES; ++i) {
            mbar_init(&a_full[i], 2 * 4);            // the group's warps of both CTAs
            mbar_init(&a_empty[i], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accf[b], 1);
            mbar_init(&acce[b], 2 * PW_EPI_WARPS);
        }
        mbar_init(drain, 1);
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        for (int i = 0; i < PW_XMAPS; ++i) prefetch_tmap(&tm_x.m[i]);
        prefetch_tmap(&tm_q);
    }
    if (warp == 1) tmem_alloc_pair<PW_TMEM_COLS>(tmem_slot);
    pdl_wait();
    pdl_trigger();
    if (warp == 2) build_pw_table(offsets, G, M, n_tiles, s_off, s_tile, s_total, dev_error);
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int total = *s_total;
    const int t_first = static_cast<int>(cluster_id_x());
    const int t_step = static_cast<int>(cluster_count_x());
    if (warp == 2)
        for (int i = lane; i < PW_MY_MAX; i += 32) {
            const int t = t_first + i * t_step;
            if (t < total) {
                const TileInfo ti = decode_pw_tile(t, s_tile, s_off, G);
                s_my[i] = make_int4(ti.g, ti.nt, ti.m0, ti.nrows);
            }
        }
    __syncthreads();
    auto tile_of = [&](int i, int t) -> TileInfo {
        if (i < PW_MY_MAX) {
            const int4 v = s_my[i];
            return TileInfo{v.x, v.y, v.z, v.w};
        }
        return decode_pw_tile(t, s_tile, s_off, G);
    };

    if (warp == 0) {
        // ------------------------------------------- token producer (each CTA)
        if (lane == 0) {
            const uint64_t pol = policy_evict_last();
            int s = 0;
            uint32_t ph = 0, filled = 0, fill_par = 0;
            bool ok = true;
            for (int t = t_first, i = 0; t < total && ok; t += t_step, ++i) {
                const TileInfo ti = tile_of(i, t);
                const int half = ((ti.nrows + 15) & ~15) >> 1;
                const int box = (half + 15) & ~15;
                const int my_cnt = leader ? min(ti.nrows, half) : ti.nrows - half;
                const CUtensorMap *tm = &tm_x.m[box / 16 - 1];
                const uint32_t bytes =
                    static_cast<uint32_t>((ti.nrows > half ? 2 : 1) * box * TC_BK * 2 * PW_KB);
                const int xrow = ti.m0 + static_cast<int>(rank) * half;
                for (int ks = 0; ks < KS; ++ks) {
                    if (!mbar_wait(&b_empty[s], ph ^ 1u, dev_error)) { ok = false; break; }
                    const uint32_t bar0 = map_to_rank(smem_u32(&b_full[s]), 0);
                    if (leader) {
                        mbar_arrive_expect_tx(&b_full[s], bytes);
                        filled |= 1u << s;
                        fill_par = (fill_par & ~(1u << s)) | (ph << s);
                    }
                    if (my_cnt > 0)
                        tma_load_3d_pair(sX + s * PW_TOK_BYTES, tm, bar0, 0, xrow, ks * PW_KB,
                                         pol);
                    if (++s == PW_TOK_STAGES) { s = 0; ph ^= 1u; }
                }
            }
            for (int j = 0; j < PW_TOK_STAGES; ++j)
                if ((filled >> j) & 1u) mbar_wait(&b_full[j], (fill_par >> j) & 1u, dev_error);
        }
        __syncwarp();
    } else if (warp == 6) {
        // ------------------------------------------- raw int8 producer (each CTA)
        if (lane == 0) {
            uint64_t pol;
            asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
            int r = 0;
            uint32_t ph = 0, filled = 0, fill_par = 0;
            bool ok = true;
            for (int t = t_first, i = 0; t < total && ok; t += t_step, ++i) {
                const TileInfo ti = tile_of(i, t);
                const int wrow = SWIGLU ? ti.nt * n_per_tile + static_cast<int>(rank) * 64
                                        : ti.g * R + ti.nt * n_per_tile + static_cast<int>(rank) * 128;
                for (int ks = 0; ks < KS; ++ks) {
                    if (!mbar_wait(&q_empty[r], ph ^ 1u, dev_error)) { ok = false; break; }
                    mbar_arrive_expect_tx(&q_full[r], PW_RAW_BYTES);
                    if (SWIGLU)
                        tma_load_4d(sQ + r * PW_RAW_BYTES, &tm_q, &q_full[r], 0, wrow, 2 * ti.g,
                                    ks * PW_KB, pol);
                    else
                        tma_load_3d(sQ + r * PW_RAW_BYTES, &tm_q, &q_full[r], 0, wrow, ks * PW_KB,
                                    pol);
                    filled |= 1u << r;
                    fill_par = (fill_par & ~(1u << r)) | (ph << r);
                    if (++r == PW_RAW_STAGES) { r = 0; ph ^= 1u; }
                }
            }
            for (int j = 0; j < PW_RAW_STAGES; ++j)
                if ((filled >> j) & 1u) mbar_wait(&q_full[j], (fill_par >> j) & 1u, dev_error);
        }
        __syncwarp();
    } else if (warp >= 7) {
        // ------------------------------------------- converters int8 -> bf16 in TMEM
        const int grp = (warp - 7) / 4;
        const int quarter = warp & 3;                 // the TMEM lanes this warp may reach
        // lane -> raw row: SwiGLU lanes of a warp are 16 features, 8 gate rows
        // then their 8 up rows twice; the raw box holds 64 gate rows then the
        // 64 matching up rows
        const int rho = SWIGLU ? ((lane >> 3) & 1) * 64 + 16 * quarter + 8 * (lane >> 4) + (lane & 7)
                               : 32 * quarter + lane;
        const int rsw = (rho >> 1) & 3;
        const uint32_t a_lane = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + PW_A_COL0;
        const uint32_t a_full0 = map_to_rank(smem_u32(&a_full[0]), 0);
        int seq = 0;
        bool ok = true;
        for (int t = t_first; t < total && ok; t += t_step) {
            for (int ks = 0; ks < KS; ++ks, ++seq) {
                if (seq % PW_NG != grp) continue;
                const int r = seq % PW_RAW_STAGES, tb = seq % PW_TOK_STAGES;
                const int s = seq % PW_A_STAGES;
                const uint32_t rph = (seq / PW_RAW_STAGES) & 1;
                const uint32_t tph = (seq / PW_TOK_STAGES) & 1;
                const uint32_t aph = (seq / PW_A_STAGES) & 1;
                if (!mbar_wait_warp(&q_full[r], rph, dev_error)) { ok = false; break; }
                uint4 v[4 * PW_KB];
#pragma unroll
                for (int p = 0; p < 4 * PW_KB; ++p)
                    v[p] = *reinterpret_cast<const uint4 *>(
                        sQ + r * PW_RAW_BYTES + (p >> 2) * (128 * TC_BK) + rho * TC_BK +
                        (((p & 3) ^ rsw) << 4));
                const uint32_t done = loads_done(v);     // 0, once the loads have landed
                __syncwarp();
                if (lane == 0) mbar_arrive(&q_empty[r + done]);
                uint32_t a[PW_KB][32];
#pragma unroll
                for (int kb = 0; kb < PW_KB; ++kb)
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        uint4 lo, hi;
                        widen16(v[4 * kb + p], lo, hi);
                        a[kb][8 * p + 0] = lo.x; a[kb][8 * p + 1] = lo.y; a[kb][8 * p + 2] = lo.z;
                        a[kb][8 * p + 3] = lo.w; a[kb][8 * p + 4] = hi.x; a[kb][8 * p + 5] = hi.y;
                        a[kb][8 * p + 6] = hi.z; a[kb][8 * p + 7] = hi.w;
                    }
                if (!mbar_wait_warp(&a_empty[s], aph ^ 1u, dev_error)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int kb = 0; kb < PW_KB; ++kb)
                    tmem_st32_pw(a_lane + static_cast<uint32_t>(s) * PW_A_COLS +
                                     static_cast<uint32_t>(kb * 32), a[kb]);
                tmem_st_wait_pw();
                // CTA 0's converters also hold the signal until the k-step's
                // token stage (both CTAs' copies) has landed, so the MMA
                // thread waits on this barrier alone
                if (leader && !mbar_wait_warp(&b_full[tb], tph, dev_error)) { ok = false; break; }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(a_full0 + static_cast<uint32_t>(s * 8));
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------- MMA issuer (CTA 0 only)
        if (leader && lane == 0) {
            int tb = 0, acc = 0, seq = 0;
            uint32_t acc_ph = 0;
            bool ok = true;
            const uint64_t dX = sw128_kmajor_desc(smem_u32(sX));
            for (int t = t_first, i = 0; t < total && ok; t += t_step, ++i) {
                const int n = (tile_of(i, t).nrows + 15) & ~15;
                const uint32_t idesc = idesc_bf16_f32(PW_W_ROWS, n);
                const uint32_t xkb1 = static_cast<uint32_t>((((n >> 1) + 15) & ~15) * TC_BK * 2);
                if (!mbar_wait(&acce[acc], acc_ph ^ 1u, dev_error)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * PW_MAX_N);
                for (int ks = 0; ks < KS; ++ks, ++seq) {
                    const int s = seq % PW_A_STAGES;
                    if (!mbar_wait(&a_full[s], (seq / PW_A_STAGES) & 1, dev_error)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = tmem_base + PW_A_COL0 + static_cast<uint32_t>(s) * PW_A_COLS;
                    const uint64_t db = dX + ((tb * PW_TOK_BYTES) >> 4);
#pragma unroll
                    for (int kk = 0; kk < TC_BK / 16; ++kk)
                        tc_mma_pair_ts(d_tmem, a0 + kk * 8, db + 2 * kk, idesc,
                                       (ks > 0 || kk > 0) ? 1u : 0u);
                    if (ks * PW_KB + 1 < KB) {
#pragma unroll
                        for (int kk = 0; kk < TC_BK / 16; ++kk)
                            tc_mma_pair_ts(d_tmem, a0 + 32 + kk * 8, db + ((xkb1 >> 4) + 2 * kk),
                                           idesc, 1u);
                    }
                    tc_commit_pair_both(&a_empty[s]);
                    tc_commit_pair_both(&b_empty[tb]);
                    if (++tb == PW_TOK_STAGES) tb = 0;
                }
                if (!ok) break;
                tc_commit_pair_both(&accf[acc]);
                acc ^= 1;
                if (acc == 0) acc_ph ^= 1u;
            }
            tc_commit_pair_local(drain);
            mbar_wait(drain, 0, dev_error);
        }
        __syncwarp();
    } else {
        // ------------------------------------------- epilogue (warps 2..5, each CTA)
        const int quarter = warp & 3;
        uint8_t *stg = staging + (warp - 2) * PW_STAGING_BYTES;
        const uint32_t acce0 = map_to_rank(smem_u32(&acce[0]), 0);
        const uint32_t acce1 = map_to_rank(smem_u32(&acce[1]), 0);
        int acc = 0;
        uint32_t acc_ph = 0;
        for (int t = t_first, i = 0; t < total; t += t_step, ++i) {
            const TileInfo ti = tile_of(i, t);
            if (!mbar_wait_warp(&accf[acc], acc_ph, dev_error)) break;
            tc_fence_after();
            const uint32_t tbase =
                tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * PW_MAX_N;
            const int64_t srow = static_cast<int64_t>(ti.g) * R;
            if (SWIGLU) {
                const bool is_up = (lane >> 3) & 1;
                const int fcol = 8 * (lane >> 4) + (lane & 7);
                const int f_warp = ti.nt * n_per_tile + static_cast<int>(rank) * 64 + 16 * quarter;
                const int f = f_warp + fcol;
                const float sc = f < NOUT ? scales[srow + (is_up ? UP_OFF : 0) + f] : 0.0f;
                const int rt = lane >> 1, rf = 8 * (lane & 1);
                const bool f_ok = f_warp + rf < NOUT;
#pragma unroll 1
                for (int c0 = 0; c0 < ti.nrows; c0 += 16) {
                    uint32_t v[16];
                    tmem_ld16(tbase + c0, v);
                    tmem_ld_wait();
                    uint16_t *hs = reinterpret_cast<uint16_t *>(stg);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float mine = __uint_as_float(is_up ? v[j] : v[8 + j]) * sc;
                        const float other = __shfl_xor_sync(FULL, mine, 8);
                        const float g = is_up ? other : __uint_as_float(v[j]) * sc;
                        const float u = is_up ? __uint_as_float(v[8 + j]) * sc : other;
                        hs[(8 * is_up + j) * 16 + fcol] =
                            __bfloat16_as_ushort(__float2bfloat16_rn(silu_fast(g) * u));
                    }
                    __syncwarp();
                    const uint4 val = *reinterpret_cast<const uint4 *>(hs + rt * 16 + rf);
                    if (c0 + rt < ti.nrows && f_ok)
                        *reinterpret_cast<uint4 *>(
                            out + static_cast<int64_t>(ti.m0 + c0 + rt) * NOUT + f_warp + rf) = val;
                    __syncwarp();
                }
            } else {
                const int n_warp = ti.nt * n_per_tile + static_cast<int>(rank) * 128 + 32 * quarter;
                const float sc = n_warp + lane < NOUT ? scales[srow + n_warp + lane] : 0.0f;
#pragma unroll 1
                for (int c0 = 0; c0 < ti.nrows; c0 += 16) {
                    uint32_t v[16];
                    tmem_ld16(tbase + c0, v);
                    tmem_ld_wait();
                    uint16_t *ys = reinterpret_cast<uint16_t *>(stg);
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        ys[j * 32 + lane] =
                            __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[j]) * sc));
                    __syncwarp();
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const int id = lane + 32 * q;
                        const int rt = id >> 2, rf = 8 * (id & 3);
                        const uint4 val = *reinterpret_cast<const uint4 *>(ys + rt * 32 + rf);
                        if (c0 + rt < ti.nrows && n_warp + rf < NOUT)
                            *reinterpret_cast<uint4 *>(
                                out + static_cast<int64_t>(ti.m0 + c0 + rt) * NOUT + n_warp + rf) =
                                val;
                    }
                    __syncwarp();
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(acc == 0 ? acce0 : acce1);
            acc ^= 1;
            if (acc == 0) acc_ph ^= 1u;
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair<PW_TMEM_COLS>(tmem_base);
    }
}

// ------------------------------------------------------------------ host

static size_t pw_smem_bytes(int G) {
    return 1024 + static_cast<size_t>(PW_RAW_STAGES) * PW_RAW_BYTES +
           static_cast<size_t>(PW_TOK_STAGES) * PW_TOK_BYTES + PW_EPI_WARPS * PW_STAGING_BYTES +
           PW_BAR_BYTES + PW_MY_MAX * sizeof(int4) + 2 * static_cast<size_t>(G + 1) * sizeof(int);
}

static bool encode_map(CUtensorMap *map, CUtensorMapDataType type, CUtensorMapSwizzle swz,
                       const void *base, int rank, const cuuint64_t *dims,
                       const cuuint64_t *strides, const cuuint32_t *box) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return enc(map, type, rank, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// K a multiple of 64 (whole k-blocks); otherwise MOE_ERR_UNSUPPORTED (the
// caller takes another tile kernel).
template <bool SWIGLU>
moe_status launch_tc_pair_w8(const void *act, const int8_t *q, const float *scales,
                             const int32_t *offsets, int G, int M, int K, int R, int NOUT,
                             int UP_OFF, uint16_t *out, int32_t *dev_error, cudaStream_t stream) {
    if (K % TC_BK != 0 || NOUT % 8 != 0) return MOE_ERR_UNSUPPORTED;
    const uint64_t K64 = static_cast<uint64_t>(K) / TC_BK;
    PairW8TokenMaps tm_x;
    for (int i = 0; i < PW_XMAPS; ++i) {
        const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(M), K64};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, 128};
        const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(16 * (i + 1)), 2};
        if (!encode_map(&tm_x.m[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, CU_TENSOR_MAP_SWIZZLE_128B,
                        act, 3, dims, strides, box))
            return MOE_ERR_CUDA;
    }
    CUtensorMap tm_q;
    if (SWIGLU) {
        // [G, 2, I, K] int8 as {64, I, 2G, K/64}: box {64, 64, 2, 2} = 64 gate
        // rows then their 64 up rows, per k-block
        const uint64_t I = static_cast<uint64_t>(UP_OFF);
        const cuuint64_t dims[4] = {64, I, 2 * static_cast<cuuint64_t>(G), K64};
        const cuuint64_t strides[3] = {static_cast<cuuint64_t>(K), I * K, 64};
        const cuuint32_t box[4] = {64, 64, 2, 2};
        if (!encode_map(&tm_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, CU_TENSOR_MAP_SWIZZLE_64B, q, 4,
                        dims, strides, box))
            return MOE_ERR_CUDA;
    } else {
        const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(G) * R, K64};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K), 64};
        const cuuint32_t box[3] = {64, 128, 2};
        if (!encode_map(&tm_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, CU_TENSOR_MAP_SWIZZLE_64B, q, 3,
                        dims, strides, box))
            return MOE_ERR_CUDA;
    }
    const size_t smem = pw_smem_bytes(G);
    if (smem > static_cast<size_t>(max_smem_optin())) return MOE_ERR_UNSUPPORTED;
    static int attr_done[64] = {0};
    if (!raise_smem_limit(tc_grouped_gemm_pair_w8<SWIGLU>, attr_done)) return MOE_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sm_count() & ~1);
    cfg.blockDim = dim3(PW_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    static int pairs_per_device[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
    if (!pairs_per_device[dev]) {
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, tc_grouped_gemm_pair_w8<SWIGLU>, &cfg) !=
                cudaSuccess ||
            clusters < 1)
            return MOE_ERR_UNSUPPORTED;
        pairs_per_device[dev] = std::min(clusters, sm_count() / 2);
    }
    cfg.gridDim = dim3(2 * pairs_per_device[dev]);
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    cudaLaunchKernelEx(&cfg, tc_grouped_gemm_pair_w8<SWIGLU>, tm_x, tm_q, scales, offsets, G, M,
                       K, R, NOUT, UP_OFF, out, dev_error);
    return launch_status();
}

template moe_status launch_tc_pair_w8<true>(const void *, const int8_t *, const float *,
                                            const int32_t *, int, int, int, int, int, int,
                                            uint16_t *, int32_t *, cudaStream_t);
template moe_status launch_tc_pair_w8<false>(const void *, const int8_t *, const float *,
                                             const int32_t *, int, int, int, int, int, int,
                                             uint16_t *, int32_t *, cudaStream_t);

}  // namespace moe
