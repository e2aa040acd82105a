// gemm_tc_pair.cu -- the grouped GEMM on CTA pairs (tcgen05 cta_group::2),
// for prefill-sized expert groups.
//
// The same computation as gemm_tc.cu (one launch for all experts, SwiGLU in
// the gate/up epilogue: "switchyard" page, 02 Kernels and dispatch, "One
// launch for all experts").  Here the operands are swapped: the MMA's M is
// 256 weight rows and its N is a block of the group's tokens,
//     D[w, j] = sum_k W_g[w, k] * X[m0 + j, k],
// so the tensor-core work of a tile follows the group's row count in steps
// of 16 (a 192-row group costs 192 columns, a group's 16-row remainder 16),
// where token rows as M padded every m-block to 256 or 128 rows: measured
// on GB300, an M = 128 pair MMA takes as long as an M = 256 one, and the
// padded blocks were a third of the tensor work at 256 rows per expert.
//
//  * A pair tile is (group g, n-tile of 256 weight rows, m-block of at most
//    256 tokens).  A group's m-blocks are balanced (equal sizes rounded up
//    to 16), so they take about equally long.
//  * CTA r (r = 0, 1 of the cluster) stages its 128 weight rows (its half of
//    A) and tokens m0 + r N/2 .. m0 + (r+1) N/2 - 1 (its half of B), 32 KB
//    per 64-deep k-step.  SwiGLU: CTA r's 128 rows are 64 features' gate and
//    up rows, in 16-row slices of 8 gate rows then the matching 8 up rows
//    (one 4-D TMA box over the [G, 2, I, K] weights), so in TMEM a warp's 32
//    lanes hold the gate and up values of 16 features, 8 lanes apart.
//  * CTA 0 issues tcgen05.mma.cta_group::2 (M = 256, N = 16 .. 256, K = 16):
//    the tensor cores of both SMs run it, and CTA r's TMEM receives its own
//    128 weight rows (lanes) by the N tokens (columns).
//  * Both CTAs' copies of a stage complete on CTA 0's stage barrier (CTA 0
//    arms it with the bytes of both); CTA 0's MMA commits arrive on the
//    stage-free and accumulator-full barriers of both CTAs (multicast);
//    both CTAs' epilogue warps arrive on CTA 0's accumulator-free barrier.
//  * Epilogue (4 warps per CTA, lane = weight row): 16 token columns at a
//    time are read from TMEM; SwiGLU exchanges gate and up values between
//    lanes 8 apart with one shuffle per token pair; a warp transposes its
//    16 tokens x 16 (SwiGLU) or 32 (down) features through 1 KB of shared
//    memory and stores whole 32- or 64-byte row segments.
//  * TMEM: 2 x 256 columns per CTA (double-buffered accumulators),
//    allocated and freed by one warp of each CTA together (cta_group::2).
// Every mbarrier wait is bounded (1 s): on running out the kernel records
// MOE_ERR_TIMEOUT, stops issuing, drains what it can observe and meets its
// peer at the closing cluster barrier before freeing TMEM.
#include <algorithm>

#include "tc_common.cuh"
#include "tc_pair.cuh"

namespace moe {

namespace {

constexpr int PAIR_MAX_N = 256;                 // tokens per pair tile (MMA N)
constexpr int PAIR_W_ROWS = 256;                // weight rows per pair tile (MMA M)
constexpr int PAIR_KB = 2;                      // 64-deep k-blocks per stage (K = 128)
constexpr int PAIR_A_KB_BYTES = 128 * TC_BK * 2;                // weights, one k-block, per CTA
constexpr int PAIR_A_BYTES = PAIR_KB * PAIR_A_KB_BYTES;        // 32 KB
constexpr int PAIR_B_BYTES = PAIR_KB * 128 * TC_BK * 2;        // tokens: up to 128 rows, 32 KB
constexpr int PAIR_STAGE_BYTES = PAIR_A_BYTES + PAIR_B_BYTES;
constexpr int PAIR_STAGES = (192 * 1024) / PAIR_STAGE_BYTES;   // 3
constexpr uint32_t PAIR_TMEM_COLS = 2 * PAIR_MAX_N;            // two accumulators
constexpr int PAIR_BAR_BYTES = 256;
constexpr int PAIR_EPI_WARPS = 4;
constexpr int PAIR_STAGING_BYTES = 1024;                        // per epilogue warp
constexpr int PAIR_XMAPS = 8;                                   // token boxes of 16 .. 128 rows
constexpr int PAIR_MY_MAX = 128;     // a pair's tiles decoded once at the start (more: on the fly)

static_assert((2 * PAIR_STAGES + 5) * 8 + 8 <= PAIR_BAR_BYTES, "barrier block");

}  // namespace

// A group of `rows` tokens in m-blocks of at most 256: nmb blocks of bs rows
// (bs a multiple of 16), the last one possibly shorter, none empty.
__device__ __forceinline__ int pair_mblocks(int rows, int &bs) {
    const int nmb0 = (rows + PAIR_MAX_N - 1) / PAIR_MAX_N;
    bs = nmb0 > 0 ? (((rows + nmb0 - 1) / nmb0 + 15) & ~15) : PAIR_MAX_N;
    return nmb0 > 0 ? (rows + bs - 1) / bs : 0;
}

// The pair tile table: group g owns n_tiles * nmb(rows_g) tiles from
// s_tile[g], n-tile major, m-block fastest.  Offsets that are negative, not
// monotone or beyond M make the launch a no-op with a device-check fault.
__device__ __forceinline__ void build_pair_table(const int32_t *offsets, int G, int M,
                                                 int n_tiles, int *s_off, int *s_tile,
                                                 int *s_total, int32_t *dev_error) {
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
                tiles = pair_mblocks(o1 - o0, bs) * n_tiles;
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

__device__ __forceinline__ TileInfo decode_pair_tile(int t, const int *s_tile, const int *s_off,
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
    const int nmb = pair_mblocks(rows, bs);
    const int u = t - s_tile[lo];
    ti.nt = u / nmb;
    const int mb = u - ti.nt * nmb;
    ti.m0 = s_off[lo] + mb * bs;
    ti.nrows = min(bs, rows - mb * bs);
    return ti;
}

// The token rows x_perm [M, K] as {64, M, K / 64} (k within a k-block, row,
// k-block): map i loads a box of 16 (i + 1) rows and two k-blocks, which
// land as two 128-byte-swizzled [rows][64] tiles one after the other.
struct PairTokenMaps {
    CUtensorMap m[PAIR_XMAPS];
};

// SWIGLU: out = h [M, NOUT = I]; weights [G, 2, I, K = H] through a 5-D map
//         (k in block, feature % 8, gate/up plane 2g + s, feature / 8, k-block).
// PLAIN : out = y [M, NOUT = H]; weights [G * H, K = I] through a 3-D map
//         (k in block, row, k-block).
// K must be a multiple of 64 (a k-block never runs into the next row).
template <bool SWIGLU>
__global__ void __launch_bounds__(TC_THREADS, 1)
    tc_grouped_gemm_pair(const __grid_constant__ PairTokenMaps tm_x,
                         const __grid_constant__ CUtensorMap tm_w,
                         const int32_t *__restrict__ offsets, int G, int M, int K, int R, int NOUT,
                         uint16_t *__restrict__ out, int32_t *dev_error) {
    constexpr int STAGES = PAIR_STAGES;
    extern __shared__ uint8_t smem_raw[];
    // the same offset in both CTAs: the MMA addresses the peer's stages by
    // the issuing CTA's shared addresses
    uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sW = smem;                                    // A: weight rows
    uint8_t *sX = smem + STAGES * PAIR_A_BYTES;            // B: token rows
    uint8_t *staging = sX + STAGES * PAIR_B_BYTES;         // epilogue transposes
    uint64_t *full = reinterpret_cast<uint64_t *>(staging + PAIR_EPI_WARPS * PAIR_STAGING_BYTES);
    uint64_t *empty = full + STAGES;
    uint64_t *accf = empty + STAGES;
    uint64_t *acce = accf + 2;
    uint64_t *drain = acce + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    int *s_total = reinterpret_cast<int *>(tmem_slot + 1);
    int4 *s_my = reinterpret_cast<int4 *>(reinterpret_cast<uint8_t *>(full) + PAIR_BAR_BYTES);
    int *s_off = reinterpret_cast<int *>(s_my + PAIR_MY_MAX);
    int *s_tile = s_off + (G + 1);

    const int warp = threadIdx.x >> 5, lane = lane_id();
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    // output columns per pair tile: 128 features (SwiGLU) or 256 rows (down)
    const int n_per_tile = SWIGLU ? PAIR_W_ROWS / 2 : PAIR_W_ROWS;
    const int n_tiles = (NOUT + n_per_tile - 1) / n_per_tile;
    const int KB = K / TC_BK;                            // 64-deep k-blocks
    const int KS = (KB + PAIR_KB - 1) / PAIR_KB;         // 128-deep k-steps

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);        // CTA 0's producer arms it for both CTAs' bytes
            mbar_init(&empty[s], 1);       // one multicast MMA commit per use
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accf[b], 1);
            mbar_init(&acce[b], 2 * PAIR_EPI_WARPS);   // the epilogue warps of both CTAs
        }
        mbar_init(drain, 1);
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        for (int i = 0; i < PAIR_XMAPS; ++i) prefetch_tmap(&tm_x.m[i]);
        prefetch_tmap(&tm_w);
    }
    if (warp == 1) tmem_alloc_pair<PAIR_TMEM_COLS>(tmem_slot);
    pdl_wait();
    pdl_trigger();
    if (warp == 2) build_pair_table(offsets, G, M, n_tiles, s_off, s_tile, s_total, dev_error);
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();           // both CTAs' barriers exist before any remote signal
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int total = *s_total;
    const int t_first = static_cast<int>(cluster_id_x());
    const int t_step = static_cast<int>(cluster_count_x());
    // This pair's tiles t_first, t_first + t_step, ... decoded once: a
    // shared-memory read by the MMA thread waits behind the MMAs it has in
    // flight, so the per-tile binary search is kept off its path.
    if (warp == 2)
        for (int i = lane; i < PAIR_MY_MAX; i += 32) {
            const int t = t_first + i * t_step;
            if (t < total) {
                const TileInfo ti = decode_pair_tile(t, s_tile, s_off, G);
                s_my[i] = make_int4(ti.g, ti.nt, ti.m0, ti.nrows);
            }
        }
    __syncthreads();
    auto tile_of = [&](int i, int t) -> TileInfo {
        if (i < PAIR_MY_MAX) {
            const int4 v = s_my[i];
            return TileInfo{v.x, v.y, v.z, v.w};
        }
        return decode_pair_tile(t, s_tile, s_off, G);
    };

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (each CTA)
        if (lane == 0) {
            // a weight tile is read once per m-block of its group, by pairs
            // running at about the same time: normal L2 priority keeps it for
            // the later readers
            uint64_t pol_w;
            asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol_w));
            const uint64_t pol_x = policy_evict_last();   // token rows: read by every n-tile
            int stage = 0;
            uint32_t phase = 0;
            uint32_t filled = 0, fill_parity = 0;     // leader: per stage ever armed / parity
            bool ok = true;
            for (int t = t_first, i = 0; t < total && ok; t += t_step, ++i) {
                const TileInfo ti = tile_of(i, t);
                const int half = ((ti.nrows + 15) & ~15) >> 1;      // N / 2 token rows per CTA
                const int box = (half + 15) & ~15;                  // the same in both CTAs
                const int my_cnt = leader ? min(ti.nrows, half) : ti.nrows - half;
                const CUtensorMap *tm = &tm_x.m[box / 16 - 1];
                const uint32_t bytes = static_cast<uint32_t>(
                    (ti.nrows > half ? 2 : 1) * box * TC_BK * 2 * PAIR_KB + 2 * PAIR_A_BYTES);
                const int xrow = ti.m0 + static_cast<int>(rank) * half;
                // SwiGLU: features f0 + 64r .. +63 as 8-feature slices (8 gate
                // rows, then their 8 up rows); down: rows 128r .. +127 of the tile
                const int wrow = SWIGLU ? (ti.nt * n_per_tile + static_cast<int>(rank) * 64) / 8
                                        : ti.g * R + ti.nt * n_per_tile + static_cast<int>(rank) * 128;
                for (int ks = 0; ks < KS; ++ks) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, dev_error)) {
                        ok = false;
                        break;
                    }
                    const uint32_t bar0 = map_to_rank(smem_u32(&full[stage]), 0);
                    if (leader) {
                        mbar_arrive_expect_tx(&full[stage], bytes);
                        filled |= 1u << stage;
                        fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
                    }
                    const int kb = ks * PAIR_KB;
                    if (SWIGLU)
                        tma_load_5d_pair(sW + stage * PAIR_A_BYTES, &tm_w, bar0, 0, 0, 2 * ti.g,
                                         wrow, kb, pol_w);
                    else
                        tma_load_3d_pair(sW + stage * PAIR_A_BYTES, &tm_w, bar0, 0, wrow, kb, pol_w);
                    if (my_cnt > 0)
                        tma_load_3d_pair(sX + stage * PAIR_B_BYTES, tm, bar0, 0, xrow, kb, pol_x);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // drain (CTA 0): every stage it armed -- both CTAs' copies -- has landed
            for (int s = 0; s < STAGES; ++s)
                if ((filled >> s) & 1u) mbar_wait(&full[s], (fill_parity >> s) & 1u, dev_error);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (CTA 0 only)
        if (leader && lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            const uint64_t dW = sw128_kmajor_desc(smem_u32(sW));
            const uint64_t dX = sw128_kmajor_desc(smem_u32(sX));
            for (int t = t_first, i = 0; t < total && ok; t += t_step, ++i) {
                const int n = (tile_of(i, t).nrows + 15) & ~15;
                const uint32_t idesc = idesc_bf16_f32(PAIR_W_ROWS, n);
                // the tokens' second k-block follows the first box in the stage
                const uint32_t xkb1 = static_cast<uint32_t>((((n >> 1) + 15) & ~15) * TC_BK * 2);
                if (!mbar_wait(&acce[acc], acc_phase ^ 1u, dev_error)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * PAIR_MAX_N);
                for (int ks = 0; ks < KS; ++ks) {
                    if (!mbar_wait(&full[stage], phase, dev_error)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // descriptors advance by (byte offset >> 4); +32 B per 16-deep slice
                    const uint64_t da = dW + ((stage * PAIR_A_BYTES) >> 4);
                    const uint64_t db = dX + ((stage * PAIR_B_BYTES) >> 4);
#pragma unroll
                    for (int kk = 0; kk < TC_BK / 16; ++kk)
                        tc_mma_pair(d_tmem, da + 2 * kk, db + 2 * kk, idesc,
                                    (ks > 0 || kk > 0) ? 1u : 0u);
                    if (ks * PAIR_KB + 1 < KB) {
#pragma unroll
                        for (int kk = 0; kk < TC_BK / 16; ++kk)
                            tc_mma_pair(d_tmem, da + ((PAIR_A_KB_BYTES >> 4) + 2 * kk),
                                        db + ((xkb1 >> 4) + 2 * kk), idesc, 1u);
                    }
                    tc_commit_pair_both(&empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit_pair_both(&accf[acc]);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            // drain: every MMA this thread issued has completed before exit
            tc_commit_pair_local(drain);
            mbar_wait(drain, 0, dev_error);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue (warps 2..5, each CTA)
        const int quarter = warp & 3;       // TMEM lanes this warp may access
        uint8_t *stg = staging + (warp - 2) * PAIR_STAGING_BYTES;
        const uint32_t acce0 = map_to_rank(smem_u32(&acce[0]), 0);
        const uint32_t acce1 = map_to_rank(smem_u32(&acce[1]), 0);
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = t_first, i = 0; t < total; t += t_step, ++i) {
            const TileInfo ti = tile_of(i, t);
            if (!mbar_wait_warp(&accf[acc], acc_phase, dev_error)) break;
            tc_fence_after();
            const uint32_t tbase =
                tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * PAIR_MAX_N;
            if (SWIGLU) {
                // lane l: feature 16 q + 8 (l >> 4) + (l & 7) of this CTA's 64,
                // gate if bit 3 of l is 0, else up.  Gate lanes form h for the
                // chunk's tokens 0..7, up lanes for tokens 8..15.
                const bool is_up = (lane >> 3) & 1;
                const int fcol = 8 * (lane >> 4) + (lane & 7);      // feature within the warp's 16
                const int f_warp = ti.nt * n_per_tile + static_cast<int>(rank) * 64 + 16 * quarter;
                // read-back: lane l stores token l >> 1, features 8 (l & 1) .. +7
                const int rt = lane >> 1, rf = 8 * (lane & 1);
                const bool f_ok = f_warp + rf < NOUT;
#pragma unroll 1
                for (int c0 = 0; c0 < ti.nrows; c0 += 16) {
                    uint32_t v[16];
                    tmem_ld16(tbase + c0, v);
                    tmem_ld_wait();
                    uint16_t *hs = reinterpret_cast<uint16_t *>(stg);     // [16 tokens][16 features]
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        // gate lanes send gate of tokens 8..15, up lanes up of tokens 0..7
                        const uint32_t mine = is_up ? v[j] : v[8 + j];
                        const float other = __uint_as_float(__shfl_xor_sync(FULL, mine, 8));
                        const float g = is_up ? other : __uint_as_float(v[j]);
                        const float u = is_up ? __uint_as_float(v[8 + j]) : other;
                        const float h = silu_fast(g) * u;
                        hs[(8 * is_up + j) * 16 + fcol] = __bfloat16_as_ushort(__float2bfloat16_rn(h));
                    }
                    __syncwarp();
                    const uint4 val = *reinterpret_cast<const uint4 *>(hs + rt * 16 + rf);
                    if (c0 + rt < ti.nrows && f_ok)
                        *reinterpret_cast<uint4 *>(
                            out + static_cast<int64_t>(ti.m0 + c0 + rt) * NOUT + f_warp + rf) = val;
                    __syncwarp();
                }
            } else {
                // lane l: output row n0 + 128 r + 32 q + l
                const int n_warp = ti.nt * n_per_tile + static_cast<int>(rank) * 128 + 32 * quarter;
#pragma unroll 1
                for (int c0 = 0; c0 < ti.nrows; c0 += 16) {
                    uint32_t v[16];
                    tmem_ld16(tbase + c0, v);
                    tmem_ld_wait();
                    uint16_t *ys = reinterpret_cast<uint16_t *>(stg);     // [16 tokens][32 rows]
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        ys[j * 32 + lane] =
                            __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[j])));
                    __syncwarp();
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const int id = lane + 32 * i;            // 64 chunks of 16 B
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
            if (lane == 0) mbar_arrive_remote(acc == 0 ? acce0 : acce1);   // CTA 0's barrier
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }

    tc_fence_before();
    __syncthreads();
    // neither CTA leaves (or frees its TMEM) while its peer may still signal
    // its barriers or run MMAs into its TMEM
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair<PAIR_TMEM_COLS>(tmem_base);
    }
}

// ------------------------------------------------------------------ host

static size_t pair_smem_bytes(int G) {
    return 1024 + static_cast<size_t>(PAIR_STAGES) * PAIR_STAGE_BYTES +
           PAIR_EPI_WARPS * PAIR_STAGING_BYTES + PAIR_BAR_BYTES + PAIR_MY_MAX * sizeof(int4) +
           2 * static_cast<size_t>(G + 1) * sizeof(int);
}

// Maps of the pair kernel.  Every one views K as (k within a 64-element
// k-block, ..., k-block) so that a box brings two k-blocks (K % 64 == 0).
//   tokens  x_perm [M, K]          -> {64, M, K/64}, box {64, rows, 2};
//   gate/up w_gu [G, 2, I, K]      -> {64, 8, 2G, I/8, K/64}: (k, feature % 8,
//           plane 2g + s with s = 0 gate / 1 up, feature / 8, k-block), box
//           {64, 8, 2, 8, 2} = 64 features as 8 slices of [8 gate][8 up] rows;
//   down    w_down [G * H, K]      -> {64, G H, K/64}, box {64, 128, 2}.
// 128-byte swizzle (each box row is 64 bf16 = 128 bytes).
static bool encode_pair_map(CUtensorMap *map, const void *base, int rank, const cuuint64_t *dims,
                            const cuuint64_t *strides, const cuuint32_t *box) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(base), dims,
               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool SWIGLU>
moe_status launch_tc_pair(const void *act, const void *w, const int32_t *offsets, int G, int M,
                          int K, int R, int NOUT, int UP_OFF, uint16_t *out, int32_t *dev_error,
                          cudaStream_t stream) {
    (void)UP_OFF;   // SwiGLU: up rows are at +I, which the 5-D map encodes
    if (K % TC_BK != 0 || NOUT % 8 != 0) return MOE_ERR_UNSUPPORTED;
    const uint64_t K64 = static_cast<uint64_t>(K) / TC_BK;
    PairTokenMaps tm_x;
    for (int i = 0; i < PAIR_XMAPS; ++i) {
        const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(M), K64};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, 128};
        const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(16 * (i + 1)), 2};
        if (!encode_pair_map(&tm_x.m[i], act, 3, dims, strides, box)) return MOE_ERR_CUDA;
    }
    CUtensorMap tm_w;
    if (SWIGLU) {
        const uint64_t I = static_cast<uint64_t>(NOUT);
        const cuuint64_t dims[5] = {64, 8, 2 * static_cast<cuuint64_t>(G), I / 8, K64};
        const cuuint64_t strides[4] = {static_cast<cuuint64_t>(K) * 2, I * K * 2, 8ull * K * 2, 128};
        const cuuint32_t box[5] = {64, 8, 2, 8, 2};
        if (!encode_pair_map(&tm_w, w, 5, dims, strides, box)) return MOE_ERR_CUDA;
    } else {
        const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(G) * R, K64};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, 128};
        const cuuint32_t box[3] = {64, 128, 2};
        if (!encode_pair_map(&tm_w, w, 3, dims, strides, box)) return MOE_ERR_CUDA;
    }
    const size_t smem = pair_smem_bytes(G);
    if (smem > static_cast<size_t>(max_smem_optin())) return MOE_ERR_UNSUPPORTED;
    static int attr_done[64] = {0};
    if (!raise_smem_limit(tc_grouped_gemm_pair<SWIGLU>, attr_done)) return MOE_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sm_count() & ~1);
    cfg.blockDim = dim3(TC_THREADS);
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
    // a persistent grid of as many pairs as can be resident at once (the
    // SMs of a GPC need not pair up evenly)
    static int pairs_per_device[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
    if (!pairs_per_device[dev]) {
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, tc_grouped_gemm_pair<SWIGLU>, &cfg) !=
                cudaSuccess ||
            clusters < 1)
            return MOE_ERR_UNSUPPORTED;
        pairs_per_device[dev] = std::min(clusters, sm_count() / 2);
    }
    cfg.gridDim = dim3(2 * pairs_per_device[dev]);
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    cudaLaunchKernelEx(&cfg, tc_grouped_gemm_pair<SWIGLU>, tm_x, tm_w, offsets, G, M, K, R, NOUT,
                       out, dev_error);
    return launch_status();
}

template moe_status launch_tc_pair<true>(const void *, const void *, const int32_t *, int, int,
                                         int, int, int, int, uint16_t *, int32_t *, cudaStream_t);
template moe_status launch_tc_pair<false>(const void *, const void *, const int32_t *, int, int,
                                          int, int, int, int, uint16_t *, int32_t *, cudaStream_t);

}  // namespace moe
