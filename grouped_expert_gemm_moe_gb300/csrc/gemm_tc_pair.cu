// gemm_tc_pair.cu -- the grouped GEMM on CTA pairs (tcgen05 cta_group::2).
//
// The same computation as gemm_tc.cu ("switchyard" page, 02 Kernels and
// dispatch, "One launch for all experts": one launch for all experts, SwiGLU
// fused into the gate/up epilogue), for prefill-sized groups.  Two CTAs of a
// cluster form a pair on two SMs and share one 256 x 256 tile:
//
//  * CTA r (r = 0, 1 in the cluster) stages token rows m0 + 128r .. +127 of
//    the tile (its half of A) and weight rows 128r .. 128r+127 of the tile
//    (its half of B: in SwiGLU mode the gate rows in CTA 0 and the matching
//    up rows in CTA 1) -- 32 KB per 64-deep k-step per SM, where a 128 x 256
//    tile on one SM stages 48 KB for the same MMA work.  With the ring bound
//    by operand bytes in flight per SM, that is 1.5x the MMA work per staged
//    byte, and the 192 KB ring holds 6 stages instead of 4;
//  * CTA 0 issues tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16): the
//    tensor cores of both SMs run it, each reading its own shared memory, and
//    CTA r's TMEM receives rows 128r .. 128r+127 of the accumulator with all
//    256 columns, so each CTA's epilogue finds gate and up values of its own
//    token rows side by side, as in the one-SM kernel;
//  * both CTAs' copies of a stage complete on CTA 0's stage barrier (CTA 0
//    arms it with the bytes of both); CTA 0's MMA commits arrive on the
//    stage-free and accumulator-full barriers of both CTAs (multicast), and
//    both CTAs' epilogue warps arrive on CTA 0's accumulator-free barrier;
//  * TMEM (2 x 256 columns per CTA: double-buffered accumulators) is
//    allocated and freed by one warp of each CTA together (cta_group::2).
// The pair tile table is the one-SM table with 256-row m-blocks; a CTA whose
// half of an m-block holds no rows of the group still stages its weight half
// (the peer needs it) and skips its token copy; its accumulator rows are
// never stored.  Every mbarrier wait is bounded (1 s): on running out the
// kernel records MOE_ERR_TIMEOUT, stops issuing, drains what it can observe
// and meets its peer at the closing cluster barrier before freeing TMEM.
#include <algorithm>

#include "tc_common.cuh"
#include "tc_pair.cuh"

namespace moe {

namespace {

constexpr int PAIR_BM = 256;                    // token rows per pair tile
constexpr int PAIR_BN = 256;                    // weight rows per pair tile (MMA N)
constexpr int PAIR_A_BYTES = 128 * TC_BK * 2;   // per CTA: 128 token rows
constexpr int PAIR_B_BYTES = 128 * TC_BK * 2;   // per CTA: 128 weight rows
constexpr int PAIR_STAGE_BYTES = PAIR_A_BYTES + PAIR_B_BYTES;
constexpr int PAIR_STAGES = (192 * 1024) / PAIR_STAGE_BYTES;   // 6
constexpr uint32_t PAIR_TMEM_COLS = 2 * PAIR_BN;               // two accumulators
constexpr int PAIR_BAR_BYTES = 256;
constexpr int PAIR_EPI_WARPS = 4;

static_assert((2 * PAIR_STAGES + 5) * 8 + 8 <= PAIR_BAR_BYTES, "barrier block");

}  // namespace

// SWIGLU: out = h [M, NOUT=I], weights [G*2I, K=H] (up rows at +UP_OFF = I).
// PLAIN : out = y [M, NOUT=H], weights [G*H,  K=I].
template <bool SWIGLU>
__global__ void __launch_bounds__(TC_THREADS, 1)
    tc_grouped_gemm_pair(const __grid_constant__ CUtensorMap tm_act16,
                         const __grid_constant__ CUtensorMap tm_act32,
                         const __grid_constant__ CUtensorMap tm_act64,
                         const __grid_constant__ CUtensorMap tm_act128,
                         const __grid_constant__ CUtensorMap tm_w,
                         const int32_t *__restrict__ offsets, int G, int M, int K, int R, int NOUT,
                         int UP_OFF, uint16_t *__restrict__ out, int32_t *dev_error) {
    constexpr int STAGES = PAIR_STAGES;
    extern __shared__ uint8_t smem_raw[];
    // the same offset in both CTAs: the MMA addresses the peer's stages by
    // the issuing CTA's shared addresses
    uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * PAIR_A_BYTES;
    uint64_t *full = reinterpret_cast<uint64_t *>(sB + STAGES * PAIR_B_BYTES);
    uint64_t *empty = full + STAGES;
    uint64_t *accf = empty + STAGES;
    uint64_t *acce = accf + 2;
    uint64_t *drain = acce + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    int *s_total = reinterpret_cast<int *>(tmem_slot + 1);
    int *s_off = reinterpret_cast<int *>(reinterpret_cast<uint8_t *>(full) + PAIR_BAR_BYTES);
    int *s_tile = s_off + (G + 1);

    const int warp = threadIdx.x >> 5, lane = lane_id();
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    const int n_per_tile = SWIGLU ? PAIR_BN / 2 : PAIR_BN;
    const int n_tiles = (NOUT + n_per_tile - 1) / n_per_tile;
    const int KB = (K + TC_BK - 1) / TC_BK;

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
        prefetch_tmap(&tm_act16);
        prefetch_tmap(&tm_act32);
        prefetch_tmap(&tm_act64);
        prefetch_tmap(&tm_act128);
        prefetch_tmap(&tm_w);
    }
    if (warp == 1) tmem_alloc_pair<PAIR_TMEM_COLS>(tmem_slot);
    pdl_wait();
    pdl_trigger();
    if (warp == 2)
        build_tile_table(offsets, G, M, n_tiles, s_off, s_tile, s_total, dev_error, PAIR_BM);
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();           // both CTAs' barriers exist before any remote signal
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int total = *s_total;
    const int t_first = static_cast<int>(cluster_id_x());
    const int t_step = static_cast<int>(cluster_count_x());

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (each CTA)
        if (lane == 0) {
            // a weight tile is read once per m-block of its group, by pairs
            // running at about the same time: normal L2 priority keeps it for
            // the later readers (evict-first measured 1-3 % slower here)
            uint64_t pol_w;
            asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol_w));
            const uint64_t pol_a = policy_evict_last();
            int stage = 0;
            uint32_t phase = 0;
            uint32_t filled = 0, fill_parity = 0;     // leader: per stage ever armed / parity
            bool ok = true;
            for (int t = t_first; t < total && ok; t += t_step) {
                const TileInfo ti = decode_tile(t, s_tile, s_off, G, PAIR_BM);
                const PairRows pr = pair_rows(ti.nrows);
                const int my_rows = leader ? pr.r0 : pr.r1;
                const int abox = abox_rows(my_rows);
                const CUtensorMap *tm_a = abox == 16 ? &tm_act16 : abox == 32 ? &tm_act32
                                        : abox == 64 ? &tm_act64 : &tm_act128;
                const uint32_t bytes = static_cast<uint32_t>(
                    (abox_rows(pr.r0) + abox_rows(pr.r1)) * TC_BK * 2 + 2 * PAIR_B_BYTES);
                // this CTA's weight rows: in SwiGLU mode the gate rows of
                // features f0 + 64r .. +63 and the matching up rows (one 3-D
                // box), else rows 128r .. 128r+127 of the tile
                const int wrow = SWIGLU ? ti.nt * n_per_tile + static_cast<int>(rank) * 64
                                        : ti.g * R + ti.nt * n_per_tile + static_cast<int>(rank) * 128;
                const int arow = ti.m0 + static_cast<int>(rank) * pr.per_cta;
                for (int kb = 0; kb < KB; ++kb) {
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
                    const int kx = kb * TC_BK;
                    if (abox > 0)
                        tma_load_2d_pair(sA + stage * PAIR_A_BYTES, tm_a, bar0, kx, arow, pol_a);
                    if (SWIGLU)
                        tma_load_3d_pair(sB + stage * PAIR_B_BYTES, &tm_w, bar0, kx, wrow,
                                         2 * ti.g, pol_w);
                    else
                        tma_load_2d_pair(sB + stage * PAIR_B_BYTES, &tm_w, bar0, kx, wrow, pol_w);
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
            constexpr uint32_t idesc_full = idesc_bf16_f32(PAIR_BM, PAIR_BN);
            constexpr uint32_t idesc_half = idesc_bf16_f32(PAIR_BM / 2, PAIR_BN);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int t = t_first; t < total && ok; t += t_step) {
                const uint32_t idesc =
                    decode_tile(t, s_tile, s_off, G, PAIR_BM).nrows <= 128 ? idesc_half : idesc_full;
                if (!mbar_wait_cluster(&acce[acc], acc_phase ^ 1u, dev_error)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * PAIR_BN);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&full[stage], phase, dev_error)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(sA + stage * PAIR_A_BYTES);
                    const uint32_t b_addr = smem_u32(sB + stage * PAIR_B_BYTES);
#pragma unroll
                    for (int kk = 0; kk < TC_BK / 16; ++kk)
                        tc_mma_pair(d_tmem, sw128_kmajor_desc(a_addr + kk * 32),
                                    sw128_kmajor_desc(b_addr + kk * 32), idesc,
                                    (kb > 0 || kk > 0) ? 1u : 0u);
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
        const int row_in_tile = quarter * 32 + lane;
        const uint32_t acce0 = map_to_rank(smem_u32(&acce[0]), 0);
        const uint32_t acce1 = map_to_rank(smem_u32(&acce[1]), 0);
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = t_first; t < total; t += t_step) {
            const TileInfo ti = decode_tile(t, s_tile, s_off, G, PAIR_BM);
            if (!mbar_wait_warp(&accf[acc], acc_phase, dev_error)) break;
            tc_fence_after();
            // Accumulator layout (per CTA, TMEM columns from tbase):
            //   M = 256 tile: lane i = row i, columns 0..255 = the tile's 256
            //     weight rows (SwiGLU: gate f0..63, up f0..63, gate f64..127,
            //     up f64..127);
            //   M = 128 tile: lane i < 64 = row i, columns 0..127 = weight rows
            //     0..127; lane 64 + i = row i, columns 0..127 = weight rows
            //     128..255.
            const PairRows pr = pair_rows(ti.nrows);
            const int my_rows = leader ? pr.r0 : pr.r1;
            const int row = pr.half ? (row_in_tile & 63) : row_in_tile;
            const int wpart = pr.half ? (row_in_tile >> 6) : 0;   // which half of the weight rows
            const bool valid = row < my_rows;
            uint16_t *orow =
                out + static_cast<int64_t>(ti.m0 + static_cast<int>(rank) * pr.per_cta + row) *
                          NOUT;
            const uint32_t tbase =
                tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * PAIR_BN;
            const int n0 = ti.nt * n_per_tile;
            if (SWIGLU) {
                // features fb .. fb + nf - 1 of this thread; gate of feature
                // fb + c at column gc(c), up at gc(c) + 64
                const int fb = wpart * 64;
                const int nf = pr.half ? 64 : 128;
#pragma unroll 1
                for (int c = 0; c < nf; c += 16) {
                    const int gcol = c < 64 ? c : c + 64;
                    uint32_t g[16], u[16];
                    tmem_ld16(tbase + gcol, g);
                    tmem_ld16(tbase + gcol + 64, u);
                    tmem_ld_wait();
                    const int f = n0 + fb + c;
                    if (valid && f < NOUT) {
                        uint32_t p[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float h0 = silu_fast(__uint_as_float(g[2 * i])) *
                                             __uint_as_float(u[2 * i]);
                            const float h1 = silu_fast(__uint_as_float(g[2 * i + 1])) *
                                             __uint_as_float(u[2 * i + 1]);
                            p[i] = pack_bf16x2(h0, h1);
                        }
                        uint4 *dst = reinterpret_cast<uint4 *>(orow + f);
                        dst[0] = make_uint4(p[0], p[1], p[2], p[3]);
                        if (f + 8 < NOUT) dst[1] = make_uint4(p[4], p[5], p[6], p[7]);
                    }
                }
            } else {
                const int cb = wpart * 128;
                const int nc = pr.half ? 128 : PAIR_BN;
#pragma unroll 1
                for (int c = 0; c < nc; c += 16) {
                    uint32_t v[16];
                    tmem_ld16(tbase + c, v);
                    tmem_ld_wait();
                    const int o = n0 + cb + c;
                    if (valid && o < NOUT) {
                        uint32_t p[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            p[i] = pack_bf16x2(__uint_as_float(v[2 * i]),
                                               __uint_as_float(v[2 * i + 1]));
                        uint4 *dst = reinterpret_cast<uint4 *>(orow + o);
                        dst[0] = make_uint4(p[0], p[1], p[2], p[3]);
                        if (o + 8 < NOUT) dst[1] = make_uint4(p[4], p[5], p[6], p[7]);
                    }
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
    return 1024 + static_cast<size_t>(PAIR_STAGES) * PAIR_STAGE_BYTES + PAIR_BAR_BYTES +
           2 * static_cast<size_t>(G + 1) * sizeof(int);
}

template <bool SWIGLU>
moe_status launch_tc_pair(const void *act, const void *w, const int32_t *offsets, int G, int M,
                          int K, int R, int NOUT, int UP_OFF, uint16_t *out, int32_t *dev_error,
                          cudaStream_t stream) {
    CUtensorMap tm_act16, tm_act32, tm_act64, tm_act128, tm_w;
    if (!encode_bf16_2d(&tm_act16, act, K, M, 16) || !encode_bf16_2d(&tm_act32, act, K, M, 32) ||
        !encode_bf16_2d(&tm_act64, act, K, M, 64) || !encode_bf16_2d(&tm_act128, act, K, M, 128) ||
        !(SWIGLU ? encode_gate_up_3d(&tm_w, w, K, UP_OFF, G, 64)
                 : encode_bf16_2d(&tm_w, w, K, static_cast<uint64_t>(G) * R, 128)))
        return MOE_ERR_CUDA;
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
    cudaLaunchKernelEx(&cfg, tc_grouped_gemm_pair<SWIGLU>, tm_act16, tm_act32, tm_act64,
                       tm_act128, tm_w, offsets, G, M, K, R, NOUT, UP_OFF, out, dev_error);
    return launch_status();
}

template moe_status launch_tc_pair<true>(const void *, const void *, const int32_t *, int, int,
                                         int, int, int, int, uint16_t *, int32_t *, cudaStream_t);
template moe_status launch_tc_pair<false>(const void *, const void *, const int32_t *, int, int,
                                          int, int, int, int, uint16_t *, int32_t *, cudaStream_t);

}  // namespace moe
