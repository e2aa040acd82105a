/*
 * moe.h -- C ABI of libmoe.so, the MoE token-dispatch hot path on one GB300
 * (sm_103a).
 *
 * The layer these calls make up is the one the pages describe: route each
 * token to its top-k experts, sort the token rows by expert, run every
 * expert's SwiGLU FFN in one grouped launch, and combine the expert outputs
 * back into token order ("switchyard" page, 02 Kernels and dispatch: "Route
 * and sort", "One launch for all experts"; "dispatch" README, Architecture
 * and Stack).  One layer is
 *
 *   moe_route -> moe_permute -> moe_grouped_gemm_swiglu | moe_grouped_gemv
 *             -> moe_combine
 *
 * (int8 weight-only experts: the *_w8 calls, weights from moe_quantize_w8;
 * a stack of layers takes its router logits from moe_router_logits).
 *
 * Conventions shared by every call
 *  - Notation: T tokens, H hidden size, E routed experts, S shared experts
 *    (always-on, weight 1), k experts per token, I expert intermediate size,
 *    G = E + S expert groups, M = T*k + S*T permuted rows.  Slot s = t*k + j
 *    is token t's j-th routed choice.
 *  - Pointers are plain device pointers unless a parameter says "host".
 *    The routing calls' logits, the combine calls' out and
 *    moe_decode_layer's logits, x and out may also be mapped pinned host
 *    memory (cudaHostAlloc), reached over NVLink-C2C on GB300.
 *    The caller owns every buffer: the library never allocates device
 *    memory, never synchronises, and enqueues all device work on `stream`
 *    (asynchronous to the host).  bf16 tensors are passed as uint16_t bit
 *    patterns.  All matrices are row-major and dense (no strides).
 *  - Every device pointer must be 16-byte aligned; H and I must be
 *    multiples of 8.  Otherwise MOE_ERR_ALIGNMENT.
 *  - Limits: 1 <= T, 1 <= k <= min(E, 32), G <= 1024, T*k < 2^31, M*H < 2^31
 *    elements.  Otherwise MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED.
 *  - The return value reports what the host can see: argument checks and
 *    launch errors (cudaGetLastError -> MOE_ERR_CUDA).  Faults in the data
 *    (an expert id outside [0,E), a non-finite logit, inconsistent offsets) are
 *    found on the device: the kernel skips the offending write and stores
 *    MOE_ERR_DEVICE_CHECK into *dev_error; a bounded wait that ran out
 *    stores MOE_ERR_TIMEOUT.  dev_error is one int32 in device memory that
 *    the caller zeroes and reads after synchronising; it may be NULL, in
 *    which case device-side faults are not reported (writes are still
 *    skipped).
 *  - Results are deterministic: the same inputs give the same bytes on
 *    every run (no atomics on any data path).
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* NULL pointer, negative size, k > E ... */
    MOE_ERR_UNSUPPORTED = 2,   /* valid but outside this build's limits */
    MOE_ERR_ALIGNMENT = 3,     /* pointer not 16-byte aligned, H or I not a multiple of 8 */
    MOE_ERR_WORKSPACE = 4,     /* workspace smaller than the *_workspace_size answer */
    MOE_ERR_CUDA = 5,          /* a CUDA runtime / driver call failed */
    MOE_ERR_DEVICE_CHECK = 6,  /* device-side data check failed (see dev_error) */
    MOE_ERR_TIMEOUT = 7        /* a bounded device-side wait ran out (see dev_error) */
} moe_status;

typedef enum moe_dtype { MOE_DTYPE_BF16 = 0, MOE_DTYPE_F32 = 1 } moe_dtype;

/* row_of_slot value of a slot that moe_permute_capped dropped (its expert
 * had no room left); moe_combine_capped adds nothing for it. */
#define MOE_ROW_DROPPED (-2)

/* Static description of a status code; never NULL. */
const char *moe_status_string(int status);

/* Library version as an integer (major*10000 + minor*100 + patch). */
int moe_version(void);

/*
 * moe_router_logits -- router logits of a bf16 activation batch.
 * logits[t,e] = sum_c x[t,c] * w_r[e,c] (+ bias[e]), fp32 accumulation in a
 * fixed order.  The pages leave the router as plain PyTorch ("dispatch"
 * README, Architecture: "Router / top-k gating"); this call exists so a
 * stack of layers (x_{l+1} = x_l + MoE_l(x_l)) can route layer l+1 on the
 * device.  x: [T,H] bf16; w_r: [E,H] bf16 (one row per expert); bias: [E]
 * fp32 or NULL (a fixed routing bias, e.g. a zipf skew); logits: [T,E] fp32.
 */
moe_status moe_router_logits(const uint16_t *x, const uint16_t *w_r, const float *bias, int T,
                             int H, int E, float *logits, cudaStream_t stream);

/*
 * moe_router_route -- moe_router_logits and moe_route in one launch: a CTA
 * forms its tokens' logits in shared memory (the same fixed summation order
 * as moe_router_logits, so the same fp32 values) and routes them there, so
 * topk_ids / topk_w equal those of the two calls bit for bit, and the
 * logits make no round trip through global memory.  logits: [T,E] fp32
 * output or NULL (not written).  Other arguments as for the two calls;
 * E <= 1024, 1 <= k <= min(E, 32).
 */
moe_status moe_router_route(const uint16_t *x, const uint16_t *w_r, const float *bias, int T,
                            int H, int E, int k, int renormalize, float *logits,
                            int32_t *topk_ids, float *topk_w, int32_t *dev_error,
                            cudaStream_t stream);

/*
 * moe_route -- top-k routing, one warp per token ("switchyard" page, "Route
 * and sort": each token routed in one warp).
 * logits: [T,E] fp32.  topk_ids: [T,k] int32, the k experts with the
 * largest logit in descending order, ties broken toward the lower expert
 * index.  topk_w: [T,k] fp32, softmax over all E logits of each chosen
 * expert; if `renormalize` is non-zero the k weights are divided by their
 * sum.  A non-finite logit (NaN or +-inf, for which the softmax has no
 * finite value) is a device-check fault (that token's outputs are
 * left untouched).  E <= 1024.
 */
moe_status moe_route(const float *logits, int T, int E, int k, int renormalize,
                     int32_t *topk_ids, float *topk_w, int32_t *dev_error, cudaStream_t stream);

/* Workspace bytes moe_permute needs: 0 for up to 1024 slots (T*k), else
 * ceil(T*k / 1024) * (E + 1) int32 chunk counts, rounded up to 256. */
size_t moe_permute_workspace_size(int T, int E, int S, int k);

/*
 * moe_permute -- stable sort of token rows by expert with a block-wide
 * prefix scan and no atomics ("switchyard" page, "Route and sort"), plus
 * the gather of activation rows into expert order.
 * topk_ids: [T,k] int32 from moe_route.  x: [T,H], bf16 (x_dtype =
 * MOE_DTYPE_BF16) or fp32 (MOE_DTYPE_F32, rounded to bf16 on the gather).
 * Outputs:
 *   offsets     [G+1] int32: group g owns permuted rows [offsets[g],
 *               offsets[g+1]); routed group e holds its slots in ascending
 *               slot order; shared group E+s holds tokens 0..T-1 in order;
 *               offsets[0] = 0, offsets[E] = T*k, offsets[G] = M.
 *   sorted_slot [T*k] int32: the slot held by routed row r.
 *   row_of_slot [T*k] int32: inverse of sorted_slot (-1 for a slot whose
 *               expert id was invalid).
 *   x_perm      [M,H] bf16: row r = x[token of row r].
 * An expert id outside [0,E) is a device-check fault: every group is left
 * empty and every row_of_slot entry -1.  workspace: device memory of at
 * least moe_permute_workspace_size(T, E, S, k) bytes (4-byte aligned; NULL
 * when that size is 0).
 */
moe_status moe_permute(const int32_t *topk_ids, int T, int E, int S, int k, const void *x,
                       int x_dtype, int H, int32_t *offsets, int32_t *sorted_slot,
                       int32_t *row_of_slot, uint16_t *x_perm, void *workspace,
                       size_t workspace_bytes, int32_t *dev_error, cudaStream_t stream);

/*
 * moe_permute_capped -- moe_permute with a capacity limit per routed expert,
 * the token-dropping variant ("switchyard" page, 03 Load balance, "What
 * dropping tokens costs": capacity limits drop the tokens an expert has no
 * room for).  Routed expert e serves at most `capacity` of its slots: the
 * first ones in slot order (t*k + j ascending: first come, first served);
 * the others are dropped.  A capacity factor CF gives capacity =
 * ceil(CF * T*k / E).  Shared experts are never capped.  Outputs as for
 * moe_permute, except:
 *   offsets     routed group e holds min(count_e, capacity) rows; the shared
 *               groups start at offsets[E] (the served routed rows), so
 *               offsets[G] = offsets[E] + S*T <= M;
 *   sorted_slot entries at positions offsets[E] .. T*k-1 are -1;
 *   row_of_slot MOE_ROW_DROPPED for a dropped slot;
 *   x_perm      rows past offsets[G] are not written;
 *   dropped     one int32 in device memory, set to the number of dropped
 *               slots (T*k - offsets[E]); must not be NULL.
 * capacity >= every expert's count gives exactly moe_permute's outputs.
 * The FFN calls take the permuted row count M = T*k + S*T as before (an
 * upper bound of the rows in use); combine with moe_combine_capped.
 */
moe_status moe_permute_capped(const int32_t *topk_ids, int T, int E, int S, int k, int capacity,
                              const void *x, int x_dtype, int H, int32_t *offsets,
                              int32_t *sorted_slot, int32_t *row_of_slot, uint16_t *x_perm,
                              int32_t *dropped, void *workspace, size_t workspace_bytes,
                              int32_t *dev_error, cudaStream_t stream);

/*
 * moe_route_permute -- moe_route followed by moe_permute in one launch, for
 * decode-sized batches (T*k <= 1024 slots, E <= 256; otherwise
 * MOE_ERR_UNSUPPORTED and nothing is launched).  Same arguments and the same
 * outputs, bit for bit, as the two calls (no permute workspace is needed);
 * a non-finite logit is a device-check fault that leaves every group empty.  The
 * pages route and sort in separate steps ("switchyard" page, "Route and
 * sort"); fusing them removes a launch and a round trip through global
 * memory from the latency-bound decode step.
 */
moe_status moe_route_permute(const float *logits, int T, int E, int S, int k, int renormalize,
                             const void *x, int x_dtype, int H, int32_t *topk_ids, float *topk_w,
                             int32_t *offsets, int32_t *sorted_slot, int32_t *row_of_slot,
                             uint16_t *x_perm, int32_t *dev_error, cudaStream_t stream);

/*
 * Tile shapes of the grouped GEMM calls.  Each call picks one from the mean
 * permuted rows per group (M / G); moe_set_gemm_tile overrides that choice
 * for every later call in the process, so that tests can run each tile
 * kernel on any batch and tuning can compare them.  bf16 weights:
 * MOE_TILE_128x128 (up to 64 rows per group), MOE_TILE_128x256 (up to 128),
 * MOE_TILE_PAIR (256 x 256 tiles on CTA pairs, above).  int8 weights:
 * 256 weight rows x 16 / 32 / 64 tokens (MOE_TILE_W8_D16 up to 10 rows per
 * group, _D32 up to 24, _D64 below 64), from 64 rows per group
 * MOE_TILE_W8_PAIR (256 weight rows widened into tensor memory x up to 192
 * tokens on CTA pairs, when H and I are multiples of 64) or else
 * MOE_TILE_W8_ROWS (128 token rows x 256 weight rows).  A forced tile of the other weight type leaves
 * that type's choice automatic.  Not synchronised with calls in flight on
 * other host threads; the results of every tile are within the same bounds
 * of the exact layer.  Returns MOE_ERR_INVALID_ARG for an unknown value.
 */
typedef enum {
    MOE_TILE_AUTO = -1,
    MOE_TILE_128x128 = 0,
    MOE_TILE_128x256 = 1,
    MOE_TILE_PAIR = 2,
    MOE_TILE_W8_D16 = 3,
    MOE_TILE_W8_D32 = 4,
    MOE_TILE_W8_D64 = 5,
    MOE_TILE_W8_ROWS = 6,
    MOE_TILE_W8_PAIR = 7
} moe_tile;
moe_status moe_set_gemm_tile(int tile);

/* Workspace bytes of the FFN calls below: the bf16 hidden rows h [M,I]. */
size_t moe_ffn_workspace_size(int M, int I);

/*
 * moe_grouped_gemm_swiglu -- every expert's SwiGLU FFN over its permuted
 * rows in one persistent launch per GEMM ("switchyard" page, "One launch
 * for all experts": a tensor-core grouped GEMM with SwiGLU fused into its
 * epilogue).  tcgen05 MMAs with TMEM accumulators fed by TMA, a per-expert
 * tile scheduler over the offsets table.
 *   h[r,:]      = bf16( silu(x_perm[r] . Wg_g^T) * (x_perm[r] . Wu_g^T) )
 *   y_perm[r,:] = bf16( h[r] . Wd_g^T )          for rows r of group g
 * x_perm: [M,H] bf16; offsets: [G+1] from moe_permute (read on the device:
 * the host never needs the per-expert counts); w_gu: [G,2I,H] bf16, rows
 * 0..I-1 of each group the gate projection, rows I..2I-1 the up projection;
 * w_down: [G,H,I] bf16; y_perm: [M,H] bf16 (unweighted: the routing weight
 * is applied by moe_combine).  workspace: at least
 * moe_ffn_workspace_size(M, I) bytes of device memory (holds h).
 * Offsets that are not monotone or exceed M are a device-check fault (no
 * output is written).  Rows beyond offsets[G] are not touched.
 */
moe_status moe_grouped_gemm_swiglu(const uint16_t *x_perm, const int32_t *offsets, int G, int M,
                                   int H, int I, const uint16_t *w_gu, const uint16_t *w_down,
                                   uint16_t *y_perm, void *workspace, size_t workspace_bytes,
                                   int32_t *dev_error, cudaStream_t stream);

/*
 * moe_grouped_gemv -- the same computation as moe_grouped_gemm_swiglu for
 * decode-sized batches: each expert weight row is streamed from HBM once
 * with coalesced 128-bit loads and dotted with the few rows of its expert
 * ("switchyard" page, "One launch for all experts": for decode, a grouped
 * GEMV).  Same arguments and results (up to fp32 summation order).  Fast
 * when the mean rows per expert is small (about <= 4); correct for any.
 */
moe_status moe_grouped_gemv(const uint16_t *x_perm, const int32_t *offsets, int G, int M, int H,
                            int I, const uint16_t *w_gu, const uint16_t *w_down,
                            uint16_t *y_perm, void *workspace, size_t workspace_bytes,
                            int32_t *dev_error, cudaStream_t stream);

/*
 * The two phases of each grouped FFN as separate calls (the combined calls
 * above are exactly gate_up followed by down), for callers that schedule
 * or time them separately:
 *   *_gate_up: h [M,I] bf16 = silu(x_perm . Wg^T) * (x_perm . Wu^T), per group;
 *   *_down   : y_perm [M,H] bf16 = h . Wd^T, per group.
 * h is caller-owned device memory (16-byte aligned, M*I bf16).
 */
moe_status moe_grouped_gemm_gate_up(const uint16_t *x_perm, const int32_t *offsets, int G, int M,
                                    int H, int I, const uint16_t *w_gu, uint16_t *h,
                                    int32_t *dev_error, cudaStream_t stream);
moe_status moe_grouped_gemm_down(const uint16_t *h, const int32_t *offsets, int G, int M, int H,
                                 int I, const uint16_t *w_down, uint16_t *y_perm,
                                 int32_t *dev_error, cudaStream_t stream);
moe_status moe_grouped_gemv_gate_up(const uint16_t *x_perm, const int32_t *offsets, int G, int M,
                                    int H, int I, const uint16_t *w_gu, uint16_t *h,
                                    int32_t *dev_error, cudaStream_t stream);
moe_status moe_grouped_gemv_down(const uint16_t *h, const int32_t *offsets, int G, int M, int H,
                                 int I, const uint16_t *w_down, uint16_t *y_perm,
                                 int32_t *dev_error, cudaStream_t stream);

/*
 * int8 weight-only variants ("dispatch" README, phase 5a: per-channel int8
 * weight-only quantisation).  q_gu: [G,2I,H] int8 with s_gu: [G,2I] fp32
 * (one scale per output row); q_down: [G,H,I] int8 with s_down: [G,H].
 * The effective weight is (float)q * scale; the kernels accumulate
 * sum x*q in fp32 and multiply by the row's scale.  H and I must be
 * multiples of 16.  Otherwise as above.
 */
moe_status moe_grouped_gemm_swiglu_w8(const uint16_t *x_perm, const int32_t *offsets, int G,
                                      int M, int H, int I, const int8_t *q_gu, const float *s_gu,
                                      const int8_t *q_down, const float *s_down,
                                      uint16_t *y_perm, void *workspace, size_t workspace_bytes,
                                      int32_t *dev_error, cudaStream_t stream);
moe_status moe_grouped_gemv_w8(const uint16_t *x_perm, const int32_t *offsets, int G, int M,
                               int H, int I, const int8_t *q_gu, const float *s_gu,
                               const int8_t *q_down, const float *s_down, uint16_t *y_perm,
                               void *workspace, size_t workspace_bytes, int32_t *dev_error,
                               cudaStream_t stream);

/*
 * moe_grouped_gemv_noalloc -- moe_grouped_gemv without a workspace argument,
 * for callers that cannot allocate device memory: code running inside a host
 * framework's execute callback that hands out no allocator, latency-critical
 * paths that cannot afford the device-wide synchronisation cudaMalloc and
 * cudaFree may cause, and processes whose device memory is already handed to
 * a pool of their own.  The pages have no counterpart of this call.
 * The hidden rows h [M,I] go to an 8 MiB scratch array built into the
 * library (every GPU that loads libmoe.so holds it until the process exits),
 * so M * I must be at most 4,194,304; a larger problem returns
 * MOE_ERR_WORKSPACE without launching anything.  The first call on a device
 * looks up the array's device address (cudaGetSymbolAddress, with that
 * device current) and caches it; make that first call before any stream
 * capture.  Every call on a device shares the one array and leaves its
 * contents behind: calls whose kernels may overlap on the GPU (different
 * streams without ordering between them) race on it and must be serialised
 * by the caller.  No part of the array needs to start at zero.  Arguments
 * and results are otherwise those of moe_grouped_gemv; no allocation of any
 * kind is made.
 */
moe_status moe_grouped_gemv_noalloc(const uint16_t *x_perm, const int32_t *offsets, int G, int M,
                                    int H, int I, const uint16_t *w_gu, const uint16_t *w_down,
                                    uint16_t *y_perm, int32_t *dev_error, cudaStream_t stream);

/*
 * moe_combine -- weighted sum of each token's expert rows back in token
 * order, by gathering (no scatter-add, so the result is the same bytes on
 * every run; the "Phase 6" pull request of "dispatch", Summary, reports
 * the atomic index_add_ combine as not bitwise deterministic).
 *   out[t] = bf16( sum_{j<k} topk_w[t,j] * y_perm[row_of_slot[t*k+j]]
 *                  + sum_{s<S} y_perm[T*k + s*T + t]  (+ residual[t]) )
 * summed in fp32 in that order.  y_perm: [M,H] bf16; row_of_slot: [T*k];
 * topk_w: [T,k] fp32; residual: [T,H] bf16 or NULL; out: [T,H] bf16 (may
 * alias residual; device memory or mapped pinned host memory, which the
 * kernel's stores reach over NVLink-C2C).  A row index outside [0, T*k) is
 * skipped.
 */
moe_status moe_combine(const uint16_t *y_perm, const int32_t *row_of_slot, const float *topk_w,
                       int T, int k, int S, int H, const uint16_t *residual, uint16_t *out,
                       int32_t *dev_error, cudaStream_t stream);

/*
 * moe_combine_capped -- moe_combine after moe_permute_capped: a slot whose
 * row_of_slot is MOE_ROW_DROPPED adds nothing (the kept weights are not
 * renormalised), and the shared rows are read from offsets[E] + s*T + t.
 *   out[t] = bf16( sum_{j<k, slot kept} topk_w[t,j] * y_perm[row_of_slot[t*k+j]]
 *                  + sum_{s<S} y_perm[offsets[E] + s*T + t]  (+ residual[t]) )
 * offsets: [E+S+1] from moe_permute_capped (read on the device; an
 * offsets[E] outside [0, T*k] is a device-check fault and the shared rows
 * are skipped).  Other arguments as for moe_combine.
 */
moe_status moe_combine_capped(const uint16_t *y_perm, const int32_t *row_of_slot,
                              const float *topk_w, const int32_t *offsets, int E, int T, int k,
                              int S, int H, const uint16_t *residual, uint16_t *out,
                              int32_t *dev_error, cudaStream_t stream);

/*
 * moe_decode_workspace_size -- bytes of device workspace moe_decode_layer
 * needs: a grid-barrier word plus the hidden rows h [M,I] and the expert
 * outputs y [M,H] (bf16), M = T*k + S*T.  0 for invalid sizes.
 */
size_t moe_decode_workspace_size(int T, int E, int S, int k, int H, int I);

/*
 * moe_decode_layer -- a whole decode-sized MoE layer in one cooperative
 * launch: moe_route, the stable sort of the T*k slots by expert, the grouped
 * GEMV gate/up + SwiGLU, the grouped GEMV down and moe_combine, with grid
 * barriers between the phases.  The pages' kernels trail most at one token
 * ("dispatch", Phase 6 pull request, Summary), where a layer is several
 * short launches around one weight stream; here it is one.
 * The result is the same bytes as moe_route -> moe_permute ->
 * moe_grouped_gemv -> moe_combine on the same inputs.
 * logits: [T,E] fp32; x: [T,H] bf16 (read by token, no gathered copy);
 * w_gu: [E+S,2I,H]; w_down: [E+S,H,I] bf16; residual: [T,H] bf16 or NULL;
 * out: [T,H] bf16 (may alias residual; device memory or mapped pinned host
 * memory, as for moe_combine); topk_ids: [T,k] int32 and
 * topk_w: [T,k] fp32 are written (NULL to skip).  workspace: at least
 * moe_decode_workspace_size bytes, 16-byte aligned, owned by the caller and
 * not shared with work in flight on another stream.
 * Limits (else MOE_ERR_UNSUPPORTED): T <= 8, T*k <= 64, S*T <= 64, S <= 32,
 * E <= 256; H and I multiples of 8.  The grid barriers wait at most 1 s:
 * on running out a CTA records MOE_ERR_TIMEOUT in dev_error and returns.
 */
moe_status moe_decode_layer(const float *logits, const uint16_t *x, int T, int E, int S, int k,
                            int renormalize, int H, int I, const uint16_t *w_gu,
                            const uint16_t *w_down, const uint16_t *residual, uint16_t *out,
                            int32_t *topk_ids, float *topk_w, void *workspace,
                            size_t workspace_bytes, int32_t *dev_error, cudaStream_t stream);

/*
 * moe_copy -- copy `bytes` bytes from src to dst with the GPU's SMs (a
 * grid-stride kernel of 16-byte loads and stores), for moving a layer's
 * inputs in and its output out of pinned host memory: pinned host memory
 * (cudaHostAlloc) is mapped into the device's address space, and on GB300
 * the SMs reach it over NVLink-C2C.  Either pointer may be device memory or
 * mapped pinned host memory; the regions must not overlap.  bytes must be a
 * multiple of 16 and both pointers 16-byte aligned (else MOE_ERR_ALIGNMENT).
 * Asynchronous on `stream`; may be captured into a CUDA graph.
 */
moe_status moe_copy(void *dst, const void *src, size_t bytes, cudaStream_t stream);

/*
 * moe_quantize_w8 -- offline, host-side int8 quantisation of expert
 * weights ("dispatch" README, phase 5a: self-computed per-channel scales).
 * w_host: [rows, K] bf16 bits in host memory; q_host: [rows, K] int8 and
 * scale_host: [rows] fp32, host memory.  Per row: scale = max|w| / 127 in
 * fp32 (1 for an all-zero row); q = clamp(round-half-even(w / scale),
 * -127, 127), the quotient taken in fp32.  Synchronous; no device work.
 */
moe_status moe_quantize_w8(const uint16_t *w_host, int64_t rows, int64_t K, int8_t *q_host,
                           float *scale_host);

/*
 * moe_ep_plan -- host-side exchange plan for expert parallelism over W
 * ranks (the "switchyard" page, Expert parallelism from the kernels up and
 * Peer-to-peer dispatch: each GPU owns part of every layer's experts, rows
 * travel to their expert's GPU after the sort and come back before the
 * combine, and the output equals one GPU's).  Rank p owns the routed
 * experts [p E/W, (p+1) E/W) (E % W == 0); shared experts are replicated
 * and their rows never move.  No device work and no communication: the
 * caller moves the rows (peer copies, a collective) as the plan says.
 *   counts: [W][E] int32, host: counts[r*E + e] = rows rank r routed to
 *           expert e (the differences of rank r's moe_permute offsets),
 *           gathered from every rank by the caller.
 *   send_offset/send_count [W]: rows [send_offset[p], +send_count[p]) of
 *           this rank's x_perm go to rank p (contiguous: the rows are sorted
 *           by expert); the results come back to the same range of y_perm.
 *   recv_offset/recv_count [W]: rank p's rows land at recv_offset[p] of a
 *           source-major receive buffer of sum(recv_count) rows.
 *   seg_src/seg_dst/seg_len [W * E/W]: segment (p, j) moves seg_len rows
 *           from row seg_src of the receive buffer to row seg_dst of the
 *           expert-major FFN input (the reverse moves bring the FFN output
 *           back to source-major order for the return trip).
 *   local_offsets [E/W + 1] int32: the offsets table of the expert-major
 *           rows for the grouped FFN over this rank's experts (append the
 *           rank's own shared rows after it for G = E/W + S groups).
 * Errors: MOE_ERR_INVALID_ARG for NULL pointers, W < 1, E % W != 0, a rank
 * outside [0, W) or a negative count; MOE_ERR_UNSUPPORTED when the
 * received rows exceed 2^31 - 1.  Nothing is written on error paths that
 * fail the argument checks.
 */
moe_status moe_ep_plan(const int32_t *counts, int W, int E, int rank, int64_t *send_offset,
                       int64_t *send_count, int64_t *recv_offset, int64_t *recv_count,
                       int64_t *seg_src, int64_t *seg_dst, int64_t *seg_len,
                       int32_t *local_offsets);

/*
 * moe_selftest_bounded_wait -- runs one of the library's bounded device
 * waits, with a short limit, on a condition that is met (satisfiable != 0)
 * or never met, so that a test can see the failure-detection path work
 * without faulting or hanging the GPU.  The pages have no counterpart: it
 * exercises this library's own rule that no device wait is unbounded.
 *   kind 0: the grid barrier of moe_decode_layer (a cooperative launch of 2
 *           CTAs; the unmet form waits for one arrival more than the grid
 *           makes);
 *   kind 1: one thread's mbarrier wait of the tensor-core kernels (the unmet
 *           form waits on an mbarrier nobody arrives at);
 *   kind 2: the warp-uniform mbarrier wait that precedes tcgen05.ld / .st.
 * limit_ns: the wait's limit in ns of %globaltimer, 1e3 .. 1e10 (the
 * kernels themselves use 1 s).  counters: 2 device words, zeroed by the
 * call; counters[0] = grid-barrier arrivals (kind 0: ends at 2),
 * counters[1] = waits that completed (kind 0: 2 CTAs, kind 1: 1, kind 2: 32
 * lanes; 0 when the limit ran out).  When a limit runs out the kernel
 * writes MOE_ERR_TIMEOUT to *dev_error and returns; nothing else is in
 * flight.  Asynchronous on `stream`.
 */
moe_status moe_selftest_bounded_wait(int kind, int satisfiable, uint64_t limit_ns,
                                     unsigned *counters, int32_t *dev_error, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
