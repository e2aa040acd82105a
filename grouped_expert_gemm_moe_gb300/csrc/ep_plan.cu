// ep_plan.cu -- host-side exchange plan for expert parallelism over W ranks.
//
// The "switchyard" page (Expert parallelism from the kernels up;
// Peer-to-peer dispatch) splits every layer's experts between GPUs: each
// GPU routes and sorts its own tokens, sends the rows routed to the other
// GPU's experts there, runs the grouped FFN over the rows it owns, and
// sends the results back before the combine; the page reports the output
// bit-identical to one GPU.  This file computes, on the host, where every
// row goes, for any W that divides E:
//
//  * rank p owns the E/W consecutive routed experts [p E/W, (p+1) E/W);
//    shared experts are replicated and applied by each rank to its own
//    tokens, so shared rows never move;
//  * a rank's permuted rows are sorted by expert (moe_permute), so the rows
//    it sends to rank p are one contiguous range of its x_perm:
//    [offsets[p E/W], offsets[(p+1) E/W]);
//  * a receiving rank lays the rows it gets out source-major (rank 0's
//    message, then rank 1's, ...) and moves them into expert-major order
//    (expert e: rank 0's rows of e, then rank 1's, ...) with W * E/W
//    segment copies, which gives the offsets table of its grouped FFN;
//  * the results travel the same way back: the inverse segment moves, then
//    each source gets back exactly the range it sent, so its y_perm holds
//    every routed row at the position a single GPU would have written it,
//    and moe_combine (fixed order) gives the single-GPU bytes.
// No device work: the data plane (peer copies or a collective) belongs to
// the caller.
#include <stdint.h>

#include "moe.h"

extern "C" moe_status moe_ep_plan(const int32_t *counts, int W, int E, int rank,
                                  int64_t *send_offset, int64_t *send_count,
                                  int64_t *recv_offset, int64_t *recv_count, int64_t *seg_src,
                                  int64_t *seg_dst, int64_t *seg_len, int32_t *local_offsets) {
    if (!counts || !send_offset || !send_count || !recv_offset || !recv_count || !seg_src ||
        !seg_dst || !seg_len || !local_offsets)
        return MOE_ERR_INVALID_ARG;
    if (W < 1 || E < 1 || E % W != 0 || rank < 0 || rank >= W) return MOE_ERR_INVALID_ARG;
    const int EL = E / W;                    // experts per rank
    for (int64_t i = 0; i < static_cast<int64_t>(W) * E; ++i)
        if (counts[i] < 0) return MOE_ERR_INVALID_ARG;

    // what this rank sends: its rows of rank p's experts, one contiguous range
    int64_t off = 0;
    for (int p = 0; p < W; ++p) {
        int64_t n = 0;
        for (int e = p * EL; e < (p + 1) * EL; ++e) n += counts[static_cast<int64_t>(rank) * E + e];
        send_offset[p] = off;
        send_count[p] = n;
        off += n;
    }
    // what it receives: rank p's rows of this rank's experts, source-major
    const int e0 = rank * EL;
    int64_t roff = 0;
    for (int p = 0; p < W; ++p) {
        int64_t n = 0;
        for (int e = e0; e < e0 + EL; ++e) n += counts[static_cast<int64_t>(p) * E + e];
        recv_offset[p] = roff;
        recv_count[p] = n;
        roff += n;
    }
    // expert-major layout of the received rows: expert e0 + j holds rank 0's
    // rows of it, then rank 1's, ...
    int64_t acc = 0;
    for (int j = 0; j < EL; ++j) {
        local_offsets[j] = static_cast<int32_t>(acc);
        for (int p = 0; p < W; ++p) acc += counts[static_cast<int64_t>(p) * E + e0 + j];
    }
    local_offsets[EL] = static_cast<int32_t>(acc);
    if (acc > INT32_MAX) return MOE_ERR_UNSUPPORTED;
    // segment (p, j): rank p's rows of expert e0 + j, from the source-major
    // buffer to the expert-major one
    for (int p = 0; p < W; ++p) {
        int64_t src = recv_offset[p];
        for (int j = 0; j < EL; ++j) {
            int64_t before = 0;              // earlier ranks' rows of the same expert
            for (int q = 0; q < p; ++q) before += counts[static_cast<int64_t>(q) * E + e0 + j];
            const int64_t n = counts[static_cast<int64_t>(p) * E + e0 + j];
            const int64_t s = static_cast<int64_t>(p) * EL + j;
            seg_src[s] = src;
            seg_dst[s] = local_offsets[j] + before;
            seg_len[s] = n;
            src += n;
        }
    }
    return MOE_OK;
}
