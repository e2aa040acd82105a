"""Expert parallelism over W ranks: the exchange plan (moe_ep_plan, host C)
and a 2-rank run of the whole data path over gloo on CPU.

The "switchyard" page (Expert parallelism from the kernels up; Peer-to-peer
dispatch) splits each layer's experts between two GPUs and reports the
output equal to one GPU's.  Here every rank routes and sorts its own tokens
(the oracle's route and permute), the plan says which rows go where, the
rows travel with all_to_all over gloo, the owning rank computes the expert
FFN of each row (the oracle's expert FFN, fp64), the results travel back,
and the rank's y_perm must equal, bit for bit, the rows one GPU computes for
the same tokens; the combined output must match the oracle's layer.  No GPU
is involved: this covers the host plan and the ordering, not a device data
plane.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


@pytest.fixture(scope="module")
def B():
    import __graft_entry__ as g
    g.build()
    from grouped_expert_gemm_moe_gb300 import binding
    return binding


def test_single_rank_plan_is_the_identity(B):
    counts = np.array([[3, 0, 5, 2]])
    p = B.moe_ep_plan(counts, 0)
    assert p["send_offset"].tolist() == [0] and p["send_count"].tolist() == [10]
    assert p["recv_count"].tolist() == [10]
    assert p["local_offsets"].tolist() == [0, 3, 3, 8, 10]
    assert p["seg_src"].tolist() == p["seg_dst"].tolist() == [0, 3, 3, 8]


@pytest.mark.parametrize("W,E", [(2, 8), (4, 64), (8, 64), (2, 2)])
def test_plan_partitions_every_row(B, W, E):
    rng = np.random.default_rng(W * 100 + E)
    counts = rng.integers(0, 9, size=(W, E))
    counts[0, 0] = 0                                     # empty experts happen
    EL = E // W
    recv_from = np.zeros((W, W), np.int64)                # [receiver, sender]
    for r in range(W):
        p = B.moe_ep_plan(counts, r)
        # what r sends to q: its rows of q's experts, contiguous and in order
        ends = np.cumsum(counts[r])
        starts = ends - counts[r]
        for q in range(W):
            assert p["send_offset"][q] == starts[q * EL]
            assert p["send_count"][q] == counts[r, q * EL:(q + 1) * EL].sum()
        assert p["send_count"].sum() == counts[r].sum()
        # what r receives: sender-major, then moved to expert-major
        total = counts[:, r * EL:(r + 1) * EL].sum()
        assert p["local_offsets"][-1] == total
        assert (np.diff(p["local_offsets"]) == counts[:, r * EL:(r + 1) * EL].sum(0)).all()
        recv_from[r] = p["recv_count"]
        src_cover = np.zeros(total, np.int64)
        dst_cover = np.zeros(total, np.int64)
        for q in range(W):
            for j in range(EL):
                s = q * EL + j
                n = p["seg_len"][s]
                assert n == counts[q, r * EL + j]
                src_cover[p["seg_src"][s]:p["seg_src"][s] + n] += 1
                dst_cover[p["seg_dst"][s]:p["seg_dst"][s] + n] += 1
                # inside expert j, sender q's rows follow those of senders < q
                assert p["seg_dst"][s] == p["local_offsets"][j] + counts[:q, r * EL + j].sum()
        assert (src_cover == 1).all() and (dst_cover == 1).all()
    # every row sent is received: send_count[r][q] == recv_count[q][r]
    for r in range(W):
        p = B.moe_ep_plan(counts, r)
        assert (p["send_count"] == recv_from[:, r]).all()


def test_plan_refuses_bad_arguments(B):
    with pytest.raises(B.MoEError):
        B.moe_ep_plan(np.zeros((3, 8)), 0)               # E % W != 0
    with pytest.raises(B.MoEError):
        B.moe_ep_plan(np.zeros((2, 8)), 2)               # rank outside [0, W)
    bad = np.zeros((2, 8))
    bad[1, 3] = -1
    with pytest.raises(B.MoEError):
        B.moe_ep_plan(bad, 0)


# ------------------------------------------------------------------ 2 ranks

H, I, E, K, S = 32, 16, 8, 2, 1


def _bits(rng, shape, std):
    t = torch.from_numpy((rng.standard_normal(shape) * std).astype(np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _val(b):
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _weights():
    rng = np.random.default_rng(7)                      # the same on every rank
    return _bits(rng, (E + S, 2 * I, H), 0.2), _bits(rng, (E + S, H, I), 0.2)


def _tokens(rank):
    rng = np.random.default_rng(100 + rank)
    T = 11 + 6 * rank
    return _bits(rng, (T, H), 1.0), rng.standard_normal((T, E)).astype(np.float32)


def _ffn(oracle, xrow_bits, e, w_gu, w_down):
    h = oracle.expert_hidden(_val(xrow_bits), w_gu[e], H, I)
    return oracle.expert_down(h, w_down[e], H, I)


def _ep_rank(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import oracle
    from grouped_expert_gemm_moe_gb300 import binding as B
    try:
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        dist.init_process_group("gloo", rank=rank, world_size=world)
        w_gu, w_down = _weights()
        x, logits = _tokens(rank)
        T = x.shape[0]
        ids, w = oracle.route(logits, K, True)
        off, ss, _ = oracle.permute(ids, E, S)
        tok = np.concatenate([ss // K] + [np.arange(T)] * S)    # token of each permuted row
        row_e = np.repeat(np.arange(E + S), np.diff(off))      # group of each permuted row
        x_perm = x[tok]
        n_routed = T * K
        # every rank's rows per routed expert
        mine = torch.from_numpy(np.diff(off)[:E].astype(np.int64))
        allc = [torch.zeros(E, dtype=torch.int64) for _ in range(world)]
        dist.all_gather(allc, mine)
        counts = torch.stack(allc).numpy()
        plan = B.moe_ep_plan(counts, rank)
        # dispatch: routed rows to their expert's rank (values as fp64)
        send = torch.from_numpy(_val(x_perm[:n_routed]))
        recv = torch.zeros((int(plan["recv_count"].sum()), H), dtype=torch.float64)
        dist.all_to_all_single(recv, send, output_split_sizes=plan["recv_count"].tolist(),
                               input_split_sizes=plan["send_count"].tolist())
        EL = E // world
        xin = torch.zeros_like(recv)
        for s in range(world * EL):
            a, d, n = plan["seg_src"][s], plan["seg_dst"][s], plan["seg_len"][s]
            xin[d:d + n] = recv[a:a + n]
        # the owner's grouped FFN, rows of local expert j at local_offsets[j]..
        lo = plan["local_offsets"]
        yin = torch.zeros_like(xin)
        for j in range(EL):
            for r in range(lo[j], lo[j + 1]):
                h = oracle.expert_hidden(xin[r].numpy(), w_gu[rank * EL + j], H, I)
                yin[r] = torch.from_numpy(oracle.expert_down(h, w_down[rank * EL + j], H, I))
        # return trip: expert-major -> sender-major -> back to each sender
        yback = torch.zeros_like(yin)
        for s in range(world * EL):
            a, d, n = plan["seg_src"][s], plan["seg_dst"][s], plan["seg_len"][s]
            yback[a:a + n] = yin[d:d + n]
        y_routed = torch.zeros((n_routed, H), dtype=torch.float64)
        dist.all_to_all_single(y_routed, yback, output_split_sizes=plan["send_count"].tolist(),
                               input_split_sizes=plan["recv_count"].tolist())
        # shared rows stay on this rank
        y_perm = np.zeros((len(tok), H))
        y_perm[:n_routed] = y_routed.numpy()
        for r in range(n_routed, len(tok)):
            y_perm[r] = _ffn(oracle, x_perm[r], row_e[r], w_gu, w_down)
        # one GPU's rows for the same tokens, computed row by row
        ref = np.stack([_ffn(oracle, x_perm[r], row_e[r], w_gu, w_down) for r in range(len(tok))])
        same_rows = bool(np.array_equal(y_perm, ref))
        # combine in the fixed order (routed j = 0..k-1, then shared) vs the oracle's layer
        ros = np.empty(n_routed, np.int64)
        ros[ss] = np.arange(n_routed)
        out = np.zeros((T, H))
        for t in range(T):
            for j in range(K):
                out[t] += w[t, j] * y_perm[ros[t * K + j]]
            for s_ in range(S):
                out[t] += y_perm[n_routed + s_ * T + t]
        layer = oracle.moe_layer(x, ids, w, E, S, w_gu, w_down)
        err = float(np.abs(out - layer).max() / np.abs(layer).max())
        moved = int(sum(plan["send_count"]) - plan["send_count"][rank])
        q.put((rank, same_rows, err, moved, None))
        dist.destroy_process_group()
    except Exception as exc:           # report to the parent instead of hanging it
        q.put((rank, False, 1.0, 0, repr(exc)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_ranks_give_one_gpus_rows(B):
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_ep_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=180) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
    for rank, same_rows, err, moved, exc in out:
        assert exc is None, f"rank {rank}: {exc}"
        assert same_rows, f"rank {rank}: y_perm differs from one GPU's rows"
        assert err <= 1e-12, f"rank {rank}: combined output off by {err:.2e}"
        assert moved > 0                                # rows really crossed ranks
    for p in procs:
        assert p.exitcode == 0
