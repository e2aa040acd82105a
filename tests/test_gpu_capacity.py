"""The capacity-limited (token-dropping) variant on the GPU against the oracle.

Reading of the "switchyard" page (03 Load balance, "What dropping tokens
costs"): routed expert e serves at most C = ceil(CF * T*k / E) of its slots,
the first ones in slot order; a dropped slot adds nothing; shared experts
are never capped.  Bars: offsets, sorted_slot, row_of_slot, the dropped
count and the gathered rows bit-exact (the same integer work); layer
outputs within the dropless layer's bounds (rel Frobenius 5e-3, max
2e-2 * max|ref|) of the oracle's capped layer.
"""
import numpy as np
import pytest
import torch

import oracle
from grouped_expert_gemm_moe_gb300 import workloads as W

from gpu_helpers import assert_close, host_inputs, sample_tokens, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def mods():
    import __graft_entry__ as g
    g.build()
    from grouped_expert_gemm_moe_gb300 import binding, layer
    return binding, layer


def _skewed_ids(T, E, k, seed, s=1.0):
    rng = np.random.default_rng(seed)
    p = np.arange(1, E + 1, dtype=np.float64) ** -s
    p /= p.sum()
    return np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,E,k,S", [(40, 16, 4, 0),      # 160 slots: one-launch path
                                     (64, 64, 8, 2),      # 512 slots, shared experts
                                     (700, 32, 3, 1),     # 2100 slots: count/place/gather path
                                     (2048, 64, 6, 2)])   # 12288 slots, DeepSeek-like
def test_capped_permute_bit_exact(mods, T, E, k, S):
    B, _ = mods
    ids = _skewed_ids(T, E, k, seed=T + E)
    H = 64
    g = torch.Generator().manual_seed(T)
    x = torch.randn((T, H), generator=g).to(torch.bfloat16)
    counts = np.bincount(ids.ravel(), minlength=E)
    caps = sorted({0, 1, B.capacity_of(1.0, T, k, E), B.capacity_of(2.0, T, k, E),
                   int(counts.max()), int(counts.max()) + 5})
    M = T * k + S * T
    pws = B.moe_permute_workspace_size(T, E, S, k)
    ws = torch.empty(max(pws, 1), dtype=torch.uint8, device=DEV) if pws else None
    err = B.new_error_word(DEV)
    for C in caps:
        off = torch.full((E + S + 1,), 7, dtype=torch.int32, device=DEV)
        ss = torch.full((T * k,), 7, dtype=torch.int32, device=DEV)
        ros = torch.full((T * k,), 7, dtype=torch.int32, device=DEV)
        xp = torch.zeros((M, H), dtype=torch.bfloat16, device=DEV)
        dropped = torch.full((1,), -5, dtype=torch.int32, device=DEV)
        B.moe_permute_capped(torch.from_numpy(ids).to(DEV), E, S, C, x.to(DEV), off, ss, ros, xp,
                             dropped, ws, err)
        B.check_device_error(err, "capped permute")
        roff, rss, rros, rdrop = oracle.permute_capped(ids, E, S, C)
        np.testing.assert_array_equal(off.cpu().numpy(), roff, err_msg=f"C={C}")
        np.testing.assert_array_equal(ss.cpu().numpy(), rss, err_msg=f"C={C}")
        np.testing.assert_array_equal(ros.cpu().numpy(), rros, err_msg=f"C={C}")
        assert int(dropped.item()) == rdrop
        rows = int(roff[-1])
        tok = np.concatenate([rss[:roff[E]] // k] + [np.arange(T)] * S)
        assert torch.equal(xp[:rows].cpu(), x[torch.from_numpy(tok).long()])


@pytest.mark.parametrize("ffn", ["gemm", "gemv"])
@pytest.mark.parametrize("name,T,routing,cf", [("olmoe", 64, "zipf", 1.0),
                                               ("olmoe", 64, "zipf", 2.0),
                                               ("deepseek", 128, "zipf", 1.0),
                                               ("deepseek", 2048, "zipf", 1.0),
                                               ("deepseek", 2048, "uniform", 1.25)])
def test_capped_layer_matches_oracle(mods, name, T, routing, cf, ffn):
    B, L = mods
    if ffn == "gemv" and T > 512:
        pytest.skip("the GEMV is for decode-sized batches")
    sh = W.CONFIGS[name]
    inp = W.make_layer(sh, T, routing, seed=0, device=DEV)
    h = host_inputs(inp)
    layer = L.MoELayer(sh.H, sh.E, sh.k, sh.I, sh.S, sh.renormalize, w_gu=inp.w_gu,
                       w_down=inp.w_down, device=DEV, capacity_factor=cf)
    out = layer.forward(inp.x, inp.logits, ffn=ffn)
    layer.check()
    b = layer.buffers(T)
    C = B.capacity_of(cf, T, sh.k, sh.E)
    assert b.capacity == C
    ids, w = oracle.route(h["logits"], sh.k, sh.renormalize)
    _, _, _, rdrop = oracle.permute_capped(ids, sh.E, sh.S, C)
    assert int(b.dropped.item()) == rdrop
    tok = sample_tokens(T)
    y = oracle.moe_layer(h["x"], ids, w, sh.E, sh.S, h["w_gu"], h["w_down"], tokens=tok,
                         capacity=C)
    rel, mx = assert_close(to_np(out)[tok], y, f"{name} T={T} {routing} CF={cf} {ffn}")
    print(f"{name} T={T} {routing} CF={cf} {ffn}: dropped {rdrop}/{T * sh.k} "
          f"({100.0 * rdrop / (T * sh.k):.1f} %), rel {rel:.2e}")


def test_large_capacity_equals_dropless_bytes(mods):
    B, L = mods
    sh = W.DEEPSEEK
    T = 512
    inp = W.make_layer(sh, T, "zipf", seed=1, device=DEV)
    free = L.MoELayer(sh.H, sh.E, sh.k, sh.I, sh.S, sh.renormalize, w_gu=inp.w_gu,
                      w_down=inp.w_down, device=DEV)
    capped = L.MoELayer(sh.H, sh.E, sh.k, sh.I, sh.S, sh.renormalize, w_gu=inp.w_gu,
                        w_down=inp.w_down, device=DEV, capacity_factor=float(sh.E))
    a = free.forward(inp.x, inp.logits).clone()
    c = capped.forward(inp.x, inp.logits).clone()
    free.check()
    capped.check()
    assert int(capped.buffers(T).dropped.item()) == 0
    assert torch.equal(a, c)
