"""The single-launch decode layer (moe_decode_layer) on the GPU.

It fuses routing, the grouped GEMV (gate/up + SwiGLU, down) and the combine
of a decode-sized batch (T <= 8) into one cooperative launch.  Bars: the
same bytes as the separate calls (moe_route + moe_permute +
moe_grouped_gemv + moe_combine) on the same inputs, routing ids bit-exact
against the oracle, and the layer within the usual bounds of the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from grouped_expert_gemm_moe_gb300 import workloads as W

from gpu_helpers import assert_close, host_inputs, oracle_out, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def mods():
    import __graft_entry__ as g
    g.build()
    from grouped_expert_gemm_moe_gb300 import binding, layer
    return binding, layer


_LAYERS = {}


def _layer(L, name):
    if name not in _LAYERS:
        _LAYERS.clear()
        sh = W.CONFIGS[name]
        inp = W.make_layer(sh, 1, "uniform", seed=0, device=DEV)
        _LAYERS[name] = (inp, L.MoELayer(sh.H, sh.E, sh.k, sh.I, sh.S, sh.renormalize,
                                         w_gu=inp.w_gu, w_down=inp.w_down, device=DEV))
    return _LAYERS[name]


def _batch(sh, inp, T, routing, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((T, sh.H), generator=g).to(torch.bfloat16)
    logits = W.router_logits_input(x, inp.w_r.cpu(), W.routing_bias(sh, routing))
    return x.to(DEV), logits.to(DEV)


@pytest.mark.parametrize("name,T,routing", [("olmoe", 1, "uniform"), ("olmoe", 2, "uniform"),
                                            ("olmoe", 4, "uniform"), ("olmoe", 8, "uniform"),
                                            ("deepseek", 1, "uniform"), ("deepseek", 4, "zipf"),
                                            ("deepseek", 8, "zipf")])
def test_decode_layer_equals_separate_calls_and_oracle(mods, name, T, routing):
    B, L = mods
    inp, layer = _layer(L, name)
    sh = inp.shape
    x, logits = _batch(sh, inp, T, routing, seed=T * 7 + 1)
    res = torch.randn((T, sh.H), generator=torch.Generator().manual_seed(5)).to(
        torch.bfloat16).to(DEV)
    for residual in (None, res):
        sep = layer.forward(x, logits, residual=residual, ffn="gemv").clone()
        layer.check()
        fused = layer.forward(x, logits, residual=residual, ffn="decode").clone()
        layer.check()
        assert torch.equal(fused, sep), f"{name} T={T} residual={residual is not None}"
    b = layer.buffers(T)
    ids, w = oracle.route(logits.cpu().numpy(), sh.k, sh.renormalize)
    np.testing.assert_array_equal(b.topk_ids.cpu().numpy(), ids)
    y = oracle.moe_layer(W.bf16_bits(x.cpu()), ids, w, sh.E, sh.S, W.bf16_bits(inp.w_gu),
                         W.bf16_bits(inp.w_down), residual_bits=W.bf16_bits(res.cpu()))
    assert_close(to_np(fused), y, f"decode layer {name} T={T}")


def test_decode_layer_repeat_and_graph_replay(mods):
    """The in-launch barrier counter is reset for every call: back-to-back
    calls and CUDA-graph replays give the same bytes."""
    B, L = mods
    inp, layer = _layer(L, "olmoe")
    x, logits = _batch(inp.shape, inp, 2, "uniform", seed=3)
    first = layer.forward(x, logits, ffn="decode").clone()
    for _ in range(5):
        again = layer.forward(x, logits, ffn="decode")
        assert torch.equal(again, first)
    cap = layer.capture(x, logits, ffn="decode")
    for _ in range(3):
        assert torch.equal(cap.replay(), first)
    layer.check()


def test_decode_layer_limits(mods):
    B, L = mods
    inp, layer = _layer(L, "olmoe")
    assert not layer.decode_layer_ok(9)
    assert not layer.decode_layer_ok(1, torch.float32)
    x, logits = _batch(inp.shape, inp, 9, "uniform", seed=4)
    ws = torch.empty(B.moe_decode_workspace_size(9, 64, 0, 8, 2048, 1024), dtype=torch.uint8,
                     device=DEV)
    out = torch.empty_like(x)
    with pytest.raises(B.MoEError):
        B.moe_decode_layer(logits, x, 8, False, 0, inp.w_gu, inp.w_down, out, ws)


def test_decode_layer_nan_logit_is_reported(mods):
    B, L = mods
    inp, layer = _layer(L, "olmoe")
    x, logits = _batch(inp.shape, inp, 3, "uniform", seed=6)
    logits[1, 5] = float("nan")
    layer.forward(x, logits, ffn="decode")
    with pytest.raises(Exception):
        layer.check()
