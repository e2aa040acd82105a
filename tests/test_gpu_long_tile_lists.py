"""CTA-pair GEMMs whose tile list is longer than the per-pair cache.

The pair kernels (bf16 `tc_grouped_gemm_pair`, int8 `tc_grouped_gemm_pair_w8`)
decode the first 128 tiles of a pair's round-robin share into shared memory
at kernel start and decode every later tile from the group table when it
comes up.  A narrow layer (H = I = 128, two experts, both chosen by every
token) with 1.4 M tokens puts 1.4 M rows on each expert: about 11 000 bf16
tiles of at most 256 tokens and 15 000 int8 tiles of at most 192 over the
GPU's pairs, so every pair runs past its cache in both kernels.  Routing and
offsets are compared bit for bit, the layer output on sampled tokens
against the oracle (fp64; bf16 weights, and the same weights quantised to
int8 by the library's host quantiser).
"""
import numpy as np
import pytest
import torch

import oracle
from grouped_expert_gemm_moe_gb300 import workloads as W

from gpu_helpers import assert_close, host_inputs, sample_tokens, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
NARROW = W.MoEShape("narrow", H=128, E=2, k=2, I=128)
T = 1_400_000
TILE_CACHE = 128          # tiles a pair decodes at kernel start


@pytest.fixture(scope="module")
def mods():
    import __graft_entry__ as g
    g.build()
    from grouped_expert_gemm_moe_gb300 import binding, layer
    return binding, layer


@pytest.fixture(scope="module")
def case():
    inp = W.make_layer(NARROW, T, "uniform", seed=11, device=DEV)
    h = host_inputs(inp)
    ids, w = oracle.route(h["logits"], NARROW.k, NARROW.renormalize)
    return inp, h, ids, w


def _pairs_at_most():
    return torch.cuda.get_device_properties(0).multi_processor_count // 2


def _check_routing(layer, ids):
    b = layer.buffers(T)
    np.testing.assert_array_equal(b.topk_ids.cpu().numpy(), ids)
    np.testing.assert_array_equal(b.offsets.cpu().numpy(),
                                  oracle.permute(ids, NARROW.E, NARROW.S)[0])


def test_bf16_pair_tile_list_past_the_cache(mods, case):
    B, L = mods
    inp, h, ids, w = case
    # every token goes to both experts: T rows per expert, m-blocks of <= 256
    assert 2 * ((T + 255) // 256) > TILE_CACHE * _pairs_at_most()
    layer = L.MoELayer(NARROW.H, NARROW.E, NARROW.k, NARROW.I, NARROW.S, NARROW.renormalize,
                       w_gu=inp.w_gu, w_down=inp.w_down, device=DEV)
    out = layer.forward(inp.x, inp.logits, ffn="gemm")
    layer.check()
    _check_routing(layer, ids)
    tok = sample_tokens(T, n=48, seed=3)
    y = oracle.moe_layer(h["x"], ids, w, NARROW.E, NARROW.S, h["w_gu"], h["w_down"], tokens=tok)
    assert_close(to_np(out[torch.from_numpy(tok).to(DEV)]), y, "bf16 pair, long tile lists")


def test_int8_pair_tile_list_past_the_cache(mods, case):
    B, L = mods
    inp, h, ids, w = case
    assert 2 * ((T + 191) // 192) > TILE_CACHE * _pairs_at_most()
    q_gu, s_gu = B.moe_quantize_w8(inp.w_gu)
    q_down, s_down = B.moe_quantize_w8(inp.w_down)
    layer = L.MoELayer(NARROW.H, NARROW.E, NARROW.k, NARROW.I, NARROW.S, NARROW.renormalize,
                       q_gu=q_gu.to(DEV), s_gu=s_gu.to(DEV), q_down=q_down.to(DEV),
                       s_down=s_down.to(DEV), device=DEV)
    out = layer.forward(inp.x, inp.logits, ffn="gemm")
    layer.check()
    _check_routing(layer, ids)
    tok = sample_tokens(T, n=48, seed=4)
    y = oracle.moe_layer_w8(h["x"], ids, w, NARROW.E, NARROW.S, q_gu.numpy(), s_gu.numpy(),
                            q_down.numpy(), s_down.numpy(), tokens=tok)
    assert_close(to_np(out[torch.from_numpy(tok).to(DEV)]), y, "int8 pair, long tile lists")
