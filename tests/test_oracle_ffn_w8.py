"""Pins of the oracle's expert FFN, whole layer and int8 path.

The expert FFN is the SwiGLU MLP of the "switchyard" page (02 Kernels and
dispatch, "One launch for all experts": grouped GEMM with SwiGLU fused in
the epilogue); shared experts come from the "dispatch" README (Stack:
shared + routed experts); int8 is the README's phase-5a per-channel int8
weight-only scheme.  Each check here compares the oracle with something
other than itself: library matmuls in fp64, closed-form special values,
exact constructions and worked examples under tests/golden/.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from grouped_expert_gemm_moe_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bits(a: np.ndarray) -> np.ndarray:
    """bf16 bit patterns of float values that are exact in bf16."""
    t = torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16)
    assert torch.equal(t.float(), torch.from_numpy(np.ascontiguousarray(a, np.float32)))
    return W.bf16_bits(t)


def val(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rand_bf16(rng, shape, std):
    t = torch.from_numpy((rng.standard_normal(shape) * std).astype(np.float32))
    return W.bf16_bits(t.to(torch.bfloat16))


def np_silu(z):
    return z / (1.0 + np.exp(-z))


def dense_ffn(x, wgu_b, wd_b):
    """numpy fp64 SwiGLU MLP: Wd (silu(Wg x) * (Wu x)) for rows of x."""
    I = wgu_b.shape[0] // 2
    wg, wu, wd = val(wgu_b[:I]), val(wgu_b[I:]), val(wd_b)
    return (np_silu(x @ wg.T) * (x @ wu.T)) @ wd.T


def test_silu_special_values():
    H = I = 1
    x = np.array([1.0])
    for z in (0.5, 1.0, 2.0, 3.5, -1.25, 8.0):
        hp = oracle.expert_hidden(x, bits(np.array([[z], [1.0]])), H, I)[0]
        hm = oracle.expert_hidden(x, bits(np.array([[-z], [1.0]])), H, I)[0]
        assert abs((hp - hm) - z) <= 1e-14 * max(1.0, abs(z))     # silu(z) - silu(-z) = z
    assert oracle.expert_hidden(x, bits(np.array([[0.0], [5.0]])), H, I)[0] == 0.0
    assert oracle.expert_hidden(x, bits(np.array([[64.0], [1.0]])), H, I)[0] == 64.0
    assert abs(oracle.expert_hidden(x, bits(np.array([[-64.0], [1.0]])), H, I)[0]) < 1e-25


def test_swiglu_gate_is_first_half():
    # gate row = 32, up row = 1, x = 2: g = 64, u = 2 -> h = silu(64) * 2 = 128.
    # Swapping the halves would give silu(2) * 64 ~ 112.7.
    h = oracle.expert_hidden(np.array([2.0]), bits(np.array([[32.0], [1.0]])), 1, 1)[0]
    assert h == 128.0


def test_down_projection_orientation():
    H = I = 5
    perm = [2, 0, 4, 1, 3]                     # not an involution
    P = np.zeros((H, I))
    P[np.arange(H), perm] = 1.0
    h = np.array([1.0, 2.0, 3.0, 4.0, 5.0])
    y = oracle.expert_down(h, bits(P), H, I)
    np.testing.assert_array_equal(y, h[perm])


@pytest.mark.parametrize("H,I", [(16, 8), (64, 96), (256, 512)])
def test_single_expert_reduces_to_dense_mlp(H, I):
    """E=1, k=1, S=0: the layer is one dense SwiGLU MLP (numpy fp64 matmul)."""
    rng = np.random.default_rng(H + I)
    T = 9
    x = rand_bf16(rng, (T, H), 1.0)
    wgu = rand_bf16(rng, (1, 2 * I, H), 0.02)
    wd = rand_bf16(rng, (1, H, I), 0.02)
    ids = np.zeros((T, 1), np.int32)
    w = np.ones((T, 1))
    y = oracle.moe_layer(x, ids, w, 1, 0, wgu, wd)
    ref = dense_ffn(val(x), wgu[0], wd[0])
    np.testing.assert_allclose(y, ref, rtol=1e-10, atol=1e-13)


def test_layer_matches_dense_all_expert_formulation():
    """y = sum_e g_e FFN_e(x) over ALL experts, g_e = routing weight of e if
    selected else 0, plus shared experts with weight 1 (numpy, fp64)."""
    rng = np.random.default_rng(42)
    T, H, I, E, S, k = 12, 32, 24, 6, 2, 3
    x = rand_bf16(rng, (T, H), 1.0)
    L = rng.standard_normal((T, E)).astype(np.float32)
    ids, w = oracle.route(L, k, renormalize=False)
    wgu = rand_bf16(rng, (E + S, 2 * I, H), 0.05)
    wd = rand_bf16(rng, (E + S, H, I), 0.05)
    res = rand_bf16(rng, (T, H), 1.0)
    y = oracle.moe_layer(x, ids, w, E, S, wgu, wd, residual_bits=res)
    xv = val(x)
    gates = np.zeros((T, E + S))
    for t in range(T):
        for j in range(k):
            gates[t, ids[t, j]] += w[t, j]
    gates[:, E:] = 1.0
    ref = val(res).copy()
    for e in range(E + S):
        ref += gates[:, e:e + 1] * dense_ffn(xv, wgu[e], wd[e])
    np.testing.assert_allclose(y, ref, rtol=1e-10, atol=1e-12)
    # a subset of tokens gives the same rows
    sub = oracle.moe_layer(x, ids, w, E, S, wgu, wd, residual_bits=res, tokens=[11, 0, 5])
    np.testing.assert_array_equal(sub, y[[11, 0, 5]])


def test_layer_fp32_activations():
    rng = np.random.default_rng(4)
    T, H, I, E, k = 4, 16, 8, 4, 2
    x = rng.standard_normal((T, H)).astype(np.float32)
    wgu = rand_bf16(rng, (E, 2 * I, H), 0.1)
    wd = rand_bf16(rng, (E, H, I), 0.1)
    ids = np.array([[0, 1], [3, 2], [1, 0], [2, 3]], np.int32)
    w = rng.random((T, k))
    y = oracle.moe_layer(x, ids, w, E, 0, wgu, wd)
    ref = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            ref[t] += w[t, j] * dense_ffn(x[t:t + 1].astype(np.float64), wgu[e], wd[e])[0]
    np.testing.assert_allclose(y, ref, rtol=1e-10, atol=1e-13)


def _read_quant_golden():
    rows = []
    with open(os.path.join(GOLDEN, "quantize_exact.txt")) as f:
        for line in f:
            if line.startswith("row"):
                parts = line.split("|")
                w = [float(v) for v in parts[0].split()[3:]]
                q = [int(v) for v in parts[1].split()[1:]]
                s = float(parts[2].split()[1])
                rows.append((w, q, s))
    return rows


def test_quantize_golden():
    rows = _read_quant_golden()
    wmat = np.array([r[0] for r in rows]) / 128.0
    q, s = oracle.quantize_w8(bits(wmat))
    np.testing.assert_array_equal(q, np.array([r[1] for r in rows], np.int8))
    np.testing.assert_array_equal(s * 128.0, np.array([r[2] for r in rows], np.float32))


def test_quantize_bounds_and_full_range():
    rng = np.random.default_rng(11)
    wb = rand_bf16(rng, (3, 40, 96), 0.02)
    q, s = oracle.quantize_w8(wb)
    wv = val(wb)
    deq = q.astype(np.float64) * s[..., None].astype(np.float64)
    # |q - W/scale| <= 1/2, plus the fp32 rounding of the quotient W/scale
    # (at most 127 * 2^-24 < 1e-5) that the rounding step sees.
    assert (np.abs(deq - wv) <= s[..., None] * (0.5 + 1e-5)).all()
    assert (np.abs(q).max(axis=-1) == 127).all()


def test_quantize_exact_power_of_two_multiples():
    rng = np.random.default_rng(12)
    m = rng.integers(-127, 128, size=(20, 64))
    m[:, 0] = 127 * rng.choice([-1, 1], size=20)        # max |m| = 127 on every row
    wmat = m / 64.0                                      # scale = 2^-6 exactly
    q, s = oracle.quantize_w8(bits(wmat))
    np.testing.assert_array_equal(q, m.astype(np.int8))
    assert (s == np.float32(1 / 64)).all()


def _exact_w8_matrix(rng, p, K):
    """[..., N, K] matrix whose row n is m * 2^-p[..., n], max |m| = 127 on
    every row, with m returned as well."""
    m = rng.integers(-127, 128, size=p.shape + (K,))
    col = rng.integers(0, K, size=p.shape)
    np.put_along_axis(m, col[..., None], (127 * rng.choice([-1, 1], size=p.shape))[..., None],
                      axis=-1)
    return m * np.exp2(-p.astype(np.float64))[..., None], m


def test_w8_layer_equals_bf16_layer_with_distinct_row_scales():
    """Weights that int8 represents exactly, with a different power-of-two
    scale on every row (gate row i, up row I+i and each down row n all
    differ): the quantiser must return q = m and scale = 2^-p exactly, and
    the w8 layer must equal the bf16 layer of the same weights.  Scales
    applied to the wrong rows (gate/up swapped, down reversed, another
    expert's) must break the equality, so the check can see such a slip."""
    rng = np.random.default_rng(13)
    T, H, I, E, S, k = 6, 32, 16, 4, 1, 2
    G = E + S
    p_gate = rng.integers(6, 11, size=(G, I))
    p_up = p_gate + rng.integers(1, 4, size=(G, I))          # up row I+i != gate row i
    p_gu = np.concatenate([p_gate, p_up], axis=1)
    p_down = rng.integers(6, 14, size=(G, H))
    assert (p_down != p_down[:, ::-1]).any() and (p_down[:-1] != p_down[1:]).any()
    wgu_v, m_gu = _exact_w8_matrix(rng, p_gu, H)
    wd_v, m_d = _exact_w8_matrix(rng, p_down, I)
    wgu, wd = bits(wgu_v), bits(wd_v)
    qg, sg = oracle.quantize_w8(wgu)
    qd, sd = oracle.quantize_w8(wd)
    np.testing.assert_array_equal(qg, m_gu.astype(np.int8))
    np.testing.assert_array_equal(qd, m_d.astype(np.int8))
    np.testing.assert_array_equal(sg, np.exp2(-p_gu).astype(np.float32))
    np.testing.assert_array_equal(sd, np.exp2(-p_down).astype(np.float32))
    x = rand_bf16(rng, (T, H), 1.0)
    L = rng.standard_normal((T, E)).astype(np.float32)
    ids, w = oracle.route(L, k, renormalize=True)
    y16 = oracle.moe_layer(x, ids, w, E, S, wgu, wd)
    y8 = oracle.moe_layer_w8(x, ids, w, E, S, qg, sg, qd, sd)
    np.testing.assert_allclose(y8, y16, rtol=1e-12, atol=1e-15)
    # negative controls: the same comparison must fail for misapplied scales
    wrong = {
        "gate/up scales swapped": (np.concatenate([sg[:, I:], sg[:, :I]], 1), sd),
        "down scales reversed": (sg, np.ascontiguousarray(sd[:, ::-1])),
        "next expert's scales": (np.roll(sg, 1, axis=0), np.roll(sd, 1, axis=0)),
    }
    for what, (sg_x, sd_x) in wrong.items():
        y_x = oracle.moe_layer_w8(x, ids, w, E, S, qg, sg_x, qd, sd_x)
        rel = np.abs(y_x - y16).max() / np.abs(y16).max()
        assert rel > 1e-3, f"{what}: not detected (max rel diff {rel:.2e})"


def test_router_logits_vs_library_matmul():
    rng = np.random.default_rng(21)
    x = rand_bf16(rng, (7, 48), 1.0)
    wr = rand_bf16(rng, (10, 48), 0.02)
    b = rng.standard_normal(10).astype(np.float32)
    L = oracle.router_logits(x, wr, b)
    np.testing.assert_allclose(L, val(x) @ val(wr).T + b.astype(np.float64), rtol=1e-12,
                               atol=1e-14)


def test_workload_inputs_are_seeded_and_shaped():
    a = W.make_layer(W.TINY, 16, seed=0)
    b = W.make_layer(W.TINY, 16, seed=0)
    assert torch.equal(a.logits, b.logits) and torch.equal(a.w_gu, b.w_gu)
    assert a.x.dtype == torch.float32 and a.x.shape == (16, 256)
    assert a.w_gu.shape == (8, 1024, 256) and a.w_down.shape == (8, 256, 512)
    assert abs(a.w_gu.float().std().item() - 0.02) < 1e-3
