"""CUDA path vs the CPU oracle on seeded inputs, through the C-ABI calls.

Bars: routing ids, permutation and offsets bit-exact (given the same fp32
logits); routing weights within 1e-6 relative; bf16 layer outputs within
relative Frobenius error 5e-3 and max |diff| <= 2e-2 * max|ref| of the
oracle's exact layer; the same bytes on every run.  Shapes are the pages'
OLMoE-1B-7B and DeepSeek-MoE-16B layers ("switchyard" page intro;
"dispatch" README, Stack) plus small shapes that span several tiles with
ragged tails.
"""
import numpy as np
import pytest
import torch

import oracle
from grouped_expert_gemm_moe_gb300 import workloads as W

from gpu_helpers import (W_RTOL, assert_close, errors, host_inputs, oracle_out, sample_tokens,
                         to_np)

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def B():
    import __graft_entry__ as g
    g.build()
    from grouped_expert_gemm_moe_gb300 import binding
    return binding


@pytest.fixture(scope="module")
def L(B):
    from grouped_expert_gemm_moe_gb300 import layer
    return layer


_CACHE = {}


def layer_case(name, T, routing):
    key = (name, T, routing)
    if key not in _CACHE:
        _CACHE.clear()                                     # keep one full-size layer resident
        sh = W.CONFIGS[name]
        big = sh.H * sh.I * sh.G > 10_000_000
        inp = W.make_layer(sh, T, routing, seed=0, device=DEV if big else "cpu")
        _CACHE[key] = (inp, host_inputs(inp))
    return _CACHE[key]


def make_layer_obj(L, inp):
    sh = inp.shape
    return L.MoELayer(sh.H, sh.E, sh.k, sh.I, sh.S, sh.renormalize,
                      w_gu=inp.w_gu.to(DEV), w_down=inp.w_down.to(DEV), device=DEV)


CASES = [("tiny", 16, "uniform"),
         ("olmoe", 1, "uniform"), ("olmoe", 8, "uniform"), ("olmoe", 64, "uniform"),
         ("deepseek", 1, "uniform"), ("deepseek", 16, "zipf"), ("deepseek", 128, "uniform"),
         ("deepseek", 512, "zipf"), ("deepseek", 2048, "uniform"), ("deepseek", 2048, "zipf")]


@pytest.mark.parametrize("name,T,routing", CASES)
def test_route_and_permute_bit_exact(B, L, name, T, routing):
    inp, h = layer_case(name, T, routing)
    sh = inp.shape
    layer = make_layer_obj(L, inp)
    b = layer.buffers(T)
    x, logits = inp.x.to(DEV), inp.logits.to(DEV)
    layer.route(logits, b)
    layer.permute(x, b)
    layer.check()
    ids_ref, w_ref = oracle.route(h["logits"], sh.k, sh.renormalize)
    np.testing.assert_array_equal(b.topk_ids.cpu().numpy(), ids_ref)
    np.testing.assert_allclose(b.topk_w.cpu().numpy().astype(np.float64), w_ref, rtol=W_RTOL)
    off, ss, ros = oracle.permute(ids_ref, sh.E, sh.S)
    np.testing.assert_array_equal(b.offsets.cpu().numpy(), off)
    np.testing.assert_array_equal(b.sorted_slot.cpu().numpy(), ss)
    np.testing.assert_array_equal(b.row_of_slot.cpu().numpy(), ros)
    # x_perm rows are the tokens' rows (rounded to bf16 for fp32 activations)
    tok = np.concatenate([ss // sh.k] + [np.arange(T)] * sh.S)
    xb = inp.x.to(torch.bfloat16).cpu()
    assert torch.equal(b.x_perm.cpu(), xb[torch.from_numpy(tok).long()])


@pytest.mark.parametrize("ffn", ["gemm", "gemv"])
@pytest.mark.parametrize("name,T,routing", CASES)
def test_layer_matches_oracle(B, L, name, T, routing, ffn):
    if ffn == "gemv" and T > 512:
        pytest.skip("the GEMV is for decode-sized batches")
    inp, h = layer_case(name, T, routing)
    layer = make_layer_obj(L, inp)
    out = layer.forward(inp.x.to(DEV), inp.logits.to(DEV), ffn=ffn)
    layer.check()
    tok = sample_tokens(T)
    _, _, y = oracle_out(inp, h, tokens=tok)
    rel, mx = assert_close(to_np(out)[tok], y, f"{name} T={T} {routing} {ffn}")
    print(f"{name} T={T} {routing} {ffn}: rel {rel:.2e} max {mx:.2e}")


def test_gemm_and_gemv_agree_and_are_deterministic(B, L):
    inp, h = layer_case("deepseek", 128, "uniform")
    layer = make_layer_obj(L, inp)
    x, logits = inp.x.to(DEV), inp.logits.to(DEV)
    outs = {}
    for ffn in ("gemm", "gemv"):
        runs = [layer.forward(x, logits, ffn=ffn).clone() for _ in range(3)]
        layer.check()
        for r in runs[1:]:
            assert torch.equal(r, runs[0]), f"{ffn} output changed between runs"
        outs[ffn] = to_np(runs[0])
    rel, mx = errors(outs["gemm"], outs["gemv"])
    assert rel < 5e-3 and mx < 2e-2


def _ffn_rows_oracle(xp_bits, off, w_gu_bits, w_down_bits, H, I):
    """Per permuted row: y = FFN_g(x_perm[r]) (unweighted), oracle fp64."""
    M = xp_bits.shape[0]
    y = np.zeros((M, H))
    xv = (xp_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for g in range(len(off) - 1):
        for r in range(off[g], off[g + 1]):
            hh = oracle.expert_hidden(xv[r], w_gu_bits[g], H, I)
            y[r] = oracle.expert_down(hh, w_down_bits[g], H, I)
    return y


@pytest.mark.parametrize("ffn", ["gemm", "gemv"])
@pytest.mark.parametrize("H,I,E,S,k,T", [(136, 200, 5, 1, 2, 300),     # K and N tails
                                          (256, 512, 4, 0, 1, 1000),   # several m-tiles + tail
                                          (512, 384, 16, 2, 4, 97),
                                          # decode-sized groups (weight-row tiles with
                                          # 16/32/64-token blocks), ragged K, N and blocks
                                          (136, 200, 5, 1, 2, 12),
                                          (136, 200, 5, 1, 2, 40),
                                          (136, 200, 5, 1, 2, 90)])
def test_grouped_ffn_rows_vs_oracle(B, L, ffn, H, I, E, S, k, T):
    """The grouped FFN alone: every permuted row against the oracle's expert
    FFN, on shapes whose tiles have ragged M, N and K tails."""
    sh = W.MoEShape("t", H=H, E=E, k=k, I=I, S=S)
    inp = W.make_layer(sh, T, "uniform", seed=1)
    layer = make_layer_obj(L, inp)
    b = layer.buffers(T)
    layer.route(inp.logits.to(DEV), b)
    layer.permute(inp.x.to(DEV), b)
    layer.ffn(b, ffn)
    layer.check()
    off = b.offsets.cpu().numpy()
    ref = _ffn_rows_oracle(W.bf16_bits(b.x_perm), off, W.bf16_bits(inp.w_gu),
                           W.bf16_bits(inp.w_down), H, I)
    got = to_np(b.y_perm)
    M = layer.rows(T)
    rel, mx = errors(got[:M], ref[:M])
    if not (rel <= 5e-3 and mx <= 2e-2):
        bad = np.abs(got - ref) > 2e-2 * np.abs(ref).max()
        rows = np.where(bad.any(1))[0]
        cols = np.where(bad.any(0))[0]
        pytest.fail(f"{ffn}: rel {rel:.3e} max {mx:.3e}; bad rows {rows[:20]}.. "
                    f"({len(rows)}), bad cols {cols[:20]}.. ({len(cols)})")


def _adversarial_logits(kind, T, E):
    if kind == "all_to_one":
        L = np.full((T, E), -3.0, np.float32)
        L[:, 5] = 4.0
        return L
    if kind == "ties":
        rng = np.random.default_rng(0)
        return rng.integers(0, 3, size=(T, E)).astype(np.float32)
    if kind == "equal":
        return np.zeros((T, E), np.float32)
    raise ValueError(kind)


@pytest.mark.parametrize("kind", ["all_to_one", "ties", "equal"])
@pytest.mark.parametrize("ffn", ["gemm", "gemv"])
def test_adversarial_routings(B, L, kind, ffn):
    sh = W.MoEShape("adv", H=256, E=16, k=4, I=256, S=1, renormalize=True)
    T = 300
    inp = W.make_layer(sh, T, "uniform", seed=2)
    inp.logits = torch.from_numpy(_adversarial_logits(kind, T, sh.E))
    h = host_inputs(inp)
    layer = make_layer_obj(L, inp)
    out = layer.forward(inp.x.to(DEV), inp.logits.to(DEV), ffn=ffn)
    layer.check()
    ids, w, y = oracle_out(inp, h)
    b = layer.buffers(T)
    np.testing.assert_array_equal(b.topk_ids.cpu().numpy(), ids)
    np.testing.assert_array_equal(b.offsets.cpu().numpy(), oracle.permute(ids, sh.E, sh.S)[0])
    assert_close(to_np(out), y, f"{kind} {ffn}")


def test_single_token_single_expert(B, L):
    sh = W.MoEShape("one", H=64, E=1, k=1, I=64)
    inp = W.make_layer(sh, 1, "uniform", seed=3)
    h = host_inputs(inp)
    layer = make_layer_obj(L, inp)
    for ffn in ("gemm", "gemv"):
        out = layer.forward(inp.x.to(DEV), inp.logits.to(DEV), ffn=ffn)
        layer.check()
        _, _, y = oracle_out(inp, h)
        assert_close(to_np(out), y, f"T=1 E=1 {ffn}")


def test_residual_and_aliasing(B, L):
    inp, h = layer_case("tiny", 16, "uniform")
    sh = inp.shape
    layer = make_layer_obj(L, inp)
    res = (torch.randn((16, sh.H), generator=torch.Generator().manual_seed(9))).to(torch.bfloat16)
    buf = res.to(DEV).clone()
    layer.forward(inp.x.to(DEV), inp.logits.to(DEV), out=buf, residual=buf, ffn="gemm")
    layer.check()
    _, _, y = oracle_out(inp, h, residual=W.bf16_bits(res))
    assert_close(to_np(buf), y, "residual")


@pytest.mark.parametrize("T", [10, 700])          # one chunk of slots / several chunks
def test_invalid_expert_id_is_reported_without_out_of_bounds(B, L, T):
    sh = W.MoEShape("bad", H=64, E=8, k=2, I=64, S=1)
    inp = W.make_layer(sh, T, "uniform", seed=4)
    layer = make_layer_obj(L, inp)
    b = layer.buffers(T)
    ids = torch.randint(0, sh.E, (T, sh.k), dtype=torch.int32)
    ids[3, 1] = sh.E                        # out of range
    b.topk_ids.copy_(ids)
    b.topk_w.fill_(0.5)
    b.y_perm.zero_()
    layer.permute(inp.x.to(DEV), b)
    torch.cuda.synchronize()
    assert int(layer.err.item()) == 6
    assert (b.offsets.cpu() == 0).all() and (b.row_of_slot.cpu() == -1).all()
    layer.err.zero_()
    for ffn in ("gemm", "gemv"):
        layer.ffn(b, ffn)                   # empty groups: no work, no error
    out = torch.empty((T, sh.H), dtype=torch.bfloat16, device=DEV)
    layer.combine(b, out)
    torch.cuda.synchronize()
    assert int(layer.err.item()) == 6       # combine skipped the unplaced slots


@pytest.mark.parametrize("bad", [float("nan"), float("inf"), float("-inf")])
def test_non_finite_logit_is_reported(B, L, bad):
    inp, _ = layer_case("tiny", 16, "uniform")
    layer = make_layer_obj(L, inp)
    b = layer.buffers(16)
    logits = inp.logits.clone()
    logits[2, 3] = bad
    layer.route(logits.to(DEV), b)
    torch.cuda.synchronize()
    assert int(layer.err.item()) == 6


@pytest.mark.parametrize("T", [1, 8, 64])
def test_w8_gemv_matches_oracle(B, L, T):
    sh = W.OLMOE
    inp = W.make_layer(sh, T, "uniform", seed=0, device=DEV)
    h = host_inputs(inp)
    q_gu, s_gu = B.moe_quantize_w8(inp.w_gu)
    q_down, s_down = B.moe_quantize_w8(inp.w_down)
    layer = L.MoELayer(sh.H, sh.E, sh.k, sh.I, sh.S, sh.renormalize, q_gu=q_gu.to(DEV),
                       s_gu=s_gu.to(DEV), q_down=q_down.to(DEV), s_down=s_down.to(DEV),
                       device=DEV)
    out = layer.forward(inp.x, inp.logits, ffn="gemv")
    layer.check()
    tok = sample_tokens(T)
    ids, w = oracle.route(h["logits"], sh.k, sh.renormalize)
    y = oracle.moe_layer_w8(h["x"], ids, w, sh.E, sh.S, q_gu.numpy(), s_gu.numpy(),
                            q_down.numpy(), s_down.numpy(), tokens=tok)
    assert_close(to_np(out)[tok], y, f"w8 gemv T={T}")


def test_router_logits_kernel(B):
    sh = W.OLMOE
    g = torch.Generator().manual_seed(5)
    x = torch.randn((77, sh.H), generator=g).to(torch.bfloat16)
    w_r = (torch.randn((sh.E, sh.H), generator=g) * 0.02).to(torch.bfloat16)
    bias = W.zipf_bias(sh.E, 0.5)
    out = torch.empty((77, sh.E), dtype=torch.float32, device=DEV)
    B.moe_router_logits(x.to(DEV), w_r.to(DEV), bias.to(DEV), out)
    ref = oracle.router_logits(W.bf16_bits(x), W.bf16_bits(w_r), bias.numpy())
    got = out.cpu().numpy().astype(np.float64)
    # fp32 accumulation of 2048 products: error << 1e-4 of the logit scale
    assert np.abs(got - ref).max() <= 1e-4 * np.abs(ref).max()


FUSED_CASES = [("tiny", 16, "uniform"), ("olmoe", 1, "uniform"), ("olmoe", 8, "uniform"),
               ("olmoe", 64, "uniform"), ("deepseek", 16, "zipf"), ("deepseek", 128, "uniform")]


@pytest.mark.parametrize("name,T,routing", FUSED_CASES)
def test_fused_route_permute_bit_exact(B, L, name, T, routing):
    """moe_route_permute gives the same bits as the oracle's route + permute."""
    inp, h = layer_case(name, T, routing)
    sh = inp.shape
    layer = make_layer_obj(L, inp)
    b = layer.buffers(T)
    for t_ in (b.topk_ids, b.offsets, b.sorted_slot, b.row_of_slot):
        t_.fill_(-7)
    b.x_perm.zero_()
    B.moe_route_permute(inp.logits.to(DEV), sh.k, sh.renormalize, sh.S, inp.x.to(DEV),
                        b.topk_ids, b.topk_w, b.offsets, b.sorted_slot, b.row_of_slot, b.x_perm,
                        layer.err)
    layer.check()
    ids_ref, w_ref = oracle.route(h["logits"], sh.k, sh.renormalize)
    np.testing.assert_array_equal(b.topk_ids.cpu().numpy(), ids_ref)
    np.testing.assert_allclose(b.topk_w.cpu().numpy().astype(np.float64), w_ref, rtol=W_RTOL)
    off, ss, ros = oracle.permute(ids_ref, sh.E, sh.S)
    np.testing.assert_array_equal(b.offsets.cpu().numpy(), off)
    np.testing.assert_array_equal(b.sorted_slot.cpu().numpy(), ss)
    np.testing.assert_array_equal(b.row_of_slot.cpu().numpy(), ros)
    tok = np.concatenate([ss // sh.k] + [np.arange(T)] * sh.S)
    xb = inp.x.to(torch.bfloat16).cpu()
    assert torch.equal(b.x_perm.cpu(), xb[torch.from_numpy(tok).long()])


def test_fused_route_permute_limits_and_nan(B, L):
    inp, _ = layer_case("tiny", 16, "uniform")
    sh = inp.shape
    layer = make_layer_obj(L, inp)
    b = layer.buffers(16)
    logits = inp.logits.clone()
    logits[5, 1] = float("nan")
    B.moe_route_permute(logits.to(DEV), sh.k, sh.renormalize, sh.S, inp.x.to(DEV), b.topk_ids,
                        b.topk_w, b.offsets, b.sorted_slot, b.row_of_slot, b.x_perm, layer.err)
    torch.cuda.synchronize()
    assert int(layer.err.item()) == 6
    assert (b.offsets.cpu() == 0).all() and (b.row_of_slot.cpu() == -1).all()
    # beyond its limits the call refuses without launching
    big = torch.zeros((600, 8), dtype=torch.float32, device=DEV)      # 600 * 2 > 1024 slots
    with pytest.raises(B.MoEError):
        B.moe_route_permute(big, 2, False, 0, torch.zeros((600, 256), dtype=torch.bfloat16,
                                                          device=DEV),
                            torch.empty((600, 2), dtype=torch.int32, device=DEV),
                            torch.empty((600, 2), dtype=torch.float32, device=DEV),
                            torch.empty(9, dtype=torch.int32, device=DEV),
                            torch.empty(1200, dtype=torch.int32, device=DEV),
                            torch.empty(1200, dtype=torch.int32, device=DEV),
                            torch.empty((1200, 256), dtype=torch.bfloat16, device=DEV))


@pytest.mark.parametrize("tile,case", [(t, ("deepseek", 512, "zipf")) for t in
                                       ("128x128", "128x256", "pair")]
                         + [("pair", ("olmoe", 2048, "uniform")), ("pair", ("olmoe", 700, "zipf"))])
def test_gemm_tile_shapes_agree(B, L, tile, case):
    """Every tile shape of the tcgen05 GEMM (128 x 128, 128 x 256, 256 x 256
    on CTA pairs; normally chosen per call from the rows per group), forced
    for every call, gives results within tolerance of the oracle on every
    token of a DeepSeek-shaped batch (zipf routing: group sizes from a few
    rows to the 512-row shared experts) and, for the pair tiles, of two
    OLMoE-shaped batches."""
    inp, h = layer_case(*case)
    layer = make_layer_obj(L, inp)
    with B.forced_gemm_tile(tile):
        out = layer.forward(inp.x.to(DEV), inp.logits.to(DEV), ffn="gemm")
        layer.check()
    tok = sample_tokens(case[1])
    _, _, y = oracle_out(inp, h, tokens=tok)
    assert_close(to_np(out)[tok], y, f"tile {tile} {case}")


def test_gemm_tile_override_is_validated(B):
    for bad in (-2, 8, 100):
        assert B._lib.moe_set_gemm_tile(bad) == 1          # MOE_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        B.moe_set_gemm_tile("dec16")
    B.moe_set_gemm_tile("auto")


@pytest.mark.parametrize("T,E,k,renorm", [(1, 64, 8, 0), (64, 64, 8, 0), (700, 96, 6, 1),
                                          (2048, 64, 6, 0), (37, 256, 4, 1)])
def test_fused_router_route_matches_the_two_calls(B, T, E, k, renorm):
    """moe_router_route: logits, ids and weights bit-identical to
    moe_router_logits followed by moe_route; logits vs the oracle (fp64)."""
    H = 2048
    g = torch.Generator().manual_seed(T + E)
    x = torch.randn((T, H), generator=g).to(torch.bfloat16).to(DEV)
    w_r = (torch.randn((E, H), generator=g) * 0.02).to(torch.bfloat16).to(DEV)
    bias = W.zipf_bias(E, 1.2).to(DEV) if E == 64 else None
    L1 = torch.empty((T, E), dtype=torch.float32, device=DEV)
    ids1 = torch.empty((T, k), dtype=torch.int32, device=DEV)
    w1 = torch.empty((T, k), dtype=torch.float32, device=DEV)
    err = B.new_error_word(DEV)
    B.moe_router_logits(x, w_r, bias, L1)
    B.moe_route(L1, k, renorm, ids1, w1, err)
    L2 = torch.empty_like(L1)
    ids2, w2 = torch.empty_like(ids1), torch.empty_like(w1)
    B.moe_router_route(x, w_r, bias, k, renorm, ids2, w2, logits=L2, dev_error=err)
    ids3, w3 = torch.empty_like(ids1), torch.empty_like(w1)
    B.moe_router_route(x, w_r, bias, k, renorm, ids3, w3, dev_error=err)   # no logits out
    B.check_device_error(err, "router_route")
    assert torch.equal(L1, L2)
    assert torch.equal(ids1, ids2) and torch.equal(ids1, ids3)
    assert torch.equal(w1.view(torch.int32), w2.view(torch.int32))
    assert torch.equal(w1.view(torch.int32), w3.view(torch.int32))
    tok = sample_tokens(T, n=16)
    ref = oracle.router_logits(W.bf16_bits(x.cpu())[tok], W.bf16_bits(w_r.cpu()),
                               None if bias is None else bias.cpu().numpy())
    assert np.abs(L2.cpu().numpy()[tok] - ref).max() <= 1e-4 * np.abs(ref).max()



@pytest.mark.parametrize("ffn", ["gemm", "gemv"])
@pytest.mark.parametrize("T", [16, 40])
def test_maximum_groups_and_k(B, L, ffn, T):
    """The limits: G = E + S = 1024 groups (1000 routed, 24 shared) and k = 32;
    T=16 uses the one-launch permute (512 slots), T=40 the chunked one."""
    sh = W.MoEShape("max", H=256, E=1000, k=32, I=128, S=24)
    inp = W.make_layer(sh, T, "uniform", seed=8)
    h = host_inputs(inp)
    layer = make_layer_obj(L, inp)
    out = layer.forward(inp.x.to(DEV), inp.logits.to(DEV), ffn=ffn)
    layer.check()
    b = layer.buffers(T)
    ids, w, y = oracle_out(inp, h)
    np.testing.assert_array_equal(b.topk_ids.cpu().numpy(), ids)
    np.testing.assert_array_equal(b.offsets.cpu().numpy(), oracle.permute(ids, sh.E, sh.S)[0])
    assert_close(to_np(out), y, f"G=1024 k=32 T={T} {ffn}")


def test_deepseek_16384_tokens(B, L):
    """A batch 8x the largest configured one (131072 permuted rows, 128
    permute chunks), checked on sampled tokens."""
    sh = W.DEEPSEEK
    T = 16384
    inp = W.make_layer(sh, T, "zipf", seed=2, device=DEV)
    layer = make_layer_obj(L, inp)
    out = layer.forward(inp.x, inp.logits, ffn="gemm")
    layer.check()
    tok = sample_tokens(T, n=24)
    h = host_inputs(inp)
    ids, w = oracle.route(h["logits"], sh.k, sh.renormalize)
    np.testing.assert_array_equal(layer.buffers(T).topk_ids.cpu().numpy(), ids)
    np.testing.assert_array_equal(layer.buffers(T).offsets.cpu().numpy(),
                                  oracle.permute(ids, sh.E, sh.S)[0])
    y = oracle.moe_layer(h["x"], ids, w, sh.E, sh.S, h["w_gu"], h["w_down"], tokens=tok)
    assert_close(to_np(out)[tok], y, "DeepSeek T=16384")


@pytest.mark.parametrize("name,T", [("olmoe", 64), ("olmoe", 1), ("deepseek", 512)])
def test_capture_host_replays_match_forward(B, L, name, T):
    """MoELayer.capture_host: the graph with the host<->device copies gives,
    for each new content of the pinned host inputs, the same bytes as a
    forward pass on device copies of them."""
    sh = W.CONFIGS[name]
    inp = W.make_layer(sh, T, "uniform", seed=2, device=DEV)
    layer = L.MoELayer(sh.H, sh.E, sh.k, sh.I, sh.S, sh.renormalize, w_gu=inp.w_gu,
                       w_down=inp.w_down, device=DEV)
    x_host = inp.x.cpu().pin_memory()
    l_host = inp.logits.cpu().pin_memory()
    cap = layer.capture_host(x_host, l_host)
    with pytest.raises(ValueError):
        layer.capture_host(inp.x.cpu(), inp.logits.cpu())      # not pinned
    g = torch.Generator().manual_seed(T)
    for _ in range(3):
        x_host.copy_(torch.randn((T, sh.H), generator=g).to(torch.bfloat16))
        l_host.copy_(torch.randn((T, sh.E), generator=g))
        out = cap.replay()
        torch.cuda.synchronize()
        ref = layer.forward(x_host.to(DEV), l_host.to(DEV)).cpu()
        layer.check()
        assert torch.equal(out, ref)


@pytest.mark.parametrize("nbytes", [16, 4096, 262144, 8 << 20])
def test_moe_copy_both_directions(B, nbytes):
    """moe_copy moves bytes exactly between pinned host memory and the device
    (both directions) and device to device; sizes off the 16-byte grid are
    refused."""
    g = torch.Generator().manual_seed(nbytes)
    src = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, generator=g).pin_memory()
    dev = torch.zeros(nbytes, dtype=torch.uint8, device=DEV)
    back = torch.zeros(nbytes, dtype=torch.uint8).pin_memory()
    B.moe_copy(dev, src)
    dev2 = torch.zeros_like(dev)
    B.moe_copy(dev2, dev)
    B.moe_copy(back, dev2)
    torch.cuda.synchronize()
    assert torch.equal(back, src)
    with pytest.raises(B.MoEError):
        B.moe_copy(dev[: nbytes - 1] if nbytes > 16 else dev[:8], src[: nbytes - 1] if nbytes > 16 else src[:8])
