"""Pins of the oracle's routing and permutation against facts fixed outside it.

Routing follows the "switchyard" page (02 Kernels and dispatch, "Route and
sort") and the "dispatch" README (Architecture, "Router / top-k gating"):
top-k of the router logits with ties to the lower expert index, softmax over
all E logits, optional renormalisation over the k chosen.  The permutation
is the page's "rows sorted by expert with a prefix scan": a stable sort of
slots s = t*k + j by expert with an exclusive-prefix offset table.
"""
import os

import numpy as np
import pytest
import scipy.special

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_kv(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out[key] = vals
    return out


def test_route_golden_closed_form():
    g = _read_kv("route_closed_form.txt")
    E, k = int(g["E"][0]), int(g["k"][0])
    L = np.log(np.array([float(v) for v in g["logits_ln"]], np.float64)).astype(np.float32)
    L = L.reshape(1, E)
    ids, w = oracle.route(L, k, renormalize=False)
    assert ids.tolist() == [[int(v) for v in g["ids"]]]
    np.testing.assert_allclose(w[0], [float(v) for v in g["weights"]], rtol=1e-6)
    ids_r, w_r = oracle.route(L, k, renormalize=True)
    assert ids_r.tolist() == ids.tolist()
    np.testing.assert_allclose(w_r[0], [float(v) for v in g["weights_renorm"]], rtol=1e-6)


def _brute_force_topk(L, k):
    """Expert e is selected iff fewer than k experts beat it (beat = larger
    logit, or equal logit and lower index); order = number of beaters."""
    T, E = L.shape
    ids = np.empty((T, k), np.int32)
    for t in range(T):
        beaten_by = []
        for e in range(E):
            n = sum(1 for f in range(E) if L[t, f] > L[t, e] or (L[t, f] == L[t, e] and f < e))
            beaten_by.append(n)
        for e in range(E):
            if beaten_by[e] < k:
                ids[t, beaten_by[e]] = e
    return ids


@pytest.mark.parametrize("E,k", [(8, 2), (6, 6), (16, 5), (64, 8)])
def test_route_brute_force_with_ties(E, k):
    rng = np.random.default_rng(1234 + E * 31 + k)
    T = 40 if E < 64 else 8
    L = rng.integers(0, 3, size=(T, E)).astype(np.float32)   # many exact ties
    ids, _ = oracle.route(L, k, renormalize=False)
    np.testing.assert_array_equal(ids, _brute_force_topk(L, k))
    Lc = rng.standard_normal((T, E)).astype(np.float32)
    ids2, _ = oracle.route(Lc, k, renormalize=False)
    np.testing.assert_array_equal(ids2, _brute_force_topk(Lc, k))


def test_route_matches_library_sort_and_softmax():
    rng = np.random.default_rng(7)
    T, E, k = 200, 64, 8
    L = (rng.standard_normal((T, E)) * 0.9).astype(np.float32)
    ids, w = oracle.route(L, k, renormalize=False)
    order = np.argsort(-L.astype(np.float64), axis=1, kind="stable")[:, :k]
    np.testing.assert_array_equal(ids, order)
    p = scipy.special.softmax(L.astype(np.float64), axis=1)
    np.testing.assert_allclose(w, np.take_along_axis(p, ids, axis=1), rtol=1e-12)
    ids_r, w_r = oracle.route(L, k, renormalize=True)
    sel = np.take_along_axis(p, ids, axis=1)
    np.testing.assert_allclose(w_r, sel / sel.sum(1, keepdims=True), rtol=1e-12)


def test_route_all_equal_and_sums():
    T, E, k = 5, 8, 3
    L = np.full((T, E), 0.75, np.float32)
    ids, w = oracle.route(L, k, renormalize=False)
    assert (ids == np.arange(k)).all()
    np.testing.assert_allclose(w, 1.0 / E, rtol=1e-15)
    _, w_r = oracle.route(L, k, renormalize=True)
    np.testing.assert_allclose(w_r, 1.0 / k, rtol=1e-15)
    rng = np.random.default_rng(3)
    L = rng.standard_normal((50, 16)).astype(np.float32)
    _, w = oracle.route(L, 4, renormalize=False)
    assert (w.sum(1) <= 1 + 1e-12).all() and (np.diff(w, axis=1) <= 0).all()
    _, w = oracle.route(L, 16, renormalize=False)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-12)
    _, w = oracle.route(L, 4, renormalize=True)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-12)


def test_route_shift_invariance():
    rng = np.random.default_rng(5)
    L = rng.integers(-20, 20, size=(30, 32)).astype(np.float32) / 4
    ids, w = oracle.route(L, 6, renormalize=False)
    ids2, w2 = oracle.route(L + np.float32(16.0), 6, renormalize=False)
    np.testing.assert_array_equal(ids, ids2)
    np.testing.assert_allclose(w, w2, rtol=1e-12)


@pytest.mark.parametrize("bad", [np.nan, np.inf, -np.inf])
def test_route_rejects_non_finite_logits(bad):
    """A NaN or infinite logit leaves the softmax without a finite value
    (inf - inf), so such a row is refused rather than given NaN weights."""
    L = np.zeros((2, 4), np.float32)
    L[1, 2] = bad
    with pytest.raises(ValueError):
        oracle.route(L, 2, renormalize=False)


def _check_permutation(ids, E, S, off, ss, ros):
    T, k = ids.shape
    n = T * k
    flat = ids.ravel()
    # a bijection on [0, T*k)
    assert sorted(ss.tolist()) == list(range(n))
    np.testing.assert_array_equal(ros[ss], np.arange(n))
    # offsets: exclusive prefix of per-expert counts, then S groups of T rows
    counts = np.bincount(flat, minlength=E)
    assert off[0] == 0 and off[E] == n
    np.testing.assert_array_equal(np.diff(off[:E + 1]), counts)
    np.testing.assert_array_equal(np.diff(off[E:]), np.full(S, T))
    # experts non-decreasing along the sort, slots increasing inside a group
    e_sorted = flat[ss]
    assert (np.diff(e_sorted) >= 0).all()
    for e in range(E):
        seg = ss[off[e]:off[e + 1]]
        assert (np.diff(seg) > 0).all()
        assert (flat[seg] == e).all()


@pytest.mark.parametrize("T,E,k,S", [(16, 8, 2, 0), (33, 64, 8, 0), (128, 64, 6, 2),
                                     (1, 64, 8, 0), (7, 5, 5, 1)])
def test_permute_invariants_and_library_sort(T, E, k, S):
    rng = np.random.default_rng(T * 131 + E)
    L = rng.standard_normal((T, E)).astype(np.float32)
    ids, _ = oracle.route(L, k, renormalize=False)
    off, ss, ros = oracle.permute(ids, E, S)
    _check_permutation(ids, E, S, off, ss, ros)
    np.testing.assert_array_equal(ss, np.argsort(ids.ravel(), kind="stable"))


def test_permute_adversarial_all_to_one_and_empty():
    T, E, k = 64, 16, 1
    ids = np.full((T, k), 11, np.int32)
    off, ss, ros = oracle.permute(ids, E, 0)
    _check_permutation(ids, E, 0, off, ss, ros)
    assert off[11] == 0 and off[12] == T
    np.testing.assert_array_equal(ss, np.arange(T))
    off0, ss0, ros0 = oracle.permute(np.zeros((0, 4), np.int32), 8, 2)
    assert (off0 == 0).all() and ss0.size == 0


def test_dropless_every_slot_served_once():
    rng = np.random.default_rng(9)
    T, E, k = 300, 64, 8
    L = rng.standard_normal((T, E)).astype(np.float32)
    ids, _ = oracle.route(L, k, renormalize=False)
    off, ss, ros = oracle.permute(ids, E, 0)
    reads = np.zeros(T * k, np.int64)
    for t in range(T):                 # the combine's reads, one per slot
        for j in range(k):
            reads[ros[t * k + j]] += 1
    assert (reads == 1).all()
    assert off[E] == T * k


def test_permute_rejects_bad_id():
    ids = np.array([[0, 9]], np.int32)
    with pytest.raises(ValueError):
        oracle.permute(ids, 8, 0)


def test_skew4_calibration_gives_four_times_mean():
    import torch
    from grouped_expert_gemm_moe_gb300 import workloads as W
    sh = W.OLMOE_STACK
    g = W.make_generator(0)
    T = 2048
    x = W._randn((T, sh.H), g, "cpu").to(torch.bfloat16)
    w_r = W._randn((sh.E, sh.H), g, "cpu", 0.02).to(torch.bfloat16)
    L = W.router_logits_input(x, w_r, W.routing_bias(sh, "skew4")).numpy()
    ids, _ = oracle.route(L, sh.k, renormalize=False)
    ratio = np.bincount(ids.ravel(), minlength=sh.E).max() / (T * sh.k / sh.E)
    assert 3.9 <= ratio <= 4.1
