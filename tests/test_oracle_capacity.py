"""Pins of the oracle's capacity-limited (token-dropping) variant.

The "switchyard" page (03 Load balance, "What dropping tokens costs") reports
what capacity limits cost: an expert drops the tokens it has no room for.
The reading used here (and by the CUDA path): routed expert e serves at most
C of its slots, the first C in slot order s = t*k + j (first come, first
served); a dropped slot adds nothing to its token's output; shared experts
are never capped.  Each check compares the oracle with something other than
itself: a pure-Python brute force, the dropless oracle in the limit of a
large capacity, closed forms for the dropped count, and a numpy dense
formulation with a keep mask.
"""
import numpy as np
import pytest

import oracle

from test_oracle_ffn_w8 import dense_ffn, rand_bf16, val


def _brute_force(ids, E, S, C):
    """Independent restatement in plain Python."""
    T, k = ids.shape
    flat = ids.reshape(-1).tolist()
    kept = {e: [s for s, ee in enumerate(flat) if ee == e][:C] for e in range(E)}
    off = [0]
    for e in range(E):
        off.append(off[-1] + len(kept[e]))
    for _ in range(S):
        off.append(off[-1] + T)
    ss = [-1] * (T * k)
    ros = [-2] * (T * k)
    for e in range(E):
        for i, s in enumerate(kept[e]):
            ss[off[e] + i] = s
            ros[s] = off[e] + i
    dropped = T * k - sum(len(v) for v in kept.values())
    return np.array(off), np.array(ss), np.array(ros), dropped


@pytest.mark.parametrize("T,E,k,S", [(7, 4, 2, 0), (33, 8, 3, 2), (64, 16, 4, 1), (5, 3, 3, 0)])
def test_capped_permute_matches_brute_force(T, E, k, S):
    rng = np.random.default_rng(T * 100 + E)
    # skewed ids so that some experts overflow at every capacity tried
    p = np.arange(1, E + 1, dtype=np.float64) ** -1.5
    p /= p.sum()
    ids = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    counts = np.bincount(ids.ravel(), minlength=E)
    for C in sorted({0, 1, 2, int(counts.max()) // 2, int(counts.max()), int(counts.max()) + 3}):
        off, ss, ros, dropped = oracle.permute_capped(ids, E, S, C)
        boff, bss, bros, bdrop = _brute_force(ids, E, S, C)
        np.testing.assert_array_equal(off, boff)
        np.testing.assert_array_equal(ss, bss)
        np.testing.assert_array_equal(ros, bros)
        assert dropped == bdrop
        # closed form of the dropped count
        assert dropped == int(np.maximum(counts - C, 0).sum())


def test_large_capacity_is_dropless():
    rng = np.random.default_rng(5)
    T, E, k, S = 50, 8, 2, 2
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    C = int(np.bincount(ids.ravel(), minlength=E).max())
    off, ss, ros, dropped = oracle.permute_capped(ids, E, S, C)
    off0, ss0, ros0 = oracle.permute(ids, E, S)
    assert dropped == 0
    np.testing.assert_array_equal(off, off0)
    np.testing.assert_array_equal(ss, ss0)
    np.testing.assert_array_equal(ros, ros0)
    # one less than the busiest expert's count drops exactly its last slot
    off, ss, ros, dropped = oracle.permute_capped(ids, E, S, C - 1)
    busiest = np.flatnonzero(np.bincount(ids.ravel(), minlength=E) == C)
    assert dropped == len(busiest)
    for e in busiest:
        last = np.flatnonzero(ids.ravel() == e)[-1]
        assert ros[last] == -2


def test_dropped_count_is_monotone_in_capacity():
    rng = np.random.default_rng(9)
    ids = rng.integers(0, 6, size=(40, 1)).astype(np.int32)
    drops = [oracle.permute_capped(ids, 6, 0, C)[3] for C in range(0, 45)]
    assert drops[0] == 40 and drops[-1] == 0
    assert all(a >= b for a, b in zip(drops, drops[1:]))


def _layer_case(rng, T=14, H=32, I=24, E=5, S=1, k=2):
    x = rand_bf16(rng, (T, H), 1.0)
    L = rng.standard_normal((T, E)).astype(np.float32)
    L[:, 0] += 2.0                           # expert 0 is chosen by most tokens
    ids, w = oracle.route(L, k, renormalize=False)
    wgu = rand_bf16(rng, (E + S, 2 * I, H), 0.05)
    wd = rand_bf16(rng, (E + S, H, I), 0.05)
    res = rand_bf16(rng, (T, H), 1.0)
    return x, ids, w, wgu, wd, res


def test_capped_layer_matches_dense_formulation_with_keep_mask():
    """y = sum over kept slots of w FFN_e(x) + shared + residual (numpy fp64)."""
    rng = np.random.default_rng(17)
    x, ids, w, wgu, wd, res = _layer_case(rng)
    T, k = ids.shape
    E, S = 5, 1
    for C in (0, 1, 3, 100):
        y = oracle.moe_layer(x, ids, w, E, S, wgu, wd, residual_bits=res, capacity=C)
        seen = np.zeros(E, int)
        keep = np.zeros(T * k, bool)
        for s, e in enumerate(ids.ravel()):
            keep[s] = seen[e] < C
            seen[e] += 1
        xv = val(x)
        ref = val(res).copy()
        for t in range(T):
            for j in range(k):
                if keep[t * k + j]:
                    ref[t] += w[t, j] * dense_ffn(xv[t:t + 1], wgu[ids[t, j]], wd[ids[t, j]])[0]
        for s in range(S):
            ref += dense_ffn(xv, wgu[E + s], wd[E + s])
        np.testing.assert_allclose(y, ref, rtol=1e-10, atol=1e-12)


def test_capped_layer_limits():
    rng = np.random.default_rng(23)
    x, ids, w, wgu, wd, res = _layer_case(rng, S=0)
    E = 5
    # capacity 0 without shared experts: every slot dropped, out = residual exactly
    y0 = oracle.moe_layer(x, ids, w, E, 0, wgu[:E], wd[:E], residual_bits=res, capacity=0)
    np.testing.assert_array_equal(y0, val(res))
    # capacity >= every count: identical to the dropless layer
    yl = oracle.moe_layer(x, ids, w, E, 0, wgu[:E], wd[:E], residual_bits=res,
                          capacity=ids.size)
    yd = oracle.moe_layer(x, ids, w, E, 0, wgu[:E], wd[:E], residual_bits=res)
    np.testing.assert_array_equal(yl, yd)
