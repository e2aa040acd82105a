"""ctypes wrapper of the plain-C MoE oracle (``moe_oracle.c``).

TEST INFRASTRUCTURE: imported only by tests, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference arm.  Inputs are numpy arrays (bf16
tensors travel as their uint16 bit patterns); outputs are numpy arrays, fp64
for every floating-point result.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

P = ctypes.c_void_p
I64 = ctypes.c_int64
I32 = ctypes.c_int


def build(force: bool = False) -> str:
    """Compile ``moe_oracle.c`` into ``liboracle.so`` with gcc (OpenMP)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            sigs = {
                "oracle_route": [P, I64, I32, I32, I32, P, P],
                "oracle_permute": [P, I64, I32, I32, I32, P, P, P],
                "oracle_permute_capped": [P, I64, I32, I32, I32, I64, P, P, P, P],
                "oracle_moe_layer_capped": [P, I32, P, P, I64, I32, I32, I32, I32, I32, I64, P,
                                            P, P, P, I64, P, I32],
                "oracle_expert_hidden": [P, P, I32, I32, P],
                "oracle_expert_down": [P, P, I32, I32, P],
                "oracle_moe_layer": [P, I32, P, P, I64, I32, I32, I32, I32, I32, P, P, P, P, I64,
                                     P, I32],
                "oracle_moe_layer_w8": [P, I32, P, P, I64, I32, I32, I32, I32, I32, P, P, P, P,
                                        P, P, I64, P, I32],
                "oracle_quantize_w8": [P, I64, I64, P, P],
                "oracle_router_logits": [P, P, P, I64, I32, I32, P],
                "oracle_num_threads": [],
            }
            for name, args in sigs.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = ctypes.c_int if name != "oracle_expert_hidden" and \
                    name != "oracle_expert_down" else None
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"{what}: oracle returned {rc} "
                         f"({'bad argument' if rc == 1 else 'bad input value'})")


def num_threads() -> int:
    return int(load().oracle_num_threads())


def route(logits, k: int, renormalize: bool):
    """Top-k by (logit desc, index asc); softmax over all E; optional renorm.

    Returns (ids int32 [T,k], w float64 [T,k])."""
    L = _c(logits, np.float32)
    T, E = L.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    _check(load().oracle_route(_p(L), T, E, k, int(renormalize), _p(ids), _p(w)), "route")
    return ids, w


def permute(ids, E: int, S: int = 0):
    """Stable counting sort of slots by expert.

    Returns (offsets int32 [E+S+1], sorted_slot int32 [T*k], row_of_slot int32 [T*k])."""
    ids = _c(ids, np.int32)
    T, k = ids.shape
    off = np.empty(E + S + 1, np.int32)
    ss = np.empty(T * k, np.int32)
    ros = np.empty(T * k, np.int32)
    _check(load().oracle_permute(_p(ids), T, E, S, k, _p(off), _p(ss), _p(ros)), "permute")
    return off, ss, ros


def permute_capped(ids, E: int, S: int, capacity: int):
    """The dropping variant: each routed expert keeps its first `capacity`
    slots in slot order.  Returns (offsets int32 [E+S+1], sorted_slot int32
    [T*k] (-1 past the kept rows), row_of_slot int32 [T*k] (-2: dropped),
    dropped: int)."""
    ids = _c(ids, np.int32)
    T, k = ids.shape
    off = np.empty(E + S + 1, np.int32)
    ss = np.empty(T * k, np.int32)
    ros = np.empty(T * k, np.int32)
    dropped = ctypes.c_int64(0)
    _check(load().oracle_permute_capped(_p(ids), T, E, S, k, int(capacity), _p(off), _p(ss),
                                        _p(ros), ctypes.byref(dropped)), "permute_capped")
    return off, ss, ros, int(dropped.value)


def expert_hidden(x_row, w_gu_e_bits, H: int, I: int):
    """h = silu(Wg x) * (Wu x) for one expert; w_gu_e_bits: uint16 [2I, H]."""
    x = _c(x_row, np.float64)
    wg = _c(w_gu_e_bits, np.uint16)
    h = np.empty(I, np.float64)
    load().oracle_expert_hidden(_p(x), _p(wg), H, I, _p(h))
    return h


def expert_down(h_row, w_down_e_bits, H: int, I: int):
    """y = Wd h for one expert; w_down_e_bits: uint16 [H, I]."""
    h = _c(h_row, np.float64)
    wd = _c(w_down_e_bits, np.uint16)
    y = np.empty(H, np.float64)
    load().oracle_expert_down(_p(h), _p(wd), H, I, _p(y))
    return y


def _x_args(x):
    if x.dtype == np.float32:
        return _c(x, np.float32), 1
    return _c(x, np.uint16), 0


def moe_layer(x, ids, w, E: int, S: int, w_gu_bits, w_down_bits, residual_bits=None,
              tokens=None, nthreads: int = 0, capacity=None):
    """Full MoE layer in fp64.  x: float32 [T,H] or bf16 bits uint16 [T,H];
    w_gu_bits uint16 [E+S, 2I, H]; w_down_bits uint16 [E+S, H, I].
    capacity: None (dropless) or the per-expert slot capacity of the
    dropping variant.  Returns float64 [T or len(tokens), H]."""
    xa, xf = _x_args(x)
    T, H = xa.shape
    ids = _c(ids, np.int32)
    w = _c(w, np.float64)
    k = ids.shape[1]
    G, twoI, H2 = w_gu_bits.shape
    I = twoI // 2
    assert G == E + S and H2 == H and w_down_bits.shape == (G, H, I)
    wgu = _c(w_gu_bits, np.uint16)
    wd = _c(w_down_bits, np.uint16)
    res = None if residual_bits is None else _c(residual_bits, np.uint16)
    tok = None if tokens is None else _c(tokens, np.int64)
    nout = T if tok is None else len(tok)
    y = np.empty((nout, H), np.float64)
    if capacity is None:
        _check(load().oracle_moe_layer(_p(xa), xf, _p(ids), _p(w), T, H, E, S, k, I, _p(wgu),
                                       _p(wd), _p(res), _p(tok), 0 if tok is None else len(tok),
                                       _p(y), nthreads), "moe_layer")
    else:
        _check(load().oracle_moe_layer_capped(_p(xa), xf, _p(ids), _p(w), T, H, E, S, k, I,
                                              int(capacity), _p(wgu), _p(wd), _p(res), _p(tok),
                                              0 if tok is None else len(tok), _p(y), nthreads),
               "moe_layer_capped")
    return y


def moe_layer_w8(x, ids, w, E: int, S: int, q_gu, s_gu, q_down, s_down, residual_bits=None,
                 tokens=None, nthreads: int = 0):
    """MoE layer with int8 weights dequantised as (float)q * scale, fp64 math."""
    xa, xf = _x_args(x)
    T, H = xa.shape
    ids = _c(ids, np.int32)
    w = _c(w, np.float64)
    k = ids.shape[1]
    G, twoI, H2 = q_gu.shape
    I = twoI // 2
    assert G == E + S and H2 == H and q_down.shape == (G, H, I)
    assert s_gu.shape == (G, 2 * I) and s_down.shape == (G, H)
    qg, qd = _c(q_gu, np.int8), _c(q_down, np.int8)
    sg, sd = _c(s_gu, np.float32), _c(s_down, np.float32)
    res = None if residual_bits is None else _c(residual_bits, np.uint16)
    tok = None if tokens is None else _c(tokens, np.int64)
    nout = T if tok is None else len(tok)
    y = np.empty((nout, H), np.float64)
    _check(load().oracle_moe_layer_w8(_p(xa), xf, _p(ids), _p(w), T, H, E, S, k, I, _p(qg),
                                      _p(sg), _p(qd), _p(sd), _p(res), _p(tok),
                                      0 if tok is None else len(tok), _p(y), nthreads),
           "moe_layer_w8")
    return y


def quantize_w8(w_bits):
    """Per-row symmetric int8 of a bf16 matrix [..., K] (bits as uint16).

    Returns (q int8 same shape, scale float32 [...])."""
    wb = _c(w_bits, np.uint16)
    K = wb.shape[-1]
    rows = wb.size // K
    q = np.empty(wb.shape, np.int8)
    s = np.empty(wb.shape[:-1], np.float32)
    _check(load().oracle_quantize_w8(_p(wb), rows, K, _p(q), _p(s)), "quantize_w8")
    return q, s


def router_logits(x_bits, w_r_bits, bias=None):
    """logits = x Wr^T (+ bias) in fp64; x uint16 [T,H], Wr uint16 [E,H]."""
    x = _c(x_bits, np.uint16)
    wr = _c(w_r_bits, np.uint16)
    T, H = x.shape
    E = wr.shape[0]
    b = None if bias is None else _c(bias, np.float32)
    out = np.empty((T, E), np.float64)
    _check(load().oracle_router_logits(_p(x), _p(wr), _p(b), T, H, E, _p(out)), "router_logits")
    return out
