"""Host-side checks of libmoe.so that need no GPU.

The library must build for sm_103a, load, export every call include/moe.h
declares, reject bad arguments before any device work, and its offline
int8 quantiser must agree bit for bit with the oracle's.  Every call here
fails validation on the host or is host-only, so none touches a device.
"""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from grouped_expert_gemm_moe_gb300 import build as b
    path = b.build()
    return ctypes.CDLL(path)


def declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            txt = open(os.path.join(inc, f)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names |= set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", txt))
    return sorted(names)


def test_header_declares_the_hot_path_calls():
    names = declared_functions()
    for n in ("moe_route", "moe_permute", "moe_grouped_gemm_swiglu", "moe_grouped_gemv",
              "moe_combine", "moe_grouped_gemm_swiglu_w8", "moe_grouped_gemv_w8",
              "moe_quantize_w8", "moe_router_logits", "moe_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_loads_and_matches_header():
    from grouped_expert_gemm_moe_gb300 import binding as B
    for n in declared_functions():
        assert hasattr(B._lib, n)
    assert B.version() >= 100
    assert "workspace" in B.status_string(4)
    assert B.status_string(99) == "unknown moe_status"


def test_status_strings(lib):
    lib.moe_status_string.restype = ctypes.c_char_p
    for code in range(8):
        assert lib.moe_status_string(code).startswith(b"MOE_")


def test_workspace_sizes(lib):
    lib.moe_ffn_workspace_size.restype = ctypes.c_size_t
    lib.moe_permute_workspace_size.restype = ctypes.c_size_t
    assert lib.moe_ffn_workspace_size(16384, 1024) == 16384 * 1024 * 2
    assert lib.moe_ffn_workspace_size(3, 8) == 256
    assert lib.moe_permute_workspace_size(128, 64, 2, 8) == 0          # <= 1024 slots
    # 12288 slots: 12 chunks x (64 + 1) int32 counts, rounded up to 256 bytes
    assert lib.moe_permute_workspace_size(2048, 64, 2, 6) == 3328


P = ctypes.c_void_p
GOOD = ctypes.c_void_p(0x1000)        # never dereferenced: each call fails validation first
ODD = ctypes.c_void_p(0x1008)         # 8-byte aligned only


def test_route_argument_checks(lib):
    lib.moe_route.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P,
                              P, P]
    assert lib.moe_route(None, 4, 8, 2, 0, GOOD, GOOD, None, None) == 1
    assert lib.moe_route(GOOD, 0, 8, 2, 0, GOOD, GOOD, None, None) == 1
    assert lib.moe_route(GOOD, 4, 8, 9, 0, GOOD, GOOD, None, None) == 1       # k > E
    assert lib.moe_route(GOOD, 4, 64, 33, 0, GOOD, GOOD, None, None) == 1     # k > 32
    assert lib.moe_route(GOOD, 4, 2048, 8, 0, GOOD, GOOD, None, None) == 2    # E > 1024


def test_permute_argument_checks(lib):
    f = lib.moe_permute
    f.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, ctypes.c_int,
                  ctypes.c_int, P, P, P, P, P, ctypes.c_size_t, P, P]
    args = dict(ids=GOOD, T=4, E=8, S=0, k=2, x=GOOD, xd=0, H=64, off=GOOD, ss=GOOD, ros=GOOD,
                xp=GOOD)

    def call(**kw):
        a = {**args, **kw}
        return f(a["ids"], a["T"], a["E"], a["S"], a["k"], a["x"], a["xd"], a["H"], a["off"],
                 a["ss"], a["ros"], a["xp"], None, 0, None, None)
    assert call(ids=None) == 1
    assert call(xd=7) == 1
    assert call(E=1000, S=100) == 2                 # G > 1024
    assert call(H=60) == 3                          # H not a multiple of 8
    assert call(x=ODD) == 3
    assert call(xp=ODD) == 3


def test_ffn_argument_checks(lib):
    for name in ("moe_grouped_gemm_swiglu", "moe_grouped_gemv"):
        f = getattr(lib, name)
        f.argtypes = [P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P, P,
                      ctypes.c_size_t, P, P]
        ws = 64 * 32 * 2
        assert f(GOOD, GOOD, 8, 64, 256, 32, GOOD, GOOD, GOOD, None, ws, None, None) == 1
        assert f(GOOD, GOOD, 8, 64, 256, 36, GOOD, GOOD, GOOD, GOOD, ws, None, None) == 3
        assert f(GOOD, GOOD, 8, 64, 256, 32, ODD, GOOD, GOOD, GOOD, ws, None, None) == 3
        assert f(GOOD, GOOD, 8, 64, 256, 32, GOOD, GOOD, GOOD, GOOD, ws - 256, None, None) == 4
        assert f(GOOD, GOOD, 2000, 64, 256, 32, GOOD, GOOD, GOOD, GOOD, ws, None, None) == 2
    f = lib.moe_grouped_gemv_w8
    f.argtypes = [P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P, P, P, P,
                  ctypes.c_size_t, P, P]
    # int8 weights need H and I multiples of 16
    assert f(GOOD, GOOD, 8, 64, 264, 32, GOOD, GOOD, GOOD, GOOD, GOOD, GOOD, 4096, None,
             None) == 3


def test_router_logits_argument_checks(lib):
    f = lib.moe_router_logits
    f.argtypes = [P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P]
    assert f(None, GOOD, None, 4, 64, 8, GOOD, None) == 1
    assert f(GOOD, GOOD, None, 0, 64, 8, GOOD, None) == 1
    assert f(GOOD, GOOD, None, 4, 60, 8, GOOD, None) == 3          # H not a multiple of 8
    assert f(ODD, GOOD, None, 4, 64, 8, GOOD, None) == 3


def test_capped_permute_and_combine_argument_checks(lib):
    f = lib.moe_permute_capped
    f.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, P,
                  ctypes.c_int, ctypes.c_int, P, P, P, P, P, P, ctypes.c_size_t, P, P]
    assert f(GOOD, 4, 8, 0, 2, -1, GOOD, 0, 64, GOOD, GOOD, GOOD, GOOD, GOOD, None, 0, None,
             None) == 1                                  # negative capacity
    assert f(GOOD, 4, 8, 0, 2, 3, GOOD, 0, 64, GOOD, GOOD, GOOD, GOOD, None, None, 0, None,
             None) == 1                                  # no dropped-count word
    assert f(GOOD, 4, 8, 0, 2, 3, GOOD, 0, 60, GOOD, GOOD, GOOD, GOOD, GOOD, None, 0, None,
             None) == 3                                  # H not a multiple of 8
    g = lib.moe_combine_capped
    g.argtypes = [P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, P, P, P, P]
    assert g(GOOD, GOOD, GOOD, None, 8, 4, 2, 0, 64, None, GOOD, None, None) == 1
    assert g(GOOD, GOOD, GOOD, GOOD, 8, 4, 2, 0, 64, ODD, GOOD, None, None) == 3


def test_combine_argument_checks(lib):
    f = lib.moe_combine
    f.argtypes = [P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P, P]
    assert f(None, GOOD, GOOD, 4, 2, 0, 64, None, GOOD, None, None) == 1
    assert f(GOOD, GOOD, GOOD, 4, 2, 0, 60, None, GOOD, None, None) == 3
    assert f(GOOD, GOOD, GOOD, 4, 2, 0, 64, ODD, GOOD, None, None) == 3


def test_quantize_matches_oracle_bit_exact(lib):
    from grouped_expert_gemm_moe_gb300 import binding as B
    g = torch.Generator().manual_seed(3)
    w = (torch.randn((5, 64, 200), generator=g) * 0.02).to(torch.bfloat16)
    w[1, 7] = 0                                      # an all-zero row
    w[2, 3, 10] = 0.5                                # a dominant element
    q, s = B.moe_quantize_w8(w)
    qo, so = oracle.quantize_w8(w.view(torch.int16).numpy().view(np.uint16))
    np.testing.assert_array_equal(q.numpy(), qo)
    np.testing.assert_array_equal(s.numpy().view(np.uint32), so.view(np.uint32))
    assert s[1, 7].item() == 1.0 and (q[1, 7] == 0).all()


def test_quantize_rejects_bad_args(lib):
    lib.moe_quantize_w8.argtypes = [P, ctypes.c_int64, ctypes.c_int64, P, P]
    assert lib.moe_quantize_w8(None, 4, 4, GOOD, GOOD) == 1
    assert lib.moe_quantize_w8(GOOD, 4, 0, GOOD, GOOD) == 1
