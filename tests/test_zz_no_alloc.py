"""moe_grouped_gemv_noalloc: the grouped GEMV for callers that cannot
allocate device memory (a framework callback with no allocator, a
latency-critical path that cannot risk cudaMalloc/cudaFree synchronising the
device, a process whose memory belongs to its own pool).  Its scratch is a
fixed 8 MiB array inside the library instead of a caller workspace.

The test calls the entry point through the C ABI (ctypes on libmoe.so) twice
in a row, on two different batches, and checks that each result has the
same bytes as the workspace-taking moe_grouped_gemv on the same inputs (the
two run the same kernels; only where the hidden rows live differs).  It also
checks that a problem larger than the built-in scratch, and one beyond the
weight-size limit of moe_grouped_gemv, are refused before any launch.  This file is named
to be collected last and works in a fresh process or after the other tests.
"""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    from grouped_expert_gemm_moe_gb300 import binding
    return binding


def _call_noalloc(B, x_perm, offsets, w_gu, w_down, y_perm, err):
    f = B._lib.moe_grouped_gemv_noalloc          # the C entry point itself
    M, H = x_perm.shape
    G = offsets.numel() - 1
    I = w_down.shape[2]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    return f(p(x_perm), p(offsets), G, M, H, I, p(w_gu), p(w_down), p(y_perm), p(err), stream)


def _batch(B, shape, T, seed, w):
    from grouped_expert_gemm_moe_gb300 import workloads as W
    from grouped_expert_gemm_moe_gb300.layer import MoELayer
    g = W.make_generator(seed)
    x = torch.randn((T, shape.H), generator=g).to(torch.bfloat16)
    logits = W.router_logits_input(x, w["w_r"], None)
    layer = MoELayer(shape.H, shape.E, shape.k, shape.I, shape.S, shape.renormalize,
                     w_gu=w["w_gu"], w_down=w["w_down"], device=DEV)
    b = layer.buffers(T)
    layer.route(logits.to(DEV), b)
    layer.permute(x.to(DEV), b)
    return layer, b


def test_noalloc_gemv_matches_workspace_gemv_on_two_calls(lib):
    B = lib
    from grouped_expert_gemm_moe_gb300 import workloads as W
    shape = W.DEEPSEEK                      # 64 routed experts top-6 + 2 shared, I = 1408
    inp = W.make_layer(shape, 1, "uniform", seed=0, device=DEV)
    w = dict(w_r=inp.w_r.cpu(), w_gu=inp.w_gu, w_down=inp.w_down)
    for call, (T, seed) in enumerate([(16, 11), (9, 12)]):
        layer, b = _batch(B, shape, T, seed, w)
        M = layer.rows(T)
        assert M * shape.I * 2 <= 8 << 20
        ws = torch.empty(B.moe_ffn_workspace_size(M, shape.I), dtype=torch.uint8, device=DEV)
        ref = torch.empty((M, shape.H), dtype=torch.bfloat16, device=DEV)
        B.moe_grouped_gemv(b.x_perm, b.offsets, w["w_gu"], w["w_down"], ref, ws, layer.err)
        got = torch.full((M, shape.H), float("nan"), dtype=torch.bfloat16, device=DEV)
        st = _call_noalloc(B, b.x_perm, b.offsets, w["w_gu"], w["w_down"], got, layer.err)
        assert st == 0, B.status_string(st)
        torch.cuda.synchronize()
        assert int(layer.err.item()) == 0
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), \
            f"call {call}: the no-allocation GEMV differs from the workspace GEMV"


def test_noalloc_gemv_refuses_problems_beyond_its_scratch(lib):
    B = lib
    H, I, G = 64, 1024, 4
    M = (8 << 20) // (I * 2) + 1            # one row more than the scratch holds
    x = torch.zeros((M, H), dtype=torch.bfloat16, device=DEV)
    off = torch.zeros(G + 1, dtype=torch.int32, device=DEV)
    wgu = torch.zeros((G, 2 * I, H), dtype=torch.bfloat16, device=DEV)
    wd = torch.zeros((G, H, I), dtype=torch.bfloat16, device=DEV)
    y = torch.zeros((M, H), dtype=torch.bfloat16, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    assert _call_noalloc(B, x, off, wgu, wd, y, err) == 4        # MOE_ERR_WORKSPACE


def test_noalloc_gemv_refuses_what_moe_grouped_gemv_refuses(lib):
    """Expert weights of 2^40 elements or more are beyond both GEMV entry
    points; the check happens on the host, so the small buffers passed here
    are never read."""
    B = lib
    G, M, H, I = 1024, 1, 65536, 8192              # G * 2I * H = 2^40
    x = torch.zeros((M, 64), dtype=torch.bfloat16, device=DEV)
    off = torch.zeros(G + 1, dtype=torch.int32, device=DEV)
    wgu = torch.zeros(64, dtype=torch.bfloat16, device=DEV)
    wd = torch.zeros(64, dtype=torch.bfloat16, device=DEV)
    y = torch.zeros((M, 64), dtype=torch.bfloat16, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    f = B._lib.moe_grouped_gemv_noalloc
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = f(p(x), p(off), G, M, H, I, p(wgu), p(wd), p(y), p(err), stream)
    assert st == 2, B.status_string(st)                          # MOE_ERR_UNSUPPORTED
    ws = torch.zeros(B.moe_ffn_workspace_size(M, I), dtype=torch.uint8, device=DEV)
    st_ws = B._lib.moe_grouped_gemv(p(x), p(off), G, M, H, I, p(wgu), p(wd), p(y), p(ws),
                                    ws.numel(), p(err), stream)
    assert st_ws == st
