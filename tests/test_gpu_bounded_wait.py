"""Failure detection on the device without a fault: every wait of the
library's kernels is bounded, and on running out it records MOE_ERR_TIMEOUT
in the caller's dev_error word and returns.  moe_selftest_bounded_wait runs
those very waits (the decode layer's grid barrier, the tensor-core kernels'
mbarrier waits) with a 1 ms limit on a condition that is never met, and on
one that is met as a control.  Afterwards the same stream must still run a
layer correctly, so the context survived.
"""
import time

import numpy as np
import pytest
import torch

from grouped_expert_gemm_moe_gb300 import workloads as W

from gpu_helpers import assert_close, host_inputs, oracle_out, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
MOE_ERR_TIMEOUT = 7
LIMIT_NS = 1_000_000                      # 1 ms
# (arrivals at the grid barrier, completed waits) when the condition is met
MET = {0: (2, 2), 1: (0, 1), 2: (0, 32)}


@pytest.fixture(scope="module")
def B():
    import __graft_entry__ as g
    g.build()
    from grouped_expert_gemm_moe_gb300 import binding
    return binding


@pytest.mark.parametrize("kind", [0, 1, 2], ids=["grid_barrier", "mbarrier", "mbarrier_warp"])
def test_met_wait_passes_and_unmet_wait_times_out(B, kind):
    err = B.new_error_word(DEV)
    cnt = torch.full((2,), -1, dtype=torch.int32, device=DEV)
    B.moe_selftest_bounded_wait(kind, True, LIMIT_NS, cnt, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert tuple(cnt.tolist()) == MET[kind]

    t0 = time.perf_counter()
    B.moe_selftest_bounded_wait(kind, False, LIMIT_NS, cnt, err)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(err.item()) == MOE_ERR_TIMEOUT
    arrivals, passed = cnt.tolist()
    assert passed == 0                                  # no wait claimed success
    assert arrivals == MET[kind][0]                     # every CTA arrived, then gave up
    assert dt < 0.5, f"a 1 ms wait took {dt:.3f} s to give up"


def test_stream_runs_a_layer_after_a_timeout(B):
    err = B.new_error_word(DEV)
    cnt = torch.zeros(2, dtype=torch.int32, device=DEV)
    for kind in (0, 1, 2):
        B.moe_selftest_bounded_wait(kind, False, LIMIT_NS, cnt, err)
    torch.cuda.synchronize()
    assert int(err.item()) == MOE_ERR_TIMEOUT
    from grouped_expert_gemm_moe_gb300.layer import MoELayer
    sh = W.TINY
    inp = W.make_layer(sh, 16, "uniform", seed=0)
    layer = MoELayer(sh.H, sh.E, sh.k, sh.I, sh.S, sh.renormalize, w_gu=inp.w_gu.to(DEV),
                     w_down=inp.w_down.to(DEV), device=DEV)
    for ffn in ("gemm", "gemv"):
        out = layer.forward(inp.x.to(DEV), inp.logits.to(DEV), ffn=ffn)
        layer.check()
        _, _, y = oracle_out(inp, host_inputs(inp))
        assert_close(to_np(out), y, f"tiny layer after timeouts ({ffn})")


def test_limit_is_validated(B):
    err = B.new_error_word(DEV)
    cnt = torch.zeros(2, dtype=torch.int32, device=DEV)
    for bad in (0, 999, 10_000_000_001):
        with pytest.raises(B.MoEError):
            B.moe_selftest_bounded_wait(0, False, bad, cnt, err)
    with pytest.raises(B.MoEError):
        B.moe_selftest_bounded_wait(3, True, LIMIT_NS, cnt, err)
