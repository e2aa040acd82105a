"""Shared helpers of the GPU parity tests (CUDA path vs the CPU oracle)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from grouped_expert_gemm_moe_gb300 import workloads as W

# bf16-output acceptance bounds: relative Frobenius error and max |diff|
# relative to max |ref|, against the oracle's exact (fp64) layer.
REL_FROB = 5e-3
MAX_REL = 2e-2
# routing weights are fp32 results of a softmax; the kernel's error is a few
# fp32 ulps of the exact value
W_RTOL = 1e-6


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def errors(out: np.ndarray, ref: np.ndarray):
    rel = float(np.linalg.norm(out - ref) / max(np.linalg.norm(ref), 1e-300))
    mx = float(np.abs(out - ref).max() / max(np.abs(ref).max(), 1e-300))
    return rel, mx


def assert_close(out: np.ndarray, ref: np.ndarray, what: str):
    rel, mx = errors(out, ref)
    assert rel <= REL_FROB and mx <= MAX_REL, f"{what}: rel Frobenius {rel:.3e}, max {mx:.3e}"
    return rel, mx


# Every token of a batch is compared against the oracle up to this size (the
# oracle runs a 2048-token DeepSeek-shaped layer in a few seconds on 16 host
# cores); only larger batches are checked on a sample.
FULL_COMPARE_T = 4096


def sample_tokens(T: int, n: int = 48, seed: int = 0) -> np.ndarray:
    """The tokens to compare: all of them up to FULL_COMPARE_T, else the
    first, the last and n-2 seeded random ones."""
    if T <= max(n, FULL_COMPARE_T):
        return np.arange(T)
    rng = np.random.default_rng(seed + T)
    mid = rng.choice(np.arange(1, T - 1), size=n - 2, replace=False)
    return np.sort(np.concatenate([[0, T - 1], mid]))


def host_inputs(inp: W.LayerInputs):
    """numpy views of a layer's inputs for the oracle."""
    x = inp.x.detach().cpu()
    xh = x.numpy() if x.dtype == torch.float32 else W.bf16_bits(x)
    return dict(x=xh, logits=inp.logits.detach().cpu().numpy(),
                w_gu=W.bf16_bits(inp.w_gu), w_down=W.bf16_bits(inp.w_down))


def oracle_out(inp: W.LayerInputs, h: dict, tokens=None, residual=None):
    sh = inp.shape
    ids, w = oracle.route(h["logits"], sh.k, sh.renormalize)
    y = oracle.moe_layer(h["x"], ids, w, sh.E, sh.S, h["w_gu"], h["w_down"],
                         residual_bits=residual, tokens=tokens)
    return ids, w, y
