"""Seeded synthetic inputs for the MoE layer shapes the pages measure.

This module only draws inputs.  It holds none of the layer's arithmetic: the
router logits it returns are an *input* of the dispatch path (they are made
here once, x . Wr^T in fp32, and handed unchanged to the CUDA path and to the
oracle).  Both sides of every parity test take their inputs from here.

Shapes follow the pages' two models:
  * OLMoE-1B-7B ("switchyard" page, intro: every token goes to 8 of 64
    experts); hidden 2048, expert intermediate 1024.
  * DeepSeek-MoE-16B ("dispatch" README, Stack: fine-grained MoE with shared
    + routed experts); hidden 2048, 64 routed experts top-6, 2 shared,
    intermediate 1408.
Values: activations N(0,1), router and expert weights N(0, 0.02) rounded to
bf16 (round to nearest even).  Zipf routing adds log p_e, p_e ~ (e+1)^-s,
to the Gaussian logits (expert 0 is the hottest); the "dispatch" README's
phase-2 work is the source of the skewed-load idea.

Draw order from one generator seeded with ``seed``: x, W_r, then W_gu of all
groups, then W_down of all groups (routed experts first, shared after), then
the next layer's weights for a stack.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class MoEShape:
    name: str
    H: int
    E: int
    k: int
    I: int
    S: int = 0
    renormalize: bool = False
    x_dtype: str = "bf16"          # "f32" for the tiny layer
    weights: str = "bf16"          # "int8": weight-only int8 experts
    layers: int = 1
    tokens: tuple = ()
    routings: tuple = ("uniform",)
    notes: str = ""

    @property
    def G(self) -> int:
        return self.E + self.S

    def rows(self, T: int) -> int:
        """Permuted rows M = T*k + S*T."""
        return T * self.k + self.S * T


TINY = MoEShape("tiny", H=256, E=8, k=2, I=512, renormalize=True, x_dtype="f32",
                tokens=(16,), notes="T=16, fp32 activations, top-2 renormalised")
OLMOE = MoEShape("olmoe", H=2048, E=64, k=8, I=1024, tokens=(1, 8, 64),
                 notes="OLMoE-shaped decode layer, top-8 of 64, no renormalisation")
DEEPSEEK = MoEShape("deepseek", H=2048, E=64, k=6, S=2, I=1408,
                    tokens=(1, 16, 128, 512, 2048), routings=("uniform", "zipf"),
                    notes="DeepSeek-MoE-16B-shaped layer, top-6 of 64 + 2 shared")
OLMOE_W8 = MoEShape("olmoe_w8", H=2048, E=64, k=8, I=1024, weights="int8",
                    tokens=(1, 8, 16, 64, 128, 512, 2048), routings=("uniform", "zipf"),
                    notes="OLMoE shapes, int8 weight-only experts")
OLMOE_STACK = MoEShape("olmoe_stack16", H=2048, E=64, k=8, I=1024, layers=16,
                       tokens=(64, 2048), routings=("skew4",),
                       notes="16 OLMoE-shaped MoE blocks with residual adds")

CONFIGS = {c.name: c for c in (TINY, OLMOE, DEEPSEEK, OLMOE_W8, OLMOE_STACK)}

ZIPF_S = 1.2
# Exponent of the zipf bias for the 16-layer stack, chosen so that on the
# seed-0, T=2048 batch of layer 0 the busiest expert receives about 4x the
# mean load (the "switchyard" page, 03 Load balance, reports 4.0x).  It was
# found by bisection over s with the oracle's routing and is checked by a test.
SKEW4_S = 0.335


def zipf_bias(E: int, s: float) -> torch.Tensor:
    """log p_e with p_e = (e+1)^-s / sum_r r^-s, as fp32 [E]."""
    r = np.arange(1, E + 1, dtype=np.float64)
    p = r ** (-s)
    p /= p.sum()
    return torch.from_numpy(np.log(p).astype(np.float32))


def routing_bias(shape: MoEShape, routing: str):
    if routing == "uniform":
        return None
    if routing == "zipf":
        return zipf_bias(shape.E, ZIPF_S)
    if routing == "skew4":
        return zipf_bias(shape.E, SKEW4_S)
    raise ValueError(f"unknown routing {routing!r}")


@dataclass
class LayerInputs:
    shape: MoEShape
    T: int
    routing: str
    x: torch.Tensor                 # [T,H] fp32 or bf16
    w_r: torch.Tensor               # [E,H] bf16
    bias: torch.Tensor | None       # [E] fp32 routing bias (zipf) or None
    logits: torch.Tensor            # [T,E] fp32 = x . Wr^T (+ bias)
    w_gu: torch.Tensor              # [G,2I,H] bf16 (rows 0..I-1 gate, I..2I-1 up)
    w_down: torch.Tensor            # [G,H,I] bf16
    extra: dict = field(default_factory=dict)


def _randn(shape, g, device, std=1.0):
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t


def make_generator(seed: int, device="cpu") -> torch.Generator:
    return torch.Generator(device=device).manual_seed(seed)


def draw_expert_weights(shape: MoEShape, g: torch.Generator, device="cpu"):
    """W_gu [G,2I,H] and W_down [G,H,I], bf16, N(0,0.02)."""
    G, H, I = shape.G, shape.H, shape.I
    w_gu = torch.empty((G, 2 * I, H), dtype=torch.bfloat16, device=device)
    w_down = torch.empty((G, H, I), dtype=torch.bfloat16, device=device)
    for e in range(G):
        w_gu[e] = _randn((2 * I, H), g, device, 0.02).to(torch.bfloat16)
    for e in range(G):
        w_down[e] = _randn((H, I), g, device, 0.02).to(torch.bfloat16)
    return w_gu, w_down


def router_logits_input(x: torch.Tensor, w_r: torch.Tensor, bias) -> torch.Tensor:
    """The router-logit input L = float(x) . float(Wr)^T (+ bias), fp32."""
    L = x.float() @ w_r.float().t()
    if bias is not None:
        L = L + bias.to(L.device)
    return L.contiguous()


def make_layer(shape: MoEShape, T: int, routing: str = "uniform", seed: int = 0,
               device="cpu") -> LayerInputs:
    """One seeded MoE layer: activations, router, logits and expert weights."""
    if device != "cpu":
        torch.backends.cuda.matmul.allow_tf32 = False
    g = make_generator(seed, device)
    x = _randn((T, shape.H), g, device)
    if shape.x_dtype == "bf16":
        x = x.to(torch.bfloat16)
    w_r = _randn((shape.E, shape.H), g, device, 0.02).to(torch.bfloat16)
    w_gu, w_down = draw_expert_weights(shape, g, device)
    bias = routing_bias(shape, routing)
    if bias is not None:
        bias = bias.to(device)
    logits = router_logits_input(x, w_r, bias)
    return LayerInputs(shape, T, routing, x, w_r, bias, logits, w_gu, w_down)


def make_stack(shape: MoEShape, T: int, routing: str = "skew4", seed: int = 0, device="cpu"):
    """x0 plus per-layer (W_r, W_gu, W_down) for an L-layer stack."""
    g = make_generator(seed, device)
    x = _randn((T, shape.H), g, device).to(torch.bfloat16)
    layers = []
    for _ in range(shape.layers):
        w_r = _randn((shape.E, shape.H), g, device, 0.02).to(torch.bfloat16)
        w_gu, w_down = draw_expert_weights(shape, g, device)
        layers.append((w_r, w_gu, w_down))
    bias = routing_bias(shape, routing)
    if bias is not None:
        bias = bias.to(device)
    return x, layers, bias


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The uint16 bit patterns of a bf16 tensor, as numpy (host copy)."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def host_array(t: torch.Tensor) -> np.ndarray:
    """numpy view of a tensor for the oracle: bf16 -> uint16 bits, else as is."""
    if t.dtype == torch.bfloat16:
        return bf16_bits(t)
    return t.detach().cpu().contiguous().numpy()


def expected_touched_experts(E: int, k: int, T: int, S: int = 0) -> float:
    """Expected number of distinct groups served under uniform routing."""
    return E * (1.0 - (1.0 - k / E) ** T) + S


def describe(shape: MoEShape) -> str:
    return (f"{shape.name}: H={shape.H} E={shape.E} k={shape.k} S={shape.S} I={shape.I} "
            f"renorm={int(shape.renormalize)} x={shape.x_dtype} weights={shape.weights} "
            f"layers={shape.layers}")

