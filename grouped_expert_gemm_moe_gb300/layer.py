"""One MoE layer (and a stack of them) on top of the C-ABI calls.

``MoELayer.forward`` runs route -> permute -> grouped FFN -> combine on the
current CUDA stream, with every buffer preallocated by PyTorch and reused
across calls, so a forward pass allocates nothing and launches only this
library's kernels.  The grouped FFN is the tcgen05 grouped GEMM, or the
grouped GEMV when the batch has only a few rows per expert.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import binding as B

# Mean permuted rows per expert group at or below which the grouped GEMV is
# used instead of the tensor-core grouped GEMM.
GEMV_MAX_ROWS_PER_GROUP = 0.25

# Largest batch for which "auto" takes the single-launch decode layer
# (measured on GB300: faster than the separate calls at T = 1 and 2, the
# tensor-core GEMM is faster from T = 4 on).
DECODE_LAYER_AUTO_MAX_T = 2


@dataclass
class LayerBuffers:
    T: int
    topk_ids: torch.Tensor
    topk_w: torch.Tensor
    offsets: torch.Tensor
    sorted_slot: torch.Tensor
    row_of_slot: torch.Tensor
    x_perm: torch.Tensor
    y_perm: torch.Tensor
    ffn_ws: torch.Tensor
    perm_ws: torch.Tensor | None
    out: torch.Tensor
    dropped: torch.Tensor            # int32 [1]: slots dropped by the capacity limit
    capacity: int | None             # slots per routed expert, or None (dropless)


class MoELayer:
    """Expert weights resident on the device plus reusable work buffers.

    bf16 experts: ``w_gu`` [G,2I,H] (gate rows then up rows) and ``w_down``
    [G,H,I].  int8 experts: ``q_gu``/``s_gu``/``q_down``/``s_down`` from
    ``binding.moe_quantize_w8``.  G = E + S; the last S groups are shared
    experts that every token visits with weight 1.
    """

    def __init__(self, H, E, k, I, S=0, renormalize=False, w_gu=None, w_down=None,
                 q_gu=None, s_gu=None, q_down=None, s_down=None, device="cuda",
                 capacity_factor=None):
        self.H, self.E, self.k, self.I, self.S = H, E, k, I, S
        self.G = E + S
        self.renormalize = bool(renormalize)
        # None: dropless; else each routed expert serves at most
        # ceil(capacity_factor * T*k / E) slots per batch (the rest are dropped)
        self.capacity_factor = capacity_factor
        self.device = torch.device(device)
        self.int8 = q_gu is not None
        if self.int8:
            self.q_gu, self.s_gu, self.q_down, self.s_down = q_gu, s_gu, q_down, s_down
        else:
            if w_gu is None or w_down is None:
                raise ValueError("bf16 weights or int8 weights are required")
            self.w_gu, self.w_down = w_gu, w_down
        self.err = B.new_error_word(self.device)
        self._bufs: dict[int, LayerBuffers] = {}
        self._decode_ws: dict[int, torch.Tensor] = {}

    def rows(self, T: int) -> int:
        return T * self.k + self.S * T

    def buffers(self, T: int) -> LayerBuffers:
        b = self._bufs.get(T)
        if b is None:
            d = self.device
            M = self.rows(T)
            ws = B.moe_ffn_workspace_size(M, self.I)
            pws = B.moe_permute_workspace_size(T, self.E, self.S, self.k)
            b = LayerBuffers(
                T=T,
                topk_ids=torch.empty((T, self.k), dtype=torch.int32, device=d),
                topk_w=torch.empty((T, self.k), dtype=torch.float32, device=d),
                offsets=torch.empty(self.G + 1, dtype=torch.int32, device=d),
                sorted_slot=torch.empty(T * self.k, dtype=torch.int32, device=d),
                row_of_slot=torch.empty(T * self.k, dtype=torch.int32, device=d),
                x_perm=torch.empty((M, self.H), dtype=torch.bfloat16, device=d),
                y_perm=torch.empty((M, self.H), dtype=torch.bfloat16, device=d),
                ffn_ws=torch.empty(max(ws, 256), dtype=torch.uint8, device=d),
                perm_ws=(torch.empty(pws, dtype=torch.uint8, device=d) if pws else None),
                out=torch.empty((T, self.H), dtype=torch.bfloat16, device=d),
                dropped=torch.zeros(1, dtype=torch.int32, device=d),
                capacity=(None if self.capacity_factor is None else
                          B.capacity_of(self.capacity_factor, T, self.k, self.E)),
            )
            self._bufs[T] = b
        return b

    def decode_layer_ok(self, T: int, x_dtype=torch.bfloat16) -> bool:
        """The single-launch decode layer applies: bf16 experts and
        activations, dropless, T <= 8, T*k <= 64, S*T <= 64, E <= 256."""
        return (not self.int8 and self.capacity_factor is None and x_dtype == torch.bfloat16
                and T <= B.DECODE_LAYER_MAX_T and T * self.k <= B.DECODE_LAYER_MAX_SLOTS
                and self.S * T <= 64 and self.S <= 32 and self.E <= B.DECODE_LAYER_MAX_E)

    def choose_path(self, T: int, x_dtype=torch.bfloat16) -> str:
        """What forward(ffn="auto") runs: "decode", "gemv" or "gemm"."""
        if T <= DECODE_LAYER_AUTO_MAX_T and self.decode_layer_ok(T, x_dtype):
            return "decode"
        return self.choose_ffn(T)

    def choose_ffn(self, T: int) -> str:
        return "gemv" if self.rows(T) / self.G <= GEMV_MAX_ROWS_PER_GROUP else "gemm"

    def route(self, logits, b: LayerBuffers, stream=None):
        B.moe_route(logits, self.k, self.renormalize, b.topk_ids, b.topk_w, self.err, stream)

    def permute(self, x, b: LayerBuffers, stream=None):
        if b.capacity is not None:
            B.moe_permute_capped(b.topk_ids, self.E, self.S, b.capacity, x, b.offsets,
                                 b.sorted_slot, b.row_of_slot, b.x_perm, b.dropped, b.perm_ws,
                                 self.err, stream)
            return
        B.moe_permute(b.topk_ids, self.E, self.S, x, b.offsets, b.sorted_slot, b.row_of_slot,
                      b.x_perm, b.perm_ws, self.err, stream)

    def fused_route_permute_ok(self, T: int) -> bool:
        # the fused kernel routes every token in every CTA, one warp per token:
        # worth it while a CTA's 32 warps route each token at most once
        return (T <= 32 and T * self.k <= B.ROUTE_PERMUTE_MAX_SLOTS
                and self.E <= B.ROUTE_PERMUTE_MAX_E and self.capacity_factor is None)

    def route_permute(self, logits, x, b: LayerBuffers, stream=None):
        """Routing and permutation: one fused launch for decode-sized batches,
        the two separate calls otherwise (identical results)."""
        if self.fused_route_permute_ok(b.T):
            B.moe_route_permute(logits, self.k, self.renormalize, self.S, x, b.topk_ids, b.topk_w,
                                b.offsets, b.sorted_slot, b.row_of_slot, b.x_perm, self.err,
                                stream)
        else:
            self.route(logits, b, stream)
            self.permute(x, b, stream)

    def hidden(self, b: LayerBuffers) -> torch.Tensor:
        """The bf16 hidden rows h [M, I] inside the FFN workspace."""
        M = self.rows(b.T)
        return b.ffn_ws[:M * self.I * 2].view(torch.bfloat16).view(M, self.I)

    def gate_up(self, b: LayerBuffers, kind: str, stream=None):
        """First FFN phase alone (bf16 experts): h = silu(x Wg^T) * (x Wu^T)."""
        fn = B.moe_grouped_gemv_gate_up if kind == "gemv" else B.moe_grouped_gemm_gate_up
        fn(b.x_perm, b.offsets, self.w_gu, self.hidden(b), self.err, stream)

    def down(self, b: LayerBuffers, kind: str, stream=None):
        """Second FFN phase alone (bf16 experts): y_perm = h Wd^T."""
        fn = B.moe_grouped_gemv_down if kind == "gemv" else B.moe_grouped_gemm_down
        fn(self.hidden(b), b.offsets, self.w_down, b.y_perm, self.err, stream)

    def ffn(self, b: LayerBuffers, kind: str, stream=None):
        if self.int8:
            fn = B.moe_grouped_gemv_w8 if kind == "gemv" else B.moe_grouped_gemm_swiglu_w8
            fn(b.x_perm, b.offsets, self.q_gu, self.s_gu, self.q_down, self.s_down, b.y_perm,
               b.ffn_ws, self.err, stream)
        else:
            fn = B.moe_grouped_gemv if kind == "gemv" else B.moe_grouped_gemm_swiglu
            fn(b.x_perm, b.offsets, self.w_gu, self.w_down, b.y_perm, b.ffn_ws, self.err, stream)

    def combine(self, b: LayerBuffers, out, residual=None, stream=None):
        if b.capacity is not None:
            B.moe_combine_capped(b.y_perm, b.row_of_slot, b.topk_w, b.offsets, self.E, self.S,
                                 out, residual, self.err, stream)
            return
        B.moe_combine(b.y_perm, b.row_of_slot, b.topk_w, self.S, out, residual, self.err, stream)

    def decode_workspace(self, T: int) -> torch.Tensor:
        ws = self._decode_ws.get(T)
        if ws is None:
            n = B.moe_decode_workspace_size(T, self.E, self.S, self.k, self.H, self.I)
            ws = self._decode_ws[T] = torch.empty(n, dtype=torch.uint8, device=self.device)
        return ws

    def forward(self, x, logits, out=None, residual=None, ffn="auto", stream=None):
        """out[t] = sum_j w[t,j] FFN_{id[t,j]}(x[t]) + sum_s FFN_{E+s}(x[t]) (+ residual[t]).
        ffn: "gemm", "gemv", "decode" (the single-launch decode layer) or
        "auto" (decode where it applies and measured fastest, else by rows
        per group)."""
        T = x.shape[0]
        b = self.buffers(T)
        kind = self.choose_path(T, x.dtype) if ffn == "auto" else ffn
        if kind == "decode":
            if not self.decode_layer_ok(T, x.dtype):
                raise ValueError("the single-launch decode layer does not apply to this batch")
            dst = b.out if out is None else out
            B.moe_decode_layer(logits, x, self.k, self.renormalize, self.S, self.w_gu,
                               self.w_down, dst, self.decode_workspace(T), residual, b.topk_ids,
                               b.topk_w, self.err, stream)
            return dst
        self.route_permute(logits, x, b, stream)
        self.ffn(b, kind, stream)
        dst = b.out if out is None else out
        self.combine(b, dst, residual, stream)
        return dst

    def forward_routed(self, x, out=None, residual=None, ffn="auto", stream=None):
        """The layer after routing: this batch's top-k ids and weights are
        already in buffers(T) (e.g. from moe_router_route)."""
        T = x.shape[0]
        b = self.buffers(T)
        kind = self.choose_ffn(T) if ffn == "auto" else ffn
        self.permute(x, b, stream)
        self.ffn(b, kind, stream)
        dst = b.out if out is None else out
        self.combine(b, dst, residual, stream)
        return dst

    def capture(self, x: torch.Tensor, logits: torch.Tensor, out=None, residual=None,
                ffn="auto") -> "CapturedForward":
        """Record one forward pass over the fixed device buffers x / logits
        into a CUDA graph; replay() then reruns it with whatever x and
        logits hold.  Decode-sized batches are launch-bound without this."""
        return CapturedForward(self, x, logits, out, residual, ffn)

    def capture_host(self, x_host: torch.Tensor, logits_host: torch.Tensor, ffn="auto",
                     residual=None) -> "CapturedHostForward":
        """Like capture(), for inputs and output in pinned host memory: the
        graph holds the copy of x to the device and the forward pass, whose
        routing reads the logits from the host buffer and whose last kernel
        stores the output straight into a pinned host buffer, so a step is
        one graph launch.
        replay() returns the pinned host output (valid after the stream is
        synchronised); it reruns the step on whatever the host inputs hold."""
        return CapturedHostForward(self, x_host, logits_host, ffn, residual)

    def check(self):
        """Synchronise and raise if any kernel reported a device-side fault."""
        B.check_device_error(self.err, "MoELayer")


class CapturedHostForward:
    """A forward pass with its host<->device copies recorded into one CUDA
    graph (see MoELayer.capture_host)."""

    def __init__(self, layer: MoELayer, x_host, logits_host, ffn, residual):
        if x_host.is_cuda or logits_host.is_cuda:
            raise ValueError("capture_host takes host tensors")
        if not (x_host.is_pinned() and logits_host.is_pinned()):
            raise ValueError("capture_host needs pinned host memory (tensor.pin_memory())")
        self.layer, self.x_host, self.logits_host = layer, x_host, logits_host
        dev = layer.device
        self.x = torch.empty(x_host.shape, dtype=x_host.dtype, device=dev)
        T = x_host.shape[0]
        self.out_host = torch.empty((T, layer.H), dtype=torch.bfloat16).pin_memory()

        # the transfers are kernels of the library (moe_copy: SMs reading and
        # writing the mapped pinned host memory over NVLink-C2C) when the
        # sizes allow 16-byte copies, else copy-engine transfers
        def transfer(dst, src):
            if dst.nbytes % 16 == 0 and dst.data_ptr() % 16 == 0 and src.data_ptr() % 16 == 0:
                B.moe_copy(dst, src)
            else:
                dst.copy_(src, non_blocking=True)

        # The layer's last kernel (combine, or the decode layer's combine
        # phase) stores the output straight into the pinned host buffer, so
        # the transfer back overlaps its own reads, and the routing reads the
        # logits straight from their host buffer.  x: the single-launch decode
        # layer reads it from the host buffer too (measured 4 us cheaper than
        # copying it at T=1); the permute's gather does not (measured 4 us
        # slower at T=64 and 260 us slower at T=2048), so x is copied there.
        kind = layer.choose_path(T, x_host.dtype) if ffn == "auto" else ffn

        def step():
            if kind == "decode":
                layer.forward(self.x_host, self.logits_host, out=self.out_host,
                              residual=residual, ffn=kind)
                return
            transfer(self.x, self.x_host)
            layer.forward(self.x, self.logits_host, out=self.out_host, residual=residual,
                          ffn=kind)

        step()                                  # eager pass: kernel attributes
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, capture_error_mode="thread_local"):
            step()
        torch.cuda.synchronize()

    def replay(self):
        self.graph.replay()
        return self.out_host


class CapturedForward:
    """A forward pass recorded into a CUDA graph (see MoELayer.capture)."""

    def __init__(self, layer: MoELayer, x, logits, out, residual, ffn):
        self.layer, self.x, self.logits = layer, x, logits
        T = x.shape[0]
        self.out = out if out is not None else torch.empty((T, layer.H), dtype=torch.bfloat16,
                                                           device=x.device)
        # one eager pass first: sets kernel attributes outside the capture
        layer.forward(x, logits, out=self.out, residual=residual, ffn=ffn)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, capture_error_mode="thread_local"):
            layer.forward(x, logits, out=self.out, residual=residual, ffn=ffn)
        torch.cuda.synchronize()

    def replay(self):
        self.graph.replay()
        return self.out


class MoEStack:
    """L MoE blocks with residual adds, x_{l+1} = bf16(x_l + MoE_l(x_l)); the
    routing of block l comes from x_l on the device, router logits and top-k
    in one launch (moe_router_route)."""

    def __init__(self, layers: list[MoELayer], routers: list[torch.Tensor], bias=None):
        self.layers = layers
        self.routers = routers
        self.bias = bias
        self._logits: dict[int, torch.Tensor] = {}
        self._x: dict[int, tuple[torch.Tensor, torch.Tensor]] = {}

    def forward(self, x, ffn="auto", stream=None, keep=None):
        """Runs all blocks; returns the final activations (a reused buffer).
        keep: optional list that receives (x_l, logits_l) clones per block."""
        T = x.shape[0]
        E = self.layers[0].E
        L = self._logits.get(T)
        if L is None:
            L = self._logits[T] = torch.empty((T, E), dtype=torch.float32, device=x.device)
        pair = self._x.get(T)
        if pair is None:
            pair = self._x[T] = (torch.empty_like(x), torch.empty_like(x))
        cur = x
        for i, (layer, w_r) in enumerate(zip(self.layers, self.routers)):
            b = layer.buffers(T)
            B.moe_router_route(cur, w_r, self.bias, layer.k, layer.renormalize, b.topk_ids,
                               b.topk_w, logits=L if keep is not None else None,
                               dev_error=layer.err, stream=stream)
            if keep is not None:
                keep.append((cur.clone(), L.clone()))
            nxt = pair[i % 2]
            layer.forward_routed(cur, out=nxt, residual=cur, ffn=ffn, stream=stream)
            cur = nxt
        return cur

    def capture(self, x: torch.Tensor, ffn="auto") -> "CapturedStack":
        """Record one pass over all blocks (router logits included) into a
        CUDA graph; replay() reruns it on whatever the fixed buffer x holds."""
        return CapturedStack(self, x, ffn)


class CapturedStack:
    """A whole-stack forward pass recorded into one CUDA graph."""

    def __init__(self, stack: MoEStack, x: torch.Tensor, ffn):
        self.stack, self.x = stack, x
        stack.forward(x, ffn=ffn)               # eager pass: buffers and kernel attributes
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, capture_error_mode="thread_local"):
            self.out = stack.forward(x, ffn=ffn)
        torch.cuda.synchronize()

    def replay(self):
        self.graph.replay()
        return self.out

