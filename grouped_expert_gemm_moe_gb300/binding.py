"""ctypes binding of libmoe.so: the same calls as include/moe.h, on torch tensors.

Argument marshalling only: every step of the layer runs in the library's
CUDA kernels.  PyTorch provides device memory and the current stream.  If
libmoe.so is missing or cannot be loaded, importing this module raises; there
is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build the CUDA library first "
        "(python -c 'import __graft_entry__ as g; g.build()')")

_lib = ctypes.CDLL(LIB_PATH)

P = ctypes.c_void_p
I = ctypes.c_int
I64 = ctypes.c_int64
SZ = ctypes.c_size_t

MOE_DTYPE_BF16 = 0
MOE_DTYPE_F32 = 1

STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
          3: "MOE_ERR_ALIGNMENT", 4: "MOE_ERR_WORKSPACE", 5: "MOE_ERR_CUDA",
          6: "MOE_ERR_DEVICE_CHECK", 7: "MOE_ERR_TIMEOUT"}

_SIGS = {
    "moe_status_string": ([I], ctypes.c_char_p),
    "moe_version": ([], I),
    "moe_router_logits": ([P, P, P, I, I, I, P, P], I),
    "moe_route": ([P, I, I, I, I, P, P, P, P], I),
    "moe_permute_workspace_size": ([I, I, I, I], SZ),
    "moe_permute": ([P, I, I, I, I, P, I, I, P, P, P, P, P, SZ, P, P], I),
    "moe_permute_capped": ([P, I, I, I, I, I, P, I, I, P, P, P, P, P, P, SZ, P, P], I),
    "moe_combine_capped": ([P, P, P, P, I, I, I, I, I, P, P, P, P], I),
    "moe_ffn_workspace_size": ([I, I], SZ),
    "moe_grouped_gemm_swiglu": ([P, P, I, I, I, I, P, P, P, P, SZ, P, P], I),
    "moe_grouped_gemv": ([P, P, I, I, I, I, P, P, P, P, SZ, P, P], I),
    "moe_grouped_gemm_swiglu_w8": ([P, P, I, I, I, I, P, P, P, P, P, P, SZ, P, P], I),
    "moe_grouped_gemv_w8": ([P, P, I, I, I, I, P, P, P, P, P, P, SZ, P, P], I),
    "moe_combine": ([P, P, P, I, I, I, I, P, P, P, P], I),
    "moe_router_route": ([P, P, P, I, I, I, I, I, P, P, P, P, P], I),
    "moe_decode_workspace_size": ([I, I, I, I, I, I], SZ),
    "moe_decode_layer": ([P, P, I, I, I, I, I, I, I, P, P, P, P, P, P, P, SZ, P, P], I),
    "moe_grouped_gemm_gate_up": ([P, P, I, I, I, I, P, P, P, P], I),
    "moe_grouped_gemm_down": ([P, P, I, I, I, I, P, P, P, P], I),
    "moe_grouped_gemv_gate_up": ([P, P, I, I, I, I, P, P, P, P], I),
    "moe_grouped_gemv_down": ([P, P, I, I, I, I, P, P, P, P], I),
    "moe_quantize_w8": ([P, I64, I64, P, P], I),
    "moe_grouped_gemv_noalloc": ([P, P, I, I, I, I, P, P, P, P, P], I),
    "moe_route_permute": ([P, I, I, I, I, I, P, I, I, P, P, P, P, P, P, P, P], I),
    "moe_copy": ([P, P, SZ, P], I),
    "moe_selftest_bounded_wait": ([I, I, ctypes.c_uint64, P, P, P], I),
    "moe_set_gemm_tile": ([I], I),
    "moe_ep_plan": ([P, I, I, I, P, P, P, P, P, P, P, P], I),
}
for _name, (_args, _res) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = _res


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib.moe_status_string(status).decode()
        super().__init__(f"{where}: {msg}")


def _ok(status: int, where: str) -> None:
    if status != 0:
        raise MoEError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t: torch.Tensor, name: str, dtype=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def _dev_or_pinned(t: torch.Tensor, name: str, dtype=None):
    """A tensor the kernels may access in device memory or in mapped pinned
    host memory (loads and stores over NVLink-C2C): the logits read once by
    the routing kernels, the output written once by the combine, the decode
    layer's x."""
    if not t.is_cuda and not t.is_pinned():
        raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def version() -> int:
    return int(_lib.moe_version())


def status_string(status: int) -> str:
    return _lib.moe_status_string(status).decode()


def new_error_word(device="cuda") -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device)


def check_device_error(err: torch.Tensor, where: str = "device check") -> None:
    """Synchronise on the word's device and raise if a kernel stored an error."""
    v = int(err.item())
    if v != 0:
        raise MoEError(v, where)


# --------------------------------------------------------------------- calls

def moe_router_logits(x, w_r, bias, logits, stream=None):
    T, H = x.shape
    E = w_r.shape[0]
    _dev(x, "x", torch.bfloat16); _dev(w_r, "w_r", torch.bfloat16)
    _dev_or_pinned(logits, "logits", torch.float32)
    if bias is not None:
        _dev(bias, "bias", torch.float32)
    _ok(_lib.moe_router_logits(_ptr(x), _ptr(w_r), _ptr(bias), T, H, E, _ptr(logits),
                               _stream(stream)), "moe_router_logits")


def moe_router_route(x, w_r, bias, k, renormalize, topk_ids, topk_w, logits=None,
                     dev_error=None, stream=None):
    """Router logits + top-k in one launch (same ids and weights as
    moe_router_logits followed by moe_route); logits: optional fp32 [T,E] output."""
    T, H = x.shape
    E = w_r.shape[0]
    _dev(x, "x", torch.bfloat16); _dev(w_r, "w_r", torch.bfloat16)
    _dev(topk_ids, "topk_ids", torch.int32); _dev(topk_w, "topk_w", torch.float32)
    if logits is not None:
        _dev_or_pinned(logits, "logits", torch.float32)
    if bias is not None:
        _dev(bias, "bias", torch.float32)
    _ok(_lib.moe_router_route(_ptr(x), _ptr(w_r), _ptr(bias), T, H, E, k, int(renormalize),
                              _ptr(logits), _ptr(topk_ids), _ptr(topk_w), _ptr(dev_error),
                              _stream(stream)), "moe_router_route")


def moe_route(logits, k, renormalize, topk_ids, topk_w, dev_error=None, stream=None):
    _dev_or_pinned(logits, "logits", torch.float32)
    T, E = logits.shape
    _dev(topk_ids, "topk_ids", torch.int32); _dev(topk_w, "topk_w", torch.float32)
    _ok(_lib.moe_route(_ptr(logits), T, E, k, int(bool(renormalize)), _ptr(topk_ids),
                       _ptr(topk_w), _ptr(dev_error), _stream(stream)), "moe_route")


def moe_permute_workspace_size(T, E, S, k) -> int:
    return int(_lib.moe_permute_workspace_size(T, E, S, k))


def moe_permute(topk_ids, E, S, x, offsets, sorted_slot, row_of_slot, x_perm, workspace=None,
                dev_error=None, stream=None):
    _dev(topk_ids, "topk_ids", torch.int32)
    T, k = topk_ids.shape
    _dev(x, "x")
    if x.dtype == torch.bfloat16:
        xd = MOE_DTYPE_BF16
    elif x.dtype == torch.float32:
        xd = MOE_DTYPE_F32
    else:
        raise ValueError("x must be bf16 or fp32")
    H = x.shape[1]
    for n, t in (("offsets", offsets), ("sorted_slot", sorted_slot),
                 ("row_of_slot", row_of_slot)):
        _dev(t, n, torch.int32)
    _dev(x_perm, "x_perm", torch.bfloat16)
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _ok(_lib.moe_permute(_ptr(topk_ids), T, E, S, k, _ptr(x), xd, H, _ptr(offsets),
                         _ptr(sorted_slot), _ptr(row_of_slot), _ptr(x_perm), _ptr(workspace),
                         wsb, _ptr(dev_error), _stream(stream)), "moe_permute")


MOE_ROW_DROPPED = -2


def capacity_of(capacity_factor: float, T: int, k: int, E: int) -> int:
    """Slots per routed expert for a capacity factor: ceil(CF * T*k / E)."""
    import math
    return int(math.ceil(capacity_factor * T * k / E))


def moe_permute_capped(topk_ids, E, S, capacity, x, offsets, sorted_slot, row_of_slot, x_perm,
                       dropped, workspace=None, dev_error=None, stream=None):
    """moe_permute with at most `capacity` slots per routed expert (the first
    in slot order); dropped: int32 [1] device tensor <- number of dropped slots."""
    _dev(topk_ids, "topk_ids", torch.int32)
    T, k = topk_ids.shape
    _dev(x, "x")
    if x.dtype == torch.bfloat16:
        xd = MOE_DTYPE_BF16
    elif x.dtype == torch.float32:
        xd = MOE_DTYPE_F32
    else:
        raise ValueError("x must be bf16 or fp32")
    H = x.shape[1]
    for n, t in (("offsets", offsets), ("sorted_slot", sorted_slot),
                 ("row_of_slot", row_of_slot), ("dropped", dropped)):
        _dev(t, n, torch.int32)
    _dev(x_perm, "x_perm", torch.bfloat16)
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _ok(_lib.moe_permute_capped(_ptr(topk_ids), T, E, S, k, int(capacity), _ptr(x), xd, H,
                                _ptr(offsets), _ptr(sorted_slot), _ptr(row_of_slot),
                                _ptr(x_perm), _ptr(dropped), _ptr(workspace), wsb,
                                _ptr(dev_error), _stream(stream)), "moe_permute_capped")


ROUTE_PERMUTE_MAX_SLOTS = 1024
ROUTE_PERMUTE_MAX_E = 256


def moe_route_permute(logits, k, renormalize, S, x, topk_ids, topk_w, offsets, sorted_slot,
                      row_of_slot, x_perm, dev_error=None, stream=None):
    """moe_route + moe_permute in one launch (T*k <= 1024, E <= 256)."""
    _dev_or_pinned(logits, "logits", torch.float32)
    T, E = logits.shape
    _dev(x, "x")
    if x.dtype == torch.bfloat16:
        xd = MOE_DTYPE_BF16
    elif x.dtype == torch.float32:
        xd = MOE_DTYPE_F32
    else:
        raise ValueError("x must be bf16 or fp32")
    _dev(topk_ids, "topk_ids", torch.int32); _dev(topk_w, "topk_w", torch.float32)
    for n, t in (("offsets", offsets), ("sorted_slot", sorted_slot),
                 ("row_of_slot", row_of_slot)):
        _dev(t, n, torch.int32)
    _dev(x_perm, "x_perm", torch.bfloat16)
    _ok(_lib.moe_route_permute(_ptr(logits), T, E, S, k, int(bool(renormalize)), _ptr(x), xd,
                               x.shape[1], _ptr(topk_ids), _ptr(topk_w), _ptr(offsets),
                               _ptr(sorted_slot), _ptr(row_of_slot), _ptr(x_perm),
                               _ptr(dev_error), _stream(stream)), "moe_route_permute")


def moe_ffn_workspace_size(M, I) -> int:
    return int(_lib.moe_ffn_workspace_size(M, I))


def _ffn_common(x_perm, offsets, y_perm, workspace):
    _dev(x_perm, "x_perm", torch.bfloat16); _dev(offsets, "offsets", torch.int32)
    _dev(y_perm, "y_perm", torch.bfloat16); _dev(workspace, "workspace")
    M, H = x_perm.shape
    G = offsets.numel() - 1
    return M, H, G, workspace.numel() * workspace.element_size()


def moe_grouped_gemm_swiglu(x_perm, offsets, w_gu, w_down, y_perm, workspace, dev_error=None,
                            stream=None):
    M, H, G, wsb = _ffn_common(x_perm, offsets, y_perm, workspace)
    _dev(w_gu, "w_gu", torch.bfloat16); _dev(w_down, "w_down", torch.bfloat16)
    I_ = w_down.shape[2]
    _ok(_lib.moe_grouped_gemm_swiglu(_ptr(x_perm), _ptr(offsets), G, M, H, I_, _ptr(w_gu),
                                     _ptr(w_down), _ptr(y_perm), _ptr(workspace), wsb,
                                     _ptr(dev_error), _stream(stream)), "moe_grouped_gemm_swiglu")


def moe_grouped_gemv(x_perm, offsets, w_gu, w_down, y_perm, workspace, dev_error=None,
                     stream=None):
    M, H, G, wsb = _ffn_common(x_perm, offsets, y_perm, workspace)
    _dev(w_gu, "w_gu", torch.bfloat16); _dev(w_down, "w_down", torch.bfloat16)
    I_ = w_down.shape[2]
    _ok(_lib.moe_grouped_gemv(_ptr(x_perm), _ptr(offsets), G, M, H, I_, _ptr(w_gu),
                              _ptr(w_down), _ptr(y_perm), _ptr(workspace), wsb, _ptr(dev_error),
                              _stream(stream)), "moe_grouped_gemv")


def _phase(name, inp, offsets, w, out, H, I_, dev_error, stream):
    _dev(inp, "input", torch.bfloat16); _dev(offsets, "offsets", torch.int32)
    _dev(w, "weights", torch.bfloat16); _dev(out, "output", torch.bfloat16)
    M = inp.shape[0]
    G = offsets.numel() - 1
    _ok(getattr(_lib, name)(_ptr(inp), _ptr(offsets), G, M, H, I_, _ptr(w), _ptr(out),
                            _ptr(dev_error), _stream(stream)), name)


def moe_grouped_gemm_gate_up(x_perm, offsets, w_gu, h, dev_error=None, stream=None):
    """h [M,I] = silu(x_perm Wg^T) * (x_perm Wu^T) per group (tcgen05)."""
    _phase("moe_grouped_gemm_gate_up", x_perm, offsets, w_gu, h, x_perm.shape[1], h.shape[1],
           dev_error, stream)


def moe_grouped_gemm_down(h, offsets, w_down, y_perm, dev_error=None, stream=None):
    """y_perm [M,H] = h Wd^T per group (tcgen05)."""
    _phase("moe_grouped_gemm_down", h, offsets, w_down, y_perm, y_perm.shape[1], h.shape[1],
           dev_error, stream)


def moe_grouped_gemv_gate_up(x_perm, offsets, w_gu, h, dev_error=None, stream=None):
    _phase("moe_grouped_gemv_gate_up", x_perm, offsets, w_gu, h, x_perm.shape[1], h.shape[1],
           dev_error, stream)


def moe_grouped_gemv_down(h, offsets, w_down, y_perm, dev_error=None, stream=None):
    _phase("moe_grouped_gemv_down", h, offsets, w_down, y_perm, y_perm.shape[1], h.shape[1],
           dev_error, stream)


def moe_grouped_gemv_noalloc(x_perm, offsets, w_gu, w_down, y_perm, dev_error=None,
                             stream=None):
    """moe_grouped_gemv with its scratch in the library's built-in 8 MiB
    array instead of a caller workspace (M * I <= 4,194,304).  Calls that
    may overlap on the GPU share that array and must be serialised."""
    _dev(x_perm, "x_perm", torch.bfloat16); _dev(offsets, "offsets", torch.int32)
    _dev(y_perm, "y_perm", torch.bfloat16)
    _dev(w_gu, "w_gu", torch.bfloat16); _dev(w_down, "w_down", torch.bfloat16)
    M, H = x_perm.shape
    G = offsets.numel() - 1
    I_ = w_down.shape[2]
    _ok(_lib.moe_grouped_gemv_noalloc(_ptr(x_perm), _ptr(offsets), G, M, H, I_, _ptr(w_gu),
                                      _ptr(w_down), _ptr(y_perm), _ptr(dev_error),
                                      _stream(stream)), "moe_grouped_gemv_noalloc")


def moe_grouped_gemm_swiglu_w8(x_perm, offsets, q_gu, s_gu, q_down, s_down, y_perm, workspace,
                               dev_error=None, stream=None):
    M, H, G, wsb = _ffn_common(x_perm, offsets, y_perm, workspace)
    for n, t, d in (("q_gu", q_gu, torch.int8), ("s_gu", s_gu, torch.float32),
                    ("q_down", q_down, torch.int8), ("s_down", s_down, torch.float32)):
        _dev(t, n, d)
    I_ = q_down.shape[2]
    _ok(_lib.moe_grouped_gemm_swiglu_w8(_ptr(x_perm), _ptr(offsets), G, M, H, I_, _ptr(q_gu),
                                        _ptr(s_gu), _ptr(q_down), _ptr(s_down), _ptr(y_perm),
                                        _ptr(workspace), wsb, _ptr(dev_error), _stream(stream)),
        "moe_grouped_gemm_swiglu_w8")


def moe_grouped_gemv_w8(x_perm, offsets, q_gu, s_gu, q_down, s_down, y_perm, workspace,
                        dev_error=None, stream=None):
    M, H, G, wsb = _ffn_common(x_perm, offsets, y_perm, workspace)
    for n, t, d in (("q_gu", q_gu, torch.int8), ("s_gu", s_gu, torch.float32),
                    ("q_down", q_down, torch.int8), ("s_down", s_down, torch.float32)):
        _dev(t, n, d)
    I_ = q_down.shape[2]
    _ok(_lib.moe_grouped_gemv_w8(_ptr(x_perm), _ptr(offsets), G, M, H, I_, _ptr(q_gu),
                                 _ptr(s_gu), _ptr(q_down), _ptr(s_down), _ptr(y_perm),
                                 _ptr(workspace), wsb, _ptr(dev_error), _stream(stream)),
        "moe_grouped_gemv_w8")


def moe_combine(y_perm, row_of_slot, topk_w, S, out, residual=None, dev_error=None,
                stream=None):
    _dev(y_perm, "y_perm", torch.bfloat16); _dev(row_of_slot, "row_of_slot", torch.int32)
    _dev(topk_w, "topk_w", torch.float32); _dev_or_pinned(out, "out", torch.bfloat16)
    if residual is not None:
        _dev(residual, "residual", torch.bfloat16)
    T, k = topk_w.shape
    H = out.shape[1]
    _ok(_lib.moe_combine(_ptr(y_perm), _ptr(row_of_slot), _ptr(topk_w), T, k, S, H,
                         _ptr(residual), _ptr(out), _ptr(dev_error), _stream(stream)),
        "moe_combine")


def moe_combine_capped(y_perm, row_of_slot, topk_w, offsets, E, S, out, residual=None,
                       dev_error=None, stream=None):
    """moe_combine after moe_permute_capped (dropped slots add nothing; the
    shared rows start at offsets[E])."""
    _dev(y_perm, "y_perm", torch.bfloat16); _dev(row_of_slot, "row_of_slot", torch.int32)
    _dev(topk_w, "topk_w", torch.float32); _dev_or_pinned(out, "out", torch.bfloat16)
    _dev(offsets, "offsets", torch.int32)
    if residual is not None:
        _dev(residual, "residual", torch.bfloat16)
    T, k = topk_w.shape
    H = out.shape[1]
    _ok(_lib.moe_combine_capped(_ptr(y_perm), _ptr(row_of_slot), _ptr(topk_w), _ptr(offsets), E,
                                T, k, S, H, _ptr(residual), _ptr(out), _ptr(dev_error),
                                _stream(stream)), "moe_combine_capped")


DECODE_LAYER_MAX_T = 8
DECODE_LAYER_MAX_SLOTS = 64
DECODE_LAYER_MAX_E = 256


def moe_decode_workspace_size(T, E, S, k, H, I) -> int:
    return int(_lib.moe_decode_workspace_size(T, E, S, k, H, I))


def moe_decode_layer(logits, x, k, renormalize, S, w_gu, w_down, out, workspace, residual=None,
                     topk_ids=None, topk_w=None, dev_error=None, stream=None):
    """The whole layer for T <= 8 tokens in one cooperative launch (route,
    grouped GEMV gate/up + down, combine); same bytes as the separate calls."""
    _dev_or_pinned(logits, "logits", torch.float32); _dev_or_pinned(x, "x", torch.bfloat16)
    _dev(w_gu, "w_gu", torch.bfloat16); _dev(w_down, "w_down", torch.bfloat16)
    _dev_or_pinned(out, "out", torch.bfloat16); _dev(workspace, "workspace")
    if residual is not None:
        _dev(residual, "residual", torch.bfloat16)
    if topk_ids is not None:
        _dev(topk_ids, "topk_ids", torch.int32)
    if topk_w is not None:
        _dev(topk_w, "topk_w", torch.float32)
    T, E = logits.shape
    H = x.shape[1]
    I = w_down.shape[2]
    wsb = workspace.numel() * workspace.element_size()
    _ok(_lib.moe_decode_layer(_ptr(logits), _ptr(x), T, E, S, k, int(renormalize), H, I,
                              _ptr(w_gu), _ptr(w_down), _ptr(residual), _ptr(out),
                              _ptr(topk_ids), _ptr(topk_w), _ptr(workspace), wsb,
                              _ptr(dev_error), _stream(stream)), "moe_decode_layer")


def moe_quantize_w8(w: torch.Tensor):
    """Host-side int8 quantisation of a bf16 tensor [..., K] (any device;
    the work runs on host copies).  Returns (q int8, scale fp32) on the CPU."""
    wc = w.detach().to("cpu").contiguous()
    if wc.dtype != torch.bfloat16:
        raise ValueError("w must be bf16")
    K = wc.shape[-1]
    rows = wc.numel() // K
    q = torch.empty(wc.shape, dtype=torch.int8)
    s = torch.empty(wc.shape[:-1], dtype=torch.float32)
    _ok(_lib.moe_quantize_w8(_ptr(wc), rows, K, _ptr(q), _ptr(s)), "moe_quantize_w8")
    return q, s


def moe_copy(dst: torch.Tensor, src: torch.Tensor, stream=None) -> None:
    """dst <- src by the GPU's SMs (either may be pinned host memory)."""
    if dst.nbytes != src.nbytes or not dst.is_contiguous() or not src.is_contiguous():
        raise ValueError("moe_copy: contiguous tensors of the same size in bytes")
    for t in (dst, src):
        if not t.is_cuda and not t.is_pinned():
            raise ValueError("moe_copy: host tensors must be pinned")
    _ok(_lib.moe_copy(_ptr(dst), _ptr(src), dst.nbytes, _stream(stream)), "moe_copy")


def moe_selftest_bounded_wait(kind: int, satisfiable: bool, limit_ns: int,
                              counters: torch.Tensor, dev_error: torch.Tensor,
                              stream=None) -> None:
    """Run one bounded device wait (0: grid barrier, 1: mbarrier, 2: warp-
    uniform mbarrier) on a condition met or never met; counters: 2 int32
    words on the device."""
    if counters.numel() < 2 or counters.dtype != torch.int32 or not counters.is_cuda:
        raise ValueError("moe_selftest_bounded_wait: counters must be >= 2 int32 device words")
    _ok(_lib.moe_selftest_bounded_wait(int(kind), int(bool(satisfiable)), int(limit_ns),
                                       _ptr(counters), _ptr(dev_error), _stream(stream)),
        "moe_selftest_bounded_wait")


# moe_tile values of include/moe.h
GEMM_TILES = {"auto": -1, "128x128": 0, "128x256": 1, "pair": 2, "w8_d16": 3, "w8_d32": 4,
              "w8_d64": 5, "w8_rows": 6, "w8_pair": 7}


def moe_set_gemm_tile(tile: str = "auto") -> None:
    """Force one tile kernel for every later grouped GEMM call ("auto":
    the per-call choice by rows per group)."""
    if tile not in GEMM_TILES:
        raise ValueError(f"unknown tile {tile!r}; one of {sorted(GEMM_TILES)}")
    _ok(_lib.moe_set_gemm_tile(GEMM_TILES[tile]), "moe_set_gemm_tile")


class forced_gemm_tile:
    """Context manager: the grouped GEMM calls inside use `tile`."""

    def __init__(self, tile: str):
        self.tile = tile

    def __enter__(self):
        moe_set_gemm_tile(self.tile)
        return self

    def __exit__(self, *exc):
        moe_set_gemm_tile("auto")
        return False


def moe_ep_plan(counts, rank: int):
    """Expert-parallel exchange plan of `rank` (host, numpy).  counts: int
    array [W, E] of every rank's rows per routed expert.  Returns a dict of
    numpy arrays: send_offset, send_count, recv_offset, recv_count [W];
    seg_src, seg_dst, seg_len [W * E/W]; local_offsets [E/W + 1]."""
    import numpy as np
    c = np.ascontiguousarray(counts, dtype=np.int32)
    if c.ndim != 2:
        raise ValueError("moe_ep_plan: counts must be [W, E]")
    W, E = c.shape
    EL = E // W if W > 0 else 0
    out = {k: np.zeros(W, np.int64) for k in ("send_offset", "send_count", "recv_offset",
                                               "recv_count")}
    for k in ("seg_src", "seg_dst", "seg_len"):
        out[k] = np.zeros(max(W * EL, 1), np.int64)
    out["local_offsets"] = np.zeros(EL + 1, np.int32)
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    _ok(_lib.moe_ep_plan(p(c), W, E, int(rank), p(out["send_offset"]), p(out["send_count"]),
                         p(out["recv_offset"]), p(out["recv_count"]), p(out["seg_src"]),
                         p(out["seg_dst"]), p(out["seg_len"]), p(out["local_offsets"])),
        "moe_ep_plan")
    return out
