"""Thin Python binding of libmoe_gb300.so (ctypes).

Every function here has the name of the C entry point it calls and only
marshals arguments: it checks dtypes, shapes and devices, allocates outputs
with ``torch.empty`` on the input's device, and passes raw pointers plus the
current CUDA stream. All arithmetic runs in the library's CUDA kernels; there
is no fallback of any kind. If the shared library has not been built, or the
tensors are not on a CUDA device, the call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_gb300.so")

# moe_status codes (include/moe_gb300.h)
MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_MISALIGNED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_UNSUPPORTED = 4
MOE_ERR_CUDA = 5
MOE_ERR_DEVICE_TIMEOUT = 6
MOE_ERR_DEVICE_CHECK = 7

MOE_OP_BUILD_PERMUTATION = 1
MOE_OP_EP_LAYOUT = 2
MOE_OP_GROUPED_FFN = 3
MOE_OP_GROUPED_FFN_BACKWARD = 4
MOE_OP_LOAD_BALANCE = 5
MOE_OP_EP_RECV_LAYOUT = 6
MOE_OP_GROUPED_FFN_FP8 = 7
MOE_OP_ROUTE_PERMUTE_EP = 8

WORKSPACE_HEADER = 256

_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t

# exported symbol -> (restype, argtypes); the single source for the loader and the tests
SIGNATURES = {
    "moe_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "moe_route_topk": (_I, [_P, _I, _I, _I, _I, _P, _P, _P]),
    "moe_route_topk_backward": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P]),
    "moe_load_balance": (_I, [_P, _P, _I, _I, _I, _P, _P, _P, _P, _SZ, _P]),
    "moe_load_balance_backward": (_I, [_P, _P, _I, _I, ctypes.c_float, _I, _P, _P]),
    "moe_build_permutation": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_build_permutation_static": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P]),
    "moe_ep_layout": (_I, [_P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_build_permutation_ep": (_I, [_P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                      _SZ, _P]),
    "moe_route_permute_ep": (_I, [_P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                  _P, _P, _SZ, _P]),
    "moe_dispatch": (_I, [_P, _I, _I, _I, _P, _P, _P]),
    "moe_dispatch_scatter": (_I, [_P, _I, _I, _I, _P, _P, _P]),
    "moe_grouped_ffn": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_grouped_ffn_backward": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P,
                                      _P, _P, _P, _SZ, _P]),
    "moe_grouped_ffn_backward_data": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P,
                                           _P, _SZ, _P]),
    "moe_grouped_ffn_backward_weights": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P,
                                              _SZ, _P]),
    "moe_combine": (_I, [_P, _P, _P, _I, _I, _I, _P, _P, _P]),
    "moe_combine_backward": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P, _P]),
    "moe_dispatch_backward": (_I, [_P, _P, _I, _I, _I, _P, _P, _P]),
    "moe_ep_recv_layout": (_I, [_P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_dispatch_slice": (_I, [_P, _I, _I, _I, _P, _P, _I, _I, _I, _P, _P, _P]),
    "moe_combine_slice": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P]),
    "moe_combine_backward_slice": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P]),
    "moe_dispatch_backward_slice": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P]),
    "moe_reduce_finish": (_I, [_P, _P, _I, _I, _P, _P]),
    "moe_mxfp8_quantize_rows": (_I, [_P, _P, _I, _I, _I, _P, _P, _P]),
    "moe_mxfp8_quantize_weights": (_I, [_P, _P, _I, _I, _I, _P, _P, _P]),
    "moe_grouped_ffn_fp8": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_debug_check_status": (_I, [ctypes.POINTER(ctypes.c_int)]),
    "moe_read_device_status": (_I, [_P, _P, ctypes.POINTER(ctypes.c_int)]),
    "moe_debug_wait_timeout": (_I, [_P, _I, _P]),
    "moe_status_string": (ctypes.c_char_p, [_I]),
    "moe_last_cuda_error": (_I, []),
    "moe_version": (_I, []),
    "moe_profile_start": (_I, [_I]),
    "moe_profile_stop": (_I, []),
    "moe_profile_record": (_I, [_I, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_float)]),
}

_lib = None


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = f"{fn} failed: status {status}"
        if _lib is not None:
            msg += f" ({_lib.moe_status_string(status).decode()})"
            if status == MOE_ERR_CUDA:
                msg += f", cudaError {_lib.moe_last_cuda_error()}"
        super().__init__(msg)


def load(path: str = LIB_PATH):
    """Loads the shared library (once) and declares every exported signature."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with grouped_gemm_moe_gb300.build.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(dev: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _check(name: str, rc: int):
    if rc != MOE_OK:
        raise MoEError(name, rc)


def _need(t: torch.Tensor, dtype, ndim: int, name: str):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def workspace_size(op: int, T: int, E: int, K: int, R: int = 1, d: int = 0, I: int = 0) -> int:
    return int(load().moe_workspace_size(op, T, E, K, R, d, I))


def new_workspace(nbytes: int, device) -> torch.Tensor:
    """A workspace with its status header zeroed (the rest is scratch)."""
    ws = torch.empty(max(int(nbytes), WORKSPACE_HEADER), dtype=torch.uint8, device=device)
    ws[:WORKSPACE_HEADER].zero_()
    return ws


def moe_workspace_size(op: int, T: int, E: int, K: int, R: int = 1, d: int = 0, I: int = 0) -> int:
    return workspace_size(op, T, E, K, R, d, I)


def moe_route_topk(logits: torch.Tensor, K: int, renorm: int = 1,
                   out: Optional[Tuple[torch.Tensor, torch.Tensor]] = None):
    _need(logits, torch.float32, 2, "logits")
    T, E = logits.shape
    if out is None:
        idx = torch.empty(T, K, dtype=torch.int32, device=logits.device)
        w = torch.empty(T, K, dtype=torch.float32, device=logits.device)
    else:
        idx, w = out
    _check("moe_route_topk", load().moe_route_topk(_ptr(logits), T, E, K, int(renorm), _ptr(idx),
                                                   _ptr(w), _stream(logits.device)))
    return idx, w


def moe_route_topk_backward(logits: Optional[torch.Tensor], topk_idx: torch.Tensor,
                            topk_w: torch.Tensor, dtopk_w: torch.Tensor, E: int, renorm: int = 1,
                            out: Optional[torch.Tensor] = None):
    _need(topk_idx, torch.int32, 2, "topk_idx")
    _need(topk_w, torch.float32, 2, "topk_w")
    _need(dtopk_w, torch.float32, 2, "dtopk_w")
    if logits is not None:
        _need(logits, torch.float32, 2, "logits")
    T, K = topk_idx.shape
    dl = out if out is not None else torch.empty(T, E, dtype=torch.float32, device=topk_idx.device)
    _check("moe_route_topk_backward", load().moe_route_topk_backward(
        _ptr(logits), _ptr(topk_idx), _ptr(topk_w), _ptr(dtopk_w), T, E, K, int(renorm), _ptr(dl),
        _stream(topk_idx.device)))
    return dl


def moe_load_balance(logits: torch.Tensor, counts: torch.Tensor, K: int,
                     ws: Optional[torch.Tensor] = None, out=None):
    """Load-balance metrics and loss: returns (load_frac [E], prob_mean [E], stats [4]) with
    stats = (loss, E * max load_frac, empty experts, sum load_frac), all fp32 on device."""
    _need(logits, torch.float32, 2, "logits")
    _need(counts, torch.int32, 1, "counts")
    T, E = logits.shape
    dev = logits.device
    if ws is None:
        ws = new_workspace(workspace_size(MOE_OP_LOAD_BALANCE, T, E, K), dev)
    if out is None:
        out = (torch.empty(E, dtype=torch.float32, device=dev),
               torch.empty(E, dtype=torch.float32, device=dev),
               torch.empty(4, dtype=torch.float32, device=dev))
    frac, pmean, stats = out
    _check("moe_load_balance", load().moe_load_balance(
        _ptr(logits), _ptr(counts), T, E, int(K), _ptr(frac), _ptr(pmean), _ptr(stats), _ptr(ws),
        ws.numel() * ws.element_size(), _stream(dev)))
    return frac, pmean, stats


def moe_load_balance_backward(logits: torch.Tensor, load_frac: torch.Tensor, scale: float,
                              dlogits: Optional[torch.Tensor] = None, accumulate: bool = True):
    """scale * d(load-balance loss)/d(logits), added into dlogits (or written if accumulate is
    False or dlogits is None)."""
    _need(logits, torch.float32, 2, "logits")
    _need(load_frac, torch.float32, 1, "load_frac")
    T, E = logits.shape
    if dlogits is None:
        dlogits = torch.empty(T, E, dtype=torch.float32, device=logits.device)
        accumulate = False
    _check("moe_load_balance_backward", load().moe_load_balance_backward(
        _ptr(logits), _ptr(load_frac), T, E, float(scale), 1 if accumulate else 0, _ptr(dlogits),
        _stream(logits.device)))
    return dlogits


def moe_build_permutation(topk_idx: torch.Tensor, E: int, ws: Optional[torch.Tensor] = None,
                          out=None):
    _need(topk_idx, torch.int32, 2, "topk_idx")
    T, K = topk_idx.shape
    dev = topk_idx.device
    nbytes = workspace_size(MOE_OP_BUILD_PERMUTATION, T, E, K)
    if ws is None:
        ws = new_workspace(nbytes, dev)
    if out is None:
        counts = torch.empty(E, dtype=torch.int32, device=dev)
        offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
        perm = torch.empty(T * K, dtype=torch.int32, device=dev)
        inv = torch.empty(T * K, dtype=torch.int32, device=dev)
    else:
        counts, offsets, perm, inv = out
    _check("moe_build_permutation", load().moe_build_permutation(
        _ptr(topk_idx), T, E, K, _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(inv), _ptr(ws),
        ws.numel(), _stream(dev)))
    return counts, offsets, perm, inv


def moe_build_permutation_static(topk_idx: torch.Tensor, E: int, out=None):
    """moe_build_permutation without a workspace: the library's fixed device
    scratch holds the chunk histogram (for callers that cannot allocate)."""
    _need(topk_idx, torch.int32, 2, "topk_idx")
    T, K = topk_idx.shape
    dev = topk_idx.device
    if out is None:
        counts = torch.empty(E, dtype=torch.int32, device=dev)
        offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
        perm = torch.empty(T * K, dtype=torch.int32, device=dev)
        inv = torch.empty(T * K, dtype=torch.int32, device=dev)
    else:
        counts, offsets, perm, inv = out
    _check("moe_build_permutation_static", load().moe_build_permutation_static(
        _ptr(topk_idx), T, E, K, _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(inv), _stream(dev)))
    return counts, offsets, perm, inv


def moe_ep_layout(topk_idx: torch.Tensor, E: int, R: int, host_splits: Optional[torch.Tensor] = None,
                  ws: Optional[torch.Tensor] = None, out=None):
    """Returns (ep_splits [R*E+R*R], send_index, a2a_index, regroup_index, host_splits).
    ``host_splits`` (pinned CPU int32 [R*E+R*R]) receives the one device-to-host copy;
    pass ``False`` to skip the copy."""
    _need(topk_idx, torch.int32, 2, "topk_idx")
    T, K = topk_idx.shape
    dev = topk_idx.device
    n = R * E + R * R
    if host_splits is None:
        host_splits = torch.empty(n, dtype=torch.int32, pin_memory=True)
    elif host_splits is False:
        host_splits = None
    if host_splits is not None:
        if host_splits.is_cuda or host_splits.dtype != torch.int32 or host_splits.numel() < n:
            raise ValueError("host_splits must be a pinned CPU int32 tensor of R*E+R*R elements")
    nbytes = workspace_size(MOE_OP_EP_LAYOUT, T, E, K, R)
    if nbytes == 0:
        raise ValueError("R must divide E and T")
    if ws is None:
        ws = new_workspace(nbytes, dev)
    if out is None:
        splits = torch.empty(n, dtype=torch.int32, device=dev)
        send = torch.empty(T * K, dtype=torch.int32, device=dev)
        a2a = torch.empty(T * K, dtype=torch.int32, device=dev)
        reg = torch.empty(T * K, dtype=torch.int32, device=dev)
    else:
        splits, send, a2a, reg = out
    _check("moe_ep_layout", load().moe_ep_layout(
        _ptr(topk_idx), T, E, K, R, _ptr(splits), _ptr(send), _ptr(a2a), _ptr(reg),
        _ptr(host_splits), _ptr(ws), ws.numel(), _stream(dev)))
    return splits, send, a2a, reg, host_splits


def moe_build_permutation_ep(topk_idx: torch.Tensor, E: int, R: int,
                             host_splits: Optional[torch.Tensor] = None,
                             ws: Optional[torch.Tensor] = None, out=None):
    """Both moe_build_permutation and moe_ep_layout from one pass. Returns
    (counts, offsets, perm, inv_perm, ep_splits, send_index, a2a_index, regroup_index,
    host_splits); ``host_splits=False`` skips the device-to-host copy."""
    _need(topk_idx, torch.int32, 2, "topk_idx")
    T, K = topk_idx.shape
    dev = topk_idx.device
    n = R * E + R * R
    if host_splits is None:
        host_splits = torch.empty(n, dtype=torch.int32, pin_memory=True)
    elif host_splits is False:
        host_splits = None
    nbytes = workspace_size(MOE_OP_EP_LAYOUT, T, E, K, R)
    if nbytes == 0:
        raise ValueError("R must divide E and T")
    if ws is None:
        ws = new_workspace(nbytes, dev)
    if out is None:
        e = lambda *s: torch.empty(*s, dtype=torch.int32, device=dev)  # noqa: E731
        out = (e(E), e(E + 1), e(T * K), e(T * K), e(n), e(T * K), e(T * K), e(T * K))
    counts, offsets, perm, inv, splits, send, a2a, reg = out
    _check("moe_build_permutation_ep", load().moe_build_permutation_ep(
        _ptr(topk_idx), T, E, K, R, _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(inv),
        _ptr(splits), _ptr(send), _ptr(a2a), _ptr(reg), _ptr(host_splits), _ptr(ws), ws.numel(),
        _stream(dev)))
    return counts, offsets, perm, inv, splits, send, a2a, reg, host_splits


def moe_route_permute_ep(logits: torch.Tensor, K: int, R: int, renorm: int = 1,
                         host_splits: Optional[torch.Tensor] = None,
                         ws: Optional[torch.Tensor] = None, out=None):
    """moe_route_topk and moe_build_permutation_ep in one launch. Returns
    (topk_idx, topk_w, counts, offsets, perm, inv_perm, ep_splits, send_index,
    a2a_index, regroup_index, host_splits); ``host_splits=False`` skips the
    device-to-host copy."""
    _need(logits, torch.float32, 2, "logits")
    T, E = logits.shape
    dev = logits.device
    n = R * E + R * R
    if host_splits is None:
        host_splits = torch.empty(n, dtype=torch.int32, pin_memory=True)
    elif host_splits is False:
        host_splits = None
    nbytes = workspace_size(MOE_OP_ROUTE_PERMUTE_EP, T, E, K, R)
    if nbytes == 0:
        raise ValueError("R must divide E and T")
    if ws is None:
        ws = new_workspace(nbytes, dev)
    if out is None:
        e = lambda *s: torch.empty(*s, dtype=torch.int32, device=dev)  # noqa: E731
        out = (e(T, K), torch.empty(T, K, dtype=torch.float32, device=dev), e(E), e(E + 1),
               e(T * K), e(T * K), e(n), e(T * K), e(T * K), e(T * K))
    idx, w, counts, offsets, perm, inv, splits, send, a2a, reg = out
    _check("moe_route_permute_ep", load().moe_route_permute_ep(
        _ptr(logits), T, E, K, int(renorm), R, _ptr(idx), _ptr(w), _ptr(counts), _ptr(offsets),
        _ptr(perm), _ptr(inv), _ptr(splits), _ptr(send), _ptr(a2a), _ptr(reg), _ptr(host_splits),
        _ptr(ws), ws.numel(), _stream(dev)))
    return idx, w, counts, offsets, perm, inv, splits, send, a2a, reg, host_splits


def moe_dispatch(x: torch.Tensor, perm: torch.Tensor, K: int, out: Optional[torch.Tensor] = None):
    _need(x, torch.bfloat16, 2, "x")
    _need(perm, torch.int32, 1, "perm")
    T, d = x.shape
    xp = out if out is not None else torch.empty(T * K, d, dtype=torch.bfloat16, device=x.device)
    _check("moe_dispatch", load().moe_dispatch(_ptr(x), T, d, K, _ptr(perm), _ptr(xp),
                                               _stream(x.device)))
    return xp


def moe_dispatch_scatter(x: torch.Tensor, inv_perm: torch.Tensor, K: int,
                         out: Optional[torch.Tensor] = None):
    """The same xp as moe_dispatch, token-major through inv_perm."""
    _need(x, torch.bfloat16, 2, "x")
    _need(inv_perm, torch.int32, 1, "inv_perm")
    T, d = x.shape
    xp = out if out is not None else torch.empty(T * K, d, dtype=torch.bfloat16, device=x.device)
    _check("moe_dispatch_scatter", load().moe_dispatch_scatter(_ptr(x), T, d, K, _ptr(inv_perm),
                                                               _ptr(xp), _stream(x.device)))
    return xp


def moe_grouped_ffn(xp: torch.Tensor, offsets: torch.Tensor, w_gate: torch.Tensor,
                    w_up: torch.Tensor, w_down: torch.Tensor, save_gu: bool = True,
                    ws: Optional[torch.Tensor] = None, out=None):
    """Returns (y [M,d], h [M,I], gu [M,2I] or None)."""
    _need(xp, torch.bfloat16, 2, "xp")
    _need(offsets, torch.int32, 1, "offsets")
    for n, t in (("w_gate", w_gate), ("w_up", w_up), ("w_down", w_down)):
        _need(t, torch.bfloat16, 3, n)
    M, d = xp.shape
    E, _, I = w_gate.shape
    dev = xp.device
    if ws is None:
        ws = new_workspace(workspace_size(MOE_OP_GROUPED_FFN, M, E, 1, 1, d, I), dev)
    if out is None:
        y = torch.empty(M, d, dtype=torch.bfloat16, device=dev)
        h = torch.empty(M, I, dtype=torch.bfloat16, device=dev)
        gu = torch.empty(M, 2 * I, dtype=torch.bfloat16, device=dev) if save_gu else None
    else:
        y, h, gu = out
    _check("moe_grouped_ffn", load().moe_grouped_ffn(
        _ptr(xp), _ptr(offsets), E, M, d, I, _ptr(w_gate), _ptr(w_up), _ptr(w_down), _ptr(y),
        _ptr(h), _ptr(gu), _ptr(ws), ws.numel(), _stream(dev)))
    return y, h, gu


def moe_grouped_ffn_backward(dy, xp, gu, h, offsets, w_gate, w_up, w_down,
                             ws: Optional[torch.Tensor] = None, out=None):
    """Returns (dxp [M,d] bf16, dw_gate, dw_up [E,d,I] fp32, dw_down [E,I,d] fp32)."""
    for n, t in (("dy", dy), ("xp", xp), ("gu", gu), ("h", h)):
        _need(t, torch.bfloat16, 2, n)
    _need(offsets, torch.int32, 1, "offsets")
    M, d = xp.shape
    E, _, I = w_gate.shape
    dev = xp.device
    if ws is None:
        ws = new_workspace(workspace_size(MOE_OP_GROUPED_FFN_BACKWARD, M, E, 1, 1, d, I), dev)
    if out is None:
        dxp = torch.empty(M, d, dtype=torch.bfloat16, device=dev)
        dwg = torch.empty(E, d, I, dtype=torch.float32, device=dev)
        dwu = torch.empty(E, d, I, dtype=torch.float32, device=dev)
        dwd = torch.empty(E, I, d, dtype=torch.float32, device=dev)
    else:
        dxp, dwg, dwu, dwd = out
    _check("moe_grouped_ffn_backward", load().moe_grouped_ffn_backward(
        _ptr(dy), _ptr(xp), _ptr(gu), _ptr(h), _ptr(offsets), E, M, d, I, _ptr(w_gate), _ptr(w_up),
        _ptr(w_down), _ptr(dxp), _ptr(dwg), _ptr(dwu), _ptr(dwd), _ptr(ws), ws.numel(),
        _stream(dev)))
    return dxp, dwg, dwu, dwd


def moe_grouped_ffn_backward_data(dy, xp, gu, h, offsets, w_gate, w_up, w_down,
                                  ws: torch.Tensor, out: Optional[torch.Tensor] = None):
    """The data part of moe_grouped_ffn_backward: returns dxp [M,d] bf16 and leaves
    [dG | dU] and the padded straddling steps in ws for the weight part."""
    for n, t in (("dy", dy), ("xp", xp), ("gu", gu), ("h", h)):
        _need(t, torch.bfloat16, 2, n)
    _need(offsets, torch.int32, 1, "offsets")
    M, d = xp.shape
    E, _, I = w_gate.shape
    dxp = out if out is not None else torch.empty(M, d, dtype=torch.bfloat16, device=xp.device)
    _check("moe_grouped_ffn_backward_data", load().moe_grouped_ffn_backward_data(
        _ptr(dy), _ptr(xp), _ptr(gu), _ptr(h), _ptr(offsets), E, M, d, I, _ptr(w_gate), _ptr(w_up),
        _ptr(w_down), _ptr(dxp), _ptr(ws), ws.numel(), _stream(xp.device)))
    return dxp


def moe_grouped_ffn_backward_weights(dy, xp, h, offsets, E: int, I: int, ws: torch.Tensor,
                                     out=None):
    """The weight part of moe_grouped_ffn_backward, after the data part on the same
    stream with the same ws: returns (dw_gate, dw_up [E,d,I], dw_down [E,I,d]) fp32."""
    for n, t in (("dy", dy), ("xp", xp), ("h", h)):
        _need(t, torch.bfloat16, 2, n)
    _need(offsets, torch.int32, 1, "offsets")
    M, d = xp.shape
    dev = xp.device
    if out is None:
        out = (torch.empty(E, d, I, dtype=torch.float32, device=dev),
               torch.empty(E, d, I, dtype=torch.float32, device=dev),
               torch.empty(E, I, d, dtype=torch.float32, device=dev))
    dwg, dwu, dwd = out
    _check("moe_grouped_ffn_backward_weights", load().moe_grouped_ffn_backward_weights(
        _ptr(dy), _ptr(xp), _ptr(h), _ptr(offsets), E, M, d, I, _ptr(dwg), _ptr(dwu), _ptr(dwd),
        _ptr(ws), ws.numel(), _stream(dev)))
    return dwg, dwu, dwd


def moe_combine(y: torch.Tensor, topk_w: torch.Tensor, inv_perm: torch.Tensor,
                shared_y: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None):
    _need(y, torch.bfloat16, 2, "y")
    _need(topk_w, torch.float32, 2, "topk_w")
    _need(inv_perm, torch.int32, 1, "inv_perm")
    T, K = topk_w.shape
    d = y.shape[1]
    o = out if out is not None else torch.empty(T, d, dtype=torch.bfloat16, device=y.device)
    _check("moe_combine", load().moe_combine(_ptr(y), _ptr(topk_w), _ptr(inv_perm), T, K, d,
                                             _ptr(shared_y), _ptr(o), _stream(y.device)))
    return o


def moe_combine_backward(dout: torch.Tensor, y: torch.Tensor, topk_w: torch.Tensor,
                         inv_perm: torch.Tensor, out=None):
    _need(dout, torch.bfloat16, 2, "dout")
    _need(y, torch.bfloat16, 2, "y")
    _need(topk_w, torch.float32, 2, "topk_w")
    _need(inv_perm, torch.int32, 1, "inv_perm")
    T, K = topk_w.shape
    d = dout.shape[1]
    if out is None:
        dy = torch.empty(T * K, d, dtype=torch.bfloat16, device=y.device)
        dw = torch.empty(T, K, dtype=torch.float32, device=y.device)
    else:
        dy, dw = out
    _check("moe_combine_backward", load().moe_combine_backward(
        _ptr(dout), _ptr(y), _ptr(topk_w), _ptr(inv_perm), T, K, d, _ptr(dy), _ptr(dw),
        _stream(y.device)))
    return dy, dw


def moe_dispatch_backward(dxp: torch.Tensor, inv_perm: torch.Tensor, T: int, K: int,
                          dx_shared: Optional[torch.Tensor] = None,
                          out: Optional[torch.Tensor] = None):
    _need(dxp, torch.bfloat16, 2, "dxp")
    _need(inv_perm, torch.int32, 1, "inv_perm")
    d = dxp.shape[1]
    dx = out if out is not None else torch.empty(T, d, dtype=torch.bfloat16, device=dxp.device)
    _check("moe_dispatch_backward", load().moe_dispatch_backward(
        _ptr(dxp), _ptr(inv_perm), T, K, d, _ptr(dx_shared), _ptr(dx), _stream(dxp.device)))
    return dx


# ---------------------------------------------------------------- expert parallelism over ranks
def moe_ep_recv_layout(counts_local: torch.Tensor, recv_counts: torch.Tensor, R: int,
                       capacity: int, host_splits: Optional[torch.Tensor] = None,
                       ws: Optional[torch.Tensor] = None, out=None):
    """Receive-side layout of the all-to-all dispatch from this rank's counts
    [E] and the exchanged counts [R*El]. Returns (splits [2R] = send then
    receive rows per peer, local_offsets [El+1], regroup_index [capacity],
    host_splits); ``host_splits`` (pinned CPU int32 [2R]) receives the one
    device-to-host copy (``False`` skips it)."""
    _need(counts_local, torch.int32, 1, "counts_local")
    _need(recv_counts, torch.int32, 1, "recv_counts")
    E = counts_local.numel()
    dev = counts_local.device
    if E % R or recv_counts.numel() != E:
        raise ValueError("R must divide E and recv_counts must hold R * (E / R) counts")
    El = E // R
    if host_splits is None:
        host_splits = torch.empty(2 * R, dtype=torch.int32, pin_memory=True)
    elif host_splits is False:
        host_splits = None
    if ws is None:
        ws = new_workspace(workspace_size(MOE_OP_EP_RECV_LAYOUT, 1, E, 1, R), dev)
    if out is None:
        out = (torch.empty(2 * R, dtype=torch.int32, device=dev),
               torch.empty(El + 1, dtype=torch.int32, device=dev),
               torch.empty(max(int(capacity), 1), dtype=torch.int32, device=dev))
    splits, loff, reg = out
    _check("moe_ep_recv_layout", load().moe_ep_recv_layout(
        _ptr(counts_local), _ptr(recv_counts), E, R, int(capacity), _ptr(splits), _ptr(loff),
        _ptr(reg), _ptr(host_splits), _ptr(ws), ws.numel(), _stream(dev)))
    return splits, loff, reg, host_splits


def moe_dispatch_slice(x: torch.Tensor, inv_perm: torch.Tensor, offsets: torch.Tensor, K: int,
                       e_lo: int, e_hi: int, out: Tuple[torch.Tensor, torch.Tensor]):
    """Local rows of the dispatch for experts [e_lo, e_hi): out = (xs [rows, d] bf16,
    local_offsets [e_hi - e_lo + 1] int32); returns out."""
    _need(x, torch.bfloat16, 2, "x")
    _need(inv_perm, torch.int32, 1, "inv_perm")
    _need(offsets, torch.int32, 1, "offsets")
    T, d = x.shape
    xs, loff = out
    _need(xs, torch.bfloat16, 2, "xs")
    _need(loff, torch.int32, 1, "local_offsets")
    _check("moe_dispatch_slice", load().moe_dispatch_slice(
        _ptr(x), T, d, K, _ptr(inv_perm), _ptr(offsets), offsets.numel() - 1, int(e_lo), int(e_hi),
        _ptr(xs), _ptr(loff), _stream(x.device)))
    return xs, loff


def moe_combine_slice(y_local: torch.Tensor, topk_w: torch.Tensor, inv_perm: torch.Tensor,
                      offsets: torch.Tensor, e_lo: int, e_hi: int,
                      out: Optional[torch.Tensor] = None):
    """fp32 partial combine [T, d] of the local experts' rows."""
    _need(y_local, torch.bfloat16, 2, "y_local")
    _need(topk_w, torch.float32, 2, "topk_w")
    _need(inv_perm, torch.int32, 1, "inv_perm")
    _need(offsets, torch.int32, 1, "offsets")
    T, K = topk_w.shape
    d = y_local.shape[1]
    o = out if out is not None else torch.empty(T, d, dtype=torch.float32, device=y_local.device)
    _check("moe_combine_slice", load().moe_combine_slice(
        _ptr(y_local), _ptr(topk_w), _ptr(inv_perm), _ptr(offsets), offsets.numel() - 1,
        int(e_lo), int(e_hi), T, K, d, _ptr(o), _stream(y_local.device)))
    return o


def moe_combine_backward_slice(dout: torch.Tensor, y_local: torch.Tensor, topk_w: torch.Tensor,
                               inv_perm: torch.Tensor, offsets: torch.Tensor, e_lo: int,
                               e_hi: int, out: Tuple[torch.Tensor, torch.Tensor]):
    """(dy_local [rows, d] bf16, dtopk_w [T, K] fp32, zero on other ranks' slots)."""
    _need(dout, torch.bfloat16, 2, "dout")
    _need(y_local, torch.bfloat16, 2, "y_local")
    _need(topk_w, torch.float32, 2, "topk_w")
    _need(inv_perm, torch.int32, 1, "inv_perm")
    _need(offsets, torch.int32, 1, "offsets")
    T, K = topk_w.shape
    d = dout.shape[1]
    dy, dw = out
    _check("moe_combine_backward_slice", load().moe_combine_backward_slice(
        _ptr(dout), _ptr(y_local), _ptr(topk_w), _ptr(inv_perm), _ptr(offsets),
        offsets.numel() - 1, int(e_lo), int(e_hi), T, K, d, _ptr(dy), _ptr(dw),
        _stream(dout.device)))
    return dy, dw


def moe_dispatch_backward_slice(dxs: torch.Tensor, inv_perm: torch.Tensor, offsets: torch.Tensor,
                                T: int, K: int, e_lo: int, e_hi: int,
                                out: Optional[torch.Tensor] = None):
    """fp32 partial input gradient [T, d] from the local experts' rows."""
    _need(dxs, torch.bfloat16, 2, "dxs")
    _need(inv_perm, torch.int32, 1, "inv_perm")
    _need(offsets, torch.int32, 1, "offsets")
    d = dxs.shape[1]
    o = out if out is not None else torch.empty(T, d, dtype=torch.float32, device=dxs.device)
    _check("moe_dispatch_backward_slice", load().moe_dispatch_backward_slice(
        _ptr(dxs), _ptr(inv_perm), _ptr(offsets), offsets.numel() - 1, int(e_lo), int(e_hi), T, K,
        d, _ptr(o), _stream(dxs.device)))
    return o


def moe_reduce_finish(partial: torch.Tensor, extra: Optional[torch.Tensor] = None,
                      out: Optional[torch.Tensor] = None):
    """bf16(partial + extra) for fp32 partial [T, d] and bf16 extra [T, d] (or None)."""
    _need(partial, torch.float32, 2, "partial")
    if extra is not None:
        _need(extra, torch.bfloat16, 2, "extra")
    T, d = partial.shape
    o = out if out is not None else torch.empty(T, d, dtype=torch.bfloat16, device=partial.device)
    _check("moe_reduce_finish", load().moe_reduce_finish(_ptr(partial), _ptr(extra), T, d, _ptr(o),
                                                         _stream(partial.device)))
    return o


# ---------------------------------------------------------------- MXFP8 grouped experts
def mxfp8_row_sf_bytes(M: int, E: int, K: int) -> int:
    """Bytes of the scale atoms of M expert-ordered rows of K elements."""
    return ((M + 127) // 128 + 2 * E) * (K // 128) * 512


def moe_mxfp8_quantize_rows(x: torch.Tensor, offsets: torch.Tensor, out=None):
    """(q [M, K] uint8 E4M3, sf uint8 scale atoms) of the expert-ordered rows x."""
    _need(x, torch.bfloat16, 2, "x")
    _need(offsets, torch.int32, 1, "offsets")
    M, K = x.shape
    E = offsets.numel() - 1
    if out is None:
        out = (torch.empty(M, K, dtype=torch.uint8, device=x.device),
               torch.empty(mxfp8_row_sf_bytes(M, E, K), dtype=torch.uint8, device=x.device))
    q, sf = out
    _check("moe_mxfp8_quantize_rows", load().moe_mxfp8_quantize_rows(
        _ptr(x), _ptr(offsets), E, M, K, _ptr(q), _ptr(sf), _stream(x.device)))
    return q, sf


def moe_mxfp8_quantize_weights(w_a: torch.Tensor, w_b: Optional[torch.Tensor] = None, out=None):
    """(q [E, Nq, K] uint8, sf) of weights [E, K, N] (gate/up interleaved when w_b is given)."""
    _need(w_a, torch.bfloat16, 3, "w_a")
    if w_b is not None:
        _need(w_b, torch.bfloat16, 3, "w_b")
        if w_b.shape != w_a.shape:
            raise ValueError("w_a and w_b must have the same shape")
    E, K, N = w_a.shape
    Nq = 2 * N if w_b is not None else N
    if out is None:
        out = (torch.empty(E, Nq, K, dtype=torch.uint8, device=w_a.device),
               torch.empty(E * (Nq // 128) * (K // 128) * 512, dtype=torch.uint8, device=w_a.device))
    q, sf = out
    _check("moe_mxfp8_quantize_weights", load().moe_mxfp8_quantize_weights(
        _ptr(w_a), _ptr(w_b), E, K, N, _ptr(q), _ptr(sf), _stream(w_a.device)))
    return q, sf


def moe_grouped_ffn_fp8(xp: torch.Tensor, offsets: torch.Tensor, wgu, wd, save_gu: bool = True,
                        ws: Optional[torch.Tensor] = None, out=None):
    """MXFP8 forward of the grouped SwiGLU experts. ``wgu`` = (q, sf) of
    moe_mxfp8_quantize_weights(w_gate, w_up), ``wd`` = (q, sf) of
    moe_mxfp8_quantize_weights(w_down). Returns (y [M,d], h [M,I], gu [M,2I] or None)."""
    _need(xp, torch.bfloat16, 2, "xp")
    _need(offsets, torch.int32, 1, "offsets")
    (gq, gsf), (dq, dsf) = wgu, wd
    for n, t in (("wgu_q", gq), ("wd_q", dq)):
        _need(t, torch.uint8, 3, n)
    M, d = xp.shape
    E, two_i, _ = gq.shape
    I = two_i // 2
    dev = xp.device
    if ws is None:
        ws = new_workspace(workspace_size(MOE_OP_GROUPED_FFN_FP8, M, E, 1, 1, d, I), dev)
    if out is None:
        out = (torch.empty(M, d, dtype=torch.bfloat16, device=dev),
               torch.empty(M, I, dtype=torch.bfloat16, device=dev),
               torch.empty(M, 2 * I, dtype=torch.bfloat16, device=dev) if save_gu else None)
    y, h, gu = out
    _check("moe_grouped_ffn_fp8", load().moe_grouped_ffn_fp8(
        _ptr(xp), _ptr(offsets), E, M, d, I, _ptr(gq), _ptr(gsf), _ptr(dq), _ptr(dsf), _ptr(y),
        _ptr(h), _ptr(gu), _ptr(ws), ws.numel(), _stream(dev)))
    return y, h, gu


def moe_profile_start(capacity: int = 4096):
    _check("moe_profile_start", load().moe_profile_start(int(capacity)))


def moe_profile_stop():
    """Stops recording; returns [(kernel name, milliseconds), ...] in launch order."""
    lib = load()
    n = lib.moe_profile_stop()
    out = []
    for i in range(n):
        name = ctypes.c_char_p()
        ms = ctypes.c_float()
        _check("moe_profile_record", lib.moe_profile_record(i, ctypes.byref(name), ctypes.byref(ms)))
        out.append((name.value.decode(), float(ms.value)))
    return out


def moe_debug_wait_timeout(ws: torch.Tensor, timeout_us: int):
    """Runs the GEMM kernels' bounded wait on a barrier nothing completes; the
    status word of ``ws`` then reads MOE_ERR_DEVICE_TIMEOUT."""
    _check("moe_debug_wait_timeout", load().moe_debug_wait_timeout(_ptr(ws), int(timeout_us),
                                                                    _stream(ws.device)))


def moe_debug_check_status() -> int:
    """The debug build's index-check record (synchronises; clears it). Raises
    MoEError(MOE_ERR_UNSUPPORTED) on a release build."""
    st = ctypes.c_int(0)
    _check("moe_debug_check_status", load().moe_debug_check_status(ctypes.byref(st)))
    return st.value


def moe_read_device_status(ws: torch.Tensor) -> int:
    st = ctypes.c_int(0)
    _check("moe_read_device_status", load().moe_read_device_status(
        _ptr(ws), _stream(ws.device), ctypes.byref(st)))
    return st.value
