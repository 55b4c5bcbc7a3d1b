"""Python binding of the GB300 attention-block library (C ABI in
``include/swa_attn.h``).

The functions named ``swa_*`` mirror the C entry points one to one and only
marshal arguments (tensor pointers, the CUDA stream, the parameter struct).
``attention_forward`` / ``attention_backward`` allocate outputs and the
workspace with PyTorch and call them. Every computation runs in the CUDA
library; if the shared library is missing, loading it raises.

Two libraries share the symbols: ``libswaattn.so`` (bf16 tensors, tcgen05
kernels) and ``libswaattn_fp32.so`` (fp32 tensors, SIMT debug kernels). The
binding picks the one matching the dtype of ``q``.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

__all__ = [
    "swa_params", "SwaError", "load",
    "swa_attn_workspace_size", "swa_attn_workspace_init", "swa_attn_fwd", "swa_attn_bwd",
    "swa_attn_fwd_ex", "swa_attn_bwd_ex",
    "swa_attn_fwd_noalloc",
    "swa_block_weights", "swa_block_workspace_size", "swa_block_fwd", "swa_block_bwd",
    "make_block_weights", "make_block_extras",
    "swa_attn_check_status", "swa_sssl_window", "swa_has_ve", "swa_strerror",
    "swa_build_info", "attention_forward", "attention_backward", "make_params",
    "SWA_OK", "SWA_ERR_INVALID_ARG", "SWA_ERR_UNSUPPORTED", "SWA_ERR_CUDA", "SWA_ERR_TIMEOUT",
    "SWA_ERR_WORKSPACE", "SWA_ERR_DEVICE_CHECK", "SWA_REUSE_PROLOGUE", "SWA_BWD_STAGE_PRE",
    "SWA_BWD_STAGE_MAIN", "SWA_BWD_STAGE_POST",
]

SWA_OK = 0
SWA_ERR_INVALID_ARG = 1
SWA_ERR_UNSUPPORTED = 2
SWA_ERR_CUDA = 3
SWA_ERR_TIMEOUT = 4
SWA_ERR_WORKSPACE = 5
SWA_ERR_DEVICE_CHECK = 6

SWA_REUSE_PROLOGUE = 1
SWA_BWD_STAGE_PRE = 2
SWA_BWD_STAGE_MAIN = 4
SWA_BWD_STAGE_POST = 8


class swa_params(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("T", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int),
        ("d", ctypes.c_int), ("window", ctypes.c_int), ("causal", ctypes.c_int),
        ("softmax_scale", ctypes.c_float), ("eps", ctypes.c_float),
        ("ve_scale", ctypes.c_float), ("vocab", ctypes.c_int),
    ]


class SwaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {swa_strerror(status)} (status {status})")
        self.status = status


class swa_extras(ctypes.Structure):
    """Extras of the _ex entry points: rotary tables, the learned
    value-embedding gate and the pipeline-wait limit (see include/swa_attn.h)."""
    _fields_ = [("rope_cos", ctypes.c_void_p), ("rope_sin", ctypes.c_void_p), ("rope_rows", ctypes.c_int),
                ("gate_x", ctypes.c_void_p), ("gate_x_stride", ctypes.c_longlong),
                ("gate_w", ctypes.c_void_p), ("gate_ch", ctypes.c_int),
                ("d_gate_w", ctypes.c_void_p), ("d_gate_x", ctypes.c_void_p),
                ("wait_limit_ns", ctypes.c_ulonglong)]


class swa_block_weights(ctypes.Structure):
    """Weights of the block calls: model width C and the four projection
    matrices in the torch.nn.Linear layout (see include/swa_attn.h)."""
    _fields_ = [("C", ctypes.c_int), ("wq", ctypes.c_void_p), ("wk", ctypes.c_void_p),
                ("wv", ctypes.c_void_p), ("wo", ctypes.c_void_p)]


_LIBS: dict = {}
_vp = ctypes.c_void_p


def load(kind: str = "bf16") -> ctypes.CDLL:
    """The ctypes handle of the bf16 or fp32 library (loaded once)."""
    if kind in _LIBS:
        return _LIBS[kind]
    path = _build.lib_path(kind)
    if not os.path.exists(path):
        raise RuntimeError(
            f"{os.path.basename(path)} is not built; run sliding_window_gqa_qk_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER(swa_params)
    lib.swa_attn_workspace_size.argtypes = [P, ctypes.c_int]
    lib.swa_attn_workspace_size.restype = ctypes.c_size_t
    lib.swa_attn_workspace_init.argtypes = [_vp, ctypes.c_size_t, _vp]
    lib.swa_attn_workspace_init.restype = ctypes.c_int
    lib.swa_attn_fwd.argtypes = [P] + [_vp] * 11 + [ctypes.c_size_t, ctypes.c_uint, _vp]
    lib.swa_attn_fwd.restype = ctypes.c_int
    lib.swa_attn_bwd.argtypes = [P] + [_vp] * 18 + [ctypes.c_size_t, ctypes.c_uint, _vp]
    lib.swa_attn_bwd.restype = ctypes.c_int
    R = ctypes.POINTER(swa_extras)
    lib.swa_attn_fwd_ex.argtypes = [P, R] + [_vp] * 11 + [ctypes.c_size_t, ctypes.c_uint, _vp]
    lib.swa_attn_fwd_ex.restype = ctypes.c_int
    lib.swa_attn_bwd_ex.argtypes = [P, R] + [_vp] * 18 + [ctypes.c_size_t, ctypes.c_uint, _vp]
    lib.swa_attn_bwd_ex.restype = ctypes.c_int
    lib.swa_attn_fwd_noalloc.argtypes = [P] + [_vp] * 10 + [_vp]
    lib.swa_attn_fwd_noalloc.restype = ctypes.c_int
    lib.swa_attn_step_host_size.argtypes = [P]
    lib.swa_attn_step_host_size.restype = ctypes.c_size_t
    lib.swa_attn_step_host.argtypes = [P, R] + [_vp] * 18 + [ctypes.c_size_t, _vp]
    lib.swa_attn_step_host.restype = ctypes.c_int
    W = ctypes.POINTER(swa_block_weights)
    lib.swa_block_workspace_size.argtypes = [P, ctypes.c_int, ctypes.c_int]
    lib.swa_block_workspace_size.restype = ctypes.c_size_t
    lib.swa_block_fwd.argtypes = [P, R, W] + [_vp] * 7 + [ctypes.c_size_t, _vp]
    lib.swa_block_fwd.restype = ctypes.c_int
    lib.swa_block_bwd.argtypes = [P, R, W] + [_vp] * 15 + [ctypes.c_size_t, _vp]
    lib.swa_block_bwd.restype = ctypes.c_int
    lib.swa_attn_check_status.argtypes = [_vp, _vp]
    lib.swa_attn_check_status.restype = ctypes.c_int
    lib.swa_sssl_window.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_char_p, ctypes.c_int]
    lib.swa_sssl_window.restype = ctypes.c_int
    lib.swa_has_ve.argtypes = [ctypes.c_int, ctypes.c_int]
    lib.swa_has_ve.restype = ctypes.c_int
    lib.swa_strerror.argtypes = [ctypes.c_int]
    lib.swa_strerror.restype = ctypes.c_char_p
    lib.swa_build_info.argtypes = []
    lib.swa_build_info.restype = ctypes.c_char_p
    _LIBS[kind] = lib
    return lib


def _kind_of(t: Optional[torch.Tensor]) -> str:
    if t is not None and t.dtype == torch.float32:
        return "fp32"
    return "bf16"


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_params(B, T, Hq, Hkv, d, window=-1, causal=True, softmax_scale=0.0, eps=1e-6,
                ve_scale=0.5, vocab=0) -> swa_params:
    return swa_params(int(B), int(T), int(Hq), int(Hkv), int(d), int(window), int(bool(causal)),
                      float(softmax_scale), float(eps), float(ve_scale), int(vocab))


# ---------------------------------------------------------------------------
# One-to-one wrappers of the C entry points
# ---------------------------------------------------------------------------

def swa_attn_workspace_size(p: swa_params, for_backward: int, kind: str = "bf16") -> int:
    return int(load(kind).swa_attn_workspace_size(ctypes.byref(p), int(for_backward)))


def swa_attn_workspace_init(ws, ws_bytes=None, stream=None, kind: str = "bf16") -> int:
    n = ws.numel() if ws_bytes is None else ws_bytes
    return int(load(kind).swa_attn_workspace_init(_ptr(ws), n, _stream(stream)))


def swa_attn_fwd(p, q, k, v, gq, gk, ve, tok, ve_gate, o, lse, ws, ws_bytes=None, flags=0,
                 stream=None, kind=None) -> int:
    kind = kind or _kind_of(q)
    n = ws.numel() if ws_bytes is None else ws_bytes
    return int(load(kind).swa_attn_fwd(
        ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(gq), _ptr(gk), _ptr(ve), _ptr(tok),
        _ptr(ve_gate), _ptr(o), _ptr(lse), _ptr(ws), n, int(flags), _stream(stream)))


def swa_attn_bwd(p, q, k, v, gq, gk, ve, tok, ve_gate, o, lse, dO, dq, dk, dv, dgq, dgk, dve,
                 ws, ws_bytes=None, flags=0, stream=None, kind=None) -> int:
    kind = kind or _kind_of(q)
    n = ws.numel() if ws_bytes is None else ws_bytes
    return int(load(kind).swa_attn_bwd(
        ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(gq), _ptr(gk), _ptr(ve), _ptr(tok),
        _ptr(ve_gate), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dgq),
        _ptr(dgk), _ptr(dve), _ptr(ws), n, int(flags), _stream(stream)))


def make_extras(rope=None, gate_x=None, gate_w=None, d_gate_w=None, d_gate_x=None,
                wait_limit_ns: int = 0) -> swa_extras:
    """swa_extras from device tensors: rope = (cos, sin) fp32 [rows, d/2] or
    None; gate_x [B, T, >= C] rows (its row stride is taken from the tensor),
    gate_w fp32 [Hkv, C] or None; backward outputs d_gate_w [Hkv, C],
    d_gate_x [B, T, C] (fp32) or None; wait_limit_ns the time limit of one
    pipeline wait of the kernels (0: the library's default)."""
    e = swa_extras()
    e.wait_limit_ns = int(wait_limit_ns)
    if rope is not None:
        e.rope_cos, e.rope_sin, e.rope_rows = _ptr(rope[0]), _ptr(rope[1]), int(rope[0].shape[0])
    if gate_w is not None:
        if gate_x.stride(-1) != 1 or gate_x.dim() != 3 or gate_x.stride(0) != gate_x.shape[1] * gate_x.stride(1):
            raise ValueError("gate_x must be [B, T, *] with unit channel stride and packed rows")
        e.gate_x = gate_x.data_ptr()
        e.gate_x_stride = int(gate_x.stride(1))
        e.gate_w = _ptr(gate_w)
        e.gate_ch = int(gate_w.shape[1])
        e.d_gate_w = _ptr(d_gate_w)
        e.d_gate_x = _ptr(d_gate_x)
    return e


def swa_attn_fwd_ex(p, ex, q, k, v, gq, gk, ve, tok, ve_gate, o, lse, ws, ws_bytes=None,
                    flags=0, stream=None, kind=None) -> int:
    kind = kind or _kind_of(q)
    n = ws.numel() if ws_bytes is None else ws_bytes
    ep = None if ex is None else ctypes.byref(ex)
    return int(load(kind).swa_attn_fwd_ex(
        ctypes.byref(p), ep, _ptr(q), _ptr(k), _ptr(v), _ptr(gq), _ptr(gk), _ptr(ve), _ptr(tok),
        _ptr(ve_gate), _ptr(o), _ptr(lse), _ptr(ws), n, int(flags), _stream(stream)))


def swa_attn_bwd_ex(p, ex, q, k, v, gq, gk, ve, tok, ve_gate, o, lse, dO, dq, dk, dv, dgq, dgk,
                    dve, ws, ws_bytes=None, flags=0, stream=None, kind=None) -> int:
    kind = kind or _kind_of(q)
    n = ws.numel() if ws_bytes is None else ws_bytes
    ep = None if ex is None else ctypes.byref(ex)
    return int(load(kind).swa_attn_bwd_ex(
        ctypes.byref(p), ep, _ptr(q), _ptr(k), _ptr(v), _ptr(gq), _ptr(gk), _ptr(ve), _ptr(tok),
        _ptr(ve_gate), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dgq),
        _ptr(dgk), _ptr(dve), _ptr(ws), n, int(flags), _stream(stream)))


def swa_attn_step_host_size(p: swa_params, kind: str = "bf16") -> int:
    return int(load(kind).swa_attn_step_host_size(ctypes.byref(p)))


def swa_attn_step_host(p, ex, q, k, v, gq, gk, ve, tok, ve_gate, dO, o, lse, dq, dk, dv, dgq, dgk,
                       dve, buf, buf_bytes=None, stream=None, kind=None) -> int:
    """One forward + backward with host tensors (inputs and outputs on the
    CPU, ideally pinned) and a device buffer of swa_attn_step_host_size
    bytes; enqueued on `stream`, returns without waiting."""
    kind = kind or _kind_of(q)
    n = buf.numel() if buf_bytes is None else buf_bytes
    ep = None if ex is None else ctypes.byref(ex)
    return int(load(kind).swa_attn_step_host(
        ctypes.byref(p), ep, _ptr(q), _ptr(k), _ptr(v), _ptr(gq), _ptr(gk), _ptr(ve), _ptr(tok),
        _ptr(ve_gate), _ptr(dO), _ptr(o), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dgq),
        _ptr(dgk), _ptr(dve), _ptr(buf), n, _stream(stream)))


def new_step_host_buffer(p: swa_params, device, kind: str, stream=None):
    """A device buffer for swa_attn_step_host, initialised."""
    n = swa_attn_step_host_size(p, kind)
    if n == 0:
        raise SwaError(SWA_ERR_INVALID_ARG, "step buffer size")
    buf = torch.empty(n, dtype=torch.uint8, device=device)
    _check(swa_attn_workspace_init(buf, n, stream, kind), "step buffer init")
    return buf


def swa_attn_fwd_noalloc(p, q, k, v, gq, gk, ve, tok, ve_gate, o, lse, stream=None,
                         kind=None) -> int:
    """Forward whose scratch is the library's fixed device array (no
    workspace argument, nothing allocated); see include/swa_attn.h."""
    kind = kind or _kind_of(q)
    return int(load(kind).swa_attn_fwd_noalloc(
        ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(gq), _ptr(gk), _ptr(ve), _ptr(tok),
        _ptr(ve_gate), _ptr(o), _ptr(lse), _stream(stream)))


def make_block_weights(wq, wk, wv, wo) -> swa_block_weights:
    """swa_block_weights from device tensors wq [Hq*d, C], wk, wv [Hkv*d, C],
    wo [C, Hq*d] (the model width C is taken from wq)."""
    return swa_block_weights(int(wq.shape[1]), _ptr(wq), _ptr(wk), _ptr(wv), _ptr(wo))


def make_block_extras(rope=None, gate_w=None, d_gate_w=None) -> swa_extras:
    """swa_extras of the block calls: rope = (cos, sin) fp32 [rows, d/2] or
    None; gate_w fp32 [Hkv, C] (the block feeds the gate its normed input);
    d_gate_w fp32 [Hkv, C] backward output or None."""
    e = make_extras(rope)
    if gate_w is not None:
        e.gate_w = _ptr(gate_w)
        e.gate_ch = int(gate_w.shape[1])
        e.d_gate_w = _ptr(d_gate_w)
    return e


def swa_block_workspace_size(p: swa_params, C: int, for_backward: int, kind: str = "bf16") -> int:
    return int(load(kind).swa_block_workspace_size(ctypes.byref(p), int(C), int(for_backward)))


def swa_block_fwd(p, ex, w, x, gq, gk, ve, tok, out, ws, ws_bytes=None, stream=None, kind=None) -> int:
    kind = kind or _kind_of(x)
    n = ws.numel() if ws_bytes is None else ws_bytes
    ep = None if ex is None else ctypes.byref(ex)
    return int(load(kind).swa_block_fwd(
        ctypes.byref(p), ep, ctypes.byref(w), _ptr(x), _ptr(gq), _ptr(gk), _ptr(ve), _ptr(tok),
        _ptr(out), _ptr(ws), n, _stream(stream)))


def swa_block_bwd(p, ex, w, x, gq, gk, ve, tok, dout, dx, dwq, dwk, dwv, dwo, dgq, dgk, dve, ws,
                  ws_bytes=None, stream=None, kind=None) -> int:
    kind = kind or _kind_of(x)
    n = ws.numel() if ws_bytes is None else ws_bytes
    ep = None if ex is None else ctypes.byref(ex)
    return int(load(kind).swa_block_bwd(
        ctypes.byref(p), ep, ctypes.byref(w), _ptr(x), _ptr(gq), _ptr(gk), _ptr(ve), _ptr(tok),
        _ptr(dout), _ptr(dx), _ptr(dwq), _ptr(dwk), _ptr(dwv), _ptr(dwo), _ptr(dgq), _ptr(dgk),
        _ptr(dve), _ptr(ws), n, _stream(stream)))


def swa_attn_check_status(ws, stream=None, kind: str = "bf16") -> int:
    return int(load(kind).swa_attn_check_status(_ptr(ws), _stream(stream)))


def swa_sssl_window(layer: int, n_layer: int, pattern: str, T: int, kind: str = "bf16") -> int:
    return int(load(kind).swa_sssl_window(layer, n_layer, pattern.encode(), T))


def swa_has_ve(layer: int, n_layer: int, kind: str = "bf16") -> int:
    return int(load(kind).swa_has_ve(layer, n_layer))


def swa_strerror(status: int, kind: str = "bf16") -> str:
    try:
        return load(kind).swa_strerror(int(status)).decode()
    except RuntimeError:
        return f"status {status}"


def swa_build_info(kind: str = "bf16") -> str:
    return load(kind).swa_build_info().decode()


# ---------------------------------------------------------------------------
# Convenience calls: allocate outputs / workspace, raise on error
# ---------------------------------------------------------------------------

def _check(status: int, what: str):
    if status != SWA_OK:
        raise SwaError(status, what)


def new_workspace(p: swa_params, for_backward: bool, device, kind: str, stream=None):
    n = swa_attn_workspace_size(p, int(for_backward), kind)
    if n == 0:
        raise SwaError(SWA_ERR_INVALID_ARG, "workspace size")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    _check(swa_attn_workspace_init(ws, n, stream, kind), "workspace init")
    return ws


def attention_forward(q, k, v, gq=None, gk=None, *, window: int = -1, causal: bool = True,
                      softmax_scale: float = 0.0, eps: float = 1e-6, ve=None, tok=None,
                      ve_gate=None, ve_scale: float = 0.5, workspace=None, stream=None,
                      rope=None, gate_x=None, gate_w=None):
    """o, lse, workspace = attention_forward(q, k, v, ...). The workspace is
    allocated for the backward too, so it can be passed on to
    ``attention_backward`` with the prologue outputs kept. ``rope``: None or
    (cos, sin) fp32 device tensors [rows >= T, d/2] (rotary before the norm).
    ``gate_x`` [B, T, >= C] and ``gate_w`` fp32 [Hkv, C]: the learned
    value-embedding gate 2 sigmoid(gate_w x[:C]) (then ve_gate must be None)."""
    B, T, Hq, d = q.shape
    Hkv = k.shape[2]
    kind = _kind_of(q)
    vocab = ve.shape[0] if ve is not None else 0
    p = make_params(B, T, Hq, Hkv, d, window, causal, softmax_scale, eps, ve_scale, vocab)
    ws = workspace if workspace is not None else new_workspace(p, True, q.device, kind, stream)
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, T, dtype=torch.float32, device=q.device)
    if rope is None and gate_w is None:
        _check(swa_attn_fwd(p, q, k, v, gq, gk, ve, tok, ve_gate, o, lse, ws, stream=stream),
               "swa_attn_fwd")
    else:
        ex = make_extras(rope, gate_x, gate_w)
        _check(swa_attn_fwd_ex(p, ex, q, k, v, gq, gk, ve, tok, ve_gate, o, lse, ws, stream=stream),
               "swa_attn_fwd_ex")
    return o, lse, ws


def attention_backward(q, k, v, gq, gk, o, lse, dO, *, window: int = -1, causal: bool = True,
                       softmax_scale: float = 0.0, eps: float = 1e-6, ve=None, tok=None,
                       ve_gate=None, ve_scale: float = 0.5, workspace=None,
                       reuse_prologue: bool = False, stream=None, rope=None, gate_x=None,
                       gate_w=None) -> dict:
    """Gradients dq, dk, dv, dgq, dgk, dve (dve None without a VE table) and,
    with the learned gate, dgate_w [Hkv, C] and dgate_x [B, T, C]."""
    B, T, Hq, d = q.shape
    Hkv = k.shape[2]
    kind = _kind_of(q)
    vocab = ve.shape[0] if ve is not None else 0
    p = make_params(B, T, Hq, Hkv, d, window, causal, softmax_scale, eps, ve_scale, vocab)
    ws = workspace if workspace is not None else new_workspace(p, True, q.device, kind, stream)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dgq = torch.empty(d, dtype=torch.float32, device=q.device)
    dgk = torch.empty(d, dtype=torch.float32, device=q.device)
    dve = torch.empty(ve.shape, dtype=torch.float32, device=q.device) if ve is not None else None
    flags = SWA_REUSE_PROLOGUE if (reuse_prologue and workspace is not None) else 0
    out = {"dq": dq, "dk": dk, "dv": dv, "dgq": dgq, "dgk": dgk, "dve": dve, "workspace": ws}
    if rope is None and gate_w is None:
        _check(swa_attn_bwd(p, q, k, v, gq, gk, ve, tok, ve_gate, o, lse, dO, dq, dk, dv, dgq, dgk,
                            dve, ws, flags=flags, stream=stream), "swa_attn_bwd")
    else:
        dgw = dgx = None
        if gate_w is not None:
            dgw = torch.empty(gate_w.shape, dtype=torch.float32, device=q.device)
            dgx = torch.empty(B, T, gate_w.shape[1], dtype=torch.float32, device=q.device)
            out["dgate_w"], out["dgate_x"] = dgw, dgx
        ex = make_extras(rope, gate_x, gate_w, dgw, dgx)
        _check(swa_attn_bwd_ex(p, ex, q, k, v, gq, gk, ve, tok, ve_gate, o, lse, dO, dq, dk, dv, dgq,
                               dgk, dve, ws, flags=flags, stream=stream), "swa_attn_bwd_ex")
    return out
