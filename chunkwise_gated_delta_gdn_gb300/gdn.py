"""Thin ctypes binding of libgdn (``include/gdn.h``), same names as the C ABI.

This module only marshals arguments: it checks tensor shapes, dtypes and
devices, allocates outputs and the workspace through PyTorch when the caller
does not pass them, and hands raw device pointers and the current CUDA stream
to the library.  Every step of the computation runs in the library's CUDA
kernels; there is no fallback.  If ``libgdn.so`` has not been built the first
call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

from . import build as _build

GDN_OK = 0
GDN_ERR_INVALID_ARG = 1
GDN_ERR_UNSUPPORTED = 2
GDN_ERR_WORKSPACE = 3
GDN_ERR_CUDA = 4

GDN_GATE_SCALAR = 0
GDN_GATE_PER_KEY = 1
GDN_F32 = 0
GDN_BF16 = 1

GDN_ACT_NONE = 0
GDN_ACT_SILU = 1

GDN_FLAG_POSITIVE_GATE = 1 << 0
GDN_FLAG_NONFINITE = 1 << 1
GDN_FLAG_BAD_SEQLENS = 1 << 2
GDN_FLAG_TIMEOUT = 1 << 3
GDN_FLAG_LAUNCH_CONFIG = 1 << 4

# every symbol include/gdn.h declares
EXPORTED = ("gdn_version", "gdn_status_string", "gdn_chunk_fwd_workspace_bytes",
            "gdn_chunk_fwd", "gdn_chunk_fwd_prep", "gdn_chunk_fwd_scan",
            "gdn_chunk_fwd_lockstep",
            "gdn_chunk_fwd_noalloc", "gdn_recurrent_fwd", "gdn_causal_conv1d_fwd",
            "gdn_l2norm_fwd", "gdn_rmsnorm_gated_fwd", "gdn_state_combine",
            "gdn_selftest_wait", "gdn_read_device_flags")

_lock = threading.Lock()
_lib = None


class GdnError(RuntimeError):
    def __init__(self, status: int, what: str = "gdn_chunk_fwd"):
        self.status = status
        super().__init__(f"{what}: {gdn_status_string(status)} ({status})")


def lib_path() -> str:
    return _build.LIB


def load(path: Optional[str] = None):
    """Load libgdn.so (it must have been built; see ``build.py``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(
                f"libgdn.so not found at {path}: build it first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(path)
        vp, sz, i32, f32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_float
        lib.gdn_version.argtypes = []
        lib.gdn_version.restype = i32
        lib.gdn_status_string.argtypes = [i32]
        lib.gdn_status_string.restype = ctypes.c_char_p
        lib.gdn_chunk_fwd_workspace_bytes.argtypes = [i32] * 10
        lib.gdn_chunk_fwd_workspace_bytes.restype = sz
        for name in ("gdn_chunk_fwd", "gdn_chunk_fwd_prep", "gdn_chunk_fwd_scan",
                     "gdn_chunk_fwd_lockstep"):
            fn = getattr(lib, name)
            fn.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32,
                           i32, i32, i32, i32, i32, f32, i32, i32, vp, sz, vp]
            fn.restype = i32
        lib.gdn_chunk_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32,
                                              i32, i32, i32, i32, i32, i32, f32, i32, i32,
                                              vp]
        lib.gdn_chunk_fwd_noalloc.restype = i32
        lib.gdn_recurrent_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32,
                                          i32, i32, i32, i32, f32, i32, i32, vp, vp]
        lib.gdn_recurrent_fwd.restype = i32
        lib.gdn_causal_conv1d_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                              i32, i32, i32, vp, vp]
        lib.gdn_causal_conv1d_fwd.restype = i32
        i64 = ctypes.c_int64
        lib.gdn_l2norm_fwd.argtypes = [vp, vp, i64, i32, f32, i32, vp]
        lib.gdn_l2norm_fwd.restype = i32
        lib.gdn_rmsnorm_gated_fwd.argtypes = [vp, vp, vp, vp, i64, i32, f32, i32, vp]
        lib.gdn_rmsnorm_gated_fwd.restype = i32
        lib.gdn_state_combine.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, vp]
        lib.gdn_state_combine.restype = i32
        lib.gdn_selftest_wait.argtypes = [vp, ctypes.c_longlong, i32, vp]
        lib.gdn_selftest_wait.restype = i32
        lib.gdn_read_device_flags.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), vp]
        lib.gdn_read_device_flags.restype = i32
        _lib = lib
    return _lib


def gdn_version() -> int:
    return int(load().gdn_version())


def gdn_status_string(status: int) -> str:
    return load().gdn_status_string(int(status)).decode()


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.bfloat16:
        return GDN_BF16
    if t == torch.float32:
        return GDN_F32
    raise TypeError(f"unsupported q/k/v dtype {t}")


def gdn_chunk_fwd_workspace_bytes(B: int, T: int, H: int, HV: int, dk: int, dv: int,
                                  chunk: int, gate_mode: int, n_seqs: int,
                                  dtype: int) -> int:
    return int(load().gdn_chunk_fwd_workspace_bytes(B, T, H, HV, dk, dv, chunk,
                                                     gate_mode, n_seqs, dtype))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call(entry: str, q, k, v, g, beta, h0, scale, chunk, cu_seqlens, o, hT,
          output_final_state, workspace, stream):
    lib = load()
    B, T, H, dk = q.shape
    HV, dv = v.shape[2], v.shape[3]
    if k.shape != q.shape or v.shape[:2] != (B, T) or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v: inconsistent shapes or dtypes")
    if g.dim() == 3:
        gate_mode = GDN_GATE_SCALAR
    elif g.dim() == 4:
        gate_mode = GDN_GATE_PER_KEY
    else:
        raise ValueError("g must be [B,T,HV] or [B,T,HV,dk]")
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("h0", h0),
                    ("cu_seqlens", cu_seqlens), ("o", o), ("hT", hT),
                    ("workspace", workspace)):
        if t is not None and (t.device != dev or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous tensor on {dev}")
    if g.dtype != torch.float32 or beta.dtype != torch.float32:
        raise TypeError("g and beta must be float32")
    if h0 is not None and h0.dtype != torch.float32:
        raise TypeError("h0 must be float32")
    if cu_seqlens is not None and cu_seqlens.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32")
    n_seqs = int(cu_seqlens.numel() - 1) if cu_seqlens is not None else B
    dt = _dtype_code(q.dtype)
    if scale is None:
        scale = dk ** -0.5
    if o is None:
        o = torch.empty((B, T, HV, dv), dtype=q.dtype, device=dev)
    if hT is None and output_final_state:
        hT = torch.empty((n_seqs, HV, dk, dv), dtype=torch.float32, device=dev)
    nbytes = gdn_chunk_fwd_workspace_bytes(B, T, H, HV, dk, dv, chunk, gate_mode, n_seqs, dt)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    status = getattr(lib, entry)(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(o), _ptr(hT),
        _ptr(cu_seqlens), n_seqs, B, T, H, HV, dk, dv, int(chunk), float(scale),
        gate_mode, dt, _ptr(workspace), workspace.numel() * workspace.element_size(),
        ctypes.c_void_p(stream.cuda_stream))
    if status != GDN_OK:
        raise GdnError(status, entry)
    return o, hT


def gdn_chunk_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                  beta: torch.Tensor, h0: Optional[torch.Tensor] = None, *,
                  scale: Optional[float] = None, chunk: int = 64,
                  cu_seqlens: Optional[torch.Tensor] = None,
                  o: Optional[torch.Tensor] = None, hT: Optional[torch.Tensor] = None,
                  output_final_state: bool = True,
                  workspace: Optional[torch.Tensor] = None,
                  stream: Optional[torch.cuda.Stream] = None
                  ) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Run the forward pass; returns ``(o, hT)`` (``hT`` None when not asked).

    q, k ``[B, T, H, dk]``; v ``[B, T, HV, dv]`` (bf16 or fp32, same dtype);
    g ``[B, T, HV]`` (scalar gate) or ``[B, T, HV, dk]`` (per-key gate), fp32;
    beta ``[B, T, HV]`` fp32; h0 ``[N, HV, dk, dv]`` fp32 or None;
    cu_seqlens int32 ``[N + 1]`` on the device for packed input (B == 1).
    """
    return _call("gdn_chunk_fwd", q, k, v, g, beta, h0, scale, chunk, cu_seqlens, o, hT,
                 output_final_state, workspace, stream)


def gdn_chunk_fwd_lockstep(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                           beta: torch.Tensor, h0: Optional[torch.Tensor] = None, *,
                           scale: Optional[float] = None, chunk: int = 64,
                           cu_seqlens: Optional[torch.Tensor] = None,
                           o: Optional[torch.Tensor] = None, hT: Optional[torch.Tensor] = None,
                           output_final_state: bool = True,
                           workspace: Optional[torch.Tensor] = None,
                           stream: Optional[torch.cuda.Stream] = None
                           ) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """gdn_chunk_fwd with prep and scan in one cooperative launch, in lockstep
    (bf16 inputs, scalar gate only); same arguments and results."""
    return _call("gdn_chunk_fwd_lockstep", q, k, v, g, beta, h0, scale, chunk, cu_seqlens, o,
                 hT, output_final_state, workspace, stream)


def gdn_chunk_fwd_prep(q, k, v, g, beta, h0=None, *, workspace: torch.Tensor,
                       o: torch.Tensor, hT: Optional[torch.Tensor] = None, scale=None,
                       chunk: int = 64, cu_seqlens=None, stream=None) -> None:
    """First half of gdn_chunk_fwd: the chunk-prep kernel (fills ``workspace``)."""
    _call("gdn_chunk_fwd_prep", q, k, v, g, beta, h0, scale, chunk, cu_seqlens, o, hT,
          hT is not None, workspace, stream)


def gdn_chunk_fwd_scan(q, k, v, g, beta, h0=None, *, workspace: torch.Tensor,
                       o: torch.Tensor, hT: Optional[torch.Tensor] = None, scale=None,
                       chunk: int = 64, cu_seqlens=None, stream=None) -> None:
    """Second half of gdn_chunk_fwd: the scan kernel (reads ``workspace``)."""
    _call("gdn_chunk_fwd_scan", q, k, v, g, beta, h0, scale, chunk, cu_seqlens, o, hT,
          hT is not None, workspace, stream)


def gdn_recurrent_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                      beta: torch.Tensor, h0: Optional[torch.Tensor] = None, *,
                      scale: Optional[float] = None,
                      cu_seqlens: Optional[torch.Tensor] = None,
                      o: Optional[torch.Tensor] = None, hT: Optional[torch.Tensor] = None,
                      output_final_state: bool = True,
                      flags: Optional[torch.Tensor] = None,
                      stream: Optional[torch.cuda.Stream] = None
                      ) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Token-serial form (the decode step when T == 1); returns ``(o, hT)``.

    Same tensors as :func:`gdn_chunk_fwd`; dv any multiple of 32 up to 1024.
    Pass ``hT=h0`` to update the state in place.  ``flags``: an int32/uint32
    device tensor of at least one element that receives the GDN_FLAG_* bits
    (read it with :func:`gdn_read_device_flags`), or None.
    """
    lib = load()
    B, T, H, dk = q.shape
    HV, dv = v.shape[2], v.shape[3]
    if k.shape != q.shape or v.shape[:2] != (B, T) or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v: inconsistent shapes or dtypes")
    if g.dim() == 3:
        gate_mode = GDN_GATE_SCALAR
    elif g.dim() == 4:
        gate_mode = GDN_GATE_PER_KEY
    else:
        raise ValueError("g must be [B,T,HV] or [B,T,HV,dk]")
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("h0", h0),
                    ("cu_seqlens", cu_seqlens), ("o", o), ("hT", hT), ("flags", flags)):
        if t is not None and (t.device != dev or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous tensor on {dev}")
    if g.dtype != torch.float32 or beta.dtype != torch.float32:
        raise TypeError("g and beta must be float32")
    if h0 is not None and h0.dtype != torch.float32:
        raise TypeError("h0 must be float32")
    if cu_seqlens is not None and cu_seqlens.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32")
    if flags is not None and (flags.element_size() != 4 or flags.numel() < 1):
        raise TypeError("flags must hold at least one 4-byte element")
    n_seqs = int(cu_seqlens.numel() - 1) if cu_seqlens is not None else B
    dt = _dtype_code(q.dtype)
    if scale is None:
        scale = dk ** -0.5
    if o is None:
        o = torch.empty((B, T, HV, dv), dtype=q.dtype, device=dev)
    if hT is None and output_final_state:
        hT = torch.empty((n_seqs, HV, dk, dv), dtype=torch.float32, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    status = lib.gdn_recurrent_fwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(o), _ptr(hT),
        _ptr(cu_seqlens), n_seqs, B, T, H, HV, dk, dv, float(scale), gate_mode, dt,
        _ptr(flags), ctypes.c_void_p(stream.cuda_stream))
    if status != GDN_OK:
        raise GdnError(status, "gdn_recurrent_fwd")
    return o, hT


def _check(t, name, dev):
    if t is not None and (t.device != dev or not t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous tensor on {dev}")


def gdn_causal_conv1d_fwd(x: torch.Tensor, w: torch.Tensor, bias: Optional[torch.Tensor] = None,
                          h0: Optional[torch.Tensor] = None, *, activation: int = GDN_ACT_NONE,
                          cu_seqlens: Optional[torch.Tensor] = None,
                          y: Optional[torch.Tensor] = None, hT: Optional[torch.Tensor] = None,
                          output_final_state: bool = True,
                          flags: Optional[torch.Tensor] = None,
                          stream: Optional[torch.cuda.Stream] = None
                          ) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Causal depthwise convolution with history; returns ``(y, hT)``.

    x ``[B, T, D]`` (bf16 or fp32; packed ``[1, Ttot, D]`` with cu_seqlens);
    w ``[D, W]`` fp32; bias ``[D]`` fp32 or None; h0 / hT ``[N, D, W-1]`` fp32
    (``hT=h0`` updates the history in place).
    """
    lib = load()
    B, T, D = x.shape
    W = w.shape[1]
    dev = x.device
    for name, t in (("x", x), ("w", w), ("bias", bias), ("h0", h0), ("cu_seqlens", cu_seqlens),
                    ("y", y), ("hT", hT), ("flags", flags)):
        _check(t, name, dev)
    for name, t in (("w", w), ("bias", bias), ("h0", h0)):
        if t is not None and t.dtype != torch.float32:
            raise TypeError(f"{name} must be float32")
    n_seqs = int(cu_seqlens.numel() - 1) if cu_seqlens is not None else B
    if y is None:
        y = torch.empty_like(x)
    if hT is None and output_final_state:
        hT = torch.empty((n_seqs, D, W - 1), dtype=torch.float32, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    status = lib.gdn_causal_conv1d_fwd(
        _ptr(x), _ptr(w), _ptr(bias), _ptr(h0), _ptr(y), _ptr(hT), _ptr(cu_seqlens), n_seqs, B,
        T, D, W, int(activation), _dtype_code(x.dtype), _ptr(flags),
        ctypes.c_void_p(stream.cuda_stream))
    if status != GDN_OK:
        raise GdnError(status, "gdn_causal_conv1d_fwd")
    return y, hT


def gdn_l2norm_fwd(x: torch.Tensor, *, eps: float = 1e-6, y: Optional[torch.Tensor] = None,
                   stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Rows of x (last axis) divided by sqrt(sum of squares + eps)."""
    lib = load()
    _check(x, "x", x.device)
    _check(y, "y", x.device)
    if y is None:
        y = torch.empty_like(x)
    if stream is None:
        stream = torch.cuda.current_stream(x.device)
    dim = x.shape[-1]
    status = lib.gdn_l2norm_fwd(_ptr(x), _ptr(y), x.numel() // max(dim, 1), dim, float(eps),
                                _dtype_code(x.dtype), ctypes.c_void_p(stream.cuda_stream))
    if status != GDN_OK:
        raise GdnError(status, "gdn_l2norm_fwd")
    return y


def gdn_rmsnorm_gated_fwd(x: torch.Tensor, weight: torch.Tensor, z: Optional[torch.Tensor] = None,
                          *, eps: float = 1e-6, y: Optional[torch.Tensor] = None,
                          stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Rows of x scaled to unit RMS, times weight (fp32), times silu(z)."""
    lib = load()
    dev = x.device
    for name, t in (("x", x), ("weight", weight), ("z", z), ("y", y)):
        _check(t, name, dev)
    if weight.dtype != torch.float32:
        raise TypeError("weight must be float32")
    if z is not None and (z.shape != x.shape or z.dtype != x.dtype):
        raise ValueError("z must match x in shape and dtype")
    if y is None:
        y = torch.empty_like(x)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    dim = x.shape[-1]
    status = lib.gdn_rmsnorm_gated_fwd(_ptr(x), _ptr(z), _ptr(weight), _ptr(y),
                                       x.numel() // max(dim, 1), dim, float(eps),
                                       _dtype_code(x.dtype), ctypes.c_void_p(stream.cuda_stream))
    if status != GDN_OK:
        raise GdnError(status, "gdn_rmsnorm_gated_fwd")
    return y


def gdn_state_combine(M: torch.Tensor, S_in: torch.Tensor, S_seg: torch.Tensor, *,
                      out: Optional[torch.Tensor] = None,
                      stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """S_out = M S_in + S_seg per (state, value head): M ``[N, HV, dk, dk]``,
    S_in and S_seg ``[N, HV, dk, dv]``, fp32 (``out=S_seg`` composes in place)."""
    lib = load()
    dev = M.device
    for name, t in (("M", M), ("S_in", S_in), ("S_seg", S_seg), ("out", out)):
        _check(t, name, dev)
        if t is not None and t.dtype != torch.float32:
            raise TypeError(f"{name} must be float32")
    N, HV, dk, dv = S_in.shape
    if M.shape != (N, HV, dk, dk) or S_seg.shape != S_in.shape:
        raise ValueError("M [N, HV, dk, dk] and S_seg [N, HV, dk, dv] must match S_in")
    if out is None:
        out = torch.empty_like(S_seg)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    status = lib.gdn_state_combine(_ptr(M), _ptr(S_in), _ptr(S_seg), _ptr(out), N, HV, dk, dv,
                                   ctypes.c_void_p(stream.cuda_stream))
    if status != GDN_OK:
        raise GdnError(status, "gdn_state_combine")
    return out


def gdn_selftest_wait(flags: torch.Tensor, budget_cycles: int, complete: bool, *,
                      stream: Optional[torch.cuda.Stream] = None) -> None:
    """Run the bounded-wait self-test into ``flags`` (a uint32-sized int32
    tensor on the device): a wait on a barrier that never completes
    (``complete=False``) must leave GDN_FLAG_TIMEOUT there; one that completes
    must leave 0.  Read it back with :func:`gdn_read_device_flags`."""
    lib = load()
    _check(flags, "flags", flags.device)
    if flags.dtype != torch.int32 or flags.numel() < 1:
        raise TypeError("flags must be an int32 tensor of at least one element")
    if stream is None:
        stream = torch.cuda.current_stream(flags.device)
    status = lib.gdn_selftest_wait(_ptr(flags), int(budget_cycles), int(bool(complete)),
                                   ctypes.c_void_p(stream.cuda_stream))
    if status != GDN_OK:
        raise GdnError(status, "gdn_selftest_wait")


def gdn_read_device_flags(workspace: torch.Tensor,
                          stream: Optional[torch.cuda.Stream] = None) -> int:
    """Status word (GDN_FLAG_*) of the last call that used ``workspace`` (or,
    for gdn_recurrent_fwd, the ``flags`` tensor)."""
    lib = load()
    if stream is None:
        stream = torch.cuda.current_stream(workspace.device)
    out = ctypes.c_uint32(0)
    status = lib.gdn_read_device_flags(_ptr(workspace), ctypes.byref(out),
                                       ctypes.c_void_p(stream.cuda_stream))
    if status != GDN_OK:
        raise GdnError(status, "gdn_read_device_flags")
    return int(out.value)
