"""fp64 CPU oracle for the gated delta rule forward pass.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
CUDA library never calls it, and it never calls the CUDA library.

Two independent walks live in ``gdn_oracle.c``:

* :func:`token_serial` -- the plain definition, one token at a time (the
  token-serial oracle of ROCm/rocm-libraries PR #11223, "Correctness").
* :func:`chunked` -- the chunk-parallel WY form (stratat pull #1296, "What this
  is"; the six state-independent tiles of PR #11223, "Summary") with pairwise
  decays formed directly, no midpoint factoring (PR #11223, "Correctness",
  tile oracle), and any chunk size.

Inputs are numpy arrays (or anything ``np.asarray`` accepts) in packed layout:
q, k ``[Ttot, H, dk]``; v ``[Ttot, HV, dv]``; g ``[Ttot, HV]`` (GDN) or
``[Ttot, HV, dk]`` (KDA); beta ``[Ttot, HV]``; h0 ``[N, HV, dk, dv]`` or None;
``cu_seqlens`` ``[N + 1]``.  They are widened to float64 before the call, so a
bf16 tensor is seen with exactly the bits the GPU sees.  Batched ``[B, T, ...]``
inputs go through :func:`pack_batched` first.

Parity status: every function here is pinned by the ``-m "not gpu"`` tests
(closed forms, invariants, brute force on tiny inputs, planted mistakes).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libgdn_oracle.so")
# negative controls: deliberately wrong copies of the token walk, a library of
# their own so that the oracle's walk carries no switch
_PLANTED_SRC = os.path.join(_HERE, "planted_walk.c")
_PLANTED_PATH = os.path.join(_BUILD_DIR, "libgdn_planted.so")
_lock = threading.Lock()
_lib = None
_planted_lib = None

GATE_SCALAR = 0  # GDN: one log-gate per (token, value head)
GATE_PER_KEY = 1  # KDA: one log-gate per (token, value head, key channel)


def _compile(src: str, out: str, force: bool, openmp: bool) -> str:
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(out)) or os.path.getmtime(out) < os.path.getmtime(src)
    if force or stale:
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O3", "-ffp-contract=off", *(["-fopenmp"] if openmp else []),
               "-fPIC", "-shared", "-std=c11", "-Wall", "-o", tmp, src, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into ``oracle/_build``; returns the .so path."""
    return _compile(_SRC, _LIB_PATH, force, openmp=True)


def _load():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            lib = ctypes.CDLL(path)
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int64)
            common = [dp, dp, dp, dp, dp, dp, dp, dp, ip, ctypes.c_int,
                      ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                      ctypes.c_double, ctypes.c_int]
            lib.gdn_oracle_token_serial.argtypes = common
            lib.gdn_oracle_token_serial.restype = ctypes.c_int
            lib.gdn_oracle_chunked.argtypes = common + [ctypes.c_int]
            lib.gdn_oracle_chunked.restype = ctypes.c_int
            lib.gdn_oracle_num_threads.argtypes = []
            lib.gdn_oracle_num_threads.restype = ctypes.c_int
            lib.gdn_oracle_set_num_threads.argtypes = [ctypes.c_int]
            lib.gdn_oracle_set_num_threads.restype = None
            _lib = lib
    return _lib


def num_threads() -> int:
    """OpenMP threads the oracle will use."""
    return int(_load().gdn_oracle_num_threads())


def set_num_threads(n: int) -> None:
    _load().gdn_oracle_set_num_threads(int(n))


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: widen on the CPU, bits preserved
        x = x.detach().to("cpu")
        x = x.double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def pack_batched(q, k, v, g, beta):
    """Flatten ``[B, T, ...]`` inputs to the packed layout; returns the arrays
    and ``cu_seqlens = [0, T, 2T, ..., B*T]``."""
    B, T = q.shape[0], q.shape[1]
    flat = [x.reshape((B * T,) + tuple(x.shape[2:])) for x in (q, k, v, g, beta)]
    cu = np.arange(B + 1, dtype=np.int64) * T
    return (*flat, cu)


def _load_planted():
    global _planted_lib
    with _lock:
        if _planted_lib is None:
            lib = ctypes.CDLL(_compile(_PLANTED_SRC, _PLANTED_PATH, False, openmp=False))
            dp = ctypes.POINTER(ctypes.c_double)
            lib.gdn_planted_token_serial.argtypes = [
                dp, dp, dp, dp, dp, dp, dp, dp, ctypes.POINTER(ctypes.c_int64), ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                ctypes.c_int, ctypes.c_int]
            lib.gdn_planted_token_serial.restype = ctypes.c_int
            _planted_lib = lib
    return _planted_lib


def _run(entry, q, k, v, g, beta, h0, cu_seqlens, scale, gate_mode, extra=(), lib=None):
    lib = lib or _load()
    q, k, v, g, beta, h0 = (_f64(x) for x in (q, k, v, g, beta, h0))
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    Ttot, H, dk = q.shape
    HV, dv = v.shape[1], v.shape[2]
    n_seqs = cu.shape[0] - 1
    if k.shape != q.shape or v.shape[0] != Ttot or beta.shape != (Ttot, HV):
        raise ValueError("oracle: inconsistent input shapes")
    want_g = (Ttot, HV) if gate_mode == GATE_SCALAR else (Ttot, HV, dk)
    if g.shape != want_g:
        raise ValueError(f"oracle: g has shape {g.shape}, expected {want_g}")
    if h0 is not None and h0.shape != (n_seqs, HV, dk, dv):
        raise ValueError("oracle: h0 shape")
    if int(cu[-1]) != Ttot:
        raise ValueError("oracle: cu_seqlens[-1] must equal the token count")
    o = np.zeros((Ttot, HV, dv), dtype=np.float64)
    hT = np.zeros((n_seqs, HV, dk, dv), dtype=np.float64)
    rc = getattr(lib, entry)(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(o),
        _ptr(hT), cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), n_seqs, H,
        HV, dk, dv, float(scale), int(gate_mode), *extra)
    if rc != 0:
        raise ValueError(f"oracle: {entry} rejected its arguments")
    return o, hT


def token_serial(q, k, v, g, beta, h0, cu_seqlens, scale, gate_mode=GATE_SCALAR):
    """The plain token-by-token recurrence; returns ``(o, hT)`` in float64."""
    return _run("gdn_oracle_token_serial", q, k, v, g, beta, h0, cu_seqlens,
                scale, gate_mode)


def token_serial_planted(q, k, v, g, beta, h0, cu_seqlens, scale, gate_mode,
                         planted):
    """A deliberately wrong token walk with one planted mistake, from
    ``planted_walk.c`` (negative controls of the pin tests only)."""
    return _run("gdn_planted_token_serial", q, k, v, g, beta, h0,
                cu_seqlens, scale, gate_mode, (int(planted),), lib=_load_planted())


def chunked(q, k, v, g, beta, h0, cu_seqlens, scale, gate_mode=GATE_SCALAR,
            chunk=64):
    """The chunked WY-form walk with chunk size ``chunk``; returns ``(o, hT)``."""
    return _run("gdn_oracle_chunked", q, k, v, g, beta, h0, cu_seqlens, scale,
                gate_mode, (int(chunk),))
