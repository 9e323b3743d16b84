"""The C ABI without a GPU: the library loads, exports every entry point that
include/gdn.h declares, and refuses malformed or unsupported requests before
touching the device (explicit refusal of unsupported inputs, logismos issue
#46 "Acceptance").  Fake device addresses are fine here: a refused call
dereferences nothing."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from chunkwise_gated_delta_gdn_gb300 import build as cuda_build
from chunkwise_gated_delta_gdn_gb300 import gdn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return gdn.load()


def declared_symbols():
    with open(os.path.join(ROOT, "include", "gdn.h")) as f:
        src = f.read()
    return sorted(set(re.findall(r"GDN_API\s+[\w\s\*]*?\b(gdn_\w+)\s*\(", src)))


def test_header_declares_the_binding_names():
    assert declared_symbols() == sorted(gdn.EXPORTED)


def test_status_flag_values_match_the_header():
    """Each GDN_FLAG_* bit of include/gdn.h has the same value in the binding."""
    with open(os.path.join(ROOT, "include", "gdn.h")) as f:
        src = f.read()
    declared = {name: 1 << int(bit) for name, bit in
                re.findall(r"\b(GDN_FLAG_\w+)\s*=\s*1u\s*<<\s*(\d+)", src)}
    assert set(declared) == {"GDN_FLAG_POSITIVE_GATE", "GDN_FLAG_NONFINITE",
                             "GDN_FLAG_BAD_SEQLENS", "GDN_FLAG_TIMEOUT",
                             "GDN_FLAG_LAUNCH_CONFIG"}
    for name, value in declared.items():
        assert getattr(gdn, name) == value, name
    assert len(set(declared.values())) == len(declared)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert gdn.gdn_version() >= 100


def test_status_strings(lib):
    assert gdn.gdn_status_string(0) == "GDN_OK"
    assert gdn.gdn_status_string(2) == "GDN_ERR_UNSUPPORTED"
    assert gdn.gdn_status_string(99) == "GDN_ERR_UNKNOWN"


def test_workspace_query(lib):
    # bf16, scalar gate: header + (T/C + N) slots x (HV x one 32 KB fp16 operand
    # image [P1; E; AqkT] + H x one 32 KB fp16 [K_next; Q] image), then one int ready flag per
    # (slot, q/k head) for the lockstep launch, padded to 256 bytes
    slots = 32768 // 64 + 1
    ws = gdn.gdn_chunk_fwd_workspace_bytes(1, 32768, 16, 48, 128, 128, 64, 0, 1, gdn.GDN_BF16)
    assert ws == (256 + slots * (48 * 256 * 128 + 16 * 2 * 128 * 128)
                  + (slots * 16 * 4 + 255) // 256 * 256)
    # bf16, per-key gate: per (slot, value head) one 24 KB image [P1; AqkT], one
    # 32 KB gated [K~; Q~] image and dk fp32 chunk decays
    ws = gdn.gdn_chunk_fwd_workspace_bytes(2, 8192, 32, 32, 128, 128, 32, 1, 2, gdn.GDN_BF16)
    assert ws == 256 + (2 * 8192 // 32 + 2) * 32 * (192 * 128 + 2 * 128 * 128 + 128 * 4)
    # fp32: header + slots x HV x (T and Aqk, C x C fp32)
    ws = gdn.gdn_chunk_fwd_workspace_bytes(1, 32768, 16, 48, 128, 128, 64, 0, 1, gdn.GDN_F32)
    assert ws == 256 + (32768 // 64 + 1) * 48 * 2 * 64 * 64 * 4
    assert gdn.gdn_chunk_fwd_workspace_bytes(1, 100, 2, 4, 96, 128, 64, 0, 1, 1) == 0
    assert gdn.gdn_chunk_fwd_workspace_bytes(1, 100, 3, 4, 128, 128, 64, 0, 1, 1) == 0


# fake, 256-byte aligned, far-apart device addresses
BASE = 1 << 40
STRIDE = 1 << 34


def addr(i):
    return ctypes.c_void_p(BASE + i * STRIDE)


def call(lib, **kw):
    a = dict(q=addr(0), k=addr(1), v=addr(2), g=addr(3), beta=addr(4), h0=addr(5),
             o=addr(6), hT=addr(7), cu=None, n_seqs=1, B=1, T=128, H=2, HV=4, dk=128,
             dv=128, chunk=64, scale=0.088, gate_mode=0, dtype=1, ws=addr(8),
             ws_bytes=1 << 30)
    a.update(kw)
    return lib.gdn_chunk_fwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["h0"], a["o"],
                             a["hT"], a["cu"], a["n_seqs"], a["B"], a["T"], a["H"],
                             a["HV"], a["dk"], a["dv"], a["chunk"], a["scale"],
                             a["gate_mode"], a["dtype"], a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("kw, status", [
    (dict(q=None), gdn.GDN_ERR_INVALID_ARG),
    (dict(v=None, T=5), gdn.GDN_ERR_INVALID_ARG),
    (dict(o=None), gdn.GDN_ERR_INVALID_ARG),
    (dict(B=0), gdn.GDN_ERR_INVALID_ARG),
    (dict(T=-1), gdn.GDN_ERR_INVALID_ARG),
    (dict(H=3), gdn.GDN_ERR_INVALID_ARG),           # HV % H != 0
    (dict(gate_mode=2), gdn.GDN_ERR_INVALID_ARG),
    (dict(dtype=7), gdn.GDN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), gdn.GDN_ERR_INVALID_ARG),
    (dict(dk=96), gdn.GDN_ERR_UNSUPPORTED),
    (dict(dv=256), gdn.GDN_ERR_UNSUPPORTED),
    (dict(chunk=16), gdn.GDN_ERR_UNSUPPORTED),
    (dict(chunk=128), gdn.GDN_ERR_UNSUPPORTED),
    (dict(q=ctypes.c_void_p(BASE + 8)), gdn.GDN_ERR_INVALID_ARG),   # misaligned
    (dict(ws=ctypes.c_void_p(BASE + 8 * STRIDE + 16)), gdn.GDN_ERR_INVALID_ARG),
    (dict(ws=None), gdn.GDN_ERR_WORKSPACE),
    (dict(ws_bytes=1000), gdn.GDN_ERR_WORKSPACE),
    (dict(hT=addr(5)), gdn.GDN_ERR_INVALID_ARG),    # hT aliases h0
    (dict(o=addr(2)), gdn.GDN_ERR_INVALID_ARG),     # o aliases v
    (dict(ws=addr(0)), gdn.GDN_ERR_INVALID_ARG),    # workspace aliases q
    (dict(cu=addr(9), B=2, n_seqs=2), gdn.GDN_ERR_INVALID_ARG),  # packed needs B == 1
    (dict(cu=addr(9), n_seqs=0), gdn.GDN_ERR_INVALID_ARG),
    (dict(B=2, n_seqs=3), gdn.GDN_ERR_INVALID_ARG),
])
def test_refusals(lib, kw, status):
    assert call(lib, **kw) == status


@pytest.mark.parametrize("kw, status", [
    (dict(dtype=0), gdn.GDN_ERR_UNSUPPORTED),       # fp32: no lockstep launch
    (dict(gate_mode=1, chunk=32), gdn.GDN_ERR_UNSUPPORTED),   # per-key gate
    (dict(q=None), gdn.GDN_ERR_INVALID_ARG),        # the same checks as gdn_chunk_fwd
    (dict(ws_bytes=1000), gdn.GDN_ERR_WORKSPACE),
    (dict(hT=addr(5)), gdn.GDN_ERR_INVALID_ARG),
])
def test_lockstep_refusals(lib, kw, status):
    a = dict(q=addr(0), k=addr(1), v=addr(2), g=addr(3), beta=addr(4), h0=addr(5),
             o=addr(6), hT=addr(7), cu=None, n_seqs=1, B=1, T=128, H=2, HV=4, dk=128,
             dv=128, chunk=64, scale=0.088, gate_mode=0, dtype=1, ws=addr(8),
             ws_bytes=1 << 30)
    a.update(kw)
    assert lib.gdn_chunk_fwd_lockstep(
        a["q"], a["k"], a["v"], a["g"], a["beta"], a["h0"], a["o"], a["hT"], a["cu"],
        a["n_seqs"], a["B"], a["T"], a["H"], a["HV"], a["dk"], a["dv"], a["chunk"],
        a["scale"], a["gate_mode"], a["dtype"], a["ws"], a["ws_bytes"], None) == status


def test_read_flags_rejects_null(lib):
    out = ctypes.c_uint32(0)
    assert lib.gdn_read_device_flags(None, ctypes.byref(out), None) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_read_device_flags(addr(8), None, None) == gdn.GDN_ERR_INVALID_ARG


def test_binding_refuses_to_run_without_library(tmp_path):
    """The product path fails loudly when the CUDA library is missing."""
    with pytest.raises(RuntimeError, match="libgdn.so not found"):
        saved = gdn._lib
        gdn._lib = None
        try:
            gdn.load(str(tmp_path / "missing.so"))
        finally:
            gdn._lib = saved


def call_rec(lib, **kw):
    a = dict(q=addr(0), k=addr(1), v=addr(2), g=addr(3), beta=addr(4), h0=addr(5),
             o=addr(6), hT=addr(7), cu=None, n_seqs=1, B=1, T=1, H=2, HV=4, dk=128,
             dv=128, scale=0.088, gate_mode=0, dtype=1, flags=addr(8))
    a.update(kw)
    return lib.gdn_recurrent_fwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["h0"], a["o"],
                                 a["hT"], a["cu"], a["n_seqs"], a["B"], a["T"], a["H"],
                                 a["HV"], a["dk"], a["dv"], a["scale"], a["gate_mode"],
                                 a["dtype"], a["flags"], None)


@pytest.mark.parametrize("kw, status", [
    (dict(q=None), gdn.GDN_ERR_INVALID_ARG),
    (dict(o=None), gdn.GDN_ERR_INVALID_ARG),
    (dict(B=0), gdn.GDN_ERR_INVALID_ARG),
    (dict(T=-1), gdn.GDN_ERR_INVALID_ARG),
    (dict(H=3), gdn.GDN_ERR_INVALID_ARG),
    (dict(gate_mode=2), gdn.GDN_ERR_INVALID_ARG),
    (dict(dtype=7), gdn.GDN_ERR_INVALID_ARG),
    (dict(scale=float("inf")), gdn.GDN_ERR_INVALID_ARG),
    (dict(dk=96), gdn.GDN_ERR_UNSUPPORTED),
    (dict(dk=256), gdn.GDN_ERR_UNSUPPORTED),
    (dict(dv=48), gdn.GDN_ERR_UNSUPPORTED),          # not a multiple of 32
    (dict(dv=2048), gdn.GDN_ERR_UNSUPPORTED),        # above 1024
    (dict(q=ctypes.c_void_p(BASE + 8)), gdn.GDN_ERR_INVALID_ARG),
    (dict(flags=ctypes.c_void_p(BASE + 8 * STRIDE + 2)), gdn.GDN_ERR_INVALID_ARG),
    (dict(hT=ctypes.c_void_p(BASE + 5 * STRIDE + 4096)), gdn.GDN_ERR_INVALID_ARG),  # partial overlap
    (dict(o=addr(2)), gdn.GDN_ERR_INVALID_ARG),     # o aliases v
    (dict(o=addr(5)), gdn.GDN_ERR_INVALID_ARG),     # o aliases h0
    (dict(flags=addr(7)), gdn.GDN_ERR_INVALID_ARG),  # status word inside hT
    (dict(hT=addr(1)), gdn.GDN_ERR_INVALID_ARG),    # hT aliases k
    (dict(cu=addr(9), B=2, n_seqs=2), gdn.GDN_ERR_INVALID_ARG),
    (dict(cu=addr(9), n_seqs=0), gdn.GDN_ERR_INVALID_ARG),
    (dict(B=2, n_seqs=3), gdn.GDN_ERR_INVALID_ARG),
])
def test_recurrent_refusals(lib, kw, status):
    assert call_rec(lib, **kw) == status


def call_conv(lib, **kw):
    a = dict(x=addr(0), w=addr(1), bias=addr(2), h0=addr(3), y=addr(4), hT=addr(5), cu=None,
             n_seqs=1, B=1, T=16, D=256, width=4, act=1, dtype=1, flags=addr(8))
    a.update(kw)
    return lib.gdn_causal_conv1d_fwd(a["x"], a["w"], a["bias"], a["h0"], a["y"], a["hT"],
                                     a["cu"], a["n_seqs"], a["B"], a["T"], a["D"], a["width"],
                                     a["act"], a["dtype"], a["flags"], None)


@pytest.mark.parametrize("kw, status", [
    (dict(x=None), gdn.GDN_ERR_INVALID_ARG),
    (dict(w=None), gdn.GDN_ERR_INVALID_ARG),
    (dict(B=0), gdn.GDN_ERR_INVALID_ARG),
    (dict(width=0), gdn.GDN_ERR_INVALID_ARG),
    (dict(act=2), gdn.GDN_ERR_INVALID_ARG),
    (dict(dtype=5), gdn.GDN_ERR_INVALID_ARG),
    (dict(width=5), gdn.GDN_ERR_UNSUPPORTED),
    (dict(D=252), gdn.GDN_ERR_UNSUPPORTED),             # not a multiple of 8
    (dict(y=addr(0)), gdn.GDN_ERR_INVALID_ARG),          # y aliases x
    (dict(hT=ctypes.c_void_p(BASE + 3 * STRIDE + 64)), gdn.GDN_ERR_INVALID_ARG),  # partial overlap
    (dict(x=ctypes.c_void_p(BASE + 4)), gdn.GDN_ERR_INVALID_ARG),
    (dict(cu=addr(9), B=2, n_seqs=2), gdn.GDN_ERR_INVALID_ARG),
])
def test_conv_refusals(lib, kw, status):
    assert call_conv(lib, **kw) == status


@pytest.mark.parametrize("entry", ["l2", "rms"])
@pytest.mark.parametrize("kw, status", [
    (dict(rows=-1), gdn.GDN_ERR_INVALID_ARG),
    (dict(dim=96), gdn.GDN_ERR_UNSUPPORTED),
    (dict(dim=512), gdn.GDN_ERR_UNSUPPORTED),
    (dict(eps=float("nan")), gdn.GDN_ERR_INVALID_ARG),
    (dict(eps=-1.0), gdn.GDN_ERR_INVALID_ARG),
    (dict(dtype=3), gdn.GDN_ERR_INVALID_ARG),
    (dict(x=None), gdn.GDN_ERR_INVALID_ARG),
    (dict(y=ctypes.c_void_p(BASE + 64)), gdn.GDN_ERR_INVALID_ARG),  # partial overlap with x
])
def test_rownorm_refusals(lib, entry, kw, status):
    a = dict(x=addr(0), z=addr(1), weight=addr(2), y=addr(3), rows=100, dim=128, eps=1e-6,
             dtype=1)
    a.update(kw)
    if entry == "l2":
        got = lib.gdn_l2norm_fwd(a["x"], a["y"], a["rows"], a["dim"], a["eps"], a["dtype"], None)
    else:
        got = lib.gdn_rmsnorm_gated_fwd(a["x"], a["z"], a["weight"], a["y"], a["rows"], a["dim"],
                                        a["eps"], a["dtype"], None)
    assert got == status


def test_rmsnorm_needs_its_weight(lib):
    assert lib.gdn_rmsnorm_gated_fwd(addr(0), None, None, addr(3), 10, 128, 1e-6, 1,
                                     None) == gdn.GDN_ERR_INVALID_ARG


@pytest.mark.parametrize("kw, status", [
    (dict(M=None), gdn.GDN_ERR_INVALID_ARG),
    (dict(HV=0), gdn.GDN_ERR_INVALID_ARG),
    (dict(n=-1), gdn.GDN_ERR_INVALID_ARG),
    (dict(dk=2048), gdn.GDN_ERR_UNSUPPORTED),
    (dict(S_out=addr(0)), gdn.GDN_ERR_INVALID_ARG),     # S_out aliases M
    (dict(S_out=addr(1)), gdn.GDN_ERR_INVALID_ARG),     # S_out aliases S_in
    (dict(S_out=ctypes.c_void_p(BASE + 2 * STRIDE + 64)), gdn.GDN_ERR_INVALID_ARG),  # partial
    (dict(M=ctypes.c_void_p(BASE + 4)), gdn.GDN_ERR_INVALID_ARG),
])
def test_state_combine_refusals(lib, kw, status):
    a = dict(M=addr(0), S_in=addr(1), S_seg=addr(2), S_out=addr(3), n=1, HV=4, dk=128, dv=128)
    a.update(kw)
    assert lib.gdn_state_combine(a["M"], a["S_in"], a["S_seg"], a["S_out"], a["n"], a["HV"],
                                 a["dk"], a["dv"], None) == status


@pytest.mark.parametrize("kw", [
    dict(flags=None),
    dict(flags=ctypes.c_void_p(BASE + 2)),   # not 4-byte aligned
    dict(budget=0),
    dict(budget=-5),
    dict(budget=4000000001),
    dict(complete=2),
])
def test_selftest_wait_refusals(lib, kw):
    a = dict(flags=addr(0), budget=1000, complete=0)
    a.update(kw)
    assert lib.gdn_selftest_wait(a["flags"], a["budget"], a["complete"], None) == \
        gdn.GDN_ERR_INVALID_ARG
