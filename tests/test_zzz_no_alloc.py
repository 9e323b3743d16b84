"""gdn_chunk_fwd_noalloc: the forward pass for callers that cannot allocate
device memory (a component whose host framework owns all device memory, or a
latency-critical loop that must not stall on an allocation).  It takes its
workspace from a fixed 64 MiB device array inside the library instead of from
the caller.  These tests call it through the C ABI on the same inputs as
gdn_chunk_fwd, for two calls in a row (the second call reuses the array the
first one left behind).  Both routes run the same kernels on the same inputs,
so their results must agree bit for bit; one case is also checked against the
fp64 oracle."""
from __future__ import annotations

import ctypes

import pytest
import torch

from chunkwise_gated_delta_gdn_gb300 import build as cuda_build
from chunkwise_gated_delta_gdn_gb300 import gdn, synth
from tests.gpu_util import gpu_heads, kind_of, run_oracle, to_dev
from tests.metrics import assert_close


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def call_noalloc(lib, c, d):
    B, T = d["q"].shape[0], d["q"].shape[1]
    n_seqs = c.num_states
    o = torch.empty((B, T, c.HV, c.dv), dtype=c.dtype, device="cuda")
    hT = torch.empty((n_seqs, c.HV, c.dk, c.dv), dtype=torch.float32, device="cuda")
    dt = gdn.GDN_BF16 if c.dtype == torch.bfloat16 else gdn.GDN_F32
    stream = torch.cuda.current_stream()
    status = lib.gdn_chunk_fwd_noalloc(
        _p(d["q"]), _p(d["k"]), _p(d["v"]), _p(d["g"]), _p(d["beta"]), _p(d["h0"]), _p(o),
        _p(hT), _p(d["cu_seqlens"]), n_seqs, B, T, c.H, c.HV, c.dk, c.dv, c.chunk, c.scale,
        c.gate_mode, dt, ctypes.c_void_p(stream.cuda_stream))
    return status, o, hT


CASES = [
    # bf16 scalar gate (GDN), grouped heads
    synth.case("gdn_bf16_t4096", T=1000, H=4, HV=12),
    # bf16 per-key gate (KDA)
    synth.case("kda_bf16_b2_t8192", T=300, H=4, HV=8),
    # packed sequences with cu_seqlens: the workspace size follows n_seqs
    synth.case("gdn_varlen_t131072", T=900, H=2, HV=6, n_seqs=5),
    # fp32 inputs: the other tile layout
    synth.case("gdn_fp32_t256"),
]


@pytest.mark.gpu
@pytest.mark.parametrize("c", CASES, ids=lambda c: c.name)
def test_noalloc_equals_gdn_chunk_fwd_twice_in_a_row(c):
    lib = gdn.load(cuda_build.build())
    d = to_dev(synth.make_inputs(c))
    o_ref, h_ref = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"],
                                     scale=c.scale, chunk=c.chunk, cu_seqlens=d["cu_seqlens"])
    for _ in range(2):
        status, o, hT = call_noalloc(lib, c, d)
        assert status == gdn.GDN_OK, gdn.gdn_status_string(status)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref), f"{c.name}: o differs from gdn_chunk_fwd"
        assert torch.equal(hT, h_ref), f"{c.name}: hT differs from gdn_chunk_fwd"


@pytest.mark.gpu
def test_noalloc_matches_the_oracle():
    lib = gdn.load(cuda_build.build())
    c = CASES[0]
    x = synth.make_inputs(c)
    status, o, hT = call_noalloc(lib, c, to_dev(x))
    assert status == gdn.GDN_OK, gdn.gdn_status_string(status)
    torch.cuda.synchronize()
    o_ref, h_ref = run_oracle(c, x)
    og, hg = gpu_heads(o, hT)
    assert_close(og, o_ref, kind_of(c), f"{c.name} o")
    assert_close(hg, h_ref, kind_of(c), f"{c.name} hT")


def test_noalloc_refuses_requests_beyond_its_array():
    """A request needing more than 64 MiB of workspace is refused before any
    device work (fake addresses: nothing is dereferenced)."""
    lib = gdn.load(cuda_build.build())
    need = gdn.gdn_chunk_fwd_workspace_bytes(1, 32768, 16, 48, 128, 128, 64, 0, 1, 1)
    assert need > 64 << 20
    a = [ctypes.c_void_p((1 << 40) + i * (1 << 34)) for i in range(8)]
    status = lib.gdn_chunk_fwd_noalloc(*a, None, 1, 1, 32768, 16, 48, 128, 128, 64, 0.088,
                                       0, gdn.GDN_BF16, None)
    assert status == gdn.GDN_ERR_WORKSPACE
