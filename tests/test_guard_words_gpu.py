"""Out-of-bounds writes: every buffer a call writes (o, hT, the workspace) is
carved out of a larger allocation whose margins hold a known byte pattern,
and the margins must be unchanged after the call.  Shapes with ragged tails,
packed sequences with empty ones, and every entry that writes device memory
(chunked forward in both launch forms, the token-serial form, the state
combination) are covered.  The kernels also check their own indices; this
catches a write that lands just outside a buffer without faulting."""
from __future__ import annotations

import pytest
import torch

from chunkwise_gated_delta_gdn_gb300 import gdn, synth
from tests.gpu_util import to_dev

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes of margin on each side, a multiple of 256
PATTERN = 0xA5


class Guarded:
    """A device byte buffer of `nbytes` with GUARD bytes of pattern either side."""

    def __init__(self, nbytes: int):
        self.nbytes = nbytes
        self.raw = torch.full((nbytes + 2 * GUARD,), PATTERN, dtype=torch.uint8, device="cuda")

    def view(self, dtype, shape):
        inner = self.raw[GUARD:GUARD + self.nbytes]
        return inner.view(dtype).view(shape)

    def intact(self) -> bool:
        torch.cuda.synchronize()
        lo, hi = self.raw[:GUARD], self.raw[GUARD + self.nbytes:]
        return bool((lo == PATTERN).all() and (hi == PATTERN).all())


def nbytes(dtype, shape):
    n = 1
    for s in shape:
        n *= s
    return n * torch.tensor([], dtype=dtype).element_size()


def run_guarded(c, x, entry):
    d = to_dev(x)
    B, T = d["q"].shape[:2]
    n_states = c.num_states
    dt = gdn.GDN_BF16 if c.dtype == torch.bfloat16 else gdn.GDN_F32
    o_shape, h_shape = (B, T, c.HV, c.dv), (n_states, c.HV, c.dk, c.dv)
    go = Guarded(nbytes(c.dtype, o_shape))
    gh = Guarded(nbytes(torch.float32, h_shape))
    ws_n = gdn.gdn_chunk_fwd_workspace_bytes(B, T, c.H, c.HV, c.dk, c.dv, c.chunk, c.gate_mode,
                                             n_states, dt)
    gw = Guarded(ws_n)  # exactly the size the library asks for
    o, hT, ws = go.view(c.dtype, o_shape), gh.view(torch.float32, h_shape), gw.view(torch.uint8, (ws_n,))
    entry(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], o=o, hT=hT, workspace=ws,
          scale=c.scale, chunk=c.chunk, cu_seqlens=d["cu_seqlens"])
    assert go.intact(), "write outside o"
    assert gh.intact(), "write outside hT"
    assert gw.intact(), "write outside the workspace"
    return o, hT


CASES = [
    synth.case("gdn_bf16_t4096", T=200, H=2, HV=6),
    synth.case("gdn_bf16_t4096", T=37, H=2, HV=4, dk=64, dv=128, chunk=32),
    synth.case("kda_bf16_b2_t8192", T=65, H=2, HV=4),
    synth.case("gdn_fp32_t256", T=150),
    synth.case("kda_bf16_b2_t8192", T=70, H=2, HV=2, dtype=torch.float32),
]


@pytest.mark.parametrize("c", CASES, ids=lambda c: f"{c.name}_T{c.T}")
def test_chunk_fwd_writes_stay_inside(c):
    run_guarded(c, synth.make_inputs(c), gdn.gdn_chunk_fwd)


def test_chunk_fwd_packed_writes_stay_inside():
    lengths = [0, 1, 63, 64, 65, 0, 17]
    c = synth.Case("guard_varlen", B=1, T=sum(lengths), H=2, HV=4, dk=128, dv=128, chunk=64,
                   dtype=torch.bfloat16, gate_mode=0, gate_dist="uniform", gate_low=-1.0,
                   h0_std=0.1, n_seqs=len(lengths), seed=9)
    x = synth.make_inputs(c, lengths=lengths)
    o1, h1 = run_guarded(c, x, gdn.gdn_chunk_fwd)
    o2, h2 = run_guarded(c, x, gdn.gdn_chunk_fwd_lockstep)
    assert torch.equal(o1, o2) and torch.equal(h1, h2)


def test_lockstep_writes_stay_inside():
    c = synth.case("gdn_bf16_t4096", T=300, H=2, HV=6)
    run_guarded(c, synth.make_inputs(c), gdn.gdn_chunk_fwd_lockstep)


def test_recurrent_writes_stay_inside():
    c = synth.case("gdn_decode_bf16_b256", B=3, T=5, H=2, HV=4)
    d = to_dev(synth.make_inputs(c))
    o_shape, h_shape = (3, 5, 4, 128), (3, 4, 128, 128)
    go, gh, gf = Guarded(nbytes(torch.bfloat16, o_shape)), Guarded(nbytes(torch.float32, h_shape)), Guarded(256)
    o, hT, flags = go.view(torch.bfloat16, o_shape), gh.view(torch.float32, h_shape), gf.view(torch.int32, (64,))
    gdn.gdn_recurrent_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], o=o, hT=hT,
                          flags=flags, scale=c.scale)
    assert go.intact() and gh.intact() and gf.intact()


def test_state_combine_writes_stay_inside():
    n, HV, dk, dv = 3, 4, 128, 64
    M = torch.randn((n, HV, dk, dk), device="cuda") * 0.1
    S_in = torch.randn((n, HV, dk, dv), device="cuda")
    S_seg = torch.randn((n, HV, dk, dv), device="cuda")
    go = Guarded(nbytes(torch.float32, (n, HV, dk, dv)))
    out = go.view(torch.float32, (n, HV, dk, dv))
    gdn.gdn_state_combine(M, S_in, S_seg, out=out)
    assert go.intact()
    ref = torch.einsum("nhij,nhjk->nhik", M.double(), S_in.double()) + S_seg.double()
    assert (out.double() - ref).abs().max() < 1e-4
