"""GPU parity of the token-serial form (gdn_recurrent_fwd, the decode step
when T == 1) against the fp64 token-serial oracle, through the C ABI.

The one-token grouped step with K-first input state and separate
output/next-state buffers, value width up to 1024 (logismos issue #46,
"Verified implementation boundary").  Tolerances as for the chunked path
(tests/metrics.py): fp32 inputs max-abs <= 1e-4; bf16 inputs max-abs <= 1e-2
and rel-Frobenius <= 2e-3.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from chunkwise_gated_delta_gdn_gb300 import gdn, synth
from tests.gpu_util import gpu_heads, kind_of, run_oracle, to_dev
from tests.metrics import assert_close

pytestmark = pytest.mark.gpu


def run_rec(c, x, *, h0=True, want_hT=True, in_place=False):
    d = to_dev(x)
    h = d["h0"] if h0 else None
    kw = dict(scale=c.scale, cu_seqlens=d["cu_seqlens"], output_final_state=want_hT)
    if in_place:
        h = h.clone()
        kw["hT"] = h
    o, hT = gdn.gdn_recurrent_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h, **kw)
    torch.cuda.synchronize()
    return o, hT


def check(c, x, heads=None, h0=True):
    o, hT = run_rec(c, x, h0=h0)
    o_ref, h_ref = run_oracle(c, x, heads, h0=h0)
    og, hg = gpu_heads(o, hT, heads)
    assert_close(og, o_ref, kind_of(c), f"{c.name} o")
    assert_close(hg, h_ref, kind_of(c), f"{c.name} hT")


def small(name, **kw):
    base = dict(B=3, T=1, H=2, HV=4, dk=128, dv=128, chunk=64, dtype=torch.bfloat16,
                gate_mode=0, gate_dist="uniform", gate_low=-5.0, h0_std=0.1, seed=21)
    base.update(kw)
    return synth.Case(name, **base)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("gate_mode", [0, 1], ids=["gdn", "kda"])
@pytest.mark.parametrize("dk,dv", [(64, 32), (64, 64), (128, 128), (128, 256), (64, 1024)])
@pytest.mark.parametrize("T", [1, 37])
def test_shapes(dtype, gate_mode, dk, dv, T):
    c = small(f"rec_{dk}_{dv}_{T}_{gate_mode}", T=T, dk=dk, dv=dv, dtype=dtype,
              gate_mode=gate_mode, gate_low=-1.0 if T > 1 else -5.0)
    check(c, synth.make_inputs(c))


@pytest.mark.parametrize("T", [1, 37, 64, 65, 200])
@pytest.mark.parametrize("low", [-0.05, -1.0, -5.0])
@pytest.mark.parametrize("gate_mode", [0, 1], ids=["gdn", "kda"])
def test_sweep(T, low, gate_mode):
    c = small(f"rec_sweep_{gate_mode}_{T}_{low}", B=1, T=T, gate_mode=gate_mode,
              gate_low=low, seed=T)
    check(c, synth.make_inputs(c))


def test_without_initial_state_and_without_final_state():
    c = small("rec_noh0", T=5)
    x = synth.make_inputs(c)
    check(c, x, h0=False)
    o, hT = run_rec(c, x, want_hT=False)
    assert hT is None
    o_ref, _ = run_oracle(c, x)
    assert_close(gpu_heads(o, None)[0], o_ref, "bf16", "o without hT")


def test_in_place_state_update_matches_separate_buffers():
    c = small("rec_inplace", B=5, T=3, gate_mode=1)
    x = synth.make_inputs(c)
    o1, h1 = run_rec(c, x)
    o2, h2 = run_rec(c, x, in_place=True)
    assert torch.equal(o1, o2) and torch.equal(h1, h2)


def test_decode_loop_in_place_equals_one_call_over_all_tokens():
    """Eight one-token steps, each updating the state in place, reproduce the
    oracle's walk over the eight tokens (partition continuation, logismos
    issue #46, Sep 10 comment)."""
    c = small("rec_loop", B=4, T=8, gate_mode=0)
    x = synth.make_inputs(c)
    d = to_dev(x)
    h = d["h0"].clone()
    outs = []
    for t in range(c.T):
        sl = {n: d[n][:, t:t + 1].contiguous() for n in ("q", "k", "v", "g", "beta")}
        o, _ = gdn.gdn_recurrent_fwd(sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"], h,
                                     hT=h, scale=c.scale)
        outs.append(o)
    torch.cuda.synchronize()
    o = torch.cat(outs, 1)
    o_ref, h_ref = run_oracle(c, x)
    og, hg = gpu_heads(o, h)
    assert_close(og, o_ref, "bf16", "looped o")
    assert_close(hg, h_ref, "bf16", "looped hT")


@pytest.mark.parametrize("gate_mode", [0, 1], ids=["gdn", "kda"])
def test_varlen_with_empty_sequences(gate_mode):
    lengths = [0, 1, 5, 0, 33, 2]
    c = synth.Case("rec_varlen", B=1, T=sum(lengths), H=2, HV=4, dk=128, dv=128, chunk=64,
                   dtype=torch.bfloat16, gate_mode=gate_mode, gate_dist="uniform",
                   gate_low=-1.0, h0_std=0.1, n_seqs=len(lengths), seed=8)
    x = synth.make_inputs(c, lengths=lengths)
    check(c, x)
    o, hT = run_rec(c, x)
    for i, L in enumerate(lengths):
        if L == 0:
            assert torch.equal(hT[i].cpu(), x["h0"][i])


def test_zero_tokens():
    c = small("rec_zero", T=0)
    x = synth.make_inputs(c)
    o, hT = run_rec(c, x)
    assert o.numel() == 0
    assert torch.equal(hT.cpu(), x["h0"])


def test_agrees_with_chunked_path():
    c = synth.case("gdn_bf16_t4096", T=300, H=2, HV=6)
    x = synth.make_inputs(c)
    d = to_dev(x)
    o1, h1 = gdn.gdn_recurrent_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"])
    o2, h2 = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], chunk=64)
    torch.cuda.synchronize()
    assert_close(o1.cpu().double().numpy(), o2.cpu().double().numpy(), "bf16", "o rec vs chunk")
    assert_close(h1.cpu().double().numpy(), h2.cpu().double().numpy(), "bf16",
                 "hT rec vs chunk")


def test_flags():
    c = small("rec_flags", T=2)
    x = synth.make_inputs(c)
    d = to_dev(x)
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_recurrent_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], flags=flags)
    assert gdn.gdn_read_device_flags(flags) == 0
    g_bad = d["g"].clone()
    g_bad[1, 1, 2] = 0.25
    gdn.gdn_recurrent_fwd(d["q"], d["k"], d["v"], g_bad, d["beta"], d["h0"], flags=flags)
    assert gdn.gdn_read_device_flags(flags) & gdn.GDN_FLAG_POSITIVE_GATE
    v_bad = d["v"].clone()
    v_bad[0, 0, 1, 5] = float("nan")
    gdn.gdn_recurrent_fwd(d["q"], d["k"], v_bad, d["g"], d["beta"], d["h0"], flags=flags)
    assert gdn.gdn_read_device_flags(flags) & gdn.GDN_FLAG_NONFINITE
    gdn.gdn_recurrent_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], flags=flags)
    assert gdn.gdn_read_device_flags(flags) == 0


def test_bad_seqlens_flagged_not_faulting():
    c = synth.Case("rec_badcu", B=1, T=10, H=2, HV=4, dk=128, dv=128, chunk=64,
                   dtype=torch.bfloat16, gate_mode=0, gate_dist="uniform", gate_low=-1.0,
                   h0_std=0.1, n_seqs=2, seed=6)
    x = to_dev(synth.make_inputs(c, lengths=[4, 6]))
    bad = torch.tensor([0, 12, 10], dtype=torch.int32, device="cuda")
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_recurrent_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], cu_seqlens=bad,
                          flags=flags)
    assert gdn.gdn_read_device_flags(flags) & gdn.GDN_FLAG_BAD_SEQLENS


@pytest.mark.parametrize("name", ["gdn_decode_bf16_b256", "kda_decode_bf16_b256"])
def test_decode_workload_all_heads(name):
    c = synth.case(name)
    check(c, synth.make_inputs(c))
