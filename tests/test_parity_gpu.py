"""GPU parity: the CUDA path (through the C ABI) against the fp64 token-serial
oracle, element by element, on the same seeded inputs.

Tolerances (tests/metrics.py): fp32 inputs max-abs <= 1e-4; bf16 inputs
max-abs <= 1e-2 and rel-Frobenius <= 2e-3; on o and hT; NaN/Inf fails.
Sweep: T in {1, 37, 64, 65, 200, 4099} x gate lower bound in {-0.05, -1, -5}
x {GDN, KDA} (stratat pull #1296, "The parity discipline"; ROCm/rocm-libraries
PR #11223, "Correctness"), then shape / edge cases, then the five workloads at
full size, every value head.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from chunkwise_gated_delta_gdn_gb300 import gdn, synth
from tests.gpu_util import gpu_heads, kind_of, run_gpu, run_oracle, to_dev
from tests.metrics import assert_close

pytestmark = pytest.mark.gpu


def check(c, x, heads=None, h0=True, chunk=None):
    o, hT = run_gpu(c, x, h0=h0, chunk=chunk)
    o_ref, h_ref = run_oracle(c, x, heads, h0=h0)
    og, hg = gpu_heads(o, hT, heads)
    r1 = assert_close(og, o_ref, kind_of(c), f"{c.name} o")
    r2 = assert_close(hg, h_ref, kind_of(c), f"{c.name} hT")
    return r1, r2


# --------------------------------------------------------------------------
# sweep
# --------------------------------------------------------------------------
@pytest.mark.parametrize("c", synth.sweep_cases(), ids=lambda c: c.name)
def test_sweep(c):
    check(c, synth.make_inputs(c))


# --------------------------------------------------------------------------
# shapes, dtypes and edge cases
# --------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("gate_mode", [0, 1], ids=["gdn", "kda"])
@pytest.mark.parametrize("chunk", [32, 64])
@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64), (128, 128)])
def test_shapes(dtype, gate_mode, chunk, dk, dv):
    c = synth.Case(f"shape_{dk}_{dv}_{chunk}_{gate_mode}", B=1, T=150, H=2, HV=6, dk=dk,
                   dv=dv, chunk=chunk, dtype=dtype, gate_mode=gate_mode,
                   gate_dist="uniform", gate_low=-2.0, h0_std=0.1, seed=3)
    check(c, synth.make_inputs(c))


@pytest.mark.parametrize("gate_mode", [0, 1], ids=["gdn", "kda"])
@pytest.mark.parametrize("chunk", [32, 64])
def test_strong_decay(gate_mode, chunk):
    """Log-gates down to -12 per token.  Within 16 tokens the decay can reach
    e^-180: a factored in-block exponent would leave the fp32 range, so the
    per-key prep must take its exact per-pair path, and cross-chunk state
    contributions vanish."""
    c = synth.Case(f"strong_decay_{gate_mode}_{chunk}", B=1, T=200, H=2, HV=4, dk=128,
                   dv=128, chunk=chunk, dtype=torch.bfloat16, gate_mode=gate_mode,
                   gate_dist="uniform", gate_low=-12.0, h0_std=0.1, seed=11)
    check(c, synth.make_inputs(c))


def test_tiny_fp32_workload():
    c = synth.case("gdn_fp32_t256")
    check(c, synth.make_inputs(c))


@pytest.mark.parametrize("gate_mode", [0, 1])
def test_varlen_with_empty_and_ragged_sequences(gate_mode):
    lengths = [0, 1, 63, 64, 65, 200, 0, 17, 129]
    c = synth.Case("varlen_small", B=1, T=sum(lengths), H=2, HV=4, dk=128, dv=128,
                   chunk=64 if gate_mode == 0 else 32, dtype=torch.bfloat16,
                   gate_mode=gate_mode, gate_dist="uniform", gate_low=-1.0,
                   h0_std=0.1, n_seqs=len(lengths), seed=4)
    x = synth.make_inputs(c, lengths=lengths)
    check(c, x)
    # empty sequences hand back their initial state exactly
    o, hT = run_gpu(c, x)
    for i, L in enumerate(lengths):
        if L == 0:
            assert torch.equal(hT[i].cpu(), x["h0"][i])


def test_batched_rows():
    c = synth.Case("batched", B=3, T=100, H=4, HV=8, dk=128, dv=128, chunk=64,
                   dtype=torch.bfloat16, gate_mode=0, gate_dist="uniform",
                   gate_low=-1.0, h0_std=0.2, seed=5)
    check(c, synth.make_inputs(c))


def test_without_initial_and_final_state():
    c = synth.case("gdn_bf16_t4096", T=300, H=2, HV=6)
    x = synth.make_inputs(c)
    check(c, x, h0=False)
    o, hT = run_gpu(c, x, want_hT=False)
    assert hT is None
    o_ref, _ = run_oracle(c, x)
    og, _ = gpu_heads(o, None)
    assert_close(og, o_ref, "bf16", "o without hT")


def test_zero_tokens():
    c = synth.case("gdn_bf16_t4096", T=0, H=2, HV=4)
    x = synth.make_inputs(c)
    o, hT = run_gpu(c, x)
    assert o.numel() == 0
    assert torch.equal(hT.cpu(), x["h0"])


def test_input_state_is_not_written():
    c = synth.case("gdn_bf16_t4096", T=200, H=2, HV=4)
    x = synth.make_inputs(c)
    d = to_dev(x)
    before = d["h0"].clone()
    gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], chunk=64)
    torch.cuda.synchronize()
    assert torch.equal(before, d["h0"])


def test_continuation_on_device():
    """Partition continuation (logismos issue #46, Sep 10 comment): [0,t) then
    [t,T) with hT fed back as h0 matches one call over [0,T)."""
    c = synth.case("gdn_bf16_t4096", T=333, H=2, HV=4)
    x = synth.make_inputs(c)
    d = to_dev(x)
    o, hT = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], chunk=64)
    t = 130
    sl = lambda a, s: a[:, s].contiguous()
    o1, h1 = gdn.gdn_chunk_fwd(*(sl(d[n], slice(0, t)) for n in ("q", "k", "v", "g", "beta")),
                               d["h0"], chunk=64)
    o2, h2 = gdn.gdn_chunk_fwd(*(sl(d[n], slice(t, None)) for n in ("q", "k", "v", "g", "beta")),
                               h1, chunk=64)
    torch.cuda.synchronize()
    assert_close(torch.cat([o1, o2], 1).cpu(), o.cpu().double(), "bf16", "continued o")
    assert_close(h2.cpu(), hT.cpu().double(), "bf16", "continued hT")


@pytest.mark.parametrize("name, over", [
    ("gdn_bf16_t4096", dict(T=300, H=2, HV=4)),            # bf16 scalar gate
    ("kda_bf16_b2_t8192", dict(T=150, H=2, HV=4)),         # bf16 per-key gate
    ("gdn_fp32_t256", dict(T=200)),                        # fp32
    ("gdn_varlen_t131072", dict(T=700, H=2, HV=4)),        # packed sequences
])
def test_halves_equal_one_call_bitwise(name, over):
    """The prep and scan halves called one after the other (as separate
    entries, on the same workspace) give the bits of the one-call entry:
    they launch the same kernels (split and fused paths sharing one scan
    body are equal bit for bit: ROCm/rocm-libraries PR #11223,
    "Correctness")."""
    c = synth.case(name, **over)
    d = to_dev(synth.make_inputs(c))
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"])
    kw = dict(scale=c.scale, chunk=c.chunk, cu_seqlens=d["cu_seqlens"])
    o1, h1 = gdn.gdn_chunk_fwd(*args, **kw)
    gate_mode = gdn.GDN_GATE_PER_KEY if d["g"].dim() == 4 else gdn.GDN_GATE_SCALAR
    nbytes = gdn.gdn_chunk_fwd_workspace_bytes(
        d["q"].shape[0], d["q"].shape[1], c.H, c.HV, c.dk, c.dv, c.chunk, gate_mode,
        h1.shape[0], gdn._dtype_code(d["q"].dtype))
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    o2 = torch.empty_like(o1)
    h2 = torch.empty_like(h1)
    gdn.gdn_chunk_fwd_prep(*args, workspace=ws, o=o2, hT=h2, **kw)
    gdn.gdn_chunk_fwd_scan(*args, workspace=ws, o=o2, hT=h2, **kw)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(h1, h2)


def test_deterministic():
    c = synth.case("kda_bf16_b2_t8192", T=200, H=2, HV=4)
    x = synth.make_inputs(c)
    a = run_gpu(c, x)
    b = run_gpu(c, x)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_device_flags():
    c = synth.case("gdn_bf16_t4096", T=100, H=2, HV=4)
    x = synth.make_inputs(c)
    d = to_dev(x)
    ws = torch.empty(gdn.gdn_chunk_fwd_workspace_bytes(1, 100, 2, 4, 128, 128, 64, 0, 1, 1),
                     dtype=torch.uint8, device="cuda")
    gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], workspace=ws)
    assert gdn.gdn_read_device_flags(ws) == 0
    g_bad = d["g"].clone()
    g_bad[0, 5, 1] = 0.5
    gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], g_bad, d["beta"], d["h0"], workspace=ws)
    assert gdn.gdn_read_device_flags(ws) & gdn.GDN_FLAG_POSITIVE_GATE
    v_bad = d["v"].clone()
    v_bad[0, 7, 2, 3] = float("inf")
    gdn.gdn_chunk_fwd(d["q"], d["k"], v_bad, d["g"], d["beta"], d["h0"], workspace=ws)
    assert gdn.gdn_read_device_flags(ws) & gdn.GDN_FLAG_NONFINITE
    # the word is cleared by the next call
    gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], workspace=ws)
    assert gdn.gdn_read_device_flags(ws) == 0


def test_bad_seqlens_flagged_not_faulting():
    lengths = [40, 60]
    c = synth.Case("badcu", B=1, T=100, H=2, HV=4, dk=128, dv=128, chunk=64,
                   dtype=torch.bfloat16, gate_mode=0, gate_dist="uniform",
                   gate_low=-1.0, h0_std=0.1, n_seqs=2, seed=6)
    x = to_dev(synth.make_inputs(c, lengths=lengths))
    bad = torch.tensor([0, 70, 50], dtype=torch.int32, device="cuda")  # decreasing
    ws = torch.empty(gdn.gdn_chunk_fwd_workspace_bytes(1, 100, 2, 4, 128, 128, 64, 0, 2, 1),
                     dtype=torch.uint8, device="cuda")
    gdn.gdn_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], cu_seqlens=bad,
                      workspace=ws)
    assert gdn.gdn_read_device_flags(ws) & gdn.GDN_FLAG_BAD_SEQLENS


# --------------------------------------------------------------------------
# the five workloads at full size
# --------------------------------------------------------------------------
def test_workload_gdn_bf16_t4096_all_heads():
    c = synth.case("gdn_bf16_t4096")
    check(c, synth.make_inputs(c))


def test_workload_gdn_bf16_t32768_all_heads():
    c = synth.case("gdn_bf16_t32768")
    check(c, synth.make_inputs(c))


def test_workload_kda_bf16_b2_t8192_all_heads():
    c = synth.case("kda_bf16_b2_t8192")
    check(c, synth.make_inputs(c))


def test_workload_gdn_varlen_t131072_all_heads():
    """All 48 value heads of all 8 packed sequences, o and the per-sequence
    hT (the oracle takes a few seconds on the host cores)."""
    c = synth.case("gdn_varlen_t131072")
    check(c, synth.make_inputs(c))
