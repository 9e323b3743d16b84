"""Seeded random parity: many small problems with shapes, dtypes, gates,
head groupings, chunk sizes and packed-sequence length mixes drawn at random
(fixed seeds, so every run checks the same cases), each through the CUDA path
and the fp64 token-serial oracle under the tolerances of tests/metrics.py."""
from __future__ import annotations

import random

import pytest
import torch

from chunkwise_gated_delta_gdn_gb300 import gdn, synth
from tests.gpu_util import gpu_heads, kind_of, run_oracle, to_dev
from tests.metrics import assert_close

pytestmark = pytest.mark.gpu


def draw_case(seed: int):
    rnd = random.Random(seed)
    gate_mode = rnd.choice([0, 1])
    dtype = rnd.choice([torch.bfloat16, torch.bfloat16, torch.float32])
    H = rnd.choice([1, 2, 3])
    HV = H * rnd.choice([1, 2, 3])
    dk = rnd.choice([64, 128])
    dv = rnd.choice([64, 128])
    chunk = rnd.choice([32, 64]) if gate_mode == 0 else 32
    n = rnd.randint(1, 6)
    lengths = [rnd.choice([0, 1, rnd.randint(1, 40), rnd.randint(30, 300)]) for _ in range(n)]
    if sum(lengths) == 0:
        lengths[-1] = 5
    c = synth.Case(f"rand{seed}", B=1, T=sum(lengths), H=H, HV=HV, dk=dk, dv=dv, chunk=chunk,
                   dtype=dtype, gate_mode=gate_mode, gate_dist="uniform",
                   gate_low=rnd.choice([-0.05, -1.0, -5.0]),
                   h0_std=rnd.choice([None, 0.1]), n_seqs=n, seed=seed)
    return c, lengths


@pytest.mark.parametrize("seed", range(24))
def test_random_chunked(seed):
    c, lengths = draw_case(seed)
    x = synth.make_inputs(c, lengths=lengths)
    d = to_dev(x)
    o, hT = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], scale=c.scale,
                              chunk=c.chunk, cu_seqlens=d["cu_seqlens"])
    torch.cuda.synchronize()
    o_ref, h_ref = run_oracle(c, x)
    og, hg = gpu_heads(o, hT)
    assert_close(og, o_ref, kind_of(c), f"{c} o")
    assert_close(hg, h_ref, kind_of(c), f"{c} hT")


@pytest.mark.parametrize("seed", range(100, 112))
def test_random_recurrent(seed):
    c, lengths = draw_case(seed)
    x = synth.make_inputs(c, lengths=lengths)
    d = to_dev(x)
    o, hT = gdn.gdn_recurrent_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"],
                                  scale=c.scale, cu_seqlens=d["cu_seqlens"])
    torch.cuda.synchronize()
    o_ref, h_ref = run_oracle(c, x)
    og, hg = gpu_heads(o, hT)
    assert_close(og, o_ref, kind_of(c), f"{c} o")
    assert_close(hg, h_ref, kind_of(c), f"{c} hT")


@pytest.mark.parametrize("seed", range(200, 216))
def test_random_lockstep_bitwise(seed):
    """The lockstep launch on random bf16 scalar-gate shapes (its head start
    sized to each one) equals the split kernels bit for bit."""
    c, lengths = draw_case(seed)
    c = synth.Case(c.name, B=1, T=c.T, H=c.H, HV=c.HV, dk=c.dk, dv=c.dv, chunk=c.chunk,
                   dtype=torch.bfloat16, gate_mode=0, gate_dist="uniform", gate_low=c.gate_low,
                   h0_std=c.h0_std, n_seqs=c.n_seqs, seed=c.seed)
    x = synth.make_inputs(c, lengths=lengths)
    d = to_dev(x)
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"])
    o, hT = gdn.gdn_chunk_fwd(*args, scale=c.scale, chunk=c.chunk, cu_seqlens=d["cu_seqlens"])
    o2, h2 = gdn.gdn_chunk_fwd_lockstep(*args, scale=c.scale, chunk=c.chunk,
                                        cu_seqlens=d["cu_seqlens"])
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(hT, h2), c.name


@pytest.mark.parametrize("seed", range(300, 312))
def test_random_per_key_chunk64(seed):
    """The per-key gate (KDA) at chunk 64, which the draws above never pick:
    the same shapes, dtypes and packed length mixes, against the oracle."""
    c, lengths = draw_case(seed)
    c = synth.Case(f"{c.name}_kda64", B=1, T=c.T, H=c.H, HV=c.HV, dk=c.dk, dv=c.dv, chunk=64,
                   dtype=c.dtype, gate_mode=1, gate_dist="uniform", gate_low=c.gate_low,
                   h0_std=c.h0_std, n_seqs=c.n_seqs, seed=c.seed)
    x = synth.make_inputs(c, lengths=lengths)
    d = to_dev(x)
    o, hT = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], scale=c.scale,
                              chunk=c.chunk, cu_seqlens=d["cu_seqlens"])
    torch.cuda.synchronize()
    o_ref, h_ref = run_oracle(c, x)
    og, hg = gpu_heads(o, hT)
    assert_close(og, o_ref, kind_of(c), f"{c} o")
    assert_close(hg, h_ref, kind_of(c), f"{c} hT")
