"""gdn_chunk_fwd_lockstep: prep and scan in one cooperative launch, in lockstep
(the fused composition of ROCm/rocm-libraries PR #11223, "Summary").  It runs
the same per-chunk and per-block device code as the split kernels, so its
results must equal gdn_chunk_fwd's bit for bit (split and fused paths sharing
one scan body are bitwise equal: PR #11223, "Correctness"); one case is also
checked against the fp64 oracle."""
from __future__ import annotations

import pytest
import torch

from chunkwise_gated_delta_gdn_gb300 import gdn, synth
from tests.gpu_util import gpu_heads, kind_of, run_oracle, to_dev
from tests.metrics import assert_close

pytestmark = pytest.mark.gpu


def both(c, x):
    d = to_dev(x)
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"])
    kw = dict(scale=c.scale, chunk=c.chunk, cu_seqlens=d["cu_seqlens"])
    o1, h1 = gdn.gdn_chunk_fwd(*args, **kw)
    o2, h2 = gdn.gdn_chunk_fwd_lockstep(*args, **kw)
    torch.cuda.synchronize()
    return (o1, h1), (o2, h2)


CASES = [
    synth.case("gdn_bf16_t4096", T=1000, H=4, HV=12),
    synth.case("gdn_bf16_t4096", T=37, H=2, HV=6),
    synth.case("gdn_bf16_t4096", T=300, H=2, HV=4, dk=64, dv=64, chunk=32),
    synth.case("gdn_bf16_t4096", T=200, H=2, HV=4, dk=64, dv=128),
    # every prep warpgroup runs several units one after another
    synth.case("gdn_bf16_t4096", T=2048),
    synth.case("gdn_bf16_t4096", T=4096),
]


@pytest.mark.parametrize("c", CASES, ids=lambda c: f"T{c.T}_H{c.H}_HV{c.HV}_dk{c.dk}_dv{c.dv}_C{c.chunk}")
def test_lockstep_equals_split_bitwise(c):
    (o1, h1), (o2, h2) = both(c, synth.make_inputs(c))
    assert torch.equal(o1, o2) and torch.equal(h1, h2)


def test_lockstep_packed_with_empty_and_ragged_sequences():
    lengths = [0, 1, 63, 64, 65, 200, 0, 17, 129]
    c = synth.Case("varlen_lock", B=1, T=sum(lengths), H=2, HV=4, dk=128, dv=128, chunk=64,
                   dtype=torch.bfloat16, gate_mode=0, gate_dist="uniform", gate_low=-1.0,
                   h0_std=0.1, n_seqs=len(lengths), seed=4)
    (o1, h1), (o2, h2) = both(c, synth.make_inputs(c, lengths=lengths))
    assert torch.equal(o1, o2) and torch.equal(h1, h2)


def test_lockstep_bench_workload_bitwise():
    c = synth.case("gdn_bf16_t32768")
    (o1, h1), (o2, h2) = both(c, synth.make_inputs(c))
    assert torch.equal(o1, o2) and torch.equal(h1, h2)


def test_lockstep_matches_the_oracle_and_reports_no_flags():
    c = CASES[0]
    x = synth.make_inputs(c)
    d = to_dev(x)
    ws = torch.empty(gdn.gdn_chunk_fwd_workspace_bytes(1, c.T, c.H, c.HV, c.dk, c.dv, c.chunk,
                                                       0, 1, gdn.GDN_BF16),
                     dtype=torch.uint8, device="cuda")
    o, hT = gdn.gdn_chunk_fwd_lockstep(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"],
                                       scale=c.scale, chunk=c.chunk, workspace=ws)
    torch.cuda.synchronize()
    assert gdn.gdn_read_device_flags(ws) == 0
    o_ref, h_ref = run_oracle(c, x)
    og, hg = gpu_heads(o, hT)
    assert_close(og, o_ref, kind_of(c), "lockstep o")
    assert_close(hg, h_ref, kind_of(c), "lockstep hT")


def test_lockstep_refuses_a_grid_with_no_room_for_the_prep():
    """Sequences x HV x dv/64 scan blocks beyond the SMs of the GPU: refused on
    the host before any launch."""
    c = synth.case("gdn_bf16_t4096", T=64, H=1, HV=200)
    d = to_dev(synth.make_inputs(c))
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_chunk_fwd_lockstep(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"],
                                   scale=c.scale, chunk=c.chunk)
    assert e.value.status == gdn.GDN_ERR_UNSUPPORTED
