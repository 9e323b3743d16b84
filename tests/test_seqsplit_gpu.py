"""GPU parity of the sequence split with a state-transfer exchange: a
sequence cut into segments, each segment's transfer (M, S_seg) composed with
gdn_state_combine, then every segment run from its true entering state, must
match the fp64 token-serial oracle over the whole sequence."""
from __future__ import annotations

import pytest
import torch

from chunkwise_gated_delta_gdn_gb300 import gdn, seqsplit, synth
from tests.gpu_util import gpu_heads, kind_of, run_oracle, to_dev
from tests.metrics import assert_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name, over", [
    ("gdn_bf16_t4096", dict(T=600, H=2, HV=6)),
    ("kda_bf16_b2_t8192", dict(B=1, T=600, H=2, HV=4)),
    ("gdn_fp32_t256", dict(T=600)),
])
@pytest.mark.parametrize("cuts", [[256], [64, 300, 511], [1, 599]])
def test_split_matches_one_pass(name, over, cuts):
    c = synth.case(name, **over)
    x = synth.make_inputs(c)
    d = to_dev(x)
    o, hT = seqsplit.split_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], cuts,
                                   scale=c.scale, chunk=c.chunk)
    torch.cuda.synchronize()
    o_ref, h_ref = run_oracle(c, x)
    og, hg = gpu_heads(o, hT)
    assert_close(og, o_ref, kind_of(c), f"{name} split {cuts} o")
    assert_close(hg, h_ref, kind_of(c), f"{name} split {cuts} hT")


def test_state_combine_against_torch():
    g = torch.Generator().manual_seed(3)
    M = torch.randn((2, 3, 128, 128), generator=g) * 0.1
    S = torch.randn((2, 3, 128, 64), generator=g)
    Sg = torch.randn((2, 3, 128, 64), generator=g)
    out = gdn.gdn_state_combine(M.cuda(), S.cuda(), Sg.cuda())
    Sg_dev = Sg.cuda()
    gdn.gdn_state_combine(M.cuda(), S.cuda(), Sg_dev, out=Sg_dev)  # in place
    torch.cuda.synchronize()
    ref = (M.double() @ S.double() + Sg.double())
    assert (out.cpu().double() - ref).abs().max() < 1e-4
    assert torch.equal(out, Sg_dev)
