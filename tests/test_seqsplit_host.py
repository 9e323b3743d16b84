"""The host logic of the sequence split (seqsplit.py) on the CPU: how it cuts a
sequence, builds each segment's transfer (M, S_seg) and composes the entering
states.  The two library calls it makes are replaced, inside this test only,
by stand-ins computed by the fp64 oracle (gdn_chunk_fwd) and by a plain
product (gdn_state_combine), so what is checked is the orchestration: the
whole sequence through split_forward must equal one oracle pass over it."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from chunkwise_gated_delta_gdn_gb300 import seqsplit, synth


def _oracle_chunk_fwd(q, k, v, g, beta, h0, *, scale=None, chunk=64, stream=None, **_):
    B, T, H, dk = q.shape
    HV, dv = v.shape[2], v.shape[3]
    scale = dk ** -0.5 if scale is None else scale
    gate_mode = 1 if g.dim() == 4 else 0
    arrs = [x.double().numpy() for x in (q, k, v, g, beta)]
    qq, kk, vv, gg, bb, cu = oracle.pack_batched(*arrs)
    h = None if h0 is None else h0.double().numpy()
    o, hT = oracle.token_serial(qq, kk, vv, gg, bb, h, cu, scale, gate_mode)
    return torch.from_numpy(o.reshape(B, T, HV, dv)), torch.from_numpy(hT)


@pytest.fixture
def cpu_library(monkeypatch):
    monkeypatch.setattr(seqsplit.gdn, "gdn_chunk_fwd", _oracle_chunk_fwd)
    monkeypatch.setattr(seqsplit.gdn, "gdn_state_combine",
                        lambda M, S, Sg: M.double() @ S.double() + Sg.double())


def _one_pass(c, x):
    return _oracle_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], scale=c.scale)


@pytest.mark.parametrize("name, over", [
    ("gdn_fp32_t256", dict(T=90)),
    ("kda_bf16_b2_t8192", dict(T=50, H=1, HV=2, dk=64, dv=64)),
    ("gdn_bf16_t4096", dict(T=70, H=1, HV=3, dk=64, dv=64)),
])
@pytest.mark.parametrize("cuts", [[30], [1, 2, 3], [45, 45, 10], [-5, 0, 20, 999], []])
def test_split_forward_equals_one_pass(cpu_library, name, over, cuts):
    """Cuts are sorted, those outside (0, T) are dropped, and a repeated cut
    makes an empty segment that must pass its entering state through."""
    c = synth.case(name, **over)
    x = synth.make_inputs(c)
    x = {kk: (vv.float() if torch.is_tensor(vv) and vv.is_floating_point() else vv)
         for kk, vv in x.items()}
    o, hT = seqsplit.split_forward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], cuts,
                                   scale=c.scale, chunk=c.chunk)
    o_ref, h_ref = _one_pass(c, x)
    np.testing.assert_allclose(o.numpy(), o_ref.numpy(), atol=1e-9)
    np.testing.assert_allclose(hT.numpy(), h_ref.numpy(), atol=1e-9)


def test_segment_transfer_shapes_and_identity(cpu_library):
    """M is dk x dk per (row, value head) and S_seg dk x dv; over a segment
    whose gates are 0 and betas 0 every token map is the identity, so M = I
    and S_seg = 0."""
    c = synth.case("gdn_fp32_t256", T=12, H=1, HV=2, dk=64, dv=64)
    x = synth.make_inputs(c)
    x["g"] = torch.zeros_like(x["g"])
    x["beta"] = torch.zeros_like(x["beta"])
    M, S_seg = seqsplit.segment_transfer(x["q"], x["k"], x["v"], x["g"], x["beta"])
    assert M.shape == (1, 2, 64, 64) and S_seg.shape == (1, 2, 64, 64)
    np.testing.assert_allclose(M.numpy(), np.broadcast_to(np.eye(64), (1, 2, 64, 64)),
                               atol=1e-12)
    assert float(S_seg.abs().max()) == 0.0


def test_compose_orders_the_transfers():
    gen = torch.Generator().manual_seed(2)
    Ms = [torch.randn((1, 1, 3, 3), generator=gen, dtype=torch.float64) for _ in range(3)]
    Ss = [torch.randn((1, 1, 3, 2), generator=gen, dtype=torch.float64) for _ in range(3)]
    starts = seqsplit.compose(list(zip(Ms, Ss)), None, combine=lambda M, S, Sg: M @ S + Sg)
    assert len(starts) == 3 and float(starts[0].abs().max()) == 0.0
    assert torch.allclose(starts[1], Ss[0])
    assert torch.allclose(starts[2], Ms[1] @ Ss[0] + Ss[1])
