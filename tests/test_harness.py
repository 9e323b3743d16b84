"""Host-side harness checks (no GPU): the tolerance comparator and its negative
control, and the seeded input generator."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from chunkwise_gated_delta_gdn_gb300 import synth
from tests.metrics import TOL, compare


@pytest.mark.parametrize("kind", ["bf16", "f32"])
def test_negative_control_fails(kind):
    """A result perturbed by 2.5x the max-abs bound in one element must FAIL
    (the +2.5 B negative control of stratat pull #1296, "The parity
    discipline"); the unperturbed result must pass."""
    c = synth.case("gdn_fp32_t256", T=64, HV=2, H=2)
    x = synth.make_inputs(c)
    o, hT = oracle.token_serial(x["q"][0], x["k"][0], x["v"][0], x["g"][0],
                                x["beta"][0], None, [0, 64], c.scale, 0)
    assert compare(o, o, kind)["ok"]
    bad = o.copy()
    bad[7, 1, 3] += 2.5 * TOL[kind]["max_abs"]
    assert not compare(bad, o, kind)["ok"]
    nan = o.copy()
    nan[0, 0, 0] = np.nan
    assert not compare(nan, o, kind)["ok"]


def test_rel_frobenius_bound_is_enforced():
    r = np.random.default_rng(0)
    ref = r.uniform(-1, 1, (100, 4, 8))
    got = ref * (1 + 3e-3)  # every element within max-abs, 3e-3 relative
    res = compare(got, ref, "bf16")
    assert res["max_abs"] < 1e-2 and res["rel_frob"] > 2e-3 and not res["ok"]


def test_bf16_output_rounding_fits_the_budget():
    """Rounding an exact result to bf16 alone must stay inside the bf16
    contract, otherwise no kernel could pass it.  This holds for outputs of
    magnitude below 4 (half an ulp of bf16 is 2^-7 on [2, 4) but 2^-6 on
    [4, 8), above the 1e-2 max-abs bound); with unit-norm q, k and
    scale = dk^-0.5 the outputs of the workloads stay far below that."""
    r = np.random.default_rng(1)
    ref = 0.5 * r.standard_normal((4096, 8, 16))
    got = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
    res = compare(got, ref, "bf16")
    assert res["ok"], res


def test_generator_is_deterministic_and_shaped():
    c = synth.case("kda_bf16_b2_t8192", T=96)
    a = synth.make_inputs(c)
    b = synth.make_inputs(c)
    for key in ("q", "k", "v", "g", "beta"):
        assert torch.equal(a[key], b[key])
    assert a["q"].shape == (2, 96, 32, 128) and a["q"].dtype == torch.bfloat16
    assert a["g"].shape == (2, 96, 32, 128) and a["g"].dtype == torch.float32
    assert float(a["g"].max()) <= 0.0 and float(a["g"].min()) >= -5.0
    n = a["k"].float().norm(dim=-1)
    assert torch.allclose(n, torch.ones_like(n), atol=1e-2)
    assert float(a["beta"].min()) > 0 and float(a["beta"].max()) < 1


def test_generator_varlen():
    c = synth.case("gdn_varlen_t131072", T=1000)
    x = synth.make_inputs(c)
    cu = x["cu_seqlens"].tolist()
    assert cu[0] == 0 and cu[-1] == 1000 and len(cu) == 9
    assert all(b - a >= 1 for a, b in zip(cu, cu[1:]))
    assert x["h0"].shape == (8, 48, 128, 128)


def test_softplus_gates_clamped():
    c = synth.case("gdn_fp32_t256")
    x = synth.make_inputs(c)
    assert float(x["g"].min()) >= -5.0 and float(x["g"].max()) <= 0.0
    assert x["q"].dtype == torch.float32 and x["h0"] is None
