"""GPU parity of the operations either side of the recurrence (causal
depthwise convolution with history, q/k L2 norm, gated RMS output norm)
against the fp64 oracle in oracle/prepost.py, through the C ABI.

Tolerance, derived from the arithmetic: each output is accumulated in fp32
and rounded once to the output dtype, so for bf16 outputs every element must
be within 2^-8 |ref| + 1e-5 (twice the half-ulp of bf16 rounding, plus fp32
accumulation) and the relative Frobenius error within 2e-3; fp32 outputs
within 1e-5 |ref| + 1e-5.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from chunkwise_gated_delta_gdn_gb300 import gdn
from oracle import prepost

pytestmark = pytest.mark.gpu


def check(got, ref, dtype, what):
    got = got.detach().double().cpu().numpy() if torch.is_tensor(got) else np.asarray(got)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), what
    d = np.abs(got - ref)
    if dtype == torch.bfloat16:
        bound = 2.0 ** -8 * np.abs(ref) + 1e-5
        rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
        assert rel <= 2e-3, (what, rel)
    else:
        bound = 1e-5 * np.abs(ref) + 1e-5
    bad = d > bound
    assert not bad.any(), (what, float(d.max()), int(bad.sum()))


def gen(seed):
    g = torch.Generator()
    g.manual_seed(seed)
    return g


def conv_inputs(lengths, D, W, dtype, seed, hist=True, bias=True):
    g = gen(seed)
    T = sum(lengths)
    x = torch.randn((1, T, D), generator=g).to(dtype)
    w = (torch.rand((D, W), generator=g) * 2 - 1) / W ** 0.5
    b = torch.randn(D, generator=g) * 0.1 if bias else None
    h0 = torch.randn((len(lengths), D, W - 1), generator=g) if hist else None
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
    return x, w, b, h0, cu


def run_conv(x, w, b, h0, cu, act, hT_in_place=False):
    d = lambda t: t.cuda() if t is not None else None
    h = d(h0)
    kw = dict(activation=act, cu_seqlens=d(cu))
    if hT_in_place:
        h = h.clone()
        kw["hT"] = h
    y, hT = gdn.gdn_causal_conv1d_fwd(d(x), d(w), d(b), h, **kw)
    torch.cuda.synchronize()
    return y, hT


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("act", [gdn.GDN_ACT_NONE, gdn.GDN_ACT_SILU], ids=["id", "silu"])
def test_conv_varlen(dtype, W, act):
    lengths = [0, 1, 2, 31, 32, 33, 100, 0, 5]
    x, w, b, h0, cu = conv_inputs(lengths, 264, W, dtype, seed=W + 10 * act)
    y, hT = run_conv(x, w, b, h0, cu, act)
    y_ref, h_ref = prepost.causal_conv1d(x[0], w, b, h0 if W > 1 else None, cu.tolist(), act)
    check(y[0], y_ref, dtype, "y")
    if W > 1:
        check(hT, h_ref, torch.float32, "hT")  # raw inputs: exact up to the fp32 copy
        assert torch.equal(hT.cpu()[0], h0[0]) and torch.equal(hT.cpu()[7], h0[7])


def test_conv_batched_without_history_or_bias():
    g = gen(3)
    x = torch.randn((3, 70, 1024), generator=g).to(torch.bfloat16)
    w = torch.randn((1024, 4), generator=g) * 0.5
    y, hT = gdn.gdn_causal_conv1d_fwd(x.cuda(), w.cuda(), activation=gdn.GDN_ACT_SILU)
    torch.cuda.synchronize()
    cu = [0, 70, 140, 210]
    y_ref, h_ref = prepost.causal_conv1d(x.reshape(210, 1024), w, None, None, cu, 1)
    check(y.reshape(210, 1024), y_ref, torch.bfloat16, "y")
    check(hT, h_ref, torch.float32, "hT")


def test_conv_in_place_history_and_decode_steps():
    """Eight one-token steps updating the history in place reproduce one call
    over the eight tokens (the staged one-token step)."""
    D, W, L = 512, 4, 8
    x, w, b, h0, _ = conv_inputs([L] * 3, D, W, torch.bfloat16, seed=5)
    xs = x.reshape(3, L, D)
    h = h0.cuda().clone()
    ys = []
    for t in range(L):
        y, _ = gdn.gdn_causal_conv1d_fwd(xs[:, t:t + 1].contiguous().cuda(), w.cuda(), b.cuda(), h,
                                         hT=h, activation=gdn.GDN_ACT_SILU)
        ys.append(y)
    torch.cuda.synchronize()
    y = torch.cat(ys, 1)
    y_ref, h_ref = prepost.causal_conv1d(x[0], w, b, h0, [0, L, 2 * L, 3 * L], 1)
    check(y.reshape(3 * L, D), y_ref, torch.bfloat16, "stepped y")
    check(h, h_ref, torch.float32, "stepped history")


def test_conv_beyond_grid_y_extent():
    """More token tiles (128 tokens each) than a grid's y extent of 65535: a
    block takes every 65535th tile.  Two packed sequences; windows at the
    start, across the sequence boundary, past the 65535th tile and at the end
    against the oracle, and both final histories (raw inputs, exact)."""
    D, W = 8, 4
    T = 65535 * 128 + 1000
    cut = 4_000_000
    x, w, b, h0, cu = conv_inputs([cut, T - cut], D, W, torch.bfloat16, seed=11)
    y, hT = run_conv(x, w, b, h0, cu, gdn.GDN_ACT_SILU)
    y, xs = y[0].cpu(), x[0]
    bounds = cu.tolist()
    for a0, a1 in ((0, 300), (cut - 150, cut + 150), (65535 * 128 - 100, 65535 * 128 + 400), (T - 300, T)):
        parts, hists, cuts = [], [], [0]
        for n in range(len(bounds) - 1):
            s, e = bounds[n], bounds[n + 1]
            lo, hi = max(a0, s), min(a1, e)
            if lo >= hi:
                continue
            ext = torch.cat([h0[n], xs[s:lo].float().T], 1) if lo - s < W - 1 else xs[lo - (W - 1):lo].float().T
            parts.append(xs[lo:hi])
            hists.append(ext[:, ext.shape[1] - (W - 1):])
            cuts.append(cuts[-1] + hi - lo)
        y_ref, _ = prepost.causal_conv1d(torch.cat(parts), w, b, torch.stack(hists), cuts, 1)
        check(y[a0:a1], y_ref, torch.bfloat16, f"y[{a0}:{a1}]")
    h_ref = torch.stack([xs[e - (W - 1):e].float().T for e in bounds[1:]])
    assert torch.equal(hT.cpu(), h_ref)


def test_conv_bad_seqlens_flagged():
    x, w, b, h0, _ = conv_inputs([10, 10], 64, 4, torch.bfloat16, seed=9)
    bad = torch.tensor([0, 15, 12], dtype=torch.int32).cuda()
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_causal_conv1d_fwd(x.cuda(), w.cuda(), b.cuda(), h0.cuda(), cu_seqlens=bad, flags=flags)
    assert gdn.gdn_read_device_flags(flags) & gdn.GDN_FLAG_BAD_SEQLENS


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("dim", [64, 128, 256])
def test_l2norm(dtype, dim):
    g = gen(dim)
    x = (torch.randn((3, 77, 5, dim), generator=g) * 3).to(dtype)
    y = gdn.gdn_l2norm_fwd(x.cuda(), eps=1e-6)
    x2 = x.cuda().clone()
    gdn.gdn_l2norm_fwd(x2, eps=1e-6, y=x2)  # in place
    torch.cuda.synchronize()
    ref = prepost.l2norm(x, 1e-6)
    check(y, ref, dtype, "l2norm")
    assert torch.equal(x2, y)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("dim", [64, 128, 256])
@pytest.mark.parametrize("gated", [False, True])
def test_rmsnorm_gated(dtype, dim, gated):
    g = gen(dim + gated)
    x = (torch.randn((200, 3, dim), generator=g) * 2).to(dtype)
    z = torch.randn((200, 3, dim), generator=g).to(dtype) if gated else None
    wt = torch.rand(dim, generator=g) + 0.5
    y = gdn.gdn_rmsnorm_gated_fwd(x.cuda(), wt.cuda(), z.cuda() if gated else None, eps=1e-6)
    torch.cuda.synchronize()
    check(y, prepost.rmsnorm_gated(x, wt, z, 1e-6), dtype, "rmsnorm")


@pytest.mark.parametrize("dim", [64, 128, 256])
def test_rmsnorm_gated_odd_row_counts(dim):
    """The gated RMS norm gives two rows side by side to each warp: with an odd
    row count one half of the last warp has no row (zeros in, nothing stored)."""
    g = gen(50 + dim)
    wt = torch.rand(dim, generator=g) + 0.5
    for rows in (1, 3, 17, 601):
        x = (torch.randn((rows, dim), generator=g) * 2).to(torch.bfloat16)
        z = torch.randn((rows, dim), generator=g).to(torch.bfloat16)
        y = torch.full((rows + 1, dim), 7.0, dtype=torch.bfloat16, device="cuda")
        gdn.gdn_rmsnorm_gated_fwd(x.cuda(), wt.cuda(), z.cuda(), eps=1e-6, y=y[:rows])
        torch.cuda.synchronize()
        # every element within one bf16 rounding of the exact value (plus fp32
        # accumulation); a flat Frobenius bound is a statistic that a handful
        # of rows can exceed even when correctly rounded, so the Frobenius error
        # is held to that of rounding the oracle's own output instead
        ref = np.asarray(prepost.rmsnorm_gated(x, wt, z, 1e-6), dtype=np.float64)
        got = y[:rows].double().cpu().numpy()
        assert np.isfinite(got).all()
        assert (np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5).all(), f"rows={rows}"
        rounded = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
        fro = lambda a: np.linalg.norm(a - ref) / np.linalg.norm(ref)
        assert fro(got) <= fro(rounded) + 1e-4, (rows, fro(got), fro(rounded))
        assert torch.all(y[rows] == 7.0), "a row past the end was written"


def test_norms_on_empty_input():
    x = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    assert gdn.gdn_l2norm_fwd(x).numel() == 0
    assert gdn.gdn_rmsnorm_gated_fwd(x, torch.ones(128, device="cuda")).numel() == 0
