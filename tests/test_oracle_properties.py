"""Property checks of the fp64 oracles over randomly drawn shapes (no GPU):
the chunked WY walk, written independently of the token walk, must agree with
it for any chunk size, head grouping, gate range, initial state and packed
length mix (all nonempty chunk cuts, logismos issue #46, Sep 6 comment); and
cutting a sequence anywhere and feeding the state back must change nothing
(partition continuation, same issue)."""
from __future__ import annotations

import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle  # noqa: E402


@st.composite
def problems(draw):
    gate_mode = draw(st.sampled_from([0, 1]))
    H = draw(st.integers(1, 2))
    HV = H * draw(st.integers(1, 3))
    dk = draw(st.integers(1, 9))
    dv = draw(st.integers(1, 9))
    lengths = draw(st.lists(st.integers(0, 40), min_size=1, max_size=4))
    low = draw(st.sampled_from([-6.0, -1.0, -0.05, 0.0]))
    with_h0 = draw(st.booleans())
    seed = draw(st.integers(0, 2 ** 31 - 1))
    r = np.random.default_rng(seed)
    T = sum(lengths)
    unit = lambda x: x / np.maximum(np.linalg.norm(x, axis=-1, keepdims=True), 1e-12)
    q = unit(r.standard_normal((T, H, dk)))
    k = unit(r.standard_normal((T, H, dk)))
    v = r.standard_normal((T, HV, dv))
    g = r.uniform(low, 0.0, (T, HV) if gate_mode == 0 else (T, HV, dk))
    beta = r.uniform(0.0, 1.0, (T, HV))
    n = len(lengths)
    h0 = r.standard_normal((n, HV, dk, dv)) * 0.5 if with_h0 else None
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    return q, k, v, g, beta, h0, cu, gate_mode


@settings(max_examples=80, deadline=None)
@given(problems(), st.integers(1, 50))
def test_chunked_walk_equals_token_walk(p, chunk):
    q, k, v, g, beta, h0, cu, gate_mode = p
    o1, h1 = oracle.token_serial(q, k, v, g, beta, h0, cu, 0.6, gate_mode)
    o2, h2 = oracle.chunked(q, k, v, g, beta, h0, cu, 0.6, gate_mode, chunk=chunk)
    np.testing.assert_allclose(o2, o1, atol=1e-9, rtol=1e-9)
    np.testing.assert_allclose(h2, h1, atol=1e-9, rtol=1e-9)


@settings(max_examples=60, deadline=None)
@given(problems(), st.floats(0.0, 1.0))
def test_continuation_at_any_cut(p, where):
    q, k, v, g, beta, h0, cu, gate_mode = p
    # the first sequence, cut at a fraction `where` of its length
    L = int(cu[1])
    t = int(round(where * L))
    sl = slice(0, L)
    h_first = None if h0 is None else h0[:1]
    o, h = oracle.token_serial(q[sl], k[sl], v[sl], g[sl], beta[sl], h_first, [0, L], 0.6,
                               gate_mode)
    a, b = slice(0, t), slice(t, L)
    oa, ha = oracle.token_serial(q[a], k[a], v[a], g[a], beta[a], h_first, [0, t], 0.6,
                                 gate_mode)
    ob, hb = oracle.token_serial(q[b], k[b], v[b], g[b], beta[b], ha, [0, L - t], 0.6,
                                 gate_mode)
    np.testing.assert_allclose(np.concatenate([oa, ob]), o, atol=1e-12)
    np.testing.assert_allclose(hb, h, atol=1e-12)
