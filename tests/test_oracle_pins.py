"""Pins of the fp64 oracle to things other than itself (no GPU needed).

Each test fixes the oracle against a closed form, a hand-worked example, an
invariant of the mathematics, or a linear-algebra library routine, chosen so
that a plausible mistake (dropped term, wrong sign or index, transposed state,
wrong decay order) fails at least one of them -- which the planted-mistake
tests at the bottom check directly.

The recurrence (the gated delta rule named by stratat pull #1296, "What this
is"; walked token by token as in ROCm/rocm-libraries PR #11223,
"Correctness"): S_t = a_t S_{t-1} + beta_t k_t (v_t - a_t S_{t-1}^T k_t)^T,
o_t = scale S_t^T q_t, K-first state (logismos issue #46).
"""
from __future__ import annotations

import json
import os

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
RNG = np.random.default_rng(1234)


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def rand_case(T, H=2, HV=4, dk=8, dv=6, gate_mode=0, low=-1.0, h0=True,
              n_seqs=1, seed=0):
    r = np.random.default_rng(seed)
    q = _unit(r.standard_normal((T, H, dk)))
    k = _unit(r.standard_normal((T, H, dk)))
    v = r.standard_normal((T, HV, dv))
    gs = (T, HV) if gate_mode == 0 else (T, HV, dk)
    g = r.uniform(low, 0.0, gs)
    beta = 1.0 / (1.0 + np.exp(-r.standard_normal((T, HV))))
    h = r.standard_normal((n_seqs, HV, dk, dv)) * 0.3 if h0 else None
    return q, k, v, g, beta, h


def run(q, k, v, g, beta, h0, cu=None, scale=0.7, gate_mode=0, fn=None):
    if cu is None:
        cu = [0, q.shape[0]]
    fn = fn or oracle.token_serial
    return fn(q, k, v, g, beta, h0, cu, scale, gate_mode)


# --------------------------------------------------------------------------
# hand-worked examples
# --------------------------------------------------------------------------
def _golden_cases():
    with open(os.path.join(HERE, "golden", "hand_worked.json")) as f:
        return json.load(f)["cases"]


def _golden_inputs(c):
    q = np.array(c["q"], dtype=np.float64)
    k = np.array(c["k"], dtype=np.float64)
    v = np.array(c["v"], dtype=np.float64)
    g = np.log(np.array(c["alpha"], dtype=np.float64))
    beta = np.array(c["beta"], dtype=np.float64)
    h0 = np.array(c["h0"], dtype=np.float64)
    return q, k, v, g, beta, h0


@pytest.mark.parametrize("c", _golden_cases(), ids=lambda c: c["name"])
@pytest.mark.parametrize("which", ["token_serial", "chunked"])
def test_hand_worked(c, which):
    q, k, v, g, beta, h0 = _golden_inputs(c)
    T = q.shape[0]
    if which == "token_serial":
        o, hT = oracle.token_serial(q, k, v, g, beta, h0, [0, T], c["scale"],
                                    c["gate_mode"])
    else:
        o, hT = oracle.chunked(q, k, v, g, beta, h0, [0, T], c["scale"],
                               c["gate_mode"], chunk=2)
    np.testing.assert_allclose(o, np.array(c["o"]), atol=1e-12)
    np.testing.assert_allclose(hT, np.array(c["hT"]), atol=1e-12)


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------
@pytest.mark.parametrize("gate_mode", [0, 1])
def test_single_token_zero_state(gate_mode):
    """T=1, h0=0: o = scale*beta*(q.k)*v and hT = beta k v^T."""
    q, k, v, g, beta, _ = rand_case(1, gate_mode=gate_mode, seed=1)
    scale = 0.37
    o, hT = run(q, k, v, g, beta, None, scale=scale, gate_mode=gate_mode)
    for hv in range(4):
        hq = hv // 2
        want_o = scale * beta[0, hv] * (q[0, hq] @ k[0, hq]) * v[0, hv]
        want_h = beta[0, hv] * np.outer(k[0, hq], v[0, hv])
        np.testing.assert_allclose(o[0, hv], want_o, atol=1e-13)
        np.testing.assert_allclose(hT[0, hv], want_h, atol=1e-13)


@pytest.mark.parametrize("gate_mode", [0, 1])
def test_single_token_with_state(gate_mode):
    """T=1, h0 != 0: hT = A h0 + beta k (v - (A h0)^T k)^T, o = scale hT^T q,
    with A = a I (GDN) or diag(a) (KDA)."""
    q, k, v, g, beta, h0 = rand_case(1, gate_mode=gate_mode, seed=2)
    scale = 0.5
    o, hT = run(q, k, v, g, beta, h0, scale=scale, gate_mode=gate_mode)
    for hv in range(4):
        hq = hv // 2
        a = np.exp(g[0, hv]) * np.ones(8) if gate_mode == 0 else np.exp(g[0, hv])
        Sd = a[:, None] * h0[0, hv]
        want_h = Sd + beta[0, hv] * np.outer(k[0, hq], v[0, hv] - Sd.T @ k[0, hq])
        np.testing.assert_allclose(hT[0, hv], want_h, atol=1e-13)
        np.testing.assert_allclose(o[0, hv], scale * want_h.T @ q[0, hq], atol=1e-13)


@pytest.mark.parametrize("gate_mode", [0, 1])
def test_beta_zero_only_decays(gate_mode):
    """beta = 0: hT = exp(sum g) h0 (per key row for KDA) and
    o_t = scale (exp(b_t) h0)^T q_t with b_t the cumulative log-gate."""
    T = 23
    q, k, v, g, beta, h0 = rand_case(T, gate_mode=gate_mode, seed=3)
    beta = np.zeros_like(beta)
    scale = 0.9
    o, hT = run(q, k, v, g, beta, h0, scale=scale, gate_mode=gate_mode)
    b = np.cumsum(g, axis=0)
    for hv in range(4):
        hq = hv // 2
        for t in range(T):
            dec = np.exp(b[t, hv]) * (np.ones(8) if gate_mode == 0 else 1.0)
            St = dec[:, None] * h0[0, hv]
            np.testing.assert_allclose(o[t, hv], scale * St.T @ q[t, hq], atol=1e-13)
        dec = np.exp(b[-1, hv]) * (np.ones(8) if gate_mode == 0 else 1.0)
        np.testing.assert_allclose(hT[0, hv], dec[:, None] * h0[0, hv], atol=1e-13)


def test_orthonormal_keys_exact_recall():
    """a = 1, beta = 1, orthonormal keys, h0 = 0: S_T^T k_j = v_j for every
    written key; writing the same key twice keeps only the last value."""
    dk, dv, T = 16, 5, 12
    r = np.random.default_rng(5)
    Qm, _ = np.linalg.qr(r.standard_normal((dk, dk)))
    keys = Qm[:T]  # orthonormal rows
    k = keys[:, None, :]
    v = r.standard_normal((T, 1, dv))
    q = k.copy()
    g = np.zeros((T, 1))
    beta = np.ones((T, 1))
    o, hT = oracle.token_serial(q, k, v, g, beta, None, [0, T], 1.0, 0)
    S = hT[0, 0]
    for j in range(T):
        np.testing.assert_allclose(S.T @ keys[j], v[j, 0], atol=1e-12)
        # reading with q = k_t right after writing it returns v_t
        np.testing.assert_allclose(o[j, 0], v[j, 0], atol=1e-12)
    # overwrite key 3 with a new value: recall returns the new value only
    k2 = np.concatenate([k, k[3:4]], axis=0)
    v_new = r.standard_normal((1, 1, dv))
    v2 = np.concatenate([v, v_new], axis=0)
    o2, hT2 = oracle.token_serial(k2, k2, v2, np.zeros((T + 1, 1)),
                                  np.ones((T + 1, 1)), None, [0, T + 1], 1.0, 0)
    np.testing.assert_allclose(hT2[0, 0].T @ keys[3], v_new[0, 0], atol=1e-12)
    np.testing.assert_allclose(hT2[0, 0].T @ keys[4], v[4, 0], atol=1e-12)


def test_scalar_state_closed_form():
    """dk = dv = 1: s_t = a_t s_{t-1} (1 - beta_t k_t^2) + beta_t k_t v_t and
    o_t = scale s_t q_t (the recurrence collapses to one scalar)."""
    T = 40
    r = np.random.default_rng(6)
    q = r.standard_normal((T, 1, 1))
    k = r.uniform(-1, 1, (T, 1, 1))
    v = r.standard_normal((T, 1, 1))
    g = r.uniform(-2, 0, (T, 1))
    beta = r.uniform(0, 1, (T, 1))
    h0 = np.array([[[[0.8]]]])
    o, hT = oracle.token_serial(q, k, v, g, beta, h0, [0, T], 1.3, 0)
    s = 0.8
    for t in range(T):
        a = np.exp(g[t, 0])
        kk = k[t, 0, 0]
        s = a * s * (1.0 - beta[t, 0] * kk * kk) + beta[t, 0] * kk * v[t, 0, 0]
        assert abs(o[t, 0, 0] - 1.3 * s * q[t, 0, 0]) < 1e-13
    assert abs(hT[0, 0, 0, 0] - s) < 1e-13


def _matrix_form(q, k, v, g, beta, h0, scale, gate_mode):
    """Whole-sequence matrix form for one head (h0 given), using a library
    linear solve:  Delta = (I + A)^-1 (diag(beta) V - diag(beta) Kg h0),
    O = scale Qg h0 + Aqk Delta, hT = diag(exp(b_T)) h0 + Kt^T Delta, with
    A = strict-lower(beta_r sum_c k_rc k_sc e^{b_rc - b_sc}), Aqk = lower
    incl. diagonal of scale sum_c q_rc k_sc e^{b_rc - b_sc}."""
    T, dk = k.shape
    b = np.cumsum(g if gate_mode == 1 else np.repeat(g[:, None], dk, 1), axis=0)
    diff = b[:, None, :] - b[None, :, :]  # [r, s, c]
    lower = np.tril(np.ones((T, T), dtype=bool))
    D = np.where(lower[:, :, None], np.exp(np.where(lower[:, :, None], diff, 0.0)), 0.0)
    KK = np.einsum("rc,sc,rsc->rs", k, k, D)
    QK = np.einsum("rc,sc,rsc->rs", q, k, D)
    A = np.tril(beta[:, None] * KK, -1)
    Aqk = scale * np.tril(QK)
    Kg = k * np.exp(b)
    rhs = beta[:, None] * (v - Kg @ h0)
    Delta = np.linalg.solve(np.eye(T) + A, rhs)
    O = scale * (q * np.exp(b)) @ h0 + Aqk @ Delta
    Kt = k * np.exp(b[-1][None, :] - b)
    hT = np.exp(b[-1])[:, None] * h0 + Kt.T @ Delta
    return O, hT


@pytest.mark.parametrize("gate_mode", [0, 1])
@pytest.mark.parametrize("low", [-0.05, -1.0, -5.0])
def test_whole_sequence_matrix_form(gate_mode, low):
    T = 57
    q, k, v, g, beta, h0 = rand_case(T, gate_mode=gate_mode, low=low, seed=7)
    scale = 0.35
    o, hT = run(q, k, v, g, beta, h0, scale=scale, gate_mode=gate_mode)
    for hv in range(4):
        hq = hv // 2
        O, H = _matrix_form(q[:, hq], k[:, hq], v[:, hv], g[:, hv], beta[:, hv],
                            h0[0, hv], scale, gate_mode)
        np.testing.assert_allclose(o[:, hv], O, atol=1e-11)
        np.testing.assert_allclose(hT[0, hv], H, atol=1e-11)


# --------------------------------------------------------------------------
# invariants
# --------------------------------------------------------------------------
@pytest.mark.parametrize("gate_mode", [0, 1])
@pytest.mark.parametrize("chunk", [1, 7, 32, 64, 200])
def test_chunked_matches_token_serial(gate_mode, chunk):
    """All nonempty chunk cuts give the same result (logismos issue #46,
    Sep 6 comment); the chunked walk is written independently."""
    T = 150
    q, k, v, g, beta, h0 = rand_case(T, gate_mode=gate_mode, low=-3.0, seed=8)
    a = run(q, k, v, g, beta, h0, gate_mode=gate_mode)
    b = oracle.chunked(q, k, v, g, beta, h0, [0, T], 0.7, gate_mode, chunk)
    np.testing.assert_allclose(b[0], a[0], atol=1e-10)
    np.testing.assert_allclose(b[1], a[1], atol=1e-10)


@pytest.mark.parametrize("gate_mode", [0, 1])
def test_continuation(gate_mode):
    """Partition continuation: [0,t) then [t,T) with hT fed back as h0."""
    T, t = 90, 41
    q, k, v, g, beta, h0 = rand_case(T, gate_mode=gate_mode, seed=9)
    o, hT = run(q, k, v, g, beta, h0, gate_mode=gate_mode)
    o1, h1 = run(q[:t], k[:t], v[:t], g[:t], beta[:t], h0, gate_mode=gate_mode)
    o2, h2 = run(q[t:], k[t:], v[t:], g[t:], beta[t:], h1, gate_mode=gate_mode)
    np.testing.assert_allclose(np.concatenate([o1, o2]), o, atol=1e-12)
    np.testing.assert_allclose(h2, hT, atol=1e-12)


@pytest.mark.parametrize("fn", ["token_serial", "chunked"])
def test_varlen_equals_separate_calls(fn):
    lengths = [5, 0, 31, 1, 64, 19]
    T = sum(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    q, k, v, g, beta, h0 = rand_case(T, n_seqs=len(lengths), seed=10)
    f = (lambda *a: oracle.chunked(*a, chunk=16)) if fn == "chunked" else oracle.token_serial
    o, hT = f(q, k, v, g, beta, h0, cu, 0.7, 0)
    for i, L in enumerate(lengths):
        s, e = cu[i], cu[i + 1]
        oi, hi = oracle.token_serial(q[s:e], k[s:e], v[s:e], g[s:e], beta[s:e],
                                     h0[i:i + 1], [0, L], 0.7, 0)
        np.testing.assert_allclose(o[s:e], oi, atol=1e-12)
        np.testing.assert_allclose(hT[i], hi[0], atol=1e-12)
    # an empty sequence leaves its state untouched
    np.testing.assert_allclose(hT[1], h0[1], atol=0)


def test_grouped_heads_equal_repeated_heads():
    """GQA: value head hv reads q/k head hv // (HV/H); the same as repeating
    each q/k head HV/H times with H = HV."""
    T = 33
    q, k, v, g, beta, h0 = rand_case(T, H=2, HV=6, seed=11)
    o, hT = run(q, k, v, g, beta, h0)
    qr = np.repeat(q, 3, axis=1)
    kr = np.repeat(k, 3, axis=1)
    o2, h2 = run(qr, kr, v, g, beta, h0)
    np.testing.assert_allclose(o, o2, atol=1e-13)
    np.testing.assert_allclose(hT, h2, atol=1e-13)


def test_per_key_gate_with_equal_channels_is_scalar_gate():
    T = 40
    q, k, v, g, beta, h0 = rand_case(T, gate_mode=0, seed=12)
    gk = np.repeat(g[:, :, None], 8, axis=2)
    a = run(q, k, v, g, beta, h0, gate_mode=0)
    b = run(q, k, v, gk, beta, h0, gate_mode=1)
    np.testing.assert_allclose(a[0], b[0], atol=1e-13)
    np.testing.assert_allclose(a[1], b[1], atol=1e-13)


@pytest.mark.parametrize("gate_mode", [0, 1])
def test_joint_linearity_in_state_and_values(gate_mode):
    """For fixed q, k, g, beta the map (h0, V) -> (o, hT) is linear."""
    T = 45
    q, k, v, g, beta, h0 = rand_case(T, gate_mode=gate_mode, seed=13)
    _, _, v2, _, _, h02 = rand_case(T, gate_mode=gate_mode, seed=14)
    a = run(q, k, v, g, beta, h0, gate_mode=gate_mode)
    b = run(q, k, v2, g, beta, h02, gate_mode=gate_mode)
    c = run(q, k, 2.0 * v - 3.0 * v2, g, beta, 2.0 * h0 - 3.0 * h02,
            gate_mode=gate_mode)
    np.testing.assert_allclose(c[0], 2.0 * a[0] - 3.0 * b[0], atol=1e-11)
    np.testing.assert_allclose(c[1], 2.0 * a[1] - 3.0 * b[1], atol=1e-11)


@pytest.mark.parametrize("gate_mode", [0, 1])
@pytest.mark.parametrize("fn", ["token_serial", "chunked"])
def test_state_transfer_is_product_of_token_maps(gate_mode, fn):
    """The reading the sequence split rests on: over a segment the state maps
    affinely, S_out = M S_in + S_seg.  A pass with every value zero and the
    identity as initial state (dv = dk) must leave M, the product of the
    per-token maps A_t = (I - beta_t k_t k_t^T) diag(a_t), formed here one
    plain matrix at a time; a pass from a zero state leaves S_seg; any other
    entering state must then give M S_in + S_seg (logismos issue #46,
    "Remaining work": later continuation)."""
    T, dk, dv = 37, 8, 6
    q, k, v, g, beta, h0 = rand_case(T, dk=dk, dv=dv, gate_mode=gate_mode, seed=21)
    f = oracle.token_serial if fn == "token_serial" else \
        (lambda *a: oracle.chunked(*a, chunk=16))  # three chunks, ragged tail
    eye = np.broadcast_to(np.eye(dk), (1, 4, dk, dk)).copy()
    v0 = np.zeros((T, 4, dk))
    _, M = run(q, k, v0, g, beta, eye, gate_mode=gate_mode, fn=f)
    _, S_seg = run(q, k, v, g, beta, None, gate_mode=gate_mode, fn=f)
    _, S_out = run(q, k, v, g, beta, h0, gate_mode=gate_mode, fn=f)
    for hv in range(4):
        P = np.eye(dk)
        for t in range(T):
            kt = k[t, hv // 2]
            a = np.exp(g[t, hv]) * np.ones(dk)
            P = (np.eye(dk) - beta[t, hv] * np.outer(kt, kt)) @ np.diag(a) @ P
        np.testing.assert_allclose(M[0, hv], P, atol=1e-12)
        np.testing.assert_allclose(S_out[0, hv], P @ h0[0, hv] + S_seg[0, hv], atol=1e-12)


def test_state_norm_bound():
    """With |k| = 1 and 0 <= beta <= 1 the transition (I - beta k k^T) diag(a)
    is a contraction, so ||S_T||_F <= ||h0||_F + sum_t beta_t ||v_t||."""
    T = 300
    q, k, v, g, beta, h0 = rand_case(T, low=-0.01, seed=15)
    _, hT = run(q, k, v, g, beta, h0)
    for hv in range(4):
        bound = np.linalg.norm(h0[0, hv]) + np.sum(beta[:, hv] * np.linalg.norm(v[:, hv], axis=-1))
        assert np.linalg.norm(hT[0, hv]) <= bound + 1e-9


def test_rejects_malformed_arguments():
    q, k, v, g, beta, h0 = rand_case(5, seed=16)
    with pytest.raises(ValueError):
        oracle.token_serial(q, k, v, g, beta, h0, [0, 3, 2, 5], 0.5, 0)
    with pytest.raises(ValueError):
        oracle.token_serial(q, k, v, g[:, :3], beta, h0, [0, 5], 0.5, 0)


# --------------------------------------------------------------------------
# planted mistakes: every plausible error in the walk fails at least one pin
# --------------------------------------------------------------------------
def _pins_pass(fn) -> bool:
    """Re-run the main pins against ``fn`` (a variant of the token walk)."""
    ok = True
    for c in _golden_cases():
        q, k, v, g, beta, h0 = _golden_inputs(c)
        T = q.shape[0]
        o, hT = fn(q, k, v, g, beta, h0, [0, T], c["scale"], c["gate_mode"])
        ok &= np.allclose(o, np.array(c["o"]), atol=1e-9)
        ok &= np.allclose(hT, np.array(c["hT"]), atol=1e-9)
    for gate_mode in (0, 1):
        T = 30
        q, k, v, g, beta, h0 = rand_case(T, gate_mode=gate_mode, seed=17)
        o, hT = fn(q, k, v, g, beta, h0, [0, T], 0.35, gate_mode)
        for hv in range(4):
            hq = hv // 2
            O, H = _matrix_form(q[:, hq], k[:, hq], v[:, hv], g[:, hv],
                                beta[:, hv], h0[0, hv], 0.35, gate_mode)
            ok &= np.allclose(o[:, hv], O, atol=1e-9)
            ok &= np.allclose(hT[0, hv], H, atol=1e-9)
    return bool(ok)


def test_pins_pass_for_the_oracle():
    assert _pins_pass(oracle.token_serial)


@pytest.mark.parametrize("planted", [1, 2, 3, 4, 5, 6])
def test_pins_catch_planted_mistakes(planted):
    def fn(q, k, v, g, beta, h0, cu, scale, gate_mode):
        return oracle.token_serial_planted(q, k, v, g, beta, h0, cu, scale,
                                           gate_mode, planted)
    assert not _pins_pass(fn)
