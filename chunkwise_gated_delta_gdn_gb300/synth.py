"""Seeded synthetic inputs for the gated delta rule forward pass.

This module holds no arithmetic of the method itself: it only draws random
tensors with the shapes and value distributions of the workloads, so that the
CUDA path and the fp64 oracle see exactly the same bits.  Both sides import it;
it imports neither.

Recipe (one torch CPU generator, seeded, draws in the order q, k, v, g, beta,
h0):

* q, k ~ N(0, 1), L2-normalised per (token, head) in fp32, then cast to the
  input dtype (the normalisation is input preparation, done before the op).
* v ~ N(0, 1), cast to the input dtype.
* g (natural-log decay, <= 0): ``"softplus"`` draws -softplus(N(0,1)) clamped
  to >= -5; ``"uniform"`` draws U[gate_low, 0] (per token and value head for
  the scalar gate, per key channel as well for the per-key gate).
* beta = sigmoid(N(0, 1)), fp32.
* h0 ~ N(0, h0_std), fp32, one state per sequence, or None.
* Variable-length packing: ``n_seqs - 1`` distinct cut points drawn uniformly
  from 1..T-1 (sorted) split T tokens into sequences of length >= 1.

The five named workloads mirror the geometries of the pages: the 32k-token,
HV = 48, dk = dv = 128 spot of stratat pull #1296 ("Measured verdict on
gfx1100"), the KDA gate range down to -5 of ROCm/rocm-libraries PR #11223
("Correctness"), and packed variable-length prefill of logismos issue #46.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import torch

GATE_SCALAR = 0
GATE_PER_KEY = 1


@dataclasses.dataclass(frozen=True)
class Case:
    """Shape, dtype and distribution of one synthetic workload."""

    name: str
    B: int
    T: int  # tokens per batch row, or total packed tokens when varlen
    H: int
    HV: int
    dk: int
    dv: int
    chunk: int
    dtype: torch.dtype
    gate_mode: int
    gate_dist: str  # "softplus" or "uniform"
    gate_low: float
    h0_std: Optional[float]  # None -> no initial state (zeros)
    n_seqs: int = 0  # > 0 -> packed variable-length input with cu_seqlens
    seed: int = 0

    @property
    def scale(self) -> float:
        return float(self.dk) ** -0.5

    @property
    def tokens(self) -> int:
        return self.T if self.n_seqs > 0 else self.B * self.T

    @property
    def varlen(self) -> bool:
        return self.n_seqs > 0

    @property
    def num_states(self) -> int:
        return self.n_seqs if self.n_seqs > 0 else self.B


WORKLOADS = {
    # tiny fp32 case, the oracle finishes in well under a second
    "gdn_fp32_t256": Case("gdn_fp32_t256", B=1, T=256, H=2, HV=2, dk=64, dv=64,
                          chunk=64, dtype=torch.float32, gate_mode=GATE_SCALAR,
                          gate_dist="softplus", gate_low=-5.0, h0_std=None),
    "gdn_bf16_t4096": Case("gdn_bf16_t4096", B=1, T=4096, H=16, HV=48, dk=128,
                           dv=128, chunk=64, dtype=torch.bfloat16,
                           gate_mode=GATE_SCALAR, gate_dist="uniform",
                           gate_low=-5.0, h0_std=0.1),
    "gdn_bf16_t32768": Case("gdn_bf16_t32768", B=1, T=32768, H=16, HV=48,
                            dk=128, dv=128, chunk=64, dtype=torch.bfloat16,
                            gate_mode=GATE_SCALAR, gate_dist="uniform",
                            gate_low=-5.0, h0_std=None),
    "kda_bf16_b2_t8192": Case("kda_bf16_b2_t8192", B=2, T=8192, H=32, HV=32,
                              dk=128, dv=128, chunk=32, dtype=torch.bfloat16,
                              gate_mode=GATE_PER_KEY, gate_dist="uniform",
                              gate_low=-5.0, h0_std=None),
    "gdn_varlen_t131072": Case("gdn_varlen_t131072", B=1, T=131072, H=16,
                               HV=48, dk=128, dv=128, chunk=64,
                               dtype=torch.bfloat16, gate_mode=GATE_SCALAR,
                               gate_dist="uniform", gate_low=-5.0, h0_std=0.1,
                               n_seqs=8),
    # one decode step (T = 1) for a batch of 256 sequences at the 32k spot's
    # head geometry: the one-token grouped step of logismos issue #46
    # ("Verified implementation boundary"); the states (805 MB) dominate
    "gdn_decode_bf16_b256": Case("gdn_decode_bf16_b256", B=256, T=1, H=16, HV=48,
                                 dk=128, dv=128, chunk=64, dtype=torch.bfloat16,
                                 gate_mode=GATE_SCALAR, gate_dist="uniform",
                                 gate_low=-5.0, h0_std=0.1),
    # the operations either side of the recurrence at the 32k spot: causal
    # convolution (width 4, SiLU) over the q, k and v channels together
    # ((2 H dk + HV dv) = 10240), L2 norm of q and k, gated RMS norm of o
    "prepost_bf16_t32768": Case("prepost_bf16_t32768", B=1, T=32768, H=16, HV=48, dk=128,
                                dv=128, chunk=64, dtype=torch.bfloat16,
                                gate_mode=GATE_SCALAR, gate_dist="uniform", gate_low=-5.0,
                                h0_std=None),
    "kda_decode_bf16_b256": Case("kda_decode_bf16_b256", B=256, T=1, H=32, HV=32,
                                 dk=128, dv=128, chunk=32, dtype=torch.bfloat16,
                                 gate_mode=GATE_PER_KEY, gate_dist="uniform",
                                 gate_low=-5.0, h0_std=0.1),
}


def case(name: str, **overrides) -> Case:
    """A named workload, optionally with fields replaced."""
    return dataclasses.replace(WORKLOADS[name], **overrides)


def _l2norm_rows(x: torch.Tensor) -> torch.Tensor:
    # input preparation only: unit-norm q/k rows, as the pages' workloads use
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-12)


def varlen_lengths(gen: torch.Generator, T: int, n_seqs: int) -> list[int]:
    """Split T tokens into n_seqs lengths >= 1 from sorted distinct cuts."""
    if n_seqs <= 1:
        return [T]
    if T < n_seqs:
        raise ValueError("need T >= n_seqs for lengths >= 1")
    cuts = torch.randperm(T - 1, generator=gen)[: n_seqs - 1] + 1
    cuts = sorted(int(c) for c in cuts)
    edges = [0] + cuts + [T]
    return [edges[i + 1] - edges[i] for i in range(n_seqs)]


def make_inputs(c: Case, lengths: Optional[Sequence[int]] = None) -> dict:
    """Draw the inputs of case ``c`` on the CPU.

    Returns a dict with q, k, v (``c.dtype``), g, beta, h0 (fp32 or None) and,
    for packed input, ``cu_seqlens`` (int32) and ``lengths``.  Batched inputs
    have shape ``[B, T, ...]``; packed ones ``[1, T, ...]``.  ``lengths``
    overrides the drawn sequence lengths of a packed case (they must sum to T).
    """
    gen = torch.Generator(device="cpu")
    gen.manual_seed(c.seed)
    Bq = 1 if c.varlen else c.B
    T = c.T
    shp_qk = (Bq, T, c.H, c.dk)
    q = _l2norm_rows(torch.randn(shp_qk, generator=gen, dtype=torch.float32)).to(c.dtype)
    k = _l2norm_rows(torch.randn(shp_qk, generator=gen, dtype=torch.float32)).to(c.dtype)
    v = torch.randn((Bq, T, c.HV, c.dv), generator=gen, dtype=torch.float32).to(c.dtype)
    g_shape = (Bq, T, c.HV) if c.gate_mode == GATE_SCALAR else (Bq, T, c.HV, c.dk)
    if c.gate_dist == "softplus":
        g = -torch.nn.functional.softplus(
            torch.randn(g_shape, generator=gen, dtype=torch.float32))
        g = g.clamp_min(c.gate_low)
    elif c.gate_dist == "uniform":
        g = torch.rand(g_shape, generator=gen, dtype=torch.float32) * c.gate_low
    elif c.gate_dist == "zero":
        g = torch.zeros(g_shape, dtype=torch.float32)
    else:
        raise ValueError(c.gate_dist)
    beta = torch.sigmoid(torch.randn((Bq, T, c.HV), generator=gen, dtype=torch.float32))
    out = dict(q=q, k=k, v=v, g=g.contiguous(), beta=beta.contiguous())
    n_states = c.num_states
    if c.h0_std is not None:
        out["h0"] = torch.randn((n_states, c.HV, c.dk, c.dv), generator=gen,
                                dtype=torch.float32) * c.h0_std
    else:
        out["h0"] = None
    if c.varlen:
        if lengths is None:
            lengths = varlen_lengths(gen, T, c.n_seqs)
        lengths = [int(x) for x in lengths]
        if sum(lengths) != T or len(lengths) != c.n_seqs:
            raise ValueError("lengths must be n_seqs entries summing to T")
        cu = [0]
        for x in lengths:
            cu.append(cu[-1] + x)
        out["cu_seqlens"] = torch.tensor(cu, dtype=torch.int32)
        out["lengths"] = lengths
    else:
        out["cu_seqlens"] = None
        out["lengths"] = [T] * c.B
    return out


def make_prepost_inputs(c: Case, width: int = 4) -> dict:
    """Seeded inputs of the pre/post operations for the geometry of ``c``:
    the convolution's input x [B, T, 2 H dk + HV dv] (q, k and v channels
    side by side) with weights [D, width], bias [D] and history
    [B, D, width - 1]; the output rows o and gate rows z [B, T, HV, dv] with
    the norm weight [dv]."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(c.seed + 1000)
    D = 2 * c.H * c.dk + c.HV * c.dv
    x = torch.randn((c.B, c.T, D), generator=gen, dtype=torch.float32).to(c.dtype)
    w = (torch.rand((D, width), generator=gen) * 2 - 1) / width ** 0.5
    bias = torch.randn(D, generator=gen) * 0.1
    h0 = torch.randn((c.B, D, width - 1), generator=gen)
    o = torch.randn((c.B, c.T, c.HV, c.dv), generator=gen, dtype=torch.float32).to(c.dtype)
    z = torch.randn((c.B, c.T, c.HV, c.dv), generator=gen, dtype=torch.float32).to(c.dtype)
    wn = torch.rand(c.dv, generator=gen) + 0.5
    return dict(x=x, w=w, bias=bias, h0=h0, o=o, z=z, norm_weight=wn)


def sweep_cases() -> list[Case]:
    """The parity sweep: T in {1, 37, 64, 65, 200, 4099} x gate lower bound in
    {-0.05, -1, -5} x {scalar gate, per-key gate} x {bf16, fp32} inputs, small
    head counts (the T sweep and decay modes of stratat pull #1296, "The parity
    discipline"; the gate range to -5 of PR #11223, "Correctness")."""
    out = []
    for dtype, tag in ((torch.bfloat16, "bf16"), (torch.float32, "f32")):
        for gate_mode in (GATE_SCALAR, GATE_PER_KEY):
            for T in (1, 37, 64, 65, 200, 4099):
                for low in (-0.05, -1.0, -5.0):
                    chunk = 64 if gate_mode == GATE_SCALAR else 32
                    out.append(Case(f"sweep_{tag}_m{gate_mode}_T{T}_L{low}", B=1, T=T,
                                    H=2, HV=4, dk=128, dv=128, chunk=chunk,
                                    dtype=dtype, gate_mode=gate_mode,
                                    gate_dist="uniform", gate_low=low, h0_std=0.1,
                                    seed=T))
    return out
