"""Helpers of the GPU parity tests: run the CUDA path through the binding and
the fp64 oracle on the same inputs (optionally on a subset of value heads, so
that full-size workloads stay cheap on the CPU)."""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np
import torch

import oracle
from chunkwise_gated_delta_gdn_gb300 import gdn, synth


def to_dev(x: dict, dev="cuda") -> dict:
    return {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in x.items()}


def run_gpu(c: synth.Case, x: dict, *, want_hT=True, h0=True, chunk=None):
    d = to_dev(x)
    o, hT = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"],
                              d["h0"] if h0 else None, scale=c.scale,
                              chunk=chunk or c.chunk, cu_seqlens=d["cu_seqlens"],
                              output_final_state=want_hT)
    torch.cuda.synchronize()
    return o, hT


def run_oracle(c: synth.Case, x: dict, heads: Optional[Sequence[int]] = None,
               h0=True):
    """Token-serial fp64 oracle on value heads ``heads`` (all by default).
    Returns o [Ttot, len(heads), dv] and hT [N, len(heads), dk, dv]."""
    group = c.HV // c.H
    heads = list(range(c.HV)) if heads is None else list(heads)
    hq = [h // group for h in heads]

    def flat(t):
        return t.reshape((-1,) + tuple(t.shape[2:]))

    q = flat(x["q"])[:, hq]
    k = flat(x["k"])[:, hq]
    v = flat(x["v"])[:, heads]
    g = flat(x["g"])[:, heads]
    beta = flat(x["beta"])[:, heads]
    h0v = x["h0"][:, heads] if (h0 and x["h0"] is not None) else None
    if x["cu_seqlens"] is not None:
        cu = x["cu_seqlens"].to(torch.int64).numpy()
    else:
        cu = np.arange(c.B + 1, dtype=np.int64) * c.T
    return oracle.token_serial(q, k, v, g, beta, h0v, cu, c.scale, c.gate_mode)


def gpu_heads(o: torch.Tensor, hT: Optional[torch.Tensor], heads=None):
    o = o.reshape((-1,) + tuple(o.shape[2:]))
    if heads is not None:
        o = o[:, list(heads)]
        hT = hT[:, list(heads)] if hT is not None else None
    return o.double().cpu().numpy(), (hT.double().cpu().numpy() if hT is not None else None)


def kind_of(c: synth.Case) -> str:
    return "bf16" if c.dtype == torch.bfloat16 else "f32"
