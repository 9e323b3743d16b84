"""Sequence split with a state-transfer exchange: one long sequence cut into
consecutive segments, each processed where it lives (its own GPU, or one after
another on one GPU), with one exchange of small per-segment transfers.

Over a segment the recurrence maps its entering state affinely,
``S_out = M S_in + S_seg``:

* ``S_seg`` is the state the segment leaves from a zero start
  (``gdn_chunk_fwd`` with ``h0=None``);
* ``M`` (``dk x dk`` per value head) is the state it leaves from the identity
  with every value zero: the value term of each update vanishes, leaving the
  product of the per-token maps ``(I - beta k k^T) diag(a)``
  (``gdn_chunk_fwd`` with ``v = 0``, ``dv = dk``, ``h0 = I``).

Segment ``p`` then starts from ``S_in(p) = M_{p-1} S_in(p-1) + S_seg_{p-1}``
(``gdn_state_combine``), and a last pass from that state gives its outputs
exactly.  This is the continuation of logismos issue #46 ("Remaining work":
later continuation across independently positioned executions) for a
sequence longer than one GPU's share.  Every step runs in the library's
kernels; this module only sequences the calls and, across ranks, gathers the
transfers with ``torch.distributed``.
"""
from __future__ import annotations

from typing import Callable, List, Optional, Sequence, Tuple

import torch

from . import gdn

Tensor = torch.Tensor


def segment_transfer(q: Tensor, k: Tensor, v: Tensor, g: Tensor, beta: Tensor, *,
                     chunk: int = 64, stream=None) -> Tuple[Tensor, Tensor]:
    """``(M, S_seg)`` of each batch row as one segment: ``M [B, HV, dk, dk]``,
    ``S_seg [B, HV, dk, dv]``, fp32."""
    B, T, H, dk = q.shape
    HV = v.shape[2]
    _, S_seg = gdn.gdn_chunk_fwd(q, k, v, g, beta, None, chunk=chunk, stream=stream)
    v0 = torch.zeros((B, T, HV, dk), dtype=v.dtype, device=v.device)
    eye = torch.eye(dk, dtype=torch.float32, device=v.device)
    ident = eye.expand(B, HV, dk, dk).contiguous()
    _, M = gdn.gdn_chunk_fwd(q, k, v0, g, beta, ident, chunk=chunk, stream=stream)
    return M, S_seg


def compose(transfers: Sequence[Tuple[Tensor, Tensor]], h0: Optional[Tensor],
            combine: Callable[[Tensor, Tensor, Tensor], Tensor] = None) -> List[Tensor]:
    """Entering state of every segment from the segments' transfers, in order:
    ``S_in(0) = h0`` (zeros when None), ``S_in(p+1) = M_p S_in(p) + S_seg_p``."""
    if combine is None:
        combine = lambda M, S, Sg: gdn.gdn_state_combine(M, S, Sg)  # noqa: E731
    M0, Sg0 = transfers[0]
    s = h0 if h0 is not None else torch.zeros_like(Sg0)
    out = [s]
    for M, Sg in transfers[:-1]:
        s = combine(M, s, Sg)
        out.append(s)
    return out


def split_forward(q: Tensor, k: Tensor, v: Tensor, g: Tensor, beta: Tensor,
                  h0: Optional[Tensor], cuts: Sequence[int], *, scale: Optional[float] = None,
                  chunk: int = 64) -> Tuple[Tensor, Tensor]:
    """One batch row's sequence cut at token positions ``cuts`` and processed
    segment by segment on this device: transfers, composition, then each
    segment's outputs from its true entering state.  Returns ``(o, hT)`` like
    ``gdn_chunk_fwd`` on the whole sequence."""
    T = q.shape[1]
    edges = [0] + sorted(int(c) for c in cuts if 0 < c < T) + [T]
    segs = [slice(edges[i], edges[i + 1]) for i in range(len(edges) - 1)]

    def part(x, s):
        # a fresh buffer: a contiguous slice would be a view whose start need
        # not be 16-byte aligned (the library refuses such pointers)
        view = x[:, s]
        return torch.empty_like(view, memory_format=torch.contiguous_format).copy_(view)

    transfers = [segment_transfer(part(q, s), part(k, s), part(v, s), part(g, s),
                                  part(beta, s), chunk=chunk) for s in segs]
    starts = compose(transfers, h0)
    outs, hT = [], None
    for s, s_in in zip(segs, starts):
        o, hT = gdn.gdn_chunk_fwd(part(q, s), part(k, s), part(v, s), part(g, s),
                                  part(beta, s), s_in, scale=scale, chunk=chunk)
        outs.append(o)
    return torch.cat(outs, 1), hT


def exchange_and_compose(M: Tensor, S_seg: Tensor, h0: Optional[Tensor], group=None,
                         combine: Callable[[Tensor, Tensor, Tensor], Tensor] = None) -> Tensor:
    """Entering state of this rank's segment, segments ordered by rank: every
    rank's ``(M, S_seg)`` is gathered (one all-gather of each), then composed
    up to this rank.  ``h0`` is the sequence's initial state (rank 0's)."""
    import torch.distributed as dist

    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    Ms = [torch.empty_like(M) for _ in range(world)]
    Ss = [torch.empty_like(S_seg) for _ in range(world)]
    dist.all_gather(Ms, M.contiguous(), group=group)
    dist.all_gather(Ss, S_seg.contiguous(), group=group)
    return compose(list(zip(Ms, Ss))[:rank + 1], h0, combine)[rank]


def distributed_forward(q: Tensor, k: Tensor, v: Tensor, g: Tensor, beta: Tensor,
                        h0: Optional[Tensor], *, scale: Optional[float] = None,
                        chunk: int = 64, group=None) -> Tuple[Tensor, Tensor]:
    """This rank's segment of one sequence (segments ordered by rank): its
    outputs, and the state after it (the last rank's is the sequence's
    final state)."""
    M, S_seg = segment_transfer(q, k, v, g, beta, chunk=chunk)
    s_in = exchange_and_compose(M, S_seg, h0, group)
    return gdn.gdn_chunk_fwd(q, k, v, g, beta, s_in, scale=scale, chunk=chunk)
