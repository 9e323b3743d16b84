"""fp64 oracle of the operations either side of the gated delta rule: the
causal depthwise convolution and the q/k L2 normalisation before it, the gated
RMS normalisation of its output after it.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU legs of ``bench.py`` may import it.
It shares nothing with the CUDA library.  Plain numpy in float64, one loop per
sequence, written from the definitions below.

Definitions and readings (the pages give the convolution's contract and name
the output norm, but print no formula for either; the plainest reading of
each is taken and listed in the design notes):

* Causal convolution (logismos issue #46, "Verified implementation
  boundary", the staged causal convolution step: channel-major
  oldest-to-newest raw history, separate next-history and output, no history
  when the width is 1).  For channel c, width W, weights w[c, 0..W-1] and a
  sequence x[0..L-1] with history h[c, 0..W-2] (h[c, W-2] is the input just
  before x[0]):
      ext = h[c, :] followed by x[:, c]        (length W - 1 + L)
      y[t, c] = act(bias[c] + sum_j w[c, j] ext[t + j])
  so w[c, W-1] weighs the current input.  act is the identity or SiLU
  (x * sigmoid(x)).  The next history is the last W - 1 entries of ext.
* L2 normalisation of q and k rows: y = x / sqrt(sum(x^2) + eps).
* Gated RMS normalisation of the output (the output norm that follows the
  recurrence in stratat pull #1296, re-base notes): per row of dv values,
      y = x / sqrt(mean(x^2) + eps) * weight * silu(z)   (z given)
      y = x / sqrt(mean(x^2) + eps) * weight             (no z).
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

ACT_NONE = 0
ACT_SILU = 1


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def _silu(x):
    return x / (1.0 + np.exp(-x))


def causal_conv1d(x, w, bias, h0, cu_seqlens: Sequence[int], activation: int = ACT_NONE):
    """x [Ttot, D] packed sequences, w [D, W], bias [D] or None, h0 [N, D, W-1]
    or None (zeros).  Returns (y [Ttot, D], hT [N, D, W-1]) in float64."""
    x, w, bias, h0 = _f64(x), _f64(w), _f64(bias), _f64(h0)
    Ttot, D = x.shape
    W = w.shape[1]
    cu = [int(c) for c in cu_seqlens]
    N = len(cu) - 1
    y = np.zeros((Ttot, D))
    hT = np.zeros((N, D, W - 1))
    for n in range(N):
        s, e = cu[n], cu[n + 1]
        hist = h0[n] if h0 is not None else np.zeros((D, W - 1))
        ext = np.concatenate([hist, x[s:e].T], axis=1)  # [D, W - 1 + L]
        for t in range(e - s):
            acc = (w * ext[:, t:t + W]).sum(axis=1)
            if bias is not None:
                acc = acc + bias
            y[s + t] = _silu(acc) if activation == ACT_SILU else acc
        hT[n] = ext[:, ext.shape[1] - (W - 1):]
    return y, hT


def l2norm(x, eps: float):
    """Rows of x (last axis) divided by sqrt(sum of squares + eps)."""
    x = _f64(x)
    return x / np.sqrt((x * x).sum(axis=-1, keepdims=True) + eps)


def rmsnorm_gated(x, weight, z: Optional[object], eps: float):
    """Rows of x (last axis) scaled to unit RMS, times weight, times silu(z)."""
    x, weight, z = _f64(x), _f64(weight), _f64(z)
    y = x / np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps) * weight
    if z is not None:
        y = y * _silu(z)
    return y
