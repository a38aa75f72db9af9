"""Test infrastructure only: fp64 CPU oracle for the mixer's fused neighbours.

Only the tests, the package's ``smoke()`` check and the benchmark's CPU
baseline leg may import this module; the library never does and shares no
code with it.

What it computes.  The Primus hybrid-LLM pretraining blog (MI355X), section
"Recipe" (table 4, "FLA fusions"), lists among the fused kernels of every
mixer block the short convolution and the gated norm around the token mixer;
the recipe's normalisation epsilon is 1e-6.  Written out (plain loops over
the definition, fp64):

* short convolution: for every channel c of a [B, T, H*D] projection, a
  causal depthwise convolution of width W over the tokens of each sequence
  (zero before the sequence start), then SiLU:
      s[t, c] = sum_{i=0}^{W-1} w[c, i] x[t - (W - 1) + i, c],   y = s * sigmoid(s);
  for the query and key projections the head's D values of each token are
  then L2-normalised and scaled (the mixer's q and k inputs), with the
  recipe's epsilon under the root so that an all-zero row stays finite:
      z[t, h, :] = scale * y[t, h, :] / sqrt(||y[t, h, :]||^2 + eps);
* gated norm: per token and head, an RMS norm of the mixer output o over its
  D values, with a learned per-dimension weight, gated by SiLU of a gate
  projection:
      out = o / sqrt(mean(o^2) + eps) * weight * gate * sigmoid(gate).

Backward passes are reverse-mode differentiation of the same loops.
Parity status: every function is pinned in tests/test_oracle_neighbours.py.
"""
from __future__ import annotations

import numpy as np


def _sig(x):
    return 1.0 / (1.0 + np.exp(-x))


def short_conv_fwd(x, w, H, l2norm=False, scale=1.0, eps=1e-6):
    """x: [B, T, H*D], w: [H*D, W].  Returns (z, s): the output [B, T, H*D]
    and the pre-activation s (kept for the backward pass)."""
    x = np.asarray(x, np.float64)
    w = np.asarray(w, np.float64)
    B, T, CH = x.shape
    W = w.shape[1]
    s = np.zeros((B, T, CH))
    for b in range(B):
        for t in range(T):
            for i in range(W):
                tt = t - (W - 1) + i
                if tt >= 0:
                    s[b, t] += w[:, i] * x[b, tt]
    y = s * _sig(s)
    if not l2norm:
        return y, s
    D = CH // H
    z = np.zeros_like(y)
    for b in range(B):
        for t in range(T):
            for h in range(H):
                seg = y[b, t, h * D:(h + 1) * D]
                z[b, t, h * D:(h + 1) * D] = scale * seg / np.sqrt(np.sum(seg * seg) + eps)
    return z, s


def short_conv_bwd(x, w, dz, H, l2norm=False, scale=1.0, eps=1e-6):
    """Gradients (dx, dw) of sum(z * dz) with respect to x and w."""
    x = np.asarray(x, np.float64)
    w = np.asarray(w, np.float64)
    dz = np.asarray(dz, np.float64)
    B, T, CH = x.shape
    W = w.shape[1]
    _, s = short_conv_fwd(x, w, H)
    sg = _sig(s)
    y = s * sg
    if l2norm:
        D = CH // H
        dy = np.zeros_like(y)
        for b in range(B):
            for t in range(T):
                for h in range(H):
                    sl = slice(h * D, (h + 1) * D)
                    r = 1.0 / np.sqrt(np.sum(y[b, t, sl] ** 2) + eps)
                    g = dz[b, t, sl]
                    # z = scale y r:  dy = scale r (g - y r^2 <y, g>)
                    dy[b, t, sl] = scale * r * (g - y[b, t, sl] * (r * r) * np.dot(y[b, t, sl], g))
    else:
        dy = dz
    ds = dy * (sg + s * sg * (1.0 - sg))     # d/ds of s sigmoid(s)
    dx = np.zeros_like(x)
    dw = np.zeros_like(w)
    for b in range(B):
        for t in range(T):
            for i in range(W):
                tt = t - (W - 1) + i
                if tt >= 0:
                    dx[b, tt] += w[:, i] * ds[b, t]
                    dw[:, i] += ds[b, t] * x[b, tt]
    return dx, dw


def gated_rmsnorm_fwd(o, gate, weight, eps=1e-6):
    """o, gate: [B, T, H, D]; weight: [D].  Returns out [B, T, H, D]."""
    o = np.asarray(o, np.float64)
    gate = np.asarray(gate, np.float64)
    weight = np.asarray(weight, np.float64)
    r = 1.0 / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)
    return o * r * weight * gate * _sig(gate)


def gated_rmsnorm_bwd(o, gate, weight, dout, eps=1e-6):
    """Gradients (do, dgate, dweight) of sum(out * dout)."""
    o = np.asarray(o, np.float64)
    gate = np.asarray(gate, np.float64)
    weight = np.asarray(weight, np.float64)
    dout = np.asarray(dout, np.float64)
    D = o.shape[-1]
    r = 1.0 / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)
    n = o * r
    sg = _sig(gate)
    a = gate * sg                               # SiLU(gate)
    dn = dout * weight * a
    do = r * (dn - n * np.sum(dn * n, axis=-1, keepdims=True) / D)
    dgate = dout * n * weight * (sg + gate * sg * (1.0 - sg))
    dweight = np.sum(dout * n * a, axis=(0, 1, 2))
    return do, dgate, dweight
