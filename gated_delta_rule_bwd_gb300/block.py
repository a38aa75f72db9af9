"""The GDN / KDA layer's token-mixing path: the mixer with its fused neighbours.

Forward (per the Primus hybrid-LLM pretraining blog, section "Recipe": the
FLA fusions of the short convolution and the gated norm around the mixer):

    q = conv_q(xq) L2-normalised per head, scaled by D^-1/2
    k = conv_k(xk) L2-normalised per head
    v = conv_v(xv)                              (conv = causal depthwise + SiLU)
    o, ht = mixer(q, k, v, g, beta, h0)         (GDN, or KDA with a per-key gate)
    out = o / sqrt(mean(o^2) + eps) * weight * SiLU(gate)

and the backward in reverse order.  Every step is a call of the C ABI (this
module only composes the binding's calls); the forward keeps the mixer's
saved context for the backward.
"""
from __future__ import annotations

import dataclasses

import torch

import gated_delta_rule_bwd_gb300 as _gdn
from gated_delta_rule_bwd_gb300 import (NORM_EPS, GdnError, gated_rmsnorm_bwd, gated_rmsnorm_fwd,
                                        new_ctx, short_conv_bwd, short_conv_fwd)


@dataclasses.dataclass
class BlockSaved:
    """What ``block_fwd`` keeps for ``block_bwd``."""
    xq: torch.Tensor
    xk: torch.Tensor
    xv: torch.Tensor
    wq: torch.Tensor
    wk: torch.Tensor
    wv: torch.Tensor
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    g: torch.Tensor
    beta: torch.Tensor
    h0: torch.Tensor | None
    o: torch.Tensor
    gate: torch.Tensor
    weight: torch.Tensor
    ctx: torch.Tensor | None
    cu_seqlens: torch.Tensor | None
    chunk: int
    kda: bool
    eps: float


def _heads(xq, g, kda):
    if xq.dim() != 3:
        raise GdnError("the projections must be [B, T, H*D]")
    H = g.shape[2]
    if xq.shape[2] % H:
        raise GdnError("H does not divide the projection width")
    return H, xq.shape[2] // H


def block_fwd(xq, xk, xv, wq, wk, wv, g, beta, gate, weight, h0=None, chunk=64, kda=False,
              ctx=None, eps=NORM_EPS, cu_seqlens=None):
    """Returns ``(out, ht, saved)``: the block output ``[B, T, H, D]``, the
    mixer's final state and what the backward needs.  ``ctx`` (optional) is a
    reusable saved-context buffer of ``new_ctx`` size; packed sequences
    (``cu_seqlens``) take the mixer's recomputing varlen calls."""
    H, D = _heads(xq, g, kda)
    B, T, _ = xq.shape
    shp = (B, T, H, D)
    q = short_conv_fwd(xq, wq, H, True, D ** -0.5, eps, cu_seqlens).view(shp)
    k = short_conv_fwd(xk, wk, H, True, 1.0, eps, cu_seqlens).view(shp)
    v = short_conv_fwd(xv, wv, H, False, 1.0, eps, cu_seqlens).view(shp)
    mixer = "kda" if kda else "gdn"
    if cu_seqlens is None:
        if ctx is None:
            ctx = new_ctx(q, v, chunk, kda)
        o, ht, ctx = getattr(_gdn, f"{mixer}_fwd_save")(q, k, v, g, beta, h0, chunk=chunk, ctx=ctx)
    else:
        o, ht = getattr(_gdn, f"{mixer}_fwd_varlen")(q, k, v, g, beta, cu_seqlens, h0, chunk=chunk)
        ctx = None
    out = gated_rmsnorm_fwd(o, gate, weight, eps)
    saved = BlockSaved(xq, xk, xv, wq, wk, wv, q, k, v, g, beta, h0, o, gate, weight, ctx,
                       cu_seqlens, chunk, kda, eps)
    return out, ht, saved


def block_bwd(saved: BlockSaved, dout, dht=None):
    """Gradients of ``block_fwd`` for the output gradient ``dout``: a dict with
    dxq, dxk, dxv, dwq, dwk, dwv, dg, dbeta, dgate, dweight and dh0."""
    s = saved
    B, T, H, D = s.q.shape
    do, dgate, dweight = gated_rmsnorm_bwd(s.o, s.gate, s.weight, dout, s.eps)
    mixer = "kda" if s.kda else "gdn"
    if s.cu_seqlens is None:
        gr = getattr(_gdn, f"{mixer}_bwd_saved")(s.q, s.k, s.v, s.g, s.beta, s.h0, do, s.ctx, dht,
                                                 chunk=s.chunk)
    else:
        gr = getattr(_gdn, f"{mixer}_bwd_varlen")(s.q, s.k, s.v, s.g, s.beta, s.cu_seqlens, s.h0,
                                                  do, dht, chunk=s.chunk)
    flat = lambda t: t.view(B, T, H * D)
    dxq, dwq = short_conv_bwd(s.xq, s.wq, flat(gr["dq"]), H, True, D ** -0.5, s.eps, s.cu_seqlens)
    dxk, dwk = short_conv_bwd(s.xk, s.wk, flat(gr["dk"]), H, True, 1.0, s.eps, s.cu_seqlens)
    dxv, dwv = short_conv_bwd(s.xv, s.wv, flat(gr["dv"]), H, False, 1.0, s.eps, s.cu_seqlens)
    return {"dxq": dxq, "dxk": dxk, "dxv": dxv, "dwq": dwq, "dwk": dwk, "dwv": dwv,
            "dg": gr["dg"], "dbeta": gr["dbeta"], "dgate": dgate, "dweight": dweight,
            "dh0": gr.get("dh0")}
