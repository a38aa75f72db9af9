"""Seeded synthetic inputs for the GDN / KDA mixers.

This module holds no arithmetic of the method itself: it only draws random
tensors and applies the input pre-processing that sits outside the mixer
(L2 normalisation of q and k, the 1/sqrt(dk) query scale, sigmoid for beta,
logsigmoid for the log forget gate).  The oracle and the CUDA path both take
their inputs from here and see identical bytes.

Recipe (one ``torch.Generator`` seeded with ``seed``; draws in this order, all
fp32 normal): q, k, v, beta-logits, g-logits, h0 (only if ``h0_std``), dO,
dht (only if ``with_dht``).

* q, k ~ N(0,1), L2-normalised over the key dimension per (b,t,h); q is then
  scaled by 1/sqrt(dk).
* v ~ N(0,1); dO ~ N(0,1); dht ~ N(0,1).
* beta = sigmoid(N(0,1)).
* g = logsigmoid(N(g_mean,1)); shape [B,T,H] (scalar gate per head, GDN) or
  [B,T,H,dk] (one gate per key dimension, KDA).
* h0 ~ N(0, h0_std) in fp32 when ``h0_std`` is given, else no initial state.

q, k, v and dO are rounded to ``dtype`` (round-to-nearest-even for bf16);
g, beta, h0 and dht stay fp32 (g is rounded to bf16 with ``g_dtype="bf16"``,
KDA's bf16-gate variant).  These are the pre-training shapes and value
ranges of the Primus hybrid-LLM pretraining blog (MI355X), sections "The
models we trained" and "Recipe": bf16, sequence length 2048; the pages' own
data set (FineWeb-Edu) is replaced by these synthetic draws.
"""
from __future__ import annotations

import dataclasses
import math

import torch
import torch.nn.functional as F


@dataclasses.dataclass
class MixerInputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    g: torch.Tensor
    beta: torch.Tensor
    h0: torch.Tensor | None
    do: torch.Tensor
    dht: torch.Tensor | None
    kda: bool

    def to(self, device) -> "MixerInputs":
        conv = lambda x: None if x is None else x.to(device).contiguous()
        return MixerInputs(conv(self.q), conv(self.k), conv(self.v), conv(self.g),
                           conv(self.beta), conv(self.h0), conv(self.do), conv(self.dht),
                           self.kda)

    def select(self, pairs) -> "MixerInputs":
        """Sub-problem holding only the (b, h) sequences listed in ``pairs``.

        The result has B = len(pairs) and H = 1 (sequences are independent)."""
        def tok(x):
            return torch.stack([x[b, :, h] for b, h in pairs], 0).unsqueeze(2).contiguous()

        def st(x):
            return None if x is None else torch.stack([x[b, h] for b, h in pairs], 0).unsqueeze(1).contiguous()

        return MixerInputs(tok(self.q), tok(self.k), tok(self.v), tok(self.g), tok(self.beta),
                           st(self.h0), tok(self.do), st(self.dht), self.kda)


_DT = {"bf16": torch.bfloat16, "f32": torch.float32, "fp32": torch.float32}


def make_inputs(B: int, T: int, H: int, dk: int, dv: int, *, kda: bool = False,
                dtype: str = "bf16", g_mean: float = 2.0, h0_std: float | None = None,
                with_dht: bool = False, seed: int = 0, device="cpu",
                t_slice: int = 1 << 16, g_dtype: str = "f32") -> MixerInputs:
    """Draw one seeded input set (see the module docstring for the recipe).

    Large tensors are drawn per batch row in slices of ``t_slice`` tokens so
    that no full fp32 temporary of a long sequence is held at once.  The bytes
    are a deterministic function of ``seed``, ``device``, the shapes and
    ``t_slice`` (leave it at its default so that every caller sees the same
    draws).
    """
    dt = _DT[dtype]
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)

    def normal_tokens(D, post, out_dtype, mean=0.0):
        out = torch.empty((B, T, H, D) if D else (B, T, H), dtype=out_dtype, device=device)
        shape_rest = (H, D) if D else (H,)
        for b in range(B):
            for t0 in range(0, T, t_slice):
                t1 = min(T, t0 + t_slice)
                x = torch.randn((t1 - t0,) + shape_rest, generator=gen, device=device,
                                dtype=torch.float32)
                if mean:
                    x += mean
                out[b, t0:t1] = post(x).to(out_dtype)
        return out

    def l2n(scale):
        return lambda x: F.normalize(x, p=2.0, dim=-1) * scale

    q = normal_tokens(dk, l2n(1.0 / math.sqrt(dk)), dt)
    k = normal_tokens(dk, l2n(1.0), dt)
    v = normal_tokens(dv, lambda x: x, dt)
    beta = normal_tokens(0, torch.sigmoid, torch.float32)
    # g_dtype "bf16" (KDA's bf16-gate variant): the same draws rounded to bf16
    g = normal_tokens(dk if kda else 0, F.logsigmoid, _DT[g_dtype], mean=g_mean)
    h0 = None
    if h0_std is not None:
        h0 = (torch.randn((B, H, dk, dv), generator=gen, device=device) * h0_std).float()
    do = normal_tokens(dv, lambda x: x, dt)
    dht = None
    if with_dht:
        dht = torch.randn((B, H, dk, dv), generator=gen, device=device).float()
    return MixerInputs(q, k, v, g, beta, h0, do, dht, kda)


@dataclasses.dataclass
class NeighbourInputs:
    """Inputs of the fused neighbours (short convolution and gated norm)."""
    x: torch.Tensor       # [B, T, H*D]  projection output (conv input)
    w: torch.Tensor       # [H*D, W]     fp32 conv taps
    dz: torch.Tensor      # [B, T, H*D]  gradient of the conv output
    o: torch.Tensor       # [B, T, H, D] mixer output (norm input)
    gate: torch.Tensor    # [B, T, H, D] gate projection
    weight: torch.Tensor  # [D]          fp32 norm weight
    dout: torch.Tensor    # [B, T, H, D] gradient of the norm output

    def to(self, device) -> "NeighbourInputs":
        return NeighbourInputs(*(getattr(self, f.name).to(device).contiguous()
                                 for f in dataclasses.fields(self)))


def make_neighbour_inputs(B: int, T: int, H: int, D: int, W: int = 4, *, dtype: str = "bf16",
                          seed: int = 0, device="cpu") -> NeighbourInputs:
    """Seeded inputs of the short convolution and the gated norm.

    Recipe (one ``torch.Generator`` seeded with ``seed``; draws in this order):
    x ~ N(0,1) [B,T,H*D]; w ~ U(-1/sqrt(W), 1/sqrt(W)) [H*D,W] (the default
    initialisation of a depthwise convolution); dz ~ N(0,1); o ~ N(0,1)
    [B,T,H,D]; gate ~ N(0,1); weight = 1 + 0.1 N(0,1) [D]; dout ~ N(0,1).
    x, dz, o, gate and dout are rounded to ``dtype``; w and weight stay fp32.
    """
    gen = torch.Generator().manual_seed(seed)
    dt = {"bf16": torch.bfloat16, "f32": torch.float32}[dtype]
    n = lambda *s: torch.randn(*s, generator=gen, dtype=torch.float32)
    x = n(B, T, H * D)
    w = (torch.rand(H * D, W, generator=gen, dtype=torch.float32) * 2 - 1) / math.sqrt(W)
    dz = n(B, T, H * D)
    o = n(B, T, H, D)
    gate = n(B, T, H, D)
    weight = 1 + 0.1 * n(D)
    dout = n(B, T, H, D)
    r = lambda t: t.to(dt).contiguous()
    out = NeighbourInputs(r(x), w.contiguous(), r(dz), r(o), r(gate), weight.contiguous(), r(dout))
    return out.to(device) if str(device) != "cpu" else out


@dataclasses.dataclass
class BlockInputs:
    """Inputs of the mixer with its neighbours: the q, k, v projections before
    their short convolutions, the gate and the norm, and the gradient of the
    block output."""
    xq: torch.Tensor      # [B, T, H*D]
    xk: torch.Tensor
    xv: torch.Tensor
    wq: torch.Tensor      # [H*D, W] fp32
    wk: torch.Tensor
    wv: torch.Tensor
    g: torch.Tensor       # [B, T, H] (GDN) or [B, T, H, D] (KDA) fp32, log forget gate
    beta: torch.Tensor    # [B, T, H] fp32
    gate: torch.Tensor    # [B, T, H, D]
    weight: torch.Tensor  # [D] fp32
    dout: torch.Tensor    # [B, T, H, D]

    def to(self, device) -> "BlockInputs":
        return BlockInputs(*(getattr(self, f.name).to(device).contiguous()
                             for f in dataclasses.fields(self)))


def make_block_inputs(B: int, T: int, H: int, D: int, W: int = 4, *, kda: bool = False,
                      dtype: str = "bf16", g_mean: float = 2.0, seed: int = 0,
                      device="cpu") -> BlockInputs:
    """Seeded inputs of the mixer block (one ``torch.Generator`` seeded with
    ``seed``; draws in this order): xq, xk, xv ~ N(0,1) [B,T,H*D]; wq, wk, wv ~
    U(-1/sqrt(W), 1/sqrt(W)) [H*D,W]; beta = sigmoid(N(0,1)) [B,T,H]; g =
    logsigmoid(N(g_mean,1)) [B,T,H] or [B,T,H,D]; gate ~ N(0,1) [B,T,H,D];
    weight = 1 + 0.1 N(0,1) [D]; dout ~ N(0,1).  Token tensors are rounded
    to ``dtype``; weights, g and beta stay fp32.  Drawn on the CPU (the same
    values on every device), then moved."""
    gen = torch.Generator().manual_seed(seed)
    dt = {"bf16": torch.bfloat16, "f32": torch.float32}[dtype]
    n = lambda *s: torch.randn(*s, generator=gen, dtype=torch.float32)
    u = lambda: (torch.rand(H * D, W, generator=gen, dtype=torch.float32) * 2 - 1) / math.sqrt(W)
    r = lambda t: t.to(dt).contiguous()
    xq, xk, xv = r(n(B, T, H * D)), r(n(B, T, H * D)), r(n(B, T, H * D))
    wq, wk, wv = u(), u(), u()
    beta = torch.sigmoid(n(B, T, H))
    g = F.logsigmoid(n(B, T, H, D) + g_mean if kda else n(B, T, H) + g_mean)
    gate = r(n(B, T, H, D))
    weight = 1 + 0.1 * n(D)
    dout = r(n(B, T, H, D))
    out = BlockInputs(xq, xk, xv, wq, wk, wv, g.contiguous(), beta.contiguous(), gate, weight, dout)
    return out.to(device) if str(device) != "cpu" else out
