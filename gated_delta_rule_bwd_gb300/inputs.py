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
g, beta, h0 and dht stay fp32.  These are the pre-training shapes and value
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
                t_slice: int = 1 << 16) -> MixerInputs:
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
    g = normal_tokens(dk if kda else 0, F.logsigmoid, torch.float32, mean=g_mean)
    h0 = None
    if h0_std is not None:
        h0 = (torch.randn((B, H, dk, dv), generator=gen, device=device) * h0_std).float()
    do = normal_tokens(dv, lambda x: x, dt)
    dht = None
    if with_dht:
        dht = torch.randn((B, H, dk, dv), generator=gen, device=device).float()
    return MixerInputs(q, k, v, g, beta, h0, do, dht, kda)
