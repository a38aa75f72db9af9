"""The synthetic workloads the mixer is checked and timed on.

Shapes follow the pre-training runs of the Primus hybrid-LLM pretraining blog
(MI355X), sections "The models we trained" and "Recipe" (bf16, sequence
length 2048, 300M and 1B pure-GDN / pure-KDA models), scaled to one GPU; the
long-context case mirrors the 1M-token context of the zebra_qwen3 7MLA+21GDN
SFT guide (section 4.2, context and training length).  Inputs come from
``inputs.make_inputs`` with seed 0.
"""
from __future__ import annotations

import dataclasses


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    H: int
    dk: int
    dv: int
    chunk: int
    kda: bool = False
    dtype: str = "bf16"
    g_mean: float = 2.0
    h0_std: float | None = None
    fwd_only: bool = False
    delta: bool = True  # False: the Mamba2 mixer (scalar gate, no delta rule)
    block: bool = False  # the mixer with its fused neighbours (short conv, gated norm)
    conv_width: int = 4
    g_dtype: str = "f32"  # "bf16": KDA's bf16-gate variant (g and dg in bf16)

    @property
    def mixer(self) -> str:
        return "kda" if self.kda else ("gdn" if self.delta else "mamba2")

    @property
    def tokens(self) -> int:
        return self.B * self.T

    def make_block(self, device="cpu", seed: int = 0, B: int | None = None):
        from .inputs import make_block_inputs
        return make_block_inputs(self.B if B is None else B, self.T, self.H, self.dk,
                                 self.conv_width, kda=self.kda, dtype=self.dtype,
                                 g_mean=self.g_mean, seed=seed, device=device)

    def make(self, device="cpu", seed: int = 0, with_dht: bool = False, T: int | None = None,
             B: int | None = None):
        from .inputs import make_inputs
        return make_inputs(self.B if B is None else B, self.T if T is None else T, self.H,
                           self.dk, self.dv, kda=self.kda, dtype=self.dtype,
                           g_mean=self.g_mean, h0_std=self.h0_std, with_dht=with_dht,
                           seed=seed, device=device, g_dtype=self.g_dtype)


GDN_TINY_FP32 = Workload("gdn_tiny_fp32_B1_T64_H2_d16_C16", 1, 64, 2, 16, 16, 16, dtype="f32")
GDN_300M_BF16 = Workload("gdn_300m_bf16_B16_T2048_H8_d128_C64", 16, 2048, 8, 128, 128, 64)
KDA_300M_BF16 = Workload("kda_300m_bf16_B16_T2048_H8_d128_C64", 16, 2048, 8, 128, 128, 64,
                         kda=True)
# KDA with the gate and its gradient in bf16 (half the gate traffic).
KDA_300M_BF16_G16 = Workload("kda_300m_bf16_g16_B16_T2048_H8_d128_C64", 16, 2048, 8, 128, 128,
                             64, kda=True, g_dtype="bf16")
# The Mamba2 mixer of the same model list (the scalar-gated state GDN extends
# with the delta rule) at the 300M pre-training shape.
MAMBA2_300M_BF16 = Workload("mamba2_300m_bf16_B16_T2048_H8_d128_C64", 16, 2048, 8, 128, 128, 64,
                            delta=False)
# The GDN layer's token-mixing path at the 300M shape: short convolutions of
# the q, k, v projections (width 4, q and k L2-normalised), the mixer, and the
# gated RMS norm of its output, forward and backward.
GDN_BLOCK_300M_BF16 = Workload("gdn_block_300m_bf16_B16_T2048_H8_d128_C64_W4", 16, 2048, 8, 128,
                               128, 64, block=True)
GDN_1B_BF16_H0 = Workload("gdn_1b_bf16_h0_B8_T2048_H16_d128_C64", 8, 2048, 16, 128, 128, 64,
                          h0_std=0.02)
GDN_1M_FWD_BF16 = Workload("gdn_1m_fwd_bf16_B1_T1048576_H16_d128_C64", 1, 1 << 20, 16, 128,
                           128, 64, g_mean=4.0, fwd_only=True)

# Single-token decode on the same state layout: a serving batch of 256
# sequences x 16 heads (the SFT guide's model has 16 heads), one token each;
# the states (268 MB fp32) exceed the L2.
GDN_DECODE_BF16 = Workload("gdn_decode_bf16_B256_T1_H16_d128", 256, 1, 16, 128, 128, 64,
                           h0_std=0.02, fwd_only=True)
KDA_DECODE_BF16 = Workload("kda_decode_bf16_B256_T1_H16_d128", 256, 1, 16, 128, 128, 64,
                           kda=True, h0_std=0.02, fwd_only=True)

ALL = [GDN_TINY_FP32, GDN_300M_BF16, KDA_300M_BF16, KDA_300M_BF16_G16, MAMBA2_300M_BF16,
       GDN_BLOCK_300M_BF16,
       GDN_1B_BF16_H0,
       GDN_1M_FWD_BF16, GDN_DECODE_BF16, KDA_DECODE_BF16]
BY_NAME = {w.name: w for w in ALL}
