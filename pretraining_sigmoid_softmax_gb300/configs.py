"""The five synthetic MoE-layer workloads, as shapes and switches only.

Each workload is one fine-grained Mixture-of-Experts layer of a decoder LLM training step
(the "Fine-grained MoE" row of "The whole stack, in the open", section "What's inside": a
sigmoid router picks the top experts, a per-expert bias balances the load without a loss
term, and experts run as grouped GEMMs). The softmax top-k router with router z-loss is the
KempnerForge README's other router ("Features", Mixture-of-Experts bullet).

Nothing here computes any part of the layer.
"""
from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int            # tokens in the step (batch x sequence)
    d: int            # d_model
    E: int            # routed experts
    k: int            # experts chosen per token
    f: int            # routed expert SwiGLU width (d_ff)
    f_shared: int     # always-on shared expert width, 0 = no shared expert
    mode: str         # "sigmoid" (bias-steered selection, renormalised gates) or "softmax"
    seed: int
    backward: bool    # forward + backward when true, forward only otherwise
    bias_update: bool # aux-loss-free bias update after backward
    gamma: float = 0.001   # bias update step
    z_coef: float = 0.0    # router z-loss coefficient (softmax mode)
    zipf: bool = False     # skewed expert popularity with a block of never-chosen experts
    bias_rule: str = "sign"  # "sign": b += gamma sign(mean - c); "proportional": gamma (mean - c)/mean
    aux_switch: float = 0.0  # Switch-style load-balancing loss coefficient (0 = off)
    aux_seq: float = 0.0     # sequence-wise load-balancing loss coefficient (0 = off)
    seq_len: int = 0         # tokens per sequence for the sequence-wise loss
    # expert GEMM operands: "bf16"; "fp8" (E4M3 rowwise forward GEMMs); "fp8_dgrad" (also the
    # backward's data-gradient GEMMs on E4M3; weight gradients stay bf16)
    precision: str = "bf16"

    @property
    def fp8(self) -> bool:
        return self.precision in ("fp8", "fp8_dgrad")

    @property
    def fp8_dgrad(self) -> bool:
        return self.precision == "fp8_dgrad"

    @property
    def has_aux(self) -> bool:
        return self.aux_switch != 0.0 or self.aux_seq != 0.0

    @property
    def N(self) -> int:
        """Routed rows: every token is sent to k experts."""
        return self.T * self.k

    @property
    def mode_id(self) -> int:
        return 0 if self.mode == "sigmoid" else 1

    def gemm_flops(self) -> float:
        """Algorithmic grouped-GEMM FLOPs of one step (routed + shared).

        A SwiGLU expert has three bias-free d x f matrices, so one row costs 3 GEMVs of
        2*d*f FLOPs forward; backward is twice the forward (data and weight gradients)."""
        fwd = 6.0 * self.N * self.d * self.f + 6.0 * self.T * self.d * self.f_shared
        return fwd * (3.0 if self.backward else 1.0)

    def with_(self, **kw) -> "MoEConfig":
        return replace(self, **kw)


# Tiny forward-only parity workload.
C0 = MoEConfig("tiny_fwd_T512_d256_E8_k2_f128", T=512, d=256, E=8, k=2, f=128, f_shared=0,
               mode="sigmoid", seed=0, backward=False, bias_update=False)
# Fine-grained sigmoid-routed layer with one shared expert and the bias update.
C1 = MoEConfig("finegrained_T8192_d1024_E64_k8_f256_shared512", T=8192, d=1024, E=64, k=8,
               f=256, f_shared=512, mode="sigmoid", seed=1, backward=True, bias_update=True)
# Softmax top-k without renormalisation, router z-loss 1e-3.
C2 = MoEConfig("softmax_zloss_T16384_d2048_E32_k4_f1024", T=16384, d=2048, E=32, k=4, f=1024,
               f_shared=0, mode="softmax", seed=2, backward=True, bias_update=False,
               z_coef=1e-3)
# Skewed expert load: ragged and empty grouped-GEMM segments.
C3 = MoEConfig("skewed_T32768_d2048_E128_k8_f768", T=32768, d=2048, E=128, k=8, f=768,
               f_shared=0, mode="sigmoid", seed=3, backward=True, bias_update=False, zipf=True)
# Large fine-grained layer with a shared expert and the bias update.
C4 = MoEConfig("large_T65536_d4096_E64_k8_f1536_shared3072", T=65536, d=4096, E=64, k=8,
               f=1536, f_shared=3072, mode="sigmoid", seed=4, backward=True, bias_update=True)

# The Apex-3 step-10 benchmark's layer ("The whole stack, in the open", "Run it yourself":
# 64 experts, expert width 1280, top-4, router bias rate 0.01 with the proportional update,
# micro-batch 6 x 8192 tokens). d_model is not printed there; 2048 is a reading.
C5 = MoEConfig("apex3_T49152_d2048_E64_k4_f1280_proportional", T=49152, d=2048, E=64, k=4,
               f=1280, f_shared=0, mode="sigmoid", seed=5, backward=True, bias_update=True,
               gamma=0.01, bias_rule="proportional")

# The large layer with the load-balancing losses the pages name: Megatron's aux_loss with
# coefficient 1e-3 (handbook summary, section 2.5) and the sequence-wise loss with
# seq_aux_alpha = 1e-3 (Apex-3 training command), over its 16 sequences of 4096 tokens.
C6 = C4.with_(name="large_T65536_d4096_E64_k8_f1536_shared3072_auxlosses", aux_switch=1e-3,
              aux_seq=1e-3, seq_len=4096)

# The large layer with the experts' forward GEMMs on E4M3 rowwise-scaled operands (the Apex-3
# stack's fp8_rowwise precision); the backward stays bf16.
C7 = C4.with_(name="large_T65536_d4096_E64_k8_f1536_shared3072_fp8fwd", precision="fp8")

# The large layer with the data-gradient GEMMs of the backward on E4M3 operands as well (the
# same fp8_rowwise precision carried to the backward; weight gradients stay bf16).
C8 = C4.with_(name="large_T65536_d4096_E64_k8_f1536_shared3072_fp8dgrad", precision="fp8_dgrad")

CONFIGS = {"C0": C0, "C1": C1, "C2": C2, "C3": C3, "C4": C4, "C5": C5, "C6": C6, "C7": C7,
           "C8": C8}
