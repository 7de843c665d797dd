"""Seeded synthetic workloads for exact attention.

This module only names shapes and draws random inputs; it holds none of the
attention arithmetic.  It is the one piece of code that both the CUDA path's
callers and the CPU oracle's callers use, so that both sides see the same bf16
bit patterns.

Recipe: every tensor is drawn iid N(0, 1) in fp32 by a CPU `torch.Generator`
seeded per tensor (Q: seed, K: seed + 1, V: seed + 2, dO: seed + 3; base
seed 0) and rounded to bf16 (round to nearest even).  Layout [B, H, N, d],
contiguous; K and V carry H_kv heads.
"""

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    N: int
    d: int
    causal: bool
    backward: bool

    @property
    def scale(self):
        return 1.0 / math.sqrt(self.d)

    def fwd_flops(self):
        """4 B Hq N^2 d, halved under the causal mask."""
        f = 4.0 * self.B * self.Hq * self.N * self.N * self.d
        return f / 2 if self.causal else f

    def bwd_flops(self):
        """10 B Hq N^2 d (five products including the recompute), halved if causal."""
        f = 10.0 * self.B * self.Hq * self.N * self.N * self.d
        return f / 2 if self.causal else f

    def describe(self):
        kind = "causal" if self.causal else "non-causal"
        heads = f"Hq{self.Hq} Hkv{self.Hkv}" if self.Hkv != self.Hq else f"H{self.Hq}"
        step = "fwd+bwd" if self.backward else "fwd"
        return f"{kind} {step} B{self.B} {heads} N{self.N} d{self.d} bf16"


# The workloads of the attention path: five at d = 64 and 128 (the training
# step and the forward targets), and forward workloads at head dimensions 96
# and 256.
WORKLOADS = {
    "single_head_n256": Workload("single_head_n256", 1, 1, 1, 256, 64, False, False),
    "causal_n4096_d64": Workload("causal_n4096_d64", 2, 8, 8, 4096, 64, True, False),
    "causal_n8192_d128": Workload("causal_n8192_d128", 4, 16, 16, 8192, 128, True, False),
    "causal_gqa_n16384_d128": Workload("causal_gqa_n16384_d128", 1, 32, 8, 16384, 128, True,
                                       False),
    "causal_train_n4096_d64": Workload("causal_train_n4096_d64", 2, 8, 8, 4096, 64, True, True),
    "causal_n8192_d96": Workload("causal_n8192_d96", 4, 16, 16, 8192, 96, True, False),
    "causal_n8192_d256": Workload("causal_n8192_d256", 2, 16, 16, 8192, 256, True, False),
    "causal_gqa_n16384_d256": Workload("causal_gqa_n16384_d256", 1, 32, 8, 16384, 256, True,
                                       False),
}


def _normal_bf16(shape, seed):
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return torch.randn(*shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def make_inputs(B, Hq, Hkv, N, d, seed=0, with_grad=False, Nk=None):
    """Seeded bf16 CPU tensors q [B,Hq,N,d], k/v [B,Hkv,Nk,d] (and dO like q)."""
    Nk = N if Nk is None else Nk
    out = {
        "q": _normal_bf16((B, Hq, N, d), seed),
        "k": _normal_bf16((B, Hkv, Nk, d), seed + 1),
        "v": _normal_bf16((B, Hkv, Nk, d), seed + 2),
    }
    if with_grad:
        out["do"] = _normal_bf16((B, Hq, N, d), seed + 3)
    return out


def workload_inputs(w, seed=0):
    return make_inputs(w.B, w.Hq, w.Hkv, w.N, w.d, seed=seed, with_grad=w.backward)


def as_f64(t):
    """Exact widening of a bf16 tensor to a float64 numpy array."""
    return t.to(torch.float64).numpy()
