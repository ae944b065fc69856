"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic (no quantisation, routing, alignment or MLP).  Both the
CUDA path and the CPU oracle consume exactly the tensors made here.

Recipe (the pages give no workloads, so these stand in for them):

* hidden states x ~ N(0, 1), rounded to bf16;
* router logits ~ N(0, 1) in fp32, plus an optional per-expert bias row:
    - ``normal``: b_e ~ N(0, 1.5), drawn once per seed (skewed prefill load);
    - ``zipf``:   b_e = -2 * s * ln(r_e) with s = 1.1 and r_e the rank of
      expert e in a seeded permutation of 1..E (Zipf-like popularity, so some
      experts receive no token at small T);
* expert weights ~ N(0, 0.02) in fp32, rounded to bf16, one expert at a
  time so that the Mixtral-sized tensors never exist twice.

Every tensor gets its own stream: torch.Generator seeded with
(seed * 1009 + tag).
"""

from __future__ import annotations

from dataclasses import dataclass, field

import torch

_TAG_X, _TAG_LOGITS, _TAG_BIAS, _TAG_W13, _TAG_W2 = 1, 2, 3, 4, 5


def _gen(seed: int, tag: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1009 + tag)
    return g


def hidden_states(T: int, H: int, seed: int = 0, device="cpu") -> torch.Tensor:
    """bf16 [T, H] ~ N(0, 1)."""
    g = _gen(seed, _TAG_X, device)
    return torch.randn(T, H, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def expert_bias(E: int, kind: str | None, seed: int = 0) -> torch.Tensor | None:
    """Per-expert logit bias (fp32 [E]) for the skewed-load workloads."""
    if kind is None or kind == "none":
        return None
    g = _gen(seed, _TAG_BIAS, "cpu")
    if kind == "normal":
        return torch.randn(E, generator=g, dtype=torch.float32) * 1.5
    if kind == "zipf":
        rank = torch.randperm(E, generator=g).to(torch.float64) + 1.0
        return (-2.0 * 1.1 * torch.log(rank)).to(torch.float32)
    raise ValueError(f"unknown bias kind {kind!r}")


def router_logits(T: int, E: int, seed: int = 0, bias: str | None = None,
                  device="cpu") -> torch.Tensor:
    """fp32 [T, E] ~ N(0, 1) (+ per-expert bias row)."""
    g = _gen(seed, _TAG_LOGITS, device)
    lg = torch.randn(T, E, generator=g, device=device, dtype=torch.float32)
    b = expert_bias(E, bias, seed)
    if b is not None:
        lg = lg + b.to(device)
    return lg


def expert_weights(E: int, N: int, K: int, seed: int = 0, which: str = "w13",
                   device="cpu", std: float = 0.02, experts=None) -> torch.Tensor:
    """bf16 [len(experts), N, K] ~ N(0, std), generated expert by expert.

    Expert e always gets the same values whatever subset is asked for (its
    generator is seeded by (seed, which, e)), so a test can regenerate one
    expert of a large layer without the others.
    """
    tag = _TAG_W13 if which == "w13" else _TAG_W2
    experts = range(E) if experts is None else experts
    experts = list(experts)
    out = torch.empty(len(experts), N, K, dtype=torch.bfloat16, device=device)
    for i, e in enumerate(experts):
        g = _gen(seed * 131 + e, tag, device)
        out[i] = (torch.randn(N, K, generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)
    return out


@dataclass(frozen=True)
class Workload:
    """One synthetic MoE layer configuration."""
    name: str
    E: int
    k: int
    H: int
    I: int
    Ts: tuple
    renormalize: bool = True
    bias: str | None = None
    bits: int = 8
    group_size: int = -1
    has_zp: bool = False
    notes: dict = field(default_factory=dict, compare=False)

    def bytes_per_expert(self) -> float:
        """Weight bytes one touched expert streams (weights + scales + zeros)."""
        n13, n2 = 2 * self.I * self.H, self.H * self.I
        if self.bits == 8:
            return n13 + n2 + 4 * (2 * self.I + self.H)
        gs = self.group_size
        q = (n13 + n2) / 2
        sc = 2 * (2 * self.I * (self.H // gs) + self.H * (self.I // gs))
        zp = (self.I * (self.H // gs) + (self.H // 2) * (self.I // gs)) if self.has_zp else 0
        return q + sc + zp

    def flops(self, T: int) -> float:
        """Algorithmic flops of the two expert GEMMs: 6 * H * I * k * T."""
        return 6.0 * self.H * self.I * self.k * T


WORKLOADS = {
    "tiny": Workload("tiny", E=8, k=2, H=128, I=256, Ts=(16,)),
    "mixtral_decode": Workload("mixtral_decode", E=8, k=2, H=4096, I=14336, Ts=(1, 8, 32, 64)),
    "mixtral_prefill": Workload("mixtral_prefill", E=8, k=2, H=4096, I=14336,
                                Ts=(1024, 4096, 8192), bias="normal"),
    "fine": Workload("fine", E=128, k=8, H=2048, I=768, Ts=(1, 64, 512, 4096), bias="zipf"),
    "w4a16": Workload("w4a16", E=64, k=6, H=2048, I=1408, Ts=(1, 32, 2048), bits=4,
                      group_size=128, has_zp=True),
}
