"""Seeded synthetic BF16 checkpoints for the delta-sync workloads (input generation only).

This module draws the inputs and nothing else: normal weights rounded to BF16, the changed
positions and the mutation mix of each workload.  It contains none of the codec's arithmetic
(no classification, position coding, packing or checksum) and imports neither the CUDA
library nor the oracle; both sides' tests and bench.py use it to build identical inputs.

Mutation mix at a changed position (the pages' observation that most BF16 updates move only
the mantissa, fewer move the exponent and sign flips are rarer still):
  0.97  XOR a uniform nonzero 7-bit value into the mantissa,
  0.029 exponent field +1 or -1 (coin flip), skipped when the result would be 0 or 255,
  0.001 flip the sign bit.
Positions are drawn as independent Bernoulli(rate) per element.

Workloads (sizes as named by the task's configurations):
  single_1m      one 1024x1024 tensor, N(0, 0.02), 2% changed
  dense7b        7B dense decoder: embed 32000x4096; 32 x (q,k,v,o 4096x4096, gate/up
                 11008x4096, down 4096x11008, two RMSNorm 4096 = 1 + N(0, 1e-3)); final norm;
                 lm_head 32000x4096; 2% per tensor
  sweep14336     one 14336x4096 tensor at 0.085%, 1%, 2%, 3%, 5%; plus a clustered 2% variant
                 with all changes in a seeded 10% of rows (20% in-row)
  moe30b         48 layers x (128 experts x gate/up 768x2048, down 2048x768; q 4096x2048,
                 k/v 512x2048, o 2048x4096, router 128x2048); embed and lm_head 151936x2048;
                 3% overall, 80% of the changed elements in 8 seeded experts per layer
  dense1g        one tensor of 2^29 elements N(0, 1); new = bf16(old + bf16(1e-3 * N(0,1)))
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

SEED = 0x5EED


@dataclass
class Spec:
    name: str
    shape: tuple
    std: float = 0.02
    mean: float = 0.0
    rate: float = 0.02
    rows_hot: float | None = None   # clustered: fraction of rows that take all changes
    kind: str = "mix"                # "mix" (mutation mix) or "additive" (dense1g rule)
    tid: int = 0                     # tensor id (part of the seed)

    @property
    def numel(self) -> int:
        n = 1
        for s in self.shape:
            n *= s
        return n


def _gen(device, seed: int, tid: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + tid * 7919 + 17) & ((1 << 63) - 1))
    return g


def bf16_normal(shape, std: float, mean: float, g: torch.Generator, device) -> torch.Tensor:
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return (x * std + mean).to(torch.bfloat16)


def mutate(old: torch.Tensor, rate: float, g: torch.Generator,
           row_mask: torch.Tensor | None = None) -> torch.Tensor:
    """Returns a copy of `old` (bfloat16) with the mutation mix applied at Bernoulli(rate)
    positions (restricted to rows where row_mask is true, when given)."""
    device = old.device
    bits = old.reshape(-1).view(torch.int16).to(torch.int32) & 0xFFFF
    n = bits.numel()
    pick = torch.rand(n, generator=g, device=device) < rate
    if row_mask is not None:
        cols = old.shape[-1]
        pick &= row_mask.repeat_interleave(cols)
    idx = pick.nonzero().squeeze(1)
    k = idx.numel()
    if k:
        kind = torch.rand(k, generator=g, device=device)
        mant = torch.randint(1, 128, (k,), generator=g, device=device, dtype=torch.int32)
        step = torch.randint(0, 2, (k,), generator=g, device=device, dtype=torch.int32) * 2 - 1
        b = bits[idx]
        e = (b >> 7) & 0xFF
        e2 = e + step
        exp_ok = (e2 > 0) & (e2 < 255)
        b_mant = b ^ mant
        b_exp = torch.where(exp_ok, (b & 0x807F) | (e2.clamp(0, 255) << 7), b)
        b_sign = b ^ 0x8000
        b = torch.where(kind < 0.97, b_mant, torch.where(kind < 0.999, b_exp, b_sign))
        bits[idx] = b
    out = (bits - ((bits >> 15) << 16)).to(torch.int16)   # [0, 65535] -> two's complement
    return out.view(torch.bfloat16).reshape(old.shape)


def make_pair(spec: Spec, seed: int = SEED, device="cuda") -> tuple[torch.Tensor, torch.Tensor]:
    """(old, new) bfloat16 tensors of one tensor spec."""
    g = _gen(device, seed, spec.tid)
    if spec.kind == "additive":
        old = torch.randn(spec.shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
        noise = torch.randn(spec.shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
        new = old + 1e-3 * noise   # bf16 tensor arithmetic: each op rounds to bf16
        return old, new
    old = bf16_normal(spec.shape, spec.std, spec.mean, g, device)
    row_mask = None
    if spec.rows_hot is not None:
        rows = spec.shape[0]
        hot = max(1, int(round(rows * spec.rows_hot)))
        perm = torch.randperm(rows, generator=g, device=device)[:hot]
        row_mask = torch.zeros(rows, dtype=torch.bool, device=device)
        row_mask[perm] = True
    new = mutate(old, spec.rate, g, row_mask)
    return old, new


# ------------------------------------------------------------------------------ workloads

def single_1m() -> list[Spec]:
    return [Spec("w", (1024, 1024))]


def dense7b(layers: int = 32) -> list[Spec]:
    h, f, v = 4096, 11008, 32000
    specs = [Spec("embed", (v, h))]
    for l in range(layers):
        p = f"layers.{l}."
        specs += [Spec(p + "q", (h, h)), Spec(p + "k", (h, h)), Spec(p + "v", (h, h)),
                  Spec(p + "o", (h, h)), Spec(p + "gate", (f, h)), Spec(p + "up", (f, h)),
                  Spec(p + "down", (h, f)),
                  Spec(p + "norm1", (h,), std=1e-3, mean=1.0),
                  Spec(p + "norm2", (h,), std=1e-3, mean=1.0)]
    specs += [Spec("norm", (h,), std=1e-3, mean=1.0), Spec("lm_head", (v, h))]
    for i, s in enumerate(specs):
        s.tid = i
    return specs


SWEEP_RATES = (0.00085, 0.01, 0.02, 0.03, 0.05)


def sweep14336() -> list[Spec]:
    specs = [Spec(f"rate{r:g}", (14336, 4096), rate=r, tid=i) for i, r in enumerate(SWEEP_RATES)]
    specs.append(Spec("clustered", (14336, 4096), rate=0.2, rows_hot=0.1, tid=len(specs)))
    return specs


def moe30b(layers: int = 48, experts: int = 128, hot_experts: int = 8,
           total_rate: float = 0.03, hot_share: float = 0.8, seed: int = SEED) -> list[Spec]:
    hdim, inter, vocab = 2048, 768, 151936
    g = torch.Generator()
    g.manual_seed(seed + 3)
    hot = [set(torch.randperm(experts, generator=g)[:hot_experts].tolist()) for _ in range(layers)]
    specs: list[Spec] = [Spec("embed", (vocab, hdim))]
    for l in range(layers):
        p = f"layers.{l}."
        for e in range(experts):
            tag = "hot" if e in hot[l] else "cold"
            specs += [Spec(p + f"experts.{e}.gate", (inter, hdim), kind=tag),
                      Spec(p + f"experts.{e}.up", (inter, hdim), kind=tag),
                      Spec(p + f"experts.{e}.down", (hdim, inter), kind=tag)]
        specs += [Spec(p + "q", (4096, hdim)), Spec(p + "k", (512, hdim)),
                  Spec(p + "v", (512, hdim)), Spec(p + "o", (hdim, 4096)),
                  Spec(p + "router", (experts, hdim))]
    specs.append(Spec("lm_head", (vocab, hdim)))
    n_tot = sum(s.numel for s in specs)
    n_hot = sum(s.numel for s in specs if s.kind == "hot")
    k = total_rate * n_tot
    hot_rate = min(1.0, hot_share * k / n_hot)
    cold_rate = (1 - hot_share) * k / (n_tot - n_hot)
    for i, s in enumerate(specs):
        s.rate = hot_rate if s.kind == "hot" else cold_rate
        s.kind = "mix"
        s.tid = i
    return specs


def dense1g() -> list[Spec]:
    return [Spec("w", (1 << 29,), kind="additive")]


WORKLOADS = {
    "single_1m": single_1m,
    "dense7b": dense7b,
    "sweep14336": sweep14336,
    "moe30b": moe30b,
    "dense1g": dense1g,
}


def specs(name: str) -> list[Spec]:
    return WORKLOADS[name]()
