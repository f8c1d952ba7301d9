"""Seeded synthetic workloads for speculative-sampling verification.

Shared by the tests and by ``bench.py``; it holds none of the verification arithmetic (no accept test,
no residual, no overlap). It only draws logits with torch's seeded normal generator and draws the draft
tokens from the draft distribution with the Gumbel-max trick (argmax of logits / T plus Gumbel noise), a
sampler independent of the inverse-CDF code under test.

Five named workloads follow the shapes and value recipes of the verification problem at the vocabularies
of Llama-3 (V = 128256) and Qwen (V = 151936). No model or dataset is involved: the logits stand in for
model outputs.

Logits tensors: target [B, K+1, V] (row K is the bonus row), draft [B, K, V] or drafters [N, B, K, V].
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    K: int
    V: int
    N: int = 1
    dtype: str = "bf16"          # "bf16" or "fp32"
    temperature: float = 1.0
    target_sigma: float = 3.0
    peaks: int = 20              # tokens per target row raised by peak_boost (0 = none)
    peak_boost: float = 8.0
    draft_sigmas: Sequence[float] = (1.5,)   # one per drafter: draft = target + N(0, sigma^2)
    selected: int = 0            # drafter whose samples are the draft tokens
    seed_base: int = 1000        # seeds[b] = seed_base + b  (seed_const overrides)
    seed_const: Optional[int] = None
    gen_seed: int = 1234
    token_seed: Optional[int] = None   # generator seed of the Gumbel noise (default gen_seed + 7)
    deltas: Sequence[float] = ()

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    @property
    def positions(self) -> int:
        """Verified draft positions per call (B * K)."""
        return self.B * self.K

    def algorithmic_bytes(self, with_bonus: bool = True) -> int:
        """One read of every logit the call consumes: target rows (with or without the bonus row)
        plus N draft rows per position."""
        rows = self.B * (self.K + (1 if with_bonus else 0)) + self.N * self.B * self.K
        return rows * self.V * self.elem_bytes

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    # Tiny standard speculative sampling (parity only): fp32, target ~ N(0, 2^2), draft = target + N(0, 1).
    "tiny_sps_v1000": Workload("tiny_sps_v1000", B=4, K=5, V=1000, dtype="fp32", target_sigma=2.0, peaks=0,
                               draft_sigmas=(1.0,), seed_const=1, token_seed=0),
    # Standard chain verify at the Llama-3 vocabulary.
    "sps_llama3_b64_k5": Workload("sps_llama3_b64_k5", B=64, K=5, V=128256, draft_sigmas=(1.5,)),
    # HedgeSpec counterfactual gamma for 7 drafters, drafts from drafter 2.
    "hedgespec_n7_b32_k5": Workload("hedgespec_n7_b32_k5", B=32, K=5, V=128256, N=7,
                                    draft_sigmas=(0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0), selected=2),
    # Cactus constrained acceptance, m = 20 draft positions at the Qwen vocabulary.
    "cactus_qwen_b128_m20": Workload("cactus_qwen_b128_m20", B=128, K=20, V=151936, draft_sigmas=(2.0,),
                                     deltas=(0.0, 0.75, 1.0)),
    # Large pool: 21 drafters with sigma spread over [0.3, 6], T = 0.7, fused verify of drafter 4.
    "hedgespec_n21_b256_k8": Workload("hedgespec_n21_b256_k8", B=256, K=8, V=151936, N=21, temperature=0.7,
                                      draft_sigmas=tuple(0.3 + i * 5.7 / 20 for i in range(21)), selected=4),
}


def _to_dtype(x: torch.Tensor, dtype: str) -> torch.Tensor:
    return x.to(torch.bfloat16) if dtype == "bf16" else x.to(torch.float32)


def _gumbel_argmax(logits: torch.Tensor, temperature: float, gen: torch.Generator) -> torch.Tensor:
    u = torch.rand(logits.shape, generator=gen, device=logits.device, dtype=torch.float32)
    u.clamp_(min=1e-20, max=1.0 - 1e-7)
    g = -torch.log(-torch.log(u))
    return torch.argmax(logits.float() / temperature + g, dim=-1).to(torch.int32)


def make(w: Workload, device="cpu"):
    """Draw the workload's tensors on `device`. Returns a dict with target, draft (N == 1) or
    drafters (N > 1; draft is then drafters[selected]), tokens [B,K] int32, seeds [B] int64 (uint64
    values), temperature, selected."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(w.gen_seed)
    B, K, V = w.B, w.K, w.V
    target = torch.randn((B, K + 1, V), generator=gen, device=device, dtype=torch.float32)
    target.mul_(w.target_sigma)
    if w.peaks > 0:
        idx = torch.randint(0, V, (B, K + 1, w.peaks), generator=gen, device=device)
        target.scatter_(-1, idx, target.gather(-1, idx) + w.peak_boost)
    target_c = _to_dtype(target, w.dtype)
    base = target[:, :K]
    drafters = []
    for sigma in w.draft_sigmas:
        d = torch.randn((B, K, V), generator=gen, device=device, dtype=torch.float32)
        d.mul_(sigma).add_(base)
        drafters.append(_to_dtype(d, w.dtype))
        del d
    del target, base
    tgen = torch.Generator(device=device)
    tgen.manual_seed(w.token_seed if w.token_seed is not None else w.gen_seed + 7)
    tokens = _gumbel_argmax(drafters[w.selected], w.temperature, tgen)
    if w.seed_const is not None:
        seeds = torch.full((B,), w.seed_const, dtype=torch.int64, device=device)
    else:
        seeds = torch.arange(B, dtype=torch.int64, device=device) + w.seed_base
    out = dict(target=target_c, tokens=tokens.contiguous(), seeds=seeds, temperature=w.temperature,
               selected=w.selected, workload=w)
    if len(drafters) == 1:
        out["draft"] = drafters[0]
    else:
        out["drafters"] = torch.stack(drafters, 0)
        out["draft"] = out["drafters"][w.selected]
    return out


def to_numpy_logits(x: torch.Tensor):
    """bf16 -> numpy uint16 bit patterns, fp32 -> numpy float32 (the oracle's input format)."""
    x = x.detach().to("cpu").contiguous()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy().view("uint16")
    return x.numpy()
