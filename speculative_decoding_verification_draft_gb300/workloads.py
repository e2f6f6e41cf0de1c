"""Seeded synthetic inputs shaped like the pages' verification workloads.

This module only builds inputs: logits, draft tokens, per-request draft
lengths and temperatures.  It holds none of the verification arithmetic, and
both the CUDA path (tests, benchmark) and the CPU oracle (tests) consume its
outputs, so the two always see the same bytes.

Drafting is simulated the way the pages describe it: the draft model proposes
gamma tokens sampled from its own distribution (greedy requests take the draft
argmax).  The pages use Llama-3.1 target/draft pairs (vocabulary 128256) and
Qwen-class models (152064); the logit recipes below stand in for them:

* ``toy_batch``      -- the 7-token Markov toy of the speculative-decoding blog
  (tables passed in by the caller), logits = ln(table), fp32, T = 1.
* ``gaussian_batch`` -- target ~ N(0, sigma_t^2) i.i.d., draft = target + N(0,
  sigma_d^2).
* ``zipf_batch``     -- target ~ N(0, 2.5^2) - 1.1 * ln(rank) with rank = 1 + a
  seeded permutation of the vocabulary shared by the batch (a Zipf(1.1) prior),
  draft = target + N(0, sigma_b^2) with sigma_b per request.
* ``ragged_batch``   -- per-request gamma in 1..gamma_max, half the requests
  greedy (T = 0) and half sampled (T = 1); rows past a request's gamma, and the
  draft rows of greedy requests, are filled with NaN (they must never be read);
  draft tokens past gamma are set to -7 (they must never be read either).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch


@dataclass
class Batch:
    """One verification batch.  Tensors live on ``device``.

    target [B, gmax+1, V], draft [B, gmax, V] (bf16 or fp32); draft_tokens
    [B, gmax] int32; temperature: float or float32 tensor [B]; gamma: None
    (uniform gmax) or int32 tensor [B].
    """
    target: torch.Tensor
    draft: torch.Tensor
    draft_tokens: torch.Tensor
    temperature: object
    gamma: Optional[torch.Tensor] = None
    meta: dict = field(default_factory=dict)

    @property
    def B(self):
        return self.target.shape[0]

    @property
    def gmax(self):
        return self.target.shape[1] - 1

    @property
    def V(self):
        return self.target.shape[2]

    def algorithmic_bytes(self) -> int:
        """Bytes of every real logit row read once: target rows 0..gamma_b, and
        draft rows 0..gamma_b-1 of sampled requests (greedy requests read no
        draft rows; padding is excluded)."""
        es = self.target.element_size()
        V = self.V
        if self.gamma is None:
            g = np.full(self.B, self.gmax, np.int64)
        else:
            g = self.gamma.cpu().numpy().astype(np.int64)
        if isinstance(self.temperature, torch.Tensor):
            t = self.temperature.cpu().numpy()
        else:
            t = np.full(self.B, float(self.temperature), np.float32)
        real = g >= 0
        rows = np.where(real, g + 1, 0) + np.where(real & (t > 0), g, 0)
        return int(rows.sum()) * V * es

    def to(self, device) -> "Batch":
        mv = lambda x: x.to(device) if isinstance(x, torch.Tensor) else x
        return Batch(mv(self.target), mv(self.draft), mv(self.draft_tokens), mv(self.temperature),
                     mv(self.gamma), dict(self.meta))

    def numpy_logits(self):
        """(target, draft) as numpy: bf16 as uint16 bit patterns, fp32 as float32."""
        def cv(x):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16)
            return x.numpy()
        return cv(self.target), cv(self.draft)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _sample_draft_tokens(draft32: torch.Tensor, temps: torch.Tensor, gen: torch.Generator) -> torch.Tensor:
    """Draft proposals: a sample from softmax(draft / T) for T > 0, the draft
    argmax for T == 0.  draft32 [B, g, V] fp32, temps [B]."""
    B, g, V = draft32.shape
    out = torch.empty(B, g, dtype=torch.int64, device=draft32.device)
    for b in range(B):
        T = float(temps[b])
        if g == 0:
            continue
        if T > 0:
            probs = torch.softmax(draft32[b] / T, dim=-1)
            out[b] = torch.multinomial(probs, 1, generator=gen).squeeze(-1)
        else:
            out[b] = torch.argmax(draft32[b], dim=-1)
    return out.to(torch.int32)


def toy_batch(tables: dict, B: int, gamma: int, seed: int, device="cpu") -> Batch:
    """The blog's Markov toy: B independent rounds, each starting from prev = 0.

    ``tables`` = {"draft": {"prev0": [...], "other": [...]}, "target": {...}}.
    Draft tokens follow the draft chain; row k of each side is the table for
    the previous token (prev = 0 for k = 0, else draft token k-1).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    d0, d1 = np.array(tables["draft"]["prev0"]), np.array(tables["draft"]["other"])
    t0, t1 = np.array(tables["target"]["prev0"]), np.array(tables["target"]["other"])
    V = d0.size
    tok = np.zeros((B, gamma), np.int32)
    prev = np.zeros(B, np.int64)
    cd0, cd1 = np.cumsum(d0), np.cumsum(d1)
    for k in range(gamma):
        u = rng.random(B)
        x0 = np.minimum(np.searchsorted(cd0, u * cd0[-1], side="right"), V - 1)
        x1 = np.minimum(np.searchsorted(cd1, u * cd1[-1], side="right"), V - 1)
        x = np.where(prev == 0, x0, x1)
        tok[:, k] = x
        prev = x
    prevs = np.concatenate([np.zeros((B, 1), np.int64), tok.astype(np.int64)], axis=1)  # [B, g+1]
    lt = np.log(np.stack([t0, t1])).astype(np.float32)
    ld = np.log(np.stack([d0, d1])).astype(np.float32)
    sel = (prevs != 0).astype(np.int64)
    target = lt[sel]                 # [B, g+1, V]
    draft = ld[sel[:, :gamma]]       # [B, g, V]
    return Batch(torch.from_numpy(np.ascontiguousarray(target)).to(device),
                 torch.from_numpy(np.ascontiguousarray(draft)).to(device),
                 torch.from_numpy(tok).to(device), 1.0, None,
                 dict(workload="toy", seed=seed))


def gaussian_batch(B: int, gamma: int, V: int, dtype=torch.bfloat16, temperature: float = 1.0,
                   seed: int = 1, sigma_t: float = 2.0, sigma_d: float = 0.5, device="cpu") -> Batch:
    """target ~ N(0, sigma_t^2) i.i.d.; draft = target + N(0, sigma_d^2)."""
    gen = _gen(seed, device)
    t32 = torch.randn(B, gamma + 1, V, generator=gen, device=device) * sigma_t
    d32 = t32[:, :gamma] + torch.randn(B, gamma, V, generator=gen, device=device) * sigma_d
    target, draft = t32.to(dtype), d32.to(dtype)
    temps = torch.full((B,), float(temperature))
    tok = _sample_draft_tokens(draft.float(), temps, gen)
    return Batch(target, draft, tok, float(temperature), None,
                 dict(workload="gaussian", seed=seed, sigma_t=sigma_t, sigma_d=sigma_d))


def _zipf_target(B, rows, V, gen, device, sigma_t, zipf_s):
    perm = torch.randperm(V, generator=gen, device=device)
    bias = -zipf_s * torch.log((perm + 1).to(torch.float32))
    return torch.randn(B, rows, V, generator=gen, device=device) * sigma_t + bias


def zipf_batch(B: int, gamma: int, V: int, dtype=torch.bfloat16, temperature: float = 0.8,
               seed: int = 2, sigma_range=(0.3, 1.2), sigma_t: float = 2.5, zipf_s: float = 1.1,
               device="cpu", sample_tokens: bool = True) -> Batch:
    """target ~ N(0, sigma_t^2) - zipf_s * ln(rank); draft = target + N(0, sigma_b^2),
    sigma_b ~ U[sigma_range] per request (a fixed sigma when lo == hi)."""
    gen = _gen(seed, device)
    t32 = _zipf_target(B, gamma + 1, V, gen, device, sigma_t, zipf_s)
    lo, hi = sigma_range
    sig = lo + (hi - lo) * torch.rand(B, generator=gen, device=device)
    d32 = t32[:, :gamma] + torch.randn(B, gamma, V, generator=gen, device=device) * sig.view(B, 1, 1)
    target, draft = t32.to(dtype), d32.to(dtype)
    del t32, d32
    temps = torch.full((B,), float(temperature))
    if sample_tokens:
        tok = _sample_draft_tokens(draft.float(), temps, gen)
    else:
        tok = torch.zeros(B, gamma, dtype=torch.int32, device=device)
    return Batch(target, draft, tok, float(temperature), None,
                 dict(workload="zipf", seed=seed, sigma=sig.cpu().tolist()))


def ragged_batch(B: int, gamma_max: int, V: int, dtype=torch.bfloat16, seed: int = 4,
                 sigma_range=(0.2, 1.5), sampled_temperature: float = 1.0,
                 sigma_t: float = 2.5, zipf_s: float = 1.1, device="cpu") -> Batch:
    """Ragged mixed batch: gamma_b ~ U{1..gamma_max}; even requests greedy (T = 0),
    odd requests sampled (T = sampled_temperature).  Unused rows are NaN."""
    gen = _gen(seed, device)
    gam = torch.randint(1, gamma_max + 1, (B,), generator=gen, device=device).to(torch.int32)
    temps = torch.where(torch.arange(B, device=device) % 2 == 0,
                        torch.zeros(B, device=device),
                        torch.full((B,), float(sampled_temperature), device=device)).to(torch.float32)
    t32 = _zipf_target(B, gamma_max + 1, V, gen, device, sigma_t, zipf_s)
    lo, hi = sigma_range
    sig = lo + (hi - lo) * torch.rand(B, generator=gen, device=device)
    d32 = t32[:, :gamma_max] + torch.randn(B, gamma_max, V, generator=gen, device=device) * sig.view(B, 1, 1)
    target, draft = t32.to(dtype), d32.to(dtype)
    del t32, d32
    tok = _sample_draft_tokens(draft.float(), temps.cpu(), gen)
    nan = float("nan")
    for b in range(B):
        g = int(gam[b])
        target[b, g + 1:] = nan
        draft[b, g:] = nan
        tok[b, g:] = -7
        if float(temps[b]) == 0.0:
            draft[b] = nan
    return Batch(target, draft, tok, temps, gam,
                 dict(workload="ragged", seed=seed, sigma=sig.cpu().tolist()))

