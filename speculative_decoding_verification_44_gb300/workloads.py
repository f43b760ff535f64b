"""Seeded synthetic inputs for the verify step: the five workload shapes.

This module holds none of the verification arithmetic.  It draws logits,
uniforms and draft tokens from fixed recipes with seeded torch generators.
Where a draft token must be drawn from the draft distribution q (sampling
workloads), the caller supplies ``draft_probs``: a callable mapping a
[rows, V] logits tensor and its sampling parameters to [rows, V]
probabilities (the tests use the float64 oracle, the benchmark the library's
own transform); the token is then drawn with ``torch.multinomial``.

Recipes (seeds: 1000+id logits, 2000+id noise, 3000+id drafts, 4000+id
uniforms), id = 1..5:
  1 tiny sampling   B=1 (rounds as batch), gamma=4, V=32 fp32, z ~ N(0, 2^2),
                    draft = z + N(0, 0.5^2), T=1, no top-k/top-p, d ~ q.
  2 small vocab     B=8, gamma=4, V=32000 fp32, z ~ N(0, 3^2) plus +6 on 20
                    random "hot" tokens per row, draft = z + N(0, 1), T=0.8,
                    top-k off, top-p 1, d ~ q.
  3 serving-shaped  B=64, gamma=5, V=128256 bf16, z = -1.1 ln(rank) + N(0, 0.5^2)
                    with ranks a random permutation per row, draft = z +
                    N(0, 0.8^2) (rounded to bf16 after the noise), T=0.7,
                    top-k 50, top-p 0.9 for p and q, d ~ q.
  4 greedy at scale B=256, gamma=8, V=152064 bf16, z ~ N(0, 2^2); d_i is the
                    row's argmax with probability 0.8, else a uniformly random
                    other token.
  5 ragged mixed    B=512, gamma_b ~ U{1..7} padded to 7, V=256000 bf16 with the
                    Zipf recipe of workload 3, T=1, top-p 0.95, top-k off;
                    sequences [0, B/2) draft = z + N(0, 1), d ~ q; sequences
                    [B/2, B) one-hot drafts proposing argmax(z + N(0, 1)).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Callable, Optional

import torch

from .api import SamplingParams


@dataclass
class Workload:
    name: str
    wid: int
    mode: str                       # "sample" or "greedy"
    B: int
    G: int
    V: int
    dtype: torch.dtype
    target_params: SamplingParams = field(default_factory=SamplingParams)
    draft_params: SamplingParams = field(default_factory=SamplingParams)
    target_logits: Optional[torch.Tensor] = None    # [B, G+1, V]
    draft_logits: Optional[torch.Tensor] = None     # [B, G, V] or None
    draft_tokens: Optional[torch.Tensor] = None     # [B, G] int32
    gamma_per_seq: Optional[torch.Tensor] = None    # [B] int32 or None
    draft_is_onehot: Optional[torch.Tensor] = None  # [B] uint8 or None
    u_accept: Optional[torch.Tensor] = None         # [B, G] float32
    u_sample: Optional[torch.Tensor] = None         # [B] float32

    def rows_used(self) -> tuple[int, int]:
        """(target rows, draft logits rows) the verifier reads."""
        g = self.gamma_per_seq.long() if self.gamma_per_seq is not None else torch.full((self.B,), self.G)
        rt = int((g + 1).sum())
        if self.mode == "greedy" or self.draft_logits is None:
            return rt, 0
        oh = self.draft_is_onehot.bool() if self.draft_is_onehot is not None else torch.zeros(self.B, dtype=torch.bool)
        rd = int(g[~oh.cpu()].sum())
        return rt, rd

    def logits_bytes(self) -> int:
        rt, rd = self.rows_used()
        return (rt + rd) * self.V * (2 if self.dtype == torch.bfloat16 else 4)

    def to(self, device) -> "Workload":
        out = Workload(**{k: getattr(self, k) for k in self.__dataclass_fields__})
        for k in ("target_logits", "draft_logits", "draft_tokens", "gamma_per_seq", "draft_is_onehot",
                  "u_accept", "u_sample"):
            t = getattr(self, k)
            if t is not None:
                setattr(out, k, t.to(device))
        return out


DraftProbs = Callable[[torch.Tensor, SamplingParams], torch.Tensor]

DEFAULTS = {
    1: dict(B=1, G=4, V=32),
    2: dict(B=8, G=4, V=32000),
    3: dict(B=64, G=5, V=128256),
    4: dict(B=256, G=8, V=152064),
    5: dict(B=512, G=7, V=256000),
}
NAMES = {1: "tiny-sampling", 2: "small-vocab-batch", 3: "serving-zipf-topk-topp",
         4: "greedy-at-scale", 5: "ragged-mixed-drafts"}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _zipf_rows(n: int, V: int, gen: torch.Generator, noise_sd: float, device, chunk: int = 64) -> torch.Tensor:
    """n rows of -1.1 ln(rank) + N(0, noise_sd^2), ranks a random permutation per row (float32)."""
    base = -1.1 * torch.log(torch.arange(1, V + 1, device=device, dtype=torch.float32))
    out = torch.empty(n, V, device=device, dtype=torch.float32)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        perm = torch.rand(e - s, V, generator=gen, device=device).argsort(dim=1)
        out[s:e].scatter_(1, perm, base.expand(e - s, V))
        out[s:e] += noise_sd * torch.randn(e - s, V, generator=gen, device=device)
    return out


def sample_from_probs(probs: torch.Tensor, gen: torch.Generator) -> torch.Tensor:
    """One token per row, drawn from the given probabilities (library multinomial)."""
    return torch.multinomial(probs.to(torch.float64 if probs.device.type == "cpu" else torch.float32),
                             1, generator=gen).squeeze(1)


def _draw_drafts(draft_logits: torch.Tensor, params: SamplingParams, rows_mask: torch.Tensor,
                 draft_probs: DraftProbs, gen: torch.Generator) -> torch.Tensor:
    """d_i ~ q_i for the masked [B, G] positions; other positions get token 0."""
    B, G, V = draft_logits.shape
    toks = torch.zeros(B, G, dtype=torch.int64, device=draft_logits.device)
    idx = rows_mask.nonzero(as_tuple=False)
    if idx.numel():
        rows = draft_logits[idx[:, 0], idx[:, 1]]
        probs = draft_probs(rows, params).to(draft_logits.device)
        gdev = torch.Generator(device=probs.device)
        gdev.manual_seed(int(torch.randint(0, 2 ** 62, (1,), generator=gen, device=gen.device).item()))
        toks[idx[:, 0], idx[:, 1]] = sample_from_probs(probs, gdev).to(draft_logits.device)
    return toks


def make(wid: int, device="cpu", draft_probs: DraftProbs | None = None, replica: int = 0,
         **overrides) -> Workload:
    """Build workload ``wid`` (1..5) on ``device``; overrides: B, G, V.

    ``replica`` > 0 shifts every seed by 10000 * replica: an independent batch of
    the same recipe (input rotation, one batch per GPU)."""
    dims = dict(DEFAULTS[wid])
    dims.update({k: v for k, v in overrides.items() if k in ("B", "G", "V")})
    B, G, V = dims["B"], dims["G"], dims["V"]
    off = 10000 * replica
    g_logit, g_noise = _gen(off + 1000 + wid, device), _gen(off + 2000 + wid, device)
    g_draft, g_unif = _gen(off + 3000 + wid, device), _gen(off + 4000 + wid, device)
    bf16 = wid in (3, 4, 5)
    w = Workload(NAMES[wid], wid, "greedy" if wid == 4 else "sample", B, G, V,
                 torch.bfloat16 if bf16 else torch.float32)

    if wid == 1:
        z = 2.0 * torch.randn(B, G + 1, V, generator=g_logit, device=device)
        dz = z[:, :G] + 0.5 * torch.randn(B, G, V, generator=g_noise, device=device)
        w.target_params = w.draft_params = SamplingParams(1.0, 0, 1.0)
    elif wid == 2:
        z = 3.0 * torch.randn(B, G + 1, V, generator=g_logit, device=device)
        hot = torch.rand(B, G + 1, V, generator=g_logit, device=device).argsort(dim=2)[..., :20]
        z.scatter_add_(2, hot, torch.full(hot.shape, 6.0, device=device))
        dz = z[:, :G] + 1.0 * torch.randn(B, G, V, generator=g_noise, device=device)
        w.target_params = w.draft_params = SamplingParams(0.8, 0, 1.0)
    elif wid in (3, 5):
        z = _zipf_rows(B * (G + 1), V, g_logit, 0.5, device).view(B, G + 1, V)
        sd = 0.8 if wid == 3 else 1.0
        dz = torch.empty(B, G, V, device=device, dtype=torch.float32)
        for s in range(0, B, 16):
            e = min(B, s + 16)
            dz[s:e] = z[s:e, :G] + sd * torch.randn(e - s, G, V, generator=g_noise, device=device)
        if wid == 3:
            w.target_params = w.draft_params = SamplingParams(0.7, 50, 0.9)
        else:
            w.target_params = w.draft_params = SamplingParams(1.0, 0, 0.95)
    else:  # wid == 4
        z = 2.0 * torch.randn(B, G + 1, V, generator=g_logit, device=device)
        dz = None

    w.target_logits = z.to(w.dtype).contiguous()
    del z
    if dz is not None:
        w.draft_logits = dz.to(w.dtype).contiguous()
        del dz

    if wid == 5:
        w.gamma_per_seq = torch.randint(1, G + 1, (B,), generator=g_draft, device=device, dtype=torch.int32)
        w.draft_is_onehot = (torch.arange(B, device=device) >= B // 2).to(torch.uint8)

    # draft tokens
    gam = (w.gamma_per_seq.long() if w.gamma_per_seq is not None
           else torch.full((B,), G, device=device, dtype=torch.long))
    pos = torch.arange(G, device=device).unsqueeze(0) < gam.unsqueeze(1)      # [B, G] used positions
    if wid == 4:
        am = w.target_logits[:, :G].float().argmax(dim=2)
        other = torch.randint(0, V - 1, (B, G), generator=g_draft, device=device)
        other = other + (other >= am).long()                                   # uniform over the other tokens
        keep = torch.rand(B, G, generator=g_draft, device=device) < 0.8
        toks = torch.where(keep, am, other)
    else:
        if draft_probs is None:
            raise ValueError(f"workload {wid} draws drafts from q: pass draft_probs")
        model_rows = pos.clone()
        if w.draft_is_onehot is not None:
            model_rows &= ~w.draft_is_onehot.bool().unsqueeze(1)
        toks = _draw_drafts(w.draft_logits, w.draft_params, model_rows, draft_probs, g_draft)
        if w.draft_is_onehot is not None:
            oh = w.draft_is_onehot.bool()
            guess = (w.target_logits[:, :G].float() +
                     torch.randn(B, G, V, generator=g_noise, device=device)).argmax(dim=2)
            toks = torch.where(oh.unsqueeze(1), guess, toks)
    w.draft_tokens = torch.where(pos, toks, torch.zeros_like(toks)).to(torch.int32).contiguous()
    if w.mode == "sample":
        w.u_accept = torch.rand(B, G, generator=g_unif, device=device)
        w.u_sample = torch.rand(B, generator=g_unif, device=device)
    return w


__all__ = ["Workload", "make", "sample_from_probs", "DEFAULTS", "NAMES"]
