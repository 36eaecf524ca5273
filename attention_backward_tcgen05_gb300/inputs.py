"""Seeded synthetic inputs for the attention backward workloads.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic, so both the CUDA path and the fp64 oracle can take their
inputs from it without sharing any computation.

Tensor shapes (torch, C order; the reverse of ggml's ne order):
    q (B, H, N, DK)   k (B, Hkv, M, DK)   v (B, Hkv, M, DV)
    d (B, N, H, DV)   -- the upstream gradient, shaped like the forward output
    mask (N, M) float16 or None  -- mask[n, m] is added to the score of query n, key m

Draw order from one ``torch.Generator`` seeded per workload: q, k, v, d, then
the mask's Bernoulli draws and finally the index of the fully masked query.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Hkv: int
    N: int
    M: int
    DK: int
    DV: int
    dtype: str            # "f32", "bf16" or "f16": the type q, k, v and d are handed over in
    dist: str             # "uniform" (lo, hi) or "normal" (std)
    scale: float
    causal: bool = False
    mask: str = "none"    # "none" | "random" (Bernoulli -inf with one fully masked query) | "pad" | "docs" | "band"
    mask_p: float = 0.1
    lo: float = -1.0
    hi: float = 1.0
    std: float = 1.0
    seed: int = 0
    parts: int = 4        # "docs": number of documents; "band": half-width in 128-key tiles
    note: str = field(default="", compare=False)

    @property
    def dims(self):
        return (self.B, self.H, self.Hkv, self.N, self.M, self.DK, self.DV)


# The five workloads the library is measured and checked on.
WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", 1, 1, 1, 128, 128, 64, 64, "f32", "uniform", 1.0 / 8, seed=11,
                         note="single head, f32 q/k/v/d uniform(-1,1), no mask"),
    "causal_d64": Workload("causal_d64", 2, 8, 8, 1024, 1024, 64, 64, "bf16", "normal", 1.0 / math.sqrt(64),
                           causal=True, seed=1002, note="causal self-attention, bf16 of N(0,1)"),
    "gqa_causal_d128": Workload("gqa_causal_d128", 4, 32, 8, 2048, 2048, 128, 128, "bf16", "normal",
                                1.0 / math.sqrt(128), causal=True, seed=1003,
                                note="grouped-query causal, groups of 4 query heads"),
    "long_seq": Workload("long_seq", 1, 16, 16, 16384, 16384, 128, 128, "bf16", "normal", 1.0 / math.sqrt(128),
                         causal=True, std=0.5, seed=1004, note="long sequence, bf16 of 0.5*N(0,1)"),
    "masked_nonsquare": Workload("masked_nonsquare", 8, 16, 4, 512, 8192, 128, 128, "bf16", "normal",
                                 1.0 / math.sqrt(128), mask="random", seed=1005,
                                 note="f16 mask [M,N]: 10% -inf, one query fully -inf, rest 0"),
    # not one of the five: the gqa shape under a padding mask, where whole
    # tiles of the mask are -inf (the tensor-core passes skip them)
    "padded_d128": Workload("padded_d128", 4, 32, 8, 2048, 2048, 128, 128, "bf16", "normal",
                            1.0 / math.sqrt(128), mask="pad", mask_p=0.05, seed=1006,
                            note="f16 padding mask: keys from 5/8 M on and queries from 7/8 N on -inf, 5% -inf elsewhere"),
    # not one of the five either: the gqa shape with four packed documents
    # (block-diagonal mask), where most tiles on both sides of each block are -inf
    "docs_d128": Workload("docs_d128", 4, 32, 8, 2048, 2048, 128, 128, "bf16", "normal",
                          1.0 / math.sqrt(128), mask="docs", mask_p=0.05, seed=1007, parts=4,
                          note="f16 block-diagonal mask of 4 documents at random cuts, 5% -inf inside"),
}

ORDER = ["tiny_f32", "causal_d64", "gqa_causal_d128", "long_seq", "masked_nonsquare"]
EXTRA = ["padded_d128", "docs_d128"]


def custom(B, H, Hkv, N, M, DK, DV=None, dtype="bf16", dist="normal", scale=None, causal=False, mask="none",
           seed=0, std=1.0, lo=-1.0, hi=1.0, mask_p=0.1, parts=4, name="custom") -> Workload:
    DV = DK if DV is None else DV
    scale = 1.0 / math.sqrt(DK) if scale is None else scale
    return Workload(name, B, H, Hkv, N, M, DK, DV, dtype, dist, scale, causal, mask, mask_p, lo, hi, std, seed,
                    parts)


def _draw(g, shape, w: Workload):
    if w.dist == "uniform":
        x = torch.rand(shape, generator=g, dtype=torch.float32) * (w.hi - w.lo) + w.lo
    elif w.dist == "normal":
        x = torch.randn(shape, generator=g, dtype=torch.float32) * w.std
    else:
        raise ValueError(w.dist)
    if w.dtype == "bf16":
        return x.to(torch.bfloat16)
    return x.to(torch.float16) if w.dtype == "f16" else x


def make(w: Workload, device="cpu"):
    """Returns dict(q, k, v, d, mask, masked_query) on `device`.

    ``masked_query`` is the index of the query row whose mask column is all
    -inf (random masks only), else None.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(int(w.seed))
    B, H, Hkv, N, M, DK, DV = w.dims
    q = _draw(g, (B, H, N, DK), w)
    k = _draw(g, (B, Hkv, M, DK), w)
    v = _draw(g, (B, Hkv, M, DV), w)
    d = _draw(g, (B, N, H, DV), w)
    mask = None
    masked_query = None
    if w.mask == "random":
        hit = torch.rand((N, M), generator=g, dtype=torch.float32) < w.mask_p
        mask = torch.zeros((N, M), dtype=torch.float32)
        mask[hit] = float("-inf")
        masked_query = int(torch.randint(0, N, (1,), generator=g).item())
        mask[masked_query, :] = float("-inf")
        mask = mask.to(torch.float16)
    elif w.mask == "pad":
        # padding: keys from 5/8 M on and queries from 7/8 N on are -inf for
        # everything (whole tiles of the mask then hold only -inf), plus
        # Bernoulli(mask_p) -inf entries elsewhere
        mv, nv = (M * 5) // 8 + 3, (N * 7) // 8 + 1
        hit = torch.rand((N, M), generator=g, dtype=torch.float32) < w.mask_p
        mask = torch.zeros((N, M), dtype=torch.float32)
        mask[hit] = float("-inf")
        mask[:, mv:] = float("-inf")
        mask[nv:, :] = float("-inf")
        mask = mask.to(torch.float16)
    elif w.mask in ("docs", "band"):
        # Bernoulli(mask_p) -inf everywhere, then
        # docs: `parts` documents cut at the same random fractions of N and M;
        #   query n and key m see each other only inside one document
        # band: key m is live for query n only within `parts` * 128 keys of
        #   the scaled diagonal n * M / N
        hit = torch.rand((N, M), generator=g, dtype=torch.float32) < w.mask_p
        mask = torch.zeros((N, M), dtype=torch.float32)
        mask[hit] = float("-inf")
        n_idx = torch.arange(N, dtype=torch.float64)[:, None]
        m_idx = torch.arange(M, dtype=torch.float64)[None, :]
        if w.mask == "docs":
            cuts = torch.sort(torch.rand((max(w.parts - 1, 0),), generator=g, dtype=torch.float64)).values
            doc_n = torch.bucketize(n_idx / N, cuts, right=True)
            doc_m = torch.bucketize(m_idx / M, cuts, right=True)
            mask[doc_n != doc_m] = float("-inf")
        else:
            mask[(m_idx - n_idx * M / N).abs() > 128 * w.parts] = float("-inf")
        mask = mask.to(torch.float16)
    elif w.mask != "none":
        raise ValueError(w.mask)
    out = dict(q=q, k=k, v=v, d=d, mask=mask, masked_query=masked_query)
    if device != "cpu":
        out = {key: (val.to(device) if isinstance(val, torch.Tensor) else val) for key, val in out.items()}
    return out
