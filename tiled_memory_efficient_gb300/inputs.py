"""Seeded synthetic inputs for the attention workloads.

This module holds the input recipes only -- random numbers, shapes, dtypes and
the outlier-key pattern -- and none of attention's arithmetic.  Both the test
suite (for the CUDA path and for the fp64 oracle) and the benchmark draw their
inputs from here, so the two sides always see the same rounded values.

Workload shapes follow the pages:
  * the isolated-attention benchmark of the noflash-attention forum post
    (ai-navigate-news, section "It's actually faster too!"): B=1, H=16, D=64,
    fp16, non-causal, N from 256 to 16384;
  * the GQA model of its LLM-inference table (Qwen 2.5 0.5B, GQA, FP16):
    14 query heads over 2 KV heads, D=64, causal prefill;
  * the video-generation case of its section "The problem" (17K and 75K-token
    self-attention, 24 heads): D=128, bf16, non-causal, with 1% of key rows
    scaled by 8 so that the softmax sees a wide range of scores;
  * the autograd tier's training use (section "Other areas where this could
    be useful"): B=2, H=16, D=128, bf16, causal, plus an upstream gradient;
  * decoding with that GQA model against a KV cache (the inference side of
    the LLM table): one new query per head, contexts of 1K to 64K cached keys,
    8 sequences at once, bottom-right causal.
Every tensor is drawn as fp32 N(0,1) from a torch CPU generator and rounded
once to the workload's dtype.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    index: int            # seed base: seed = 1000 * index + N
    B: int
    Hq: int
    Hkv: int
    D: int
    dtype: torch.dtype
    causal: object        # False, True (top-left) or "bottom_right"
    seq_lens: tuple       # key counts Nk (and query counts, unless nq is set)
    outlier_keys: bool = False   # scale 1% of key rows by 8
    with_grad: bool = False      # also draw an upstream gradient dO
    nq: int | None = None        # fixed query count (decode); None: Nq = Nk = n
    note: str = ""

    def queries(self, n: int) -> int:
        return n if self.nq is None else self.nq

    def flops_fwd(self, n: int) -> float:
        """Algorithmic forward FLOPs 4*B*Hq*Nq*Nk*D, halved under the causal
        mask when Nq = Nk; with a fixed query count, 4*D per visible
        (query, key) pair."""
        if self.nq is None:
            f = 4.0 * self.B * self.Hq * n * n * self.D
            return f / 2 if self.causal else f
        nq = self.nq
        if self.causal == "bottom_right":   # query i sees n - nq + i + 1 keys
            pairs = nq * (n - nq) + nq * (nq + 1) / 2
        elif self.causal:                   # top-left: query i sees min(i + 1, n)
            pairs = sum(min(i + 1, n) for i in range(nq))
        else:
            pairs = nq * n
        return 4.0 * self.B * self.Hq * pairs * self.D

    def bytes_fwd(self, n: int) -> float:
        """Algorithmic forward bytes: read Q, K, V once, write O and LSE."""
        e = 2  # fp16 / bf16
        nq = self.queries(n)
        return (2.0 * self.B * self.Hq * nq * self.D * e + 2.0 * self.B * self.Hkv * n * self.D * e
                + 4.0 * self.B * self.Hq * nq)


WORKLOADS = {
    "tiny": Workload("tiny", 0, 1, 2, 2, 64, torch.float16, False, (256,),
                     note="tiny non-causal MHA, fp16"),
    "sweep": Workload("sweep", 1, 1, 16, 16, 64, torch.float16, False,
                      (256, 512, 1024, 2048, 4096, 8192, 16384),
                      note="isolated attention sweep B=1 H=16 D=64 fp16 non-causal"),
    "gqa_prefill": Workload("gqa_prefill", 2, 1, 14, 2, 64, torch.float16, True,
                            (1024, 2048, 4096, 8192, 16384),
                            note="GQA causal prefill Hq=14 Hkv=2 D=64 fp16"),
    "video_dit": Workload("video_dit", 3, 1, 24, 24, 128, torch.bfloat16, False,
                          (17600, 75600), outlier_keys=True,
                          note="video-DiT self-attention H=24 D=128 bf16, 1% keys x8"),
    "training": Workload("training", 4, 2, 16, 16, 128, torch.bfloat16, True, (8192,),
                         with_grad=True, note="training fwd+bwd B=2 H=16 D=128 bf16 causal"),
    "gqa_decode": Workload("gqa_decode", 5, 8, 14, 2, 64, torch.float16, "bottom_right",
                           (1024, 4096, 16384, 65536), nq=1,
                           note="GQA KV-cache decode B=8 Hq=14 Hkv=2 D=64 fp16, 1 query, "
                                "bottom-right causal"),
}


def seed_for(w: Workload, n: int) -> int:
    return 1000 * w.index + n


def make_inputs(w: Workload, n: int, nk: int | None = None, seed: int | None = None):
    """Return dict(q, k, v[, do]) as CPU tensors of the workload's dtype.

    q: [B,Hq,nq,D] with nq = w.nq or n; k, v: [B,Hkv,nk,D] (nk defaults to n).
    """
    nk = n if nk is None else nk
    nq = w.queries(n)
    g = torch.Generator(device="cpu")
    g.manual_seed(seed_for(w, n) if seed is None else seed)
    q = torch.randn((w.B, w.Hq, nq, w.D), generator=g, dtype=torch.float32)
    k = torch.randn((w.B, w.Hkv, nk, w.D), generator=g, dtype=torch.float32)
    v = torch.randn((w.B, w.Hkv, nk, w.D), generator=g, dtype=torch.float32)
    if w.outlier_keys:
        n_out = int(0.01 * nk)
        for b in range(w.B):
            for h in range(w.Hkv):
                idx = torch.randperm(nk, generator=g)[:n_out]
                k[b, h, idx, :] *= 8.0
    out = {"q": q.to(w.dtype), "k": k.to(w.dtype), "v": v.to(w.dtype)}
    if w.with_grad:
        out["do"] = torch.randn((w.B, w.Hq, nq, w.D), generator=g,
                                dtype=torch.float32).to(w.dtype)
    return out


def make_custom(B, Hq, Hkv, Nq, Nk, D, dtype=torch.float16, seed=0, with_grad=False,
                std: float = 1.0, v_std: float = 1.0):
    """Ad-hoc shapes for parity tests: q, k i.i.d. N(0, std^2), v N(0, v_std^2),
    rounded to dtype."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    q = (torch.randn((B, Hq, Nq, D), generator=g) * std).to(dtype)
    k = (torch.randn((B, Hkv, Nk, D), generator=g) * std).to(dtype)
    v = (torch.randn((B, Hkv, Nk, D), generator=g) * v_std).to(dtype)
    out = {"q": q, "k": k, "v": v}
    if with_grad:
        out["do"] = torch.randn((B, Hq, Nq, D), generator=g).to(dtype)
    return out


def sample_rows(B, H, Nq, per_head: int, seed: int = 0, tile: int = 128):
    """Seeded sample of flattened row ids (b*H + h)*Nq + i for oracle checks.

    Always includes rows 0 and Nq-1 and the rows on each side of the first
    few 128-row tile edges of every head, plus ``per_head`` random rows.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    fixed = {0, Nq - 1}
    for e in range(tile, min(Nq, 4 * tile + 1), tile):
        fixed.update({e - 1, e})
    rows = []
    for bh in range(B * H):
        rnd = torch.randint(0, Nq, (per_head,), generator=g).tolist()
        for i in sorted(fixed.union(rnd)):
            if 0 <= i < Nq:
                rows.append(bh * Nq + i)
    return torch.tensor(rows, dtype=torch.int64)
