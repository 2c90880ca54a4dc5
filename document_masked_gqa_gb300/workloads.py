"""Seeded synthetic inputs for the document-masked GQA workloads.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic, no chunk assignment and no mask logic.  Both the CUDA
path (tests, bench) and the float64 oracle are fed from it, so the two sides
see bit-identical bf16 tensors.

Workload shapes follow the configurations the Llama 3 infrastructure pages
discuss: an 8K-token layer with 8 KV heads ("Paper notes: The Llama 3 Herd of
Models", "Two architectural choices"), the 70B and 405B per-GPU tensor-parallel
shards, a 128K-token context-parallel shard of 16 ranks ("The Llama 3 Herd of
Models - part 3/16", section 3.3.2, "Context parallelism for long sequences"),
plus a tiny case and a many-short-documents stress case.

Recipe (stated once, used everywhere):

* document lengths per sample: drawn with ``numpy.random.default_rng(seed)``
  until their sum reaches ``seq_len``; the last one is truncated so the sum is
  exactly ``seq_len``.  ``uniform``: integers uniform in [lo, hi];
  ``loguniform``: ``round(exp(U[ln lo, ln hi]))`` clamped to [lo, hi];
  ``single``: one document of ``seq_len`` tokens.
* ``cu_doc_lens``: cumulative document offsets over the flattened
  ``batch * seq_len`` token stream (varlen convention), starting at 0 and
  containing every sample boundary ``b * seq_len``.
* tensors: ``torch.Generator('cpu').manual_seed(seed)``, then, in this order,
  q [B, S, Hq, D], k [B, S, Hkv, D], v [B, S, Hkv, D], dO [B, S, Hq, D], each
  drawn fp32 ~ N(0, 1), q multiplied by ``q_prescale``, then cast to bf16
  (round to nearest even).  The tensors are in natural sequence order over
  the full sequence; the per-rank query chunks are cut from them by each side
  with its own code.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    seq_len: int
    cp_size: int
    ranks: tuple
    batch: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    doc_dist: str  # 'uniform' | 'loguniform' | 'single' | 'fixed'
    doc_lo: int = 0
    doc_hi: int = 0
    q_prescale: float = 1.0
    seed: int = 0
    fixed_docs: tuple = field(default=())  # per-sample doc lengths for 'fixed'

    @property
    def chunk(self) -> int:
        return self.seq_len // (2 * self.cp_size)

    @property
    def local_len(self) -> int:
        return 2 * self.chunk

    @property
    def group(self) -> int:
        return self.n_heads // self.n_kv_heads


WORKLOADS = {
    "tiny": Workload("tiny", 256, 2, (0, 1), 1, 4, 1, 64, "uniform", 16, 128,
                     1.0, 1001),
    "8b": Workload("8b-layer", 8192, 1, (0,), 2, 32, 8, 128, "loguniform",
                   256, 8192, 1.0 / math.sqrt(128.0), 1002),
    "70b": Workload("70b-tp8-shard", 8192, 2, (0, 1), 1, 8, 1, 128,
                    "loguniform", 128, 8192, 1.0, 1003),
    "405b-1doc": Workload("405b-cp16-one-doc", 131072, 16, (0, 7, 15), 1, 16,
                          1, 128, "single", 0, 0, 1.0, 1004),
    "405b-logu": Workload("405b-cp16-loguniform-docs", 131072, 16, (0, 7, 15),
                          1, 16, 1, 128, "loguniform", 1024, 65536, 1.0, 1014),
    "sparse": Workload("sparse-stress", 32768, 4, (0, 1, 2, 3), 1, 16, 1, 128,
                       "uniform", 32, 512, 1.0, 1005),
    # plain causal attention (one document) at 128K on a single rank: the
    # long-sequence case of the pages' Figure 11 without CP
    "causal-128k": Workload("causal-128k-cp1", 131072, 1, (0,), 1, 16, 1, 128,
                            "single", 0, 0, 1.0, 1006),
}


def doc_lengths(w: Workload) -> list:
    """Per-sample lists of document lengths, each summing to ``seq_len``."""
    rng = np.random.default_rng(w.seed)
    out = []
    for b in range(w.batch):
        if w.doc_dist == "single":
            out.append([w.seq_len])
            continue
        if w.doc_dist == "fixed":
            lens = list(w.fixed_docs[b])
            assert sum(lens) == w.seq_len
            out.append(lens)
            continue
        lens, total = [], 0
        while total < w.seq_len:
            if w.doc_dist == "uniform":
                n = int(rng.integers(w.doc_lo, w.doc_hi + 1))
            elif w.doc_dist == "loguniform":
                x = rng.uniform(math.log(w.doc_lo), math.log(w.doc_hi))
                n = int(min(max(round(math.exp(x)), w.doc_lo), w.doc_hi))
            else:
                raise ValueError(w.doc_dist)
            n = min(n, w.seq_len - total)
            lens.append(n)
            total += n
        out.append(lens)
    return out


def cu_doc_lens(w: Workload) -> np.ndarray:
    """int32 cumulative offsets over the flattened batch*seq_len stream."""
    offs = [0]
    for lens in doc_lengths(w):
        for n in lens:
            offs.append(offs[-1] + n)
    return np.asarray(offs, dtype=np.int32)


def tensors(w: Workload, with_grad: bool = True) -> dict:
    """bf16 CPU tensors over the full sequence: q, k, v and (optionally) dO."""
    g = torch.Generator(device="cpu").manual_seed(w.seed)
    B, S, Hq, Hkv, D = w.batch, w.seq_len, w.n_heads, w.n_kv_heads, w.head_dim
    q = torch.randn(B, S, Hq, D, generator=g, dtype=torch.float32)
    if w.q_prescale != 1.0:
        q.mul_(w.q_prescale)
    out = {"q": q.to(torch.bfloat16)}
    del q
    out["k"] = torch.randn(B, S, Hkv, D, generator=g).to(torch.bfloat16)
    out["v"] = torch.randn(B, S, Hkv, D, generator=g).to(torch.bfloat16)
    if with_grad:
        out["do"] = torch.randn(B, S, Hq, D, generator=g).to(torch.bfloat16)
    return out


def custom(name: str, seq_len: int, cp_size: int, batch: int, n_heads: int,
           n_kv_heads: int, head_dim: int, doc_dist: str = "uniform",
           doc_lo: int = 16, doc_hi: int = 128, seed: int = 7,
           ranks=None, q_prescale: float = 1.0, fixed_docs=()) -> Workload:
    """A workload of arbitrary shape (test sweeps, edge cases)."""
    if ranks is None:
        ranks = tuple(range(cp_size))
    return Workload(name, seq_len, cp_size, tuple(ranks), batch, n_heads,
                    n_kv_heads, head_dim, doc_dist, doc_lo, doc_hi,
                    q_prescale, seed, tuple(tuple(x) for x in fixed_docs))
