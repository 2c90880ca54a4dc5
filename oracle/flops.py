"""Unmasked pair counts and the FLOP convention.

Oracle (test infrastructure only; see ``oracle/__init__``).

Only (query, key) pairs the mask allows are counted.  Per head, the forward
does two contractions over D per pair (q.k and p.v: 4*D FLOPs) and the
backward five (recomputed q.k, dO.v, dV, dQ, dK: 10*D FLOPs).  This is the
hardware-FLOPs style count the review of "Scaling Llama 3 Training with
Efficient Parallelism Strategies" uses for attention (Figure 11, relative
HFU); "Training Infrastructure and Systems" ("Model FLOPs Utilization")
separates the model count (no recompute: 4*D + 8*D) from the hardware count.
"""
from __future__ import annotations

import numpy as np

from . import cp as _cp


def pairs_per_head(cu_doc_lens, batch: int, seq_len: int, cp_size: int,
                   cp_rank: int) -> np.ndarray:
    """[B] number of allowed (query, key) pairs of this rank, per head:
    sum over local queries p of (p - start of p's document + 1)."""
    qpos = _cp.local_positions(seq_len, cp_size, cp_rank)
    start = _cp.doc_start(cu_doc_lens, batch, seq_len)
    return np.array([int((qpos - start[b, qpos] + 1).sum()) for b in range(batch)],
                    dtype=np.int64)


def single_doc_pairs_closed_form(chunk: int, cp_size: int) -> int:
    """One document spanning the sequence: a rank holding chunks i and
    2CP-1-i sees C*(iC) + C(C+1)/2 + C*((2CP-1-i)C) + C(C+1)/2 pairs, which is
    C^2 (2CP-1) + C(C+1) whatever i is: the balance the chunk rule is for."""
    c = chunk
    return c * c * (2 * cp_size - 1) + c * (c + 1)


def counted_flops(pairs_total: int, n_heads: int, head_dim: int,
                  backward: bool = True) -> float:
    """Hardware-style count: Hq * pairs * (4D fwd + 10D bwd)."""
    per = 4 * head_dim + (10 * head_dim if backward else 0)
    return float(n_heads) * float(pairs_total) * per


def model_flops(pairs_total: int, n_heads: int, head_dim: int) -> float:
    """Model-style count, no recompute: Hq * pairs * (4D + 8D)."""
    return float(n_heads) * float(pairs_total) * 12 * head_dim
