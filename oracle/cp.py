"""Context-parallel sharding of one sequence, written from the pages.

Oracle (test infrastructure only; see ``oracle/__init__``).

Sources:
* "The Llama 3 Herd of Models - part 3/16", section 3.3.2, paragraph
  "Context parallelism for long sequences": the input is split into 2*CP
  chunks; rank i holds chunks i and 2*CP-1-i.
* "Scaling Llama 3 Training with Efficient Parallelism Strategies" (review),
  section "Context Parallelism (CP)", subsection on implementation details
  (the same i / 2*cp-i-1 rule), and its integration notes: every CP rank sees
  the whole sequence's document boundaries so it can build the mask.
* "Paper notes: The Llama 3 Herd of Models", "Two architectural choices":
  document masking keeps a token's attention inside its own document.

Readings taken where the pages are silent:
* within a rank, chunk i comes first, then chunk 2*CP-1-i;
* the global chunk order (used to re-assemble a full sequence from all ranks)
  is rank-major: rank 0's two chunks, then rank 1's, and so on;
* ``cu_doc_lens`` holds cumulative document offsets over the flattened
  batch*seq_len token stream and contains every sample boundary.
"""
from __future__ import annotations

import numpy as np


def rank_chunks(cp_size: int, cp_rank: int) -> tuple:
    """The two chunk indices rank ``cp_rank`` holds: i and 2*CP-1-i."""
    return (cp_rank, 2 * cp_size - 1 - cp_rank)


def chunk_order(cp_size: int) -> list:
    """Chunk indices in rank-major order (rank 0's pair, rank 1's pair, ...)."""
    order = []
    for r in range(cp_size):
        order.extend(rank_chunks(cp_size, r))
    return order


def local_positions(seq_len: int, cp_size: int, cp_rank: int) -> np.ndarray:
    """Global sequence position of each local query row of this rank."""
    n_chunks = 2 * cp_size
    assert seq_len % n_chunks == 0
    c = seq_len // n_chunks
    a, b = rank_chunks(cp_size, cp_rank)
    return np.concatenate([np.arange(a * c, (a + 1) * c),
                           np.arange(b * c, (b + 1) * c)]).astype(np.int64)


def gather_local(x_full, seq_len: int, cp_size: int, cp_rank: int):
    """Cut this rank's query rows out of a [B, S, ...] tensor."""
    return x_full[:, local_positions(seq_len, cp_size, cp_rank)]


def assemble_full(locals_by_rank: dict, seq_len: int, cp_size: int):
    """Inverse of ``gather_local`` over all ranks: put every rank's rows back
    at their global positions.  ``locals_by_rank[r]`` is [B, 2C, ...]."""
    first = next(iter(locals_by_rank.values()))
    full = np.zeros((first.shape[0], seq_len) + tuple(first.shape[2:]),
                    dtype=first.dtype)
    seen = np.zeros(seq_len, dtype=bool)
    for r, x in locals_by_rank.items():
        pos = local_positions(seq_len, cp_size, r)
        full[:, pos] = x
        seen[pos] = True
    assert seen.all(), "not every rank was given"
    return full


def doc_ids(cu_doc_lens, batch: int, seq_len: int) -> np.ndarray:
    """Explicit document index of every token, [B, S] (int64)."""
    cu = np.asarray(cu_doc_lens, dtype=np.int64)
    ids = np.full(batch * seq_len, -1, dtype=np.int64)
    for d in range(len(cu) - 1):
        ids[cu[d]:cu[d + 1]] = d
    assert (ids >= 0).all(), "cu_doc_lens does not cover the token stream"
    return ids.reshape(batch, seq_len)


def doc_start(cu_doc_lens, batch: int, seq_len: int) -> np.ndarray:
    """Position (within its sample) of the first token of each token's
    document, [B, S]."""
    cu = np.asarray(cu_doc_lens, dtype=np.int64)
    ids = doc_ids(cu, batch, seq_len)
    base = (np.arange(batch, dtype=np.int64) * seq_len)[:, None]
    return cu[ids] - base


def docs_valid(cu_doc_lens, batch: int, seq_len: int) -> bool:
    """The input contract on ``cu_doc_lens``: starts at 0, strictly
    increasing, ends at batch*seq_len, and contains every b*seq_len."""
    cu = [int(x) for x in np.asarray(cu_doc_lens).ravel()]
    if len(cu) < 2 or cu[0] != 0 or cu[-1] != batch * seq_len:
        return False
    if any(cu[i + 1] <= cu[i] for i in range(len(cu) - 1)):
        return False
    s = set(cu)
    return all(b * seq_len in s for b in range(batch + 1))
