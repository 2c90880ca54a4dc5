"""Brute-force (query tile, key tile) classification from the explicit mask.

Oracle (test infrastructure only; see ``oracle/__init__``).

The pages motivate skipping work that a document mask removes (review of
"Scaling Llama 3 Training with Efficient Parallelism Strategies": all-gather
CP supports arbitrary masks; the document mask makes ranks' attention work
uneven, Figure 11 and Figure 14 discussion) but describe no tile scheme.
The plainest reading, used here: a query tile holds ``P = 128 // g``
consecutive local query rows of all ``g`` query heads of one K/V group, a key
tile holds ``n_key_tile`` consecutive key positions, and a pair of tiles is

* SKIP    (0) - no element of the explicit mask is true,
* FULL    (1) - every element is true,
* PARTIAL (2) - anything else.

Rows of the same position but different heads share the mask, so the tile
is classified over its positions.  Classes come from an element-by-element
look at the explicit mask (``oracle.attention.allowed``), not from any
interval reasoning.

The derived lists:
* row list of (b, query tile): ascending key-tile indices with class != SKIP;
* column list of (b, key tile): ascending query-tile indices with
  class != SKIP.
"""
from __future__ import annotations

import numpy as np

from . import cp as _cp
from .attention import allowed

SKIP, FULL, PARTIAL = 0, 1, 2


def tile_classes(cu_doc_lens, batch: int, seq_len: int, cp_size: int,
                 cp_rank: int, group: int, n_key_tile: int = 128) -> np.ndarray:
    """uint8 [B, n_query_tiles, n_key_tiles]."""
    P = 128 // group
    qpos = _cp.local_positions(seq_len, cp_size, cp_rank)
    Lq = len(qpos)
    assert Lq % P == 0 and seq_len % n_key_tile == 0
    nqt, nkt = Lq // P, seq_len // n_key_tile
    ids = _cp.doc_ids(cu_doc_lens, batch, seq_len)
    keys = np.arange(seq_len)
    cls = np.empty((batch, nqt, nkt), dtype=np.uint8)
    for b in range(batch):
        for t in range(nqt):
            m = allowed(ids[b], qpos[t * P:(t + 1) * P], keys)
            m = m.reshape(P, nkt, n_key_tile)
            any_ = m.any(axis=(0, 2))
            all_ = m.all(axis=(0, 2))
            c = np.full(nkt, PARTIAL, dtype=np.uint8)
            c[~any_] = SKIP
            c[all_] = FULL
            cls[b, t] = c
    return cls


def row_lists(cls: np.ndarray) -> list:
    """Per (b, query tile), flattened b-major: ascending non-skip key tiles."""
    B, nqt, _ = cls.shape
    return [np.nonzero(cls[b, t] != SKIP)[0] for b in range(B) for t in range(nqt)]


def col_lists(cls: np.ndarray) -> list:
    """Per (b, key tile), flattened b-major: ascending non-skip query tiles."""
    B, _, nkt = cls.shape
    return [np.nonzero(cls[b, :, j] != SKIP)[0] for b in range(B) for j in range(nkt)]


def allowed_count_in_partials(cu_doc_lens, batch, seq_len, cp_size, cp_rank,
                              group, cls, n_key_tile=128) -> int:
    """Number of true mask elements (per head) inside PARTIAL tiles."""
    P = 128 // group
    qpos = _cp.local_positions(seq_len, cp_size, cp_rank)
    ids = _cp.doc_ids(cu_doc_lens, batch, seq_len)
    total = 0
    for b, t, j in zip(*np.nonzero(cls == PARTIAL)):
        m = allowed(ids[b], qpos[t * P:(t + 1) * P],
                    np.arange(j * n_key_tile, (j + 1) * n_key_tile))
        total += int(m.sum())
    return total
