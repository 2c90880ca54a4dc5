"""Cross-rank load balance of context parallelism under document masks.

The review of "Scaling Llama 3 Training with Efficient Parallelism
Strategies" (Figure 14 and its limitations) reports that with document masks
the slowest CP rank's compute was 1.44x the fastest's, entirely from the
attention kernels, because the static CP shards are not aligned with document
boundaries.  This module is the cost model behind that statement for one
sequence split the way "The Llama 3 Herd of Models - part 3/16" (3.3.2,
"Context parallelism for long sequences") splits it: 2*CP equal chunks, rank
r holding chunks r and 2*CP-1-r.  A rank's attention work is its number of
(query, key) pairs allowed by the causal + document mask (the FLOP count of
the forward and backward is proportional to it).

It also reports a document-aware alternative.  The pairing of chunks stays
the same, but the 2*CP chunk boundaries of each sample are placed, on a grid
of `granule` positions, so that every chunk carries about the same work.
That alternative is a report only: the kernels of this package run the
pages' equal-length chunks.

Host-side planning arithmetic (numpy), no device work.
"""
from __future__ import annotations

import numpy as np


def _docs_of_sample(cu_doc_lens, b: int, seq_len: int) -> list:
    """(start, end) of every document of sample b, positions within the sample."""
    cu = np.asarray(cu_doc_lens, dtype=np.int64)
    lo, hi = b * seq_len, (b + 1) * seq_len
    out = []
    for a, e in zip(cu[:-1], cu[1:]):
        if e <= lo or a >= hi:
            continue
        out.append((int(max(a, lo) - lo), int(min(e, hi) - lo)))
    return out


def _segment_work(docs: list, x0: int, x1: int) -> int:
    """Allowed pairs of the queries at positions [x0, x1): a query at
    position p of a document starting at a sees keys a..p, i.e. p - a + 1."""
    total = 0
    for a, e in docs:
        u0, u1 = max(a, x0), min(e, x1)
        if u1 <= u0:
            continue
        # sum over p in [u0, u1) of (p - a + 1) = sum of k for k in [u0-a+1, u1-a]
        k0, k1 = u0 - a + 1, u1 - a
        total += (k0 + k1) * (k1 - k0 + 1) // 2
    return total


def _prefix_work(docs: list, points) -> np.ndarray:
    """Work of the queries at positions [0, x) for every x in `points`."""
    return np.array([_segment_work(docs, 0, int(x)) for x in points], dtype=np.int64)


def rank_work(cu_doc_lens, batch: int, seq_len: int, cp_size: int, bounds=None) -> np.ndarray:
    """[cp_size, batch] allowed pairs per head of each rank and sample.

    `bounds`: optional [batch, 2*cp_size + 1] chunk boundaries per sample;
    default: the pages' equal chunks of seq_len / (2*cp_size) positions."""
    n_chunks = 2 * cp_size
    out = np.zeros((cp_size, batch), dtype=np.int64)
    for b in range(batch):
        docs = _docs_of_sample(cu_doc_lens, b, seq_len)
        if bounds is None:
            edges = [c * (seq_len // n_chunks) for c in range(n_chunks + 1)]
        else:
            edges = [int(x) for x in bounds[b]]
        for r in range(cp_size):
            for c in (r, n_chunks - 1 - r):
                out[r, b] += _segment_work(docs, edges[c], edges[c + 1])
    return out


def balanced_bounds(cu_doc_lens, batch: int, seq_len: int, cp_size: int,
                    granule: int = 128) -> np.ndarray:
    """[batch, 2*cp_size + 1] chunk boundaries, multiples of `granule`, that
    split each sample into 2*cp_size chunks of about equal work: boundary c
    is the grid point where the cumulative work comes closest to c/(2*cp_size)
    of the sample's total, kept strictly increasing."""
    if seq_len % granule != 0:
        raise ValueError("seq_len must be a multiple of granule")
    n_chunks = 2 * cp_size
    n_grid = seq_len // granule
    if n_grid < n_chunks:
        raise ValueError("fewer grid points than chunks")
    out = np.zeros((batch, n_chunks + 1), dtype=np.int64)
    for b in range(batch):
        docs = _docs_of_sample(cu_doc_lens, b, seq_len)
        grid = np.arange(n_grid + 1) * granule
        cum = _prefix_work(docs, grid)
        total = int(cum[-1])
        edges = [0]
        for c in range(1, n_chunks):
            target = total * c / n_chunks
            j = int(np.argmin(np.abs(cum - target)))
            # strictly increasing, and room left for the remaining chunks
            j = max(j, edges[-1] // granule + 1)
            j = min(j, n_grid - (n_chunks - c))
            edges.append(int(grid[j]))
        edges.append(seq_len)
        out[b] = edges
    return out


def imbalance(work_per_rank) -> dict:
    """max / mean and slowest / fastest of per-rank work (summed over samples)."""
    w = np.asarray(work_per_rank, dtype=np.float64)
    if w.ndim == 2:
        w = w.sum(axis=1)
    mean = float(w.mean())
    return {"max_over_mean": float(w.max() / mean) if mean > 0 else 1.0,
            "slowest_over_fastest": float(w.max() / w.min()) if w.min() > 0 else float("inf")}


def doc_aware_bounds(cu_doc_lens, batch: int, seq_len: int, cp_size: int,
                     granule: int = 128) -> np.ndarray:
    """The document-aware alternative: per sample, the equal-work chunks of
    `balanced_bounds` or the pages' equal-length chunks, whichever gives that
    sample the smaller slowest rank (the mirrored pairing balances a single
    document exactly with equal lengths); the pages' chunks throughout if
    that leaves the whole batch less balanced, or if the grid of `granule`
    positions has fewer points than chunks."""
    n_chunks = 2 * cp_size
    equal = np.tile(np.arange(n_chunks + 1, dtype=np.int64) * (seq_len // n_chunks), (batch, 1))
    if seq_len % granule != 0 or seq_len // granule < n_chunks:
        return equal  # the grid is too coarse to place the chunks otherwise
    work_eq = rank_work(cu_doc_lens, batch, seq_len, cp_size, equal)
    cand = balanced_bounds(cu_doc_lens, batch, seq_len, cp_size, granule)
    work_bal = rank_work(cu_doc_lens, batch, seq_len, cp_size, cand)
    out = np.where((work_bal.max(axis=0) < work_eq.max(axis=0))[:, None], cand, equal)
    alt = rank_work(cu_doc_lens, batch, seq_len, cp_size, out)
    if imbalance(alt)["max_over_mean"] > imbalance(work_eq)["max_over_mean"]:
        return equal
    return out


def report(cu_doc_lens, batch: int, seq_len: int, cp_size: int, granule: int = 128) -> dict:
    """Per-rank work and imbalance of the pages' chunking and of the
    document-aware alternative."""
    pages = rank_work(cu_doc_lens, batch, seq_len, cp_size)
    bounds = doc_aware_bounds(cu_doc_lens, batch, seq_len, cp_size, granule)
    alt = rank_work(cu_doc_lens, batch, seq_len, cp_size, bounds)
    return {
        "cp_size": cp_size,
        "pairs_per_rank": pages.sum(axis=1).tolist(),
        "imbalance": imbalance(pages),
        "doc_aware": {"granule": granule, "bounds": bounds.tolist(),
                      "pairs_per_rank": alt.sum(axis=1).tolist(),
                      "imbalance": imbalance(alt)},
    }


def _main(argv=None) -> int:
    import argparse
    import json

    from . import workloads as wl

    ap = argparse.ArgumentParser(description="CP load-balance report for a workload")
    ap.add_argument("workload", choices=sorted(wl.WORKLOADS))
    ap.add_argument("--cp-size", type=int, default=None, help="override the workload's CP size")
    ap.add_argument("--granule", type=int, default=128)
    args = ap.parse_args(argv)
    w = wl.WORKLOADS[args.workload]
    cp = args.cp_size or w.cp_size
    rep = report(wl.cu_doc_lens(w), w.batch, w.seq_len, cp, args.granule)
    rep["workload"] = w.name
    print(json.dumps(rep))
    return 0


if __name__ == "__main__":
    raise SystemExit(_main())
