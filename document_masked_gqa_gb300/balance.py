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

A second model counts what the kernels actually do: the block-mask
builder's classes of (query tile, key tile) pairs.  A full or a partial pair
costs a whole 128 x 128 tile of tensor work whatever its number of allowed
pairs, partial pairs add the masking, and every work item has a fixed cost
(its first loads, its epilogue).  ``rank_costs`` counts, per rank, the
non-skipped and partial tile pairs and the work items; ``fit_costs`` fits
the per-tile and per-item constants to measured per-rank step times by
least squares; ``predict_ms`` applies them.

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


def report(cu_doc_lens, batch: int, seq_len: int, cp_size: int, granule: int = 128,
           n_heads: int | None = None, n_kv_heads: int | None = None) -> dict:
    """Per-rank work and imbalance of the pages' chunking and of the
    document-aware alternative; with the head counts also the tile-cost
    model's predicted step time per rank (COST_MS_GB300)."""
    pages = rank_work(cu_doc_lens, batch, seq_len, cp_size)
    bounds = doc_aware_bounds(cu_doc_lens, batch, seq_len, cp_size, granule)
    alt = rank_work(cu_doc_lens, batch, seq_len, cp_size, bounds)
    out = {
        "cp_size": cp_size,
        "pairs_per_rank": pages.sum(axis=1).tolist(),
        "imbalance": imbalance(pages),
        "doc_aware": {"granule": granule, "bounds": bounds.tolist(),
                      "pairs_per_rank": alt.sum(axis=1).tolist(),
                      "imbalance": imbalance(alt)},
    }
    if n_heads and n_kv_heads:
        feats = [rank_costs(cu_doc_lens, batch, seq_len, cp_size, r, n_heads, n_kv_heads)
                 for r in range(cp_size)]
        ms = predict_ms(feats)
        out["tile_cost_model"] = {"predicted_ms_per_rank": [round(float(x), 4) for x in ms],
                                  "imbalance": imbalance(ms)}
    return out


TILE = 128  # positions per key tile; a query tile holds TILE rows (TILE / g positions)
# the dK/dV list cutting rule of the planner: segments of at least SEG_MIN
# query tiles; cut when the greedy-makespan bound exceeds SPLIT_ON = 23/20
# times the mean work per SM, to within SPLIT_TARGET = 11/10 of it; at most
# SORT_MAX units
SEG_MIN, SORT_MAX = 16, 2048
SPLIT_ON, SPLIT_TARGET = (23, 20), (11, 10)


def kv_pool_slots(batch: int, seq_len: int, n_kv_heads: int, n_qtiles: int) -> int:
    """Slots of the plan's pool of partial dK, dV: one per (sample, key tile)
    unit, at least 512 / Hkv where the lists are long enough to be cut."""
    units = batch * (seq_len // TILE)
    max_extra = units * (-(-n_qtiles // SEG_MIN) - 1)
    floor_slots = min(-(-512 // n_kv_heads), max_extra)
    return max(0, max(units, floor_slots))


def kv_work_list(col_counts, n_kv_heads: int, n_sms: int, pool_slots: int) -> dict:
    """The dK/dV work list the planner lays out from the column-list lengths
    of the units (sample, key tile), in the same steps and arithmetic.

    Greedy list scheduling runs each item, in order, on the SM that frees
    first, so an item ends no later than the work before it over the SMs
    plus its own length.  Units sorted longest list first, heads side by side:
    unit o ends by E_o = (Hkv pre_o + (Hkv - 1) c_o) / P + c_o against the
    mean m = Hkv sum(c) / P.  When max E_o > SPLIT_ON m, every list longer
    than L is cut into k = ceil(c / L) contiguous segments (the first c mod k
    of them one query tile longer), L = the length at the first position
    from which every E_o <= SPLIT_TARGET m (at least SEG_MIN),
    lengthened by an eighth while the segments after the first of each cut
    list need more than pool_slots slots.  Slices are then ordered by length,
    longest first, ties by unit.

    Returns {"L": L or None, "slices": [(unit, first, n, seg, split, slot)],
    "splits": [(unit, slot0, segs)]}; `first` is the offset in the unit's
    list."""
    cnt = np.asarray(col_counts, dtype=np.int64)
    n = len(cnt)
    order = sorted(range(n), key=lambda i: (-int(cnt[i]), i))
    L = None
    if 0 < n <= SORT_MAX:
        c = cnt[order]
        P = max(int(n_sms), 1)
        h = int(n_kv_heads)
        pre = np.concatenate([[0], np.cumsum(c)[:-1]]).astype(np.int64)
        total = int(c.sum())
        pm = h * total                                   # P m
        pe = h * pre + (h - 1) * c + P * c               # P E_o, exact
        if total > 0 and SPLIT_ON[1] * int(pe.max()) > SPLIT_ON[0] * pm:
            over = np.nonzero(SPLIT_TARGET[1] * pe > SPLIT_TARGET[0] * pm)[0]
            o_star = min(int(over.max()) + 1 if len(over) else 0, n - 1)
            cand = max(SEG_MIN, int(c[o_star]))
            fits = False
            for _ in range(4096):
                if cand >= int(c[0]):
                    break
                need = int(sum(-(-int(x) // cand) - 1 for x in c if x > cand))
                if need <= pool_slots:
                    fits = True
                    break
                cand += max(1, cand // 8)
            L = cand if fits else None

    def segs_of(x):
        return -(-int(x) // L) if (L is not None and x > L) else 1

    def seg_len(u):
        return -(-int(cnt[u]) // segs_of(cnt[u]))

    if L is not None:
        order = sorted(order, key=lambda u: (-seg_len(u), u))
    slices, splits, slot = [], [], 0
    for u in order:
        c_u, k = int(cnt[u]), segs_of(cnt[u])
        if k == 1:
            slices.append((u, 0, c_u, 0, -1, -1))
            continue
        split = len(splits)
        splits.append((u, slot, k))
        q, r = divmod(c_u, k)  # the first r segments take one more query tile
        lo = 0
        for sg in range(k):
            n_sg = q + (1 if sg < r else 0)
            slices.append((u, lo, n_sg, sg, split, slot + sg - 1 if sg > 0 else -1))
            lo += n_sg
        slot += k - 1
    return {"L": L, "slices": slices, "splits": splits}


def _doc_starts(cu_doc_lens, batch: int, seq_len: int, pos: np.ndarray) -> np.ndarray:
    """[batch, len(pos)] first position (within the sample) of the document
    holding each position."""
    cu = np.asarray(cu_doc_lens, dtype=np.int64)
    out = np.empty((batch, len(pos)), dtype=np.int64)
    for b in range(batch):
        g = b * seq_len + pos
        d = np.searchsorted(cu, g, side="right") - 1
        out[b] = cu[d] - b * seq_len
    return out


def tile_counts(cu_doc_lens, batch: int, seq_len: int, cp_size: int, cp_rank: int,
                group: int) -> dict:
    """Full and partial (query tile, key tile) pairs of one rank, summed over
    samples (per K/V head), and the longest row list (key tiles of one query
    tile) and column list (query tiles of one key tile).  A query tile is TILE / group consecutive local
    positions, whose allowed keys are [start of its document, position]; both
    ends grow with the position, so the tile meets key tile [k0, k1] iff its
    first row whose position reaches k0 starts its document at or before
    k1, and covers it fully iff its last row's document starts at or before
    k0 and its first position is at or past k1."""
    P = TILE // group
    n = 2 * cp_size
    C = seq_len // n
    pos = np.concatenate([np.arange(cp_rank * C, (cp_rank + 1) * C),
                          np.arange((n - 1 - cp_rank) * C, (n - cp_rank) * C)])
    nqt, nkt = len(pos) // P, seq_len // TILE
    lo = _doc_starts(cu_doc_lens, batch, seq_len, pos)
    k0 = (np.arange(nkt) * TILE)[None, :]
    k1 = k0 + TILE - 1
    q_first = pos[::P][:, None]
    full = partial = 0
    max_row = max_col = 0
    col_counts = []
    for b in range(batch):
        lo_b = lo[b].reshape(nqt, P)
        r_star = np.clip(k0 - q_first, 0, P)                  # first row with position >= k0
        meets = r_star < P
        lo_at = np.take_along_axis(lo_b, np.minimum(r_star, P - 1), axis=1)
        meets &= lo_at <= k1
        covers = (lo_b[:, -1:] <= k0) & (k1 <= q_first)
        full += int((meets & covers).sum())
        partial += int((meets & ~covers).sum())
        max_row = max(max_row, int(meets.sum(axis=1).max()))
        max_col = max(max_col, int(meets.sum(axis=0).max()))
        col_counts.append(meets.sum(axis=0))
    return {"full": full, "partial": partial, "max_row": max_row, "max_col": max_col,
            "col_counts": np.concatenate(col_counts).astype(np.int64)}


def rank_costs(cu_doc_lens, batch: int, seq_len: int, cp_size: int, cp_rank: int,
               n_heads: int, n_kv_heads: int, n_sms: int = 152) -> np.ndarray:
    """Cost features of one rank's step: [tile-pair makespan, partial pairs,
    work items, 1].  The makespan counts, for each of the three attention
    kernels, the tile pairs the busiest of n_sms persistent CTAs must run at
    least: the kernel's tile pairs (all samples and K/V heads) shared evenly,
    or its longest work item, whichever is more (the forward and dQ walk row
    lists, dK/dV the slices of its work list, kv_work_list).  Items: the
    forward's and dQ's (query tile, K/V head) pairs and dK/dV's (slice, K/V
    head) pairs."""
    g = n_heads // n_kv_heads
    c = tile_counts(cu_doc_lens, batch, seq_len, cp_size, cp_rank, g)
    nqt = (seq_len // cp_size) // (TILE // g)
    work = kv_work_list(c["col_counts"], n_kv_heads, n_sms,
                        kv_pool_slots(batch, seq_len, n_kv_heads, nqt))
    longest_slice = max((sl[2] for sl in work["slices"]), default=0)
    items = 2 * batch * nqt * n_kv_heads + len(work["slices"]) * n_kv_heads
    tiles = (c["full"] + c["partial"]) * n_kv_heads
    makespan = 2 * max(tiles / n_sms, c["max_row"]) + max(tiles / n_sms, longest_slice)
    return np.array([makespan, c["partial"] * n_kv_heads, items, 1.0], dtype=np.float64)


def fit_costs(features, times_ms) -> np.ndarray:
    """Non-negative least-squares constants (ms per tile pair of makespan,
    per partial pair, per item, and a fixed part) from rows of rank_costs
    features and measured step times of those ranks."""
    from scipy.optimize import nnls
    a = np.asarray(features, dtype=np.float64)
    t = np.asarray(times_ms, dtype=np.float64)
    coef, _ = nnls(a, t)
    return coef


# Constants fitted (fit_costs) to the measured per-rank step times of the
# 8B, 70B, sparse-stress and both 405B workloads on one GB300 (152 SMs), with
# the kernels' dynamic work distribution and the planner's cut dK/dV lists:
# ms per tile pair of makespan, per partial pair, per work item, fixed.
COST_MS_GB300 = np.array([1.25330e-03, 5.51287e-07, 0.0, 1.28789e-01])


def predict_ms(features, coef=None) -> np.ndarray:
    """Step time (ms) of each row of rank_costs features; default constants:
    COST_MS_GB300."""
    c = COST_MS_GB300 if coef is None else coef
    return np.asarray(features, dtype=np.float64) @ np.asarray(c, dtype=np.float64)


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
    rep = report(wl.cu_doc_lens(w), w.batch, w.seq_len, cp, args.granule, w.n_heads,
                 w.n_kv_heads)
    rep["workload"] = w.name
    print(json.dumps(rep))
    return 0


if __name__ == "__main__":
    raise SystemExit(_main())
