"""Explicit-softmax causal + document-masked GQA attention in float64.

Oracle (test infrastructure only; see ``oracle/__init__``).

What is computed, and where the pages fix it:

* Mask.  Query at global position p may see key position k iff k <= p
  (causal, "The Llama 3 Herd of Models - part 3/16", 3.3.2 "Context
  parallelism for long sequences": the full causal mask) and k lies in the
  same document as p ("Paper notes: The Llama 3 Herd of Models", "Two
  architectural choices"; the review "Scaling Llama 3 Training with Efficient
  Parallelism Strategies", CP design, Figure 7(b)/(c) document masks).  It
  is built here as an explicit boolean matrix from explicit document ids.
* GQA.  Several query heads share one K/V head (part 3/16, 3.3.2, citing
  Ainslie et al.; "Paper notes", 8 key-value heads).  Reading: contiguous
  groups, query head h uses K/V head h // (Hq / Hkv).
* Context parallelism.  The rank's queries are its two chunks (``oracle.cp``)
  against the full, all-gathered K and V (part 3/16, 3.3.2).
* Softmax attention.  O = softmax(scale * q k^T + mask) v, with the
  per-row log-sum-exp kept for the backward ("Training Infrastructure and
  Systems", "FlashAttention: never write the score matrix", sections
  "Online softmax" and "Tiling": the blocked method is exact, so its oracle
  is the plain definition written out here).  LSE is the natural log of the
  sum of exp of the scaled, masked logits.
* Backward.  The analytic gradient of that definition:
  dV = P^T dO, dP = dO V^T, Delta = rowsum(P * dP), dS = P * (dP - Delta),
  dQ = scale * dS K, dK = scale * dS^T Q, summed over the query heads of a
  group for dK and dV.  dK / dV are this rank's partial contribution (only
  its own query rows), the reading the pages leave for the reduction step.

The only liberty taken over the literal definition: a block of rows only
multiplies against the contiguous key range its mask touches.  Keys outside
that range are masked for every row of the block and contribute exactly 0
(exp(-inf) = 0), so dropping them changes no value.
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from . import cp as _cp


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor (bf16 upcasts exactly)
        import torch
        return x.detach().to(torch.float64).cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def allowed(ids_b: np.ndarray, qpos: np.ndarray, kpos: np.ndarray) -> np.ndarray:
    """Explicit mask [len(qpos), len(kpos)]: same document and key <= query."""
    same_doc = ids_b[qpos][:, None] == ids_b[kpos][None, :]
    causal = kpos[None, :] <= qpos[:, None]
    return same_doc & causal


def _rows_block(qb, kc, vc, mask, scale, dob):
    """One block of query rows of one head against its key columns."""
    x = scale * (qb @ kc.T)
    x = np.where(mask, x, -np.inf)
    m = x.max(axis=1, keepdims=True)          # every row has >= 1 key (k = p)
    e = np.exp(x - m)
    ell = e.sum(axis=1, keepdims=True)
    p = e / ell
    o = p @ vc
    lse = m[:, 0] + np.log(ell[:, 0])
    if dob is None:
        return o, lse, None, None, None
    dp = dob @ vc.T
    delta = (p * dp).sum(axis=1, keepdims=True)
    ds = p * (dp - delta)
    dq = scale * (ds @ kc)
    dk_c = scale * (ds.T @ qb)
    dv_c = p.T @ dob
    return o, lse, dq, dk_c, dv_c


def attention(q_local, k, v, cu_doc_lens, cp_size: int, cp_rank: int,
              scale: float | None = None, do_local=None, rows=None,
              block: int = 256, threads: int = 1,
              kv_grads_from_rows: bool = False) -> dict:
    """Forward (and, with ``do_local``, backward) for one CP rank.

    q_local, do_local : [B, Lq, Hq, D], this rank's query rows in local order
                        (chunk i, then chunk 2*CP-1-i).
    k, v              : [B, S, Hkv, D], full sequence, natural order.
    threads           : worker threads, each taking (head, row block) units
    rows              : optional local row indices; then only o / lse / dq
                        of those rows are computed (others are NaN) and no
                        dk / dv is returned (they need every row), unless
                        kv_grads_from_rows: then dk / dv are the contribution
                        of the selected rows alone.
    Returns float64 arrays: o [B,Lq,Hq,D], lse [B,Hq,Lq]; with do_local also
    dq [B,Lq,Hq,D], dk and dv [B,S,Hkv,D].
    """
    q = _f64(q_local)
    kk = _f64(k)
    vv = _f64(v)
    do = None if do_local is None else _f64(do_local)
    B, Lq, Hq, D = q.shape
    S, Hkv = kk.shape[1], kk.shape[2]
    assert Hq % Hkv == 0
    g = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    qpos_all = _cp.local_positions(S, cp_size, cp_rank)
    assert len(qpos_all) == Lq
    ids = _cp.doc_ids(cu_doc_lens, B, S)
    sel = np.arange(Lq) if rows is None else np.sort(np.asarray(rows))
    full = rows is None or kv_grads_from_rows

    o = np.full((B, Lq, Hq, D), np.nan)
    lse = np.full((B, Hq, Lq), np.nan)
    dq = None if do is None else np.full((B, Lq, Hq, D), np.nan)

    blocks = []
    for b in range(B):
        for s0 in range(0, len(sel), block):
            lr = sel[s0:s0 + block]
            qp = qpos_all[lr]
            mask_all = allowed(ids[b], qp, np.arange(S))
            cols = np.nonzero(mask_all.any(axis=0))[0]
            c0, c1 = int(cols[0]), int(cols[-1]) + 1
            blocks.append((b, lr, c0, c1, mask_all[:, c0:c1]))

    # work units (head, row block), dealt round-robin to the threads; each
    # thread keeps its own dK / dV partial sums, added at the end
    units = [(h, i) for h in range(Hq) for i in range(len(blocks))]

    def run_units(mine):
        dk_part = np.zeros((B, S, Hkv, D)) if (do is not None and full) else None
        dv_part = np.zeros((B, S, Hkv, D)) if (do is not None and full) else None
        for h, i in mine:
            kvh = h // g
            b, lr, c0, c1, mask = blocks[i]
            qb = q[b, lr, h]
            kc = kk[b, c0:c1, kvh]
            vc = vv[b, c0:c1, kvh]
            dob = None if do is None else do[b, lr, h]
            ob, lb, dqb, dkc, dvc = _rows_block(qb, kc, vc, mask, scale, dob)
            o[b, lr, h] = ob
            lse[b, h, lr] = lb
            if dob is not None:
                dq[b, lr, h] = dqb
                if full:
                    dk_part[b, c0:c1, kvh] += dkc
                    dv_part[b, c0:c1, kvh] += dvc
        return dk_part, dv_part

    nthreads = max(1, min(threads, len(units)))
    shares = [units[w::nthreads] for w in range(nthreads)]
    if nthreads == 1:
        parts = [run_units(shares[0])]
    else:
        with ThreadPoolExecutor(nthreads) as ex:
            parts = list(ex.map(run_units, shares))

    out = {"o": o, "lse": lse}
    if rows is not None and full and do is not None:
        out["kv_grads_rows"] = sel
    if do is not None:
        out["dq"] = dq
        if full:
            out["dk"] = sum(p[0] for p in parts)
            out["dv"] = sum(p[1] for p in parts)
    return out


def delta_rowsum_do_o(o, do) -> np.ndarray:
    """Delta[b, h, l] = sum_d dO * O, the rowsum the backward preprocess of a
    blocked backward computes (equal to rowsum(P * dP) of the definition,
    since rowsum(P * (dO V^T)) = dO . (P V) = dO . O).  [B, Hq, Lq]."""
    return np.einsum("blhd,blhd->bhl", _f64(o), _f64(do))
