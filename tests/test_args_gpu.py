"""Argument values and inputs the workload configurations leave untried, on
the GPU against the float64 oracle:

* a softmax scale other than 1/sqrt(D): the 8B-layer inputs (q already
  multiplied by 1/sqrt(128)) with softmax_scale = 1, the alternative reading
  of that configuration in which the pre-scale is the softmax scale;
* large logits (q x 6, logit std 6 nats) with documents several key tiles
  long, so that the forward's lazy running-max update, which rescales the
  partial O when a row's max grows by more than 2^8, does so on many rows
  with a nonzero O (a host replay of the tile walk counts them);
* V holding +-1e5 and one NaN: the finite out-of-range values saturate in the
  forward's fp16 copy of V and the plan reports DMA_WARN_V_SATURATED; the NaN
  reaches O in its column for every row that attends its key, as it would
  in bf16 arithmetic; everything else matches the oracle.
"""
import math

import numpy as np
import pytest
import torch

from document_masked_gqa_gb300 import workloads as wl
from helpers import TOL_GRAD, TOL_LSE, TOL_O, gpu_rank, max_abs, oracle_rank, rel_fro

pytestmark = pytest.mark.gpu


def _full_parity(w, scale_arg, scale_oracle):
    cu = wl.cu_doc_lens(w)
    inp = wl.tensors(w)
    for r in w.ranks:
        g, _ = gpu_rank(w, r, inp, cu, backward=True, scale=scale_arg)
        ref = oracle_rank(w, r, inp, cu, backward=True, scale=scale_oracle, threads=8)
        assert max_abs(g["o"].numpy(), ref["o"]) <= TOL_O, (w.name, r)
        assert max_abs(g["lse"].numpy(), ref["lse"]) <= TOL_LSE, (w.name, r)
        for key in ("dq", "dk", "dv"):
            x = g[key].numpy()
            assert np.isfinite(x).all(), (w.name, r, key)
            assert rel_fro(x, ref[key]) <= TOL_GRAD, (w.name, r, key)


def test_softmax_scale_one_on_prescaled_8b_inputs():
    _full_parity(wl.WORKLOADS["8b"], 1.0, 1.0)


LARGE_LOGITS = wl.custom("large-logits", 4096, 2, 1, 8, 1, 128, "loguniform", 256, 4096,
                         seed=21, q_prescale=6.0)


def _rescales_with_nonzero_o(w, inp, cu, rank):
    """Replay of the forward's per-row tile walk on the host: for each query
    row (all heads), walk the key tiles that hold an allowed key in ascending
    order, take the tile's row max of the scaled logits in base 2, and move
    the reference max only when it grows by more than 8; count the rows
    where it moves after the first such tile (O already nonzero)."""
    from oracle import cp as ocp
    C, Lq, g = w.chunk, w.local_len, w.group
    qpos = ocp.local_positions(w.seq_len, w.cp_size, rank)
    ids = ocp.doc_ids(cu, w.batch, w.seq_len)[0]
    q = ocp.gather_local(inp["q"], w.seq_len, w.cp_size, rank)[0].double().numpy()
    k = inp["k"][0, :, 0].double().numpy()
    sl2 = (1.0 / math.sqrt(w.head_dim)) / math.log(2.0)
    count = 0
    for l in range(Lq):
        p = int(qpos[l])
        lo = int(np.searchsorted(ids, ids[p], side="left"))
        x = (q[l] @ k[lo:p + 1].T) * sl2           # [g, keys]
        t_first, t_last = lo // 128, p // 128
        for h in range(g):
            m = -np.inf
            for t in range(t_first, t_last + 1):
                a, b = max(lo, 128 * t), min(p + 1, 128 * t + 128)
                mx = float(x[h, a - lo:b - lo].max())
                if mx > m + 8.0:
                    if t > t_first:
                        count += 1
                        break
                    m = mx
    return count


def test_large_logits_lazy_rescale():
    w = LARGE_LOGITS
    cu = wl.cu_doc_lens(w)
    inp = wl.tensors(w)
    hits = sum(_rescales_with_nonzero_o(w, inp, cu, r) for r in w.ranks)
    assert hits >= 500, hits  # the rescale path runs on many rows
    _full_parity(w, 0.0, None)


def test_v_saturation_and_nan_propagation():
    import document_masked_gqa_gb300 as dma
    from oracle import cp as ocp
    w = wl.WORKLOADS["tiny"]
    cu = wl.cu_doc_lens(w)
    inp = wl.tensors(w, with_grad=False)
    v = inp["v"].clone()
    ka, kb = 97, 250          # key positions: +-1e5 at ka, NaN at kb
    v[0, ka, 0, 7] = 1.0e5
    v[0, ka, 0, 9] = -1.0e5
    v[0, kb, 0, 5] = float("nan")
    inp_v = dict(inp, v=v)
    dev = torch.device("cuda:0")
    cu_d = torch.from_numpy(cu).to(dev)
    ids = ocp.doc_ids(cu, w.batch, w.seq_len)[0]
    # the oracle sees V as the kernel's fp16 copy holds it: +-65504 at ka
    v_sat = v.clone()
    v_sat[0, ka, 0, 7] = 65504.0
    v_sat[0, ka, 0, 9] = -65504.0
    for r in w.ranks:
        plan = dma.dma_plan(cu_d, w.batch, w.seq_len, w.cp_size, r, w.n_heads, w.n_kv_heads,
                            w.head_dim)
        q = dma.dma_cp_gather(plan, inp["q"].to(dev))
        o, lse = dma.dma_attn_fwd(plan, q, inp["k"].to(dev), v.to(dev))
        torch.cuda.synchronize()
        assert dma.dma_plan_check(plan) == dma.DMA_WARN_V_SATURATED
        o = o.cpu().numpy()
        lse = lse.cpu().numpy()
        ref = oracle_rank(w, r, dict(inp_v, v=v_sat), cu, backward=False)
        qpos = ocp.local_positions(w.seq_len, w.cp_size, r)
        sees = lambda key: (ids[qpos] == ids[key]) & (qpos >= key)  # noqa: E731
        # LSE does not depend on V
        assert np.isfinite(lse).all() and max_abs(lse, ref["lse"]) <= TOL_LSE
        # every column without the NaN or a saturated value matches the
        # oracle on the saturated V
        cols = [c for c in range(w.head_dim) if c not in (5, 7, 9)]
        assert max_abs(o[..., cols], ref["o"][..., cols]) <= TOL_O, r
        # the saturated columns too, within the fp16 rounding of P times
        # 65504 (relative 2^-11 of the term that value contributes)
        for c in (7, 9):
            err = np.abs(o[..., c].astype(np.float64) - ref["o"][..., c])
            assert (err <= TOL_O + 2.0 ** -10 * np.abs(ref["o"][..., c])).all(), (r, c)
        # the NaN reaches column 5 of every row that attends its key ...
        rows_b = np.nonzero(sees(kb))[0]
        assert len(rows_b) > 0 or r == 1
        assert np.isnan(o[0, rows_b, :, 5]).all()
        # ... and no row of a query tile that lies wholly before its key tile
        tp = 128 // w.group
        early = [l for l in range(w.local_len)
                 if qpos[(l // tp) * tp:(l // tp + 1) * tp].max() < (kb // 128) * 128]
        assert len(early) > 0
        assert np.isfinite(o[0, early]).all()
        # rows that attend the saturated key see +-65504 there
        rows_a = np.nonzero(sees(ka))[0]
        assert len(rows_a) > 0 or r == 0
        assert np.isfinite(o[0, rows_a][..., [c for c in range(w.head_dim) if c != 5]]).all()
