"""Forward parity on the GPU against the float64 oracle: O max-abs <= 1e-2,
LSE max-abs <= 1e-3 per rank, on the seeded workloads (full outputs where the
oracle is quick, sampled rows at the 405B size) and on edge shapes."""
import numpy as np
import pytest

from document_masked_gqa_gb300 import workloads as wl
from helpers import TOL_LSE, TOL_O, gpu_rank, max_abs, oracle_rank
from test_plan_gpu import EDGE

pytestmark = pytest.mark.gpu


def _fwd_case(w, rank, rows=None):
    cu = wl.cu_doc_lens(w)
    inp = wl.tensors(w, with_grad=False)
    g, _ = gpu_rank(w, rank, inp, cu, backward=False)
    ref = oracle_rank(w, rank, inp, cu, backward=False, rows=rows)
    if rows is None:
        eo = max_abs(g["o"].numpy(), ref["o"])
        el = max_abs(g["lse"].numpy(), ref["lse"])
    else:
        eo = max_abs(g["o"].numpy()[:, rows], ref["o"][:, rows])
        el = max_abs(g["lse"].numpy()[:, :, rows], ref["lse"][:, :, rows])
    assert np.isfinite(g["o"].numpy()).all() and np.isfinite(g["lse"].numpy()).all()
    assert eo <= TOL_O, (w.name, rank, "o", eo)
    assert el <= TOL_LSE, (w.name, rank, "lse", el)
    return eo, el


@pytest.mark.parametrize("name", ["tiny", "70b", "sparse", "8b"])
def test_fwd_parity_full(name):
    w = wl.WORKLOADS[name]
    for r in w.ranks:
        _fwd_case(w, r)


@pytest.mark.parametrize("name", list(EDGE))
def test_fwd_parity_edge(name):
    w = EDGE[name]
    for r in w.ranks:
        _fwd_case(w, r)


@pytest.mark.parametrize("name", ["405b-logu", "405b-1doc", "causal-128k"])
def test_fwd_parity_405b_sampled_rows(name):
    w = wl.WORKLOADS[name]
    rng = np.random.default_rng(99)
    for r in w.ranks:
        rows = np.unique(np.concatenate([[0, w.chunk - 1, w.chunk, w.local_len - 1],
                                         rng.integers(0, w.local_len, 60)]))
        _fwd_case(w, r, rows=rows)
