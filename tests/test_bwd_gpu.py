"""Backward parity on the GPU against the float64 oracle: dQ, dK, dV relative
Frobenius error <= 2e-2 per tensor per rank (full tensors where the oracle is
quick), CP re-assembly of the per-rank partial gradients against the CP=1
oracle, and at the 405B size sampled dQ rows plus identities that hold at any
size."""
import numpy as np
import pytest
import torch

from document_masked_gqa_gb300 import workloads as wl
from helpers import TOL_GRAD, TOL_LSE, TOL_O, gpu_rank, max_abs, oracle_rank, rel_fro
from oracle import attention as oa
from oracle import cp as ocp
from test_plan_gpu import EDGE

pytestmark = pytest.mark.gpu


def _bwd_case(w, rank, inp=None, cu=None):
    cu = wl.cu_doc_lens(w) if cu is None else cu
    inp = wl.tensors(w) if inp is None else inp
    g, _ = gpu_rank(w, rank, inp, cu, backward=True)
    ref = oracle_rank(w, rank, inp, cu, backward=True)
    assert max_abs(g["o"].numpy(), ref["o"]) <= TOL_O
    assert max_abs(g["lse"].numpy(), ref["lse"]) <= TOL_LSE
    errs = {}
    for key in ("dq", "dk", "dv"):
        x = g[key].numpy()
        assert np.isfinite(x).all(), (w.name, rank, key)
        errs[key] = rel_fro(x, ref[key])
        assert errs[key] <= TOL_GRAD, (w.name, rank, key, errs[key])
    return g, ref, errs


@pytest.mark.parametrize("name", ["tiny", "70b", "sparse", "8b"])
def test_bwd_parity_full(name):
    w = wl.WORKLOADS[name]
    cu = wl.cu_doc_lens(w)
    inp = wl.tensors(w)
    for r in w.ranks:
        _bwd_case(w, r, inp, cu)


@pytest.mark.parametrize("name", list(EDGE))
def test_bwd_parity_edge(name):
    w = EDGE[name]
    cu = wl.cu_doc_lens(w)
    inp = wl.tensors(w)
    for r in w.ranks:
        _bwd_case(w, r, inp, cu)


@pytest.mark.parametrize("name", ["tiny", "70b", "sparse"])
def test_cp_reassembly_against_cp1_oracle(name):
    """All ranks of the GPU path, put back together, equal the oracle run on
    the whole sequence as one rank (CP=1); partial dK/dV sum to the full."""
    w = wl.WORKLOADS[name]
    assert tuple(w.ranks) == tuple(range(w.cp_size))
    cu = wl.cu_doc_lens(w)
    inp = wl.tensors(w)
    outs = {r: gpu_rank(w, r, inp, cu)[0] for r in w.ranks}
    full = oa.attention(inp["q"], inp["k"], inp["v"], cu, 1, 0, do_local=inp["do"], threads=4)
    o = ocp.assemble_full({r: outs[r]["o"].numpy() for r in outs}, w.seq_len, w.cp_size)
    dq = ocp.assemble_full({r: outs[r]["dq"].numpy() for r in outs}, w.seq_len, w.cp_size)
    lse = ocp.assemble_full({r: outs[r]["lse"].numpy().transpose(0, 2, 1) for r in outs},
                            w.seq_len, w.cp_size).transpose(0, 2, 1)
    assert max_abs(o, full["o"]) <= TOL_O
    assert max_abs(lse, full["lse"]) <= TOL_LSE
    assert rel_fro(dq, full["dq"]) <= TOL_GRAD
    dk = sum(outs[r]["dk"].numpy() for r in outs)
    dv = sum(outs[r]["dv"].numpy() for r in outs)
    assert rel_fro(dk, full["dk"]) <= TOL_GRAD
    assert rel_fro(dv, full["dv"]) <= TOL_GRAD


def test_bwd_parity_405b_logu_rank15_full():
    """Full outputs at the 405B size for the lightest emulated rank."""
    w = wl.WORKLOADS["405b-logu"]
    cu = wl.cu_doc_lens(w)
    inp = wl.tensors(w)
    g, _ = gpu_rank(w, 15, inp, cu, backward=True)
    ref = oracle_rank(w, 15, inp, cu, backward=True, threads=8)
    assert max_abs(g["o"].numpy(), ref["o"]) <= TOL_O
    assert max_abs(g["lse"].numpy(), ref["lse"]) <= TOL_LSE
    for key in ("dq", "dk", "dv"):
        assert rel_fro(g[key].numpy(), ref[key]) <= TOL_GRAD, key


@pytest.mark.parametrize("name", ["405b-logu", "405b-1doc", "causal-128k"])
def test_bwd_405b_sampled_rows_and_tail_keys(name):
    """Every emulated rank at full size: sampled query rows (O, LSE, dQ), the
    exact dK/dV of the last key tile the rank reaches (only its last 128
    local rows attend those keys, so the oracle restricted to those rows
    gives them exactly), and sum_k dV = sum of dO over rows and heads."""
    w = wl.WORKLOADS[name]
    cu = wl.cu_doc_lens(w)
    inp = wl.tensors(w)
    rng = np.random.default_rng(7)
    for r in w.ranks:
        g, _ = gpu_rank(w, r, inp, cu, backward=True)
        rows = np.unique(np.concatenate([[0, w.chunk - 1, w.chunk, w.local_len - 1],
                                         rng.integers(0, w.local_len, 28)]))
        ref = oracle_rank(w, r, inp, cu, backward=True, rows=rows, threads=8)
        assert max_abs(g["o"].numpy()[:, rows], ref["o"][:, rows]) <= TOL_O
        assert max_abs(g["lse"].numpy()[:, :, rows], ref["lse"][:, :, rows]) <= TOL_LSE
        assert rel_fro(g["dq"].numpy()[:, rows], ref["dq"][:, rows]) <= TOL_GRAD
        dk, dv = g["dk"].numpy(), g["dv"].numpy()
        assert np.isfinite(dk).all() and np.isfinite(dv).all()
        # last key tile this rank reaches: positions [k_end - 128, k_end)
        k_end = (2 * w.cp_size - r) * w.chunk
        tail = np.arange(w.local_len - 128, w.local_len)
        from oracle import attention as oa
        q_l = ocp.gather_local(inp["q"], w.seq_len, w.cp_size, r)
        do_l = ocp.gather_local(inp["do"], w.seq_len, w.cp_size, r)
        ref_t = oa.attention(q_l, inp["k"], inp["v"], cu, w.cp_size, r, do_local=do_l,
                             rows=tail, kv_grads_from_rows=True, threads=8)
        ks = slice(k_end - 128, k_end)
        assert rel_fro(dk[:, ks], ref_t["dk"][:, ks]) <= TOL_GRAD
        assert rel_fro(dv[:, ks], ref_t["dv"][:, ks]) <= TOL_GRAD
        # no key beyond the rank's last position receives gradient
        assert not dk[:, k_end:].any() and not dv[:, k_end:].any()
        # every row's P sums to one: sum over keys of dV = sum of dO over the
        # rank's rows and the group's heads
        lhs = dv.astype(np.float64).sum(axis=1)                       # [B, Hkv, D]
        rhs = do_l.double().numpy().reshape(w.batch, w.local_len, w.n_kv_heads, w.group,
                                            w.head_dim).sum(axis=(1, 3))
        assert rel_fro(lhs, rhs) <= TOL_GRAD


@pytest.mark.parametrize("name", ["70b", "8b"])
def test_split_backward_entry_points(name):
    """The backward's parts called one by one: Delta by its own pass, then
    dQ reading it, then dK/dV, against the oracle; and the fused dQ + Delta
    launch gives the same dQ up to the order of Delta's sum."""
    import document_masked_gqa_gb300 as dma
    w = wl.WORKLOADS[name]
    cu = wl.cu_doc_lens(w)
    inp = wl.tensors(w)
    dev = torch.device("cuda:0")
    cu_d = torch.from_numpy(cu).to(dev)
    k, v = inp["k"].to(dev), inp["v"].to(dev)
    r = w.ranks[-1]
    plan = dma.dma_plan(cu_d, w.batch, w.seq_len, w.cp_size, r, w.n_heads, w.n_kv_heads,
                        w.head_dim)
    q = dma.dma_cp_gather(plan, inp["q"].to(dev))
    do = dma.dma_cp_gather(plan, inp["do"].to(dev))
    o, lse = dma.dma_attn_fwd(plan, q, k, v)
    dq = torch.empty_like(q)
    dk = torch.empty(w.batch, w.seq_len, w.n_kv_heads, w.head_dim, device=dev)
    dv = torch.empty_like(dk)
    dma.dma_attn_bwd_delta(plan, o, do)
    dma.dma_attn_bwd_dq(plan, q, k, v, lse, do, dq)
    dma.dma_attn_bwd_dkdv(plan, q, k, v, lse, do, dk, dv)
    torch.cuda.synchronize()
    assert dma.dma_plan_check(plan) == 0
    ref = oracle_rank(w, r, inp, cu, backward=True, threads=8)
    for key, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert rel_fro(got.float().cpu().numpy(), ref[key]) <= TOL_GRAD, (name, key)
    # the fused launch gives the same gradients up to the order of Delta's sum
    dq2 = torch.empty_like(q)
    dma.dma_attn_bwd_dq_delta(plan, q, k, v, o, lse, do, dq2)
    torch.cuda.synchronize()
    assert rel_fro(dq2.float().cpu().numpy(), dq.float().cpu().numpy()) <= 1e-3
