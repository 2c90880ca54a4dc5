"""Pins for the float64 oracle: checks against what the pages and the
mathematics fix, never against the oracle's own formulas retyped.

* golden worked examples (tests/golden/*.json, hand-derived, cited there);
* library routine: torch scaled_dot_product_attention in float64 (causal),
  forward and autograd backward;
* finite differences of the forward for the analytic backward;
* GQA against MHA on K/V heads repeated with repeat_interleave;
* context-parallel re-assembly of all ranks against the CP=1 result;
* the single-document load-balance closed form and brute-force counts.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import attention as oa
from oracle import blockmask as ob
from oracle import cp as ocp
from oracle import flops as ofl
from document_masked_gqa_gb300 import workloads as wl

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


def _val(x):
    if isinstance(x, (int, float)):
        return float(x)
    table = {"ln3": math.log(3.0), "ln4": math.log(4.0), "0.75*ln3": 0.75 * math.log(3.0),
             "(10*e5+30)/(e5+1)": (10 * math.exp(5) + 30) / (math.exp(5) + 1),
             "ln(e5+1)": math.log(math.exp(5) + 1)}
    return table[x]


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def _rand(shape, seed, dtype=torch.float64):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=dtype)


# ----------------------------------------------------------------- CP rules

def test_golden_cp_chunks(golden_dir):
    for case in _load(golden_dir, "cp_chunks.json")["cases"]:
        assert list(ocp.rank_chunks(case["cp_size"], case["rank"])) == case["chunks"]


@pytest.mark.parametrize("cp_size", [1, 2, 3, 4, 16])
def test_local_positions_partition_sequence(cp_size):
    S = 2 * cp_size * 8
    allpos = np.concatenate([ocp.local_positions(S, cp_size, r) for r in range(cp_size)])
    assert sorted(allpos.tolist()) == list(range(S))
    order = ocp.chunk_order(cp_size)
    assert sorted(order) == list(range(2 * cp_size))
    # the rank-major order lays the ranks' positions end to end
    C = S // (2 * cp_size)
    expect = np.concatenate([np.arange(c * C, (c + 1) * C) for c in order])
    assert (allpos == expect).all()


def test_docs_valid():
    assert ocp.docs_valid([0, 3, 8], 1, 8)
    assert not ocp.docs_valid([1, 3, 8], 1, 8)       # must start at 0
    assert not ocp.docs_valid([0, 3, 3, 8], 1, 8)    # strictly increasing
    assert not ocp.docs_valid([0, 3, 7], 1, 8)       # must end at B*S
    assert not ocp.docs_valid([0, 5, 11, 16], 2, 8)  # boundary 8 missing
    assert ocp.docs_valid([0, 5, 8, 11, 16], 2, 8)


# ---------------------------------------------------------- worked examples

def test_golden_worked_attention(golden_dir):
    for case in _load(golden_dir, "worked_attention.json")["cases"]:
        S = case["seq_len"]
        q = np.array([_val(x) for x in case["q"]]).reshape(1, S, 1, 1)
        k = np.array([_val(x) for x in case["k"]]).reshape(1, S, 1, 1)
        v = np.array([_val(x) for x in case["v"]]).reshape(1, S, 1, 1)
        do = np.array([_val(x) for x in case["do"]]).reshape(1, S, 1, 1)
        r = oa.attention(q, k, v, case["cu_doc_lens"], 1, 0, scale=1.0, do_local=do)
        np.testing.assert_allclose(r["o"].ravel(), [_val(x) for x in case["o"]], rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(r["lse"].ravel(), [_val(x) for x in case["lse"]], rtol=1e-13, atol=1e-13)
        for key in ("dq", "dk", "dv"):
            if key in case:
                np.testing.assert_allclose(r[key].ravel(), [_val(x) for x in case[key]],
                                           rtol=1e-13, atol=1e-13)


def test_uniform_scores_closed_form():
    """q = 0 makes every allowed logit 0: O is the plain mean of the allowed
    v rows and LSE = ln(number of allowed keys) = ln(p - doc_start + 1)."""
    B, S, Hq, Hkv, D, cp = 2, 64, 4, 2, 8, 2
    cu = np.array([0, 5, 30, 64, 64 + 17, 128])
    k = _rand((B, S, Hkv, D), 1).numpy()
    v = _rand((B, S, Hkv, D), 2).numpy()
    start = ocp.doc_start(cu, B, S)
    for r in range(cp):
        Lq = S // cp
        q = np.zeros((B, Lq, Hq, D))
        res = oa.attention(q, k, v, cu, cp, r)
        qpos = ocp.local_positions(S, cp, r)
        for b in range(B):
            for i, p in enumerate(qpos):
                s0 = start[b, p]
                for h in range(Hq):
                    mean = v[b, s0:p + 1, h // (Hq // Hkv)].mean(axis=0)
                    np.testing.assert_allclose(res["o"][b, i, h], mean, rtol=1e-12, atol=1e-12)
                    assert abs(res["lse"][b, h, i] - math.log(p - s0 + 1)) < 1e-12


# -------------------------------------------- library routine: torch SDPA

def _sdpa_causal(q, k, v):
    """torch SDPA, float64, causal, q/k/v [S, H, D] -> [S, H, D]."""
    o = torch.nn.functional.scaled_dot_product_attention(
        q.transpose(0, 1), k.transpose(0, 1), v.transpose(0, 1), is_causal=True)
    return o.transpose(0, 1)


def test_single_doc_cp1_equals_sdpa_fwd_bwd():
    B, S, H, D = 2, 48, 3, 16
    q, k, v, do = (_rand((B, S, H, D), s) for s in (10, 11, 12, 13))
    cu = [0, S, 2 * S]
    res = oa.attention(q, k, v, cu, 1, 0, do_local=do)
    for b in range(B):
        qq, kk, vv = (t[b].clone().requires_grad_(True) for t in (q, k, v))
        o = _sdpa_causal(qq, kk, vv)
        o.backward(do[b])
        np.testing.assert_allclose(res["o"][b], o.detach().numpy(), rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(res["dq"][b], qq.grad.numpy(), rtol=1e-10, atol=1e-11)
        np.testing.assert_allclose(res["dk"][b], kk.grad.numpy(), rtol=1e-10, atol=1e-11)
        np.testing.assert_allclose(res["dv"][b], vv.grad.numpy(), rtol=1e-10, atol=1e-11)
        # LSE: logsumexp of the causal logits, through torch's own routine
        logits = torch.einsum("qhd,khd->hqk", q[b], k[b]) / math.sqrt(D)
        logits = logits.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), float("-inf"))
        np.testing.assert_allclose(res["lse"][b], torch.logsumexp(logits, -1).numpy(),
                                   rtol=1e-12, atol=1e-12)


def test_documents_equal_per_document_sdpa():
    """Document masking = causal attention run on each document on its own."""
    B, S, H, D = 2, 64, 2, 8
    q, k, v, do = (_rand((B, S, H, D), s) for s in (20, 21, 22, 23))
    lens = [[10, 1, 30, 23], [64]]
    cu = [0]
    for ls in lens:
        for n in ls:
            cu.append(cu[-1] + n)
    res = oa.attention(q, k, v, cu, 1, 0, do_local=do)
    for b in range(B):
        s0 = 0
        for n in lens[b]:
            sl = slice(s0, s0 + n)
            qq, kk, vv = (t[b, sl].clone().requires_grad_(True) for t in (q, k, v))
            o = _sdpa_causal(qq, kk, vv)
            o.backward(do[b, sl])
            np.testing.assert_allclose(res["o"][b, sl], o.detach().numpy(), rtol=1e-11, atol=1e-12)
            np.testing.assert_allclose(res["dq"][b, sl], qq.grad.numpy(), rtol=1e-10, atol=1e-11)
            np.testing.assert_allclose(res["dk"][b, sl], kk.grad.numpy(), rtol=1e-10, atol=1e-11)
            np.testing.assert_allclose(res["dv"][b, sl], vv.grad.numpy(), rtol=1e-10, atol=1e-11)
            s0 += n


# ------------------------------------------------------------------- GQA

def test_gqa_equals_mha_on_repeated_kv():
    B, S, Hq, Hkv, D, cp = 1, 32, 6, 2, 8, 2
    g = Hq // Hkv
    cu = [0, 7, 19, 32]
    qf, kf, vf, dof = (_rand((B, S, H, D), s) for s, H in ((30, Hq), (31, Hkv), (32, Hkv), (33, Hq)))
    kr = kf.repeat_interleave(g, dim=2)
    vr = vf.repeat_interleave(g, dim=2)
    for r in range(cp):
        ql = ocp.gather_local(qf.numpy(), S, cp, r)
        dol = ocp.gather_local(dof.numpy(), S, cp, r)
        a = oa.attention(ql, kf, vf, cu, cp, r, do_local=dol)
        m = oa.attention(ql, kr, vr, cu, cp, r, do_local=dol)
        np.testing.assert_allclose(a["o"], m["o"], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(a["lse"], m["lse"], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(a["dq"], m["dq"], rtol=1e-12, atol=1e-13)
        dk_sum = m["dk"].reshape(B, S, Hkv, g, D).sum(axis=3)
        dv_sum = m["dv"].reshape(B, S, Hkv, g, D).sum(axis=3)
        np.testing.assert_allclose(a["dk"], dk_sum, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(a["dv"], dv_sum, rtol=1e-12, atol=1e-13)


# ------------------------------------------------------ finite differences

def test_backward_matches_finite_differences():
    B, S, Hq, Hkv, D, cp, r = 1, 16, 2, 1, 4, 2, 1
    cu = [0, 5, 12, 16]
    rng = np.random.default_rng(5)
    q = rng.standard_normal((B, S // cp, Hq, D))
    k = rng.standard_normal((B, S, Hkv, D))
    v = rng.standard_normal((B, S, Hkv, D))
    do = rng.standard_normal((B, S // cp, Hq, D))
    res = oa.attention(q, k, v, cu, cp, r, do_local=do)

    def loss(qq, kk, vv):
        return float((oa.attention(qq, kk, vv, cu, cp, r)["o"] * do).sum())

    eps = 1e-6
    for name, arr, key in (("q", q, "dq"), ("k", k, "dk"), ("v", v, "dv")):
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            plus, minus = arr.copy(), arr.copy()
            plus[idx] += eps
            minus[idx] -= eps
            args = {"q": q, "k": k, "v": v}
            args[name] = plus
            lp = loss(args["q"], args["k"], args["v"])
            args[name] = minus
            lm = loss(args["q"], args["k"], args["v"])
            num[idx] = (lp - lm) / (2 * eps)
        err = np.linalg.norm(num - res[key]) / np.linalg.norm(num)
        assert err < 1e-6, (name, err)


# ------------------------------------------------------- CP re-assembly

@pytest.mark.parametrize("cp_size", [2, 4])
def test_cp_reassembly_equals_full_sequence(cp_size):
    B, S, Hq, Hkv, D = 2, 64, 4, 2, 8
    cu = [0, 9, 40, 64, 70, 128]
    qf, kf, vf, dof = (_rand((B, S, H, D), s) for s, H in ((40, Hq), (41, Hkv), (42, Hkv), (43, Hq)))
    full = oa.attention(qf, kf, vf, cu, 1, 0, do_local=dof)
    per = {}
    for r in range(cp_size):
        ql = ocp.gather_local(qf.numpy(), S, cp_size, r)
        dol = ocp.gather_local(dof.numpy(), S, cp_size, r)
        per[r] = oa.attention(ql, kf, vf, cu, cp_size, r, do_local=dol)
    for key in ("o", "dq"):
        got = ocp.assemble_full({r: per[r][key] for r in per}, S, cp_size)
        np.testing.assert_allclose(got, full[key], rtol=1e-12, atol=1e-13)
    lse = ocp.assemble_full({r: per[r]["lse"].transpose(0, 2, 1) for r in per}, S, cp_size)
    np.testing.assert_allclose(lse.transpose(0, 2, 1), full["lse"], rtol=1e-12, atol=1e-13)
    for key in ("dk", "dv"):
        np.testing.assert_allclose(sum(per[r][key] for r in per), full[key], rtol=1e-11, atol=1e-12)


def test_row_sampled_mode_matches_full():
    B, S, Hq, Hkv, D, cp = 1, 128, 4, 1, 8, 2
    cu = [0, 20, 21, 100, 128]
    qf, kf, vf, dof = (_rand((B, S, H, D), s) for s, H in ((50, Hq), (51, Hkv), (52, Hkv), (53, Hq)))
    ql = ocp.gather_local(qf.numpy(), S, cp, 1)
    dol = ocp.gather_local(dof.numpy(), S, cp, 1)
    full = oa.attention(ql, kf, vf, cu, cp, 1, do_local=dol)
    rows = [0, 3, 17, 31, 32, 63]
    part = oa.attention(ql, kf, vf, cu, cp, 1, do_local=dol, rows=rows, block=4)
    np.testing.assert_allclose(part["o"][:, rows], full["o"][:, rows], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(part["dq"][:, rows], full["dq"][:, rows], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(part["lse"][:, :, rows], full["lse"][:, :, rows], rtol=1e-13, atol=1e-14)
    # the threaded path gives the same numbers
    thr = oa.attention(ql, kf, vf, cu, cp, 1, do_local=dol, threads=3)
    for key in ("o", "lse", "dq", "dk", "dv"):
        np.testing.assert_allclose(thr[key], full[key], rtol=1e-13, atol=1e-14)


def test_delta_identity():
    """rowsum(dO * O) equals rowsum(P * dP) of the definition (the oracle's
    backward uses the latter; the library's preprocess the former)."""
    B, S, Hq, Hkv, D = 1, 32, 2, 1, 8
    cu = [0, 11, 32]
    q, k, v, do = (_rand((B, S, H, D), s) for s, H in ((60, Hq), (61, Hkv), (62, Hkv), (63, Hq)))
    res = oa.attention(q, k, v, cu, 1, 0, do_local=do)
    d1 = oa.delta_rowsum_do_o(res["o"], do)
    # rowsum(P * dP) with P recovered through the library routine softmax
    ids = ocp.doc_ids(cu, B, S)
    for h in range(Hq):
        x = (q[0, :, h] @ k[0, :, 0].T).numpy() / math.sqrt(D)
        m = oa.allowed(ids[0], np.arange(S), np.arange(S))
        p = torch.softmax(torch.from_numpy(np.where(m, x, -np.inf)), -1).numpy()
        dp = do[0, :, h].numpy() @ v[0, :, 0].numpy().T
        np.testing.assert_allclose(d1[0, h], (p * dp).sum(1), rtol=1e-11, atol=1e-12)


# --------------------------------------------------- load balance, counts

def test_golden_load_balance(golden_dir):
    for case in _load(golden_dir, "load_balance.json")["cases"]:
        S, cp = case["seq_len"], case["cp_size"]
        assert ofl.single_doc_pairs_closed_form(case["chunk"], cp) == case["pairs_per_rank_per_head"]
        for r in sorted({0, cp // 2, cp - 1}):
            got = ofl.pairs_per_head([0, S], 1, S, cp, r)
            assert int(got[0]) == case["pairs_per_rank_per_head"]


def test_pair_count_equals_explicit_mask_sum():
    B, S, cp = 2, 96, 3
    cu = [0, 13, 14, 50, 96, 96 + 40, 192]
    ids = ocp.doc_ids(cu, B, S)
    for r in range(cp):
        qp = ocp.local_positions(S, cp, r)
        got = ofl.pairs_per_head(cu, B, S, cp, r)
        for b in range(B):
            assert int(got[b]) == int(oa.allowed(ids[b], qp, np.arange(S)).sum())


# ---------------------------------------------------------- tile classes

def test_golden_tile_classes(golden_dir):
    for case in _load(golden_dir, "tile_classes.json")["cases"]:
        cu = case["cu_doc_lens"]
        if isinstance(cu, str):
            cu = list(range(0, case["seq_len"] + 1))
        got = ob.tile_classes(cu, case["batch"], case["seq_len"], case["cp_size"],
                              case["rank"], case["group"])
        assert got.tolist() == case["classes"], case["name"]


@pytest.mark.parametrize("group", [1, 4, 16])
def test_tile_classes_account_for_every_pair(group):
    w = wl.custom("t", 1024, 2, 2, 16, 16 // group, 64, "uniform", 20, 300, seed=3)
    cu = wl.cu_doc_lens(w)
    P = 128 // group
    for r in range(2):
        cls = ob.tile_classes(cu, w.batch, w.seq_len, 2, r, group)
        pairs = int(ofl.pairs_per_head(cu, w.batch, w.seq_len, 2, r).sum())
        n_full = int((cls == ob.FULL).sum())
        in_partial = ob.allowed_count_in_partials(cu, w.batch, w.seq_len, 2, r, group, cls)
        assert n_full * P * 128 + in_partial == pairs
        # a partial tile holds at least one allowed and one masked element
        n_part = int((cls == ob.PARTIAL).sum())
        assert in_partial >= n_part and in_partial < n_part * P * 128 or n_part == 0


# -------------------------------------------------------------- workloads

@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_workload_doc_lengths(name):
    w = wl.WORKLOADS[name]
    lens = wl.doc_lengths(w)
    assert len(lens) == w.batch
    for ls in lens:
        assert sum(ls) == w.seq_len
        if w.doc_dist != "single":
            assert all(1 <= n <= w.doc_hi for n in ls)
            assert all(n >= w.doc_lo for n in ls[:-1])
    cu = wl.cu_doc_lens(w)
    assert ocp.docs_valid(cu, w.batch, w.seq_len)
    assert (wl.cu_doc_lens(w) == cu).all()  # deterministic
    assert w.seq_len % (2 * w.cp_size) == 0


def test_workload_tensors_deterministic():
    w = wl.WORKLOADS["tiny"]
    a, b = wl.tensors(w), wl.tensors(w)
    for key in a:
        assert a[key].dtype == torch.bfloat16
        assert torch.equal(a[key], b[key])
    assert a["q"].shape == (1, 256, 4, 64) and a["k"].shape == (1, 256, 1, 64)
