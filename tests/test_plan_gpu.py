"""Planner and block-mask builder on the GPU, bit-exact against the oracle:
query positions, document starts, chunk order, tile classes, row and column
lists (with the partial bit), launch orders (validity), the CP gather /
scatter copies, malformed document tables and the bounded-wait probe."""
import numpy as np
import pytest
import torch

from document_masked_gqa_gb300 import workloads as wl
from oracle import blockmask as ob
from oracle import cp as ocp

pytestmark = pytest.mark.gpu

EDGE = {
    "docs-of-one": wl.custom("docs-of-one", 512, 2, 1, 4, 1, 64, "fixed",
                             fixed_docs=[[1] * 512]),
    "cp1-single-g1": wl.custom("cp1-single-g1", 512, 1, 2, 2, 2, 128, "fixed",
                               fixed_docs=[[512], [512]]),
    "g2-d64": wl.custom("g2-d64", 1024, 2, 2, 4, 2, 64, "uniform", 1, 300, seed=11),
    "g16-d64": wl.custom("g16-d64", 2048, 4, 1, 16, 1, 64, "uniform", 5, 700, seed=12),
    "g8-hkv2": wl.custom("g8-hkv2", 1024, 2, 1, 16, 2, 128, "loguniform", 16, 1024, seed=13),
}


# plan-only cases whose launch orders have more than 2048 units (rows: 4096
# query tiles of 8 positions; rows and columns: 17 samples x 128 tiles), which
# the planner orders with its separate ranking kernel
LONG_ORDERS = {
    "long-row-order": wl.custom("long-row-order", 32768, 1, 1, 16, 1, 64, "uniform", 64, 4096,
                                seed=14),
    "long-col-order": wl.custom("long-col-order", 16384, 1, 17, 2, 2, 64, "uniform", 64, 4096,
                                seed=15),
}


def _cases():
    out = []
    for name in ["tiny", "8b", "70b", "sparse", "405b-logu", "405b-1doc"]:
        w = wl.WORKLOADS[name]
        for r in w.ranks:
            out.append((name, w, r))
    for name, w in list(EDGE.items()) + list(LONG_ORDERS.items()):
        for r in w.ranks:
            out.append((name, w, r))
    return out


def _plan(w, rank, cu):
    import document_masked_gqa_gb300 as dma
    cu_d = torch.from_numpy(np.asarray(cu, dtype=np.int32)).cuda()
    plan = dma.dma_plan(cu_d, w.batch, w.seq_len, w.cp_size, rank, w.n_heads,
                        w.n_kv_heads, w.head_dim)
    return plan, dma.plan_arrays(plan)


def _check_order(order, lengths):
    order = np.asarray(order)
    assert sorted(order.tolist()) == list(range(len(lengths)))
    c = np.asarray(lengths)[order]
    assert (np.diff(c) <= 0).all()
    # ties broken by ascending index
    for a, b in zip(order[:-1], order[1:]):
        if lengths[a] == lengths[b]:
            assert a < b


@pytest.mark.parametrize("name,w,rank", _cases(), ids=lambda x: str(x) if not hasattr(x, "name") else "")
def test_plan_bit_exact(name, w, rank):
    cu = wl.cu_doc_lens(w)
    plan, a = _plan(w, rank, cu)
    assert int(a["status"][0]) == 0
    qpos = ocp.local_positions(w.seq_len, w.cp_size, rank)
    assert np.array_equal(a["qpos"].numpy(), qpos)
    start = ocp.doc_start(cu, w.batch, w.seq_len)
    assert np.array_equal(a["doc_lo"].numpy(), start[:, qpos])
    assert a["chunk_order"].tolist() == ocp.chunk_order(w.cp_size)
    cls = ob.tile_classes(cu, w.batch, w.seq_len, w.cp_size, rank, w.group)
    assert np.array_equal(a["tile_class"].numpy(), cls)
    rows = ob.row_lists(cls)
    rp = a["row_ptr"].numpy()
    ri = a["row_idx"].numpy().view(np.uint32)
    flat_cls = cls.reshape(len(rows), -1)
    for i, lst in enumerate(rows):
        got = ri[rp[i]:rp[i + 1]]
        assert np.array_equal(got & 0x7FFFFFFF, lst)
        assert np.array_equal((got >> 31) == 1, flat_cls[i, lst] == ob.PARTIAL)
    cols = ob.col_lists(cls)
    cp_ = a["col_ptr"].numpy()
    ci = a["col_idx"].numpy().view(np.uint32)
    B, nqt, nkt = cls.shape
    for j, lst in enumerate(cols):
        b, kt = divmod(j, nkt)
        got = ci[cp_[j]:cp_[j + 1]]
        assert np.array_equal(got & 0x7FFFFFFF, lst)
        assert np.array_equal((got >> 31) == 1, cls[b, lst, kt] == ob.PARTIAL)
    _check_order(a["fwd_order"].numpy(), [len(x) for x in rows])
    _check_order(a["bwd_order"].numpy(), [len(x) for x in cols])
    _check_kv_work_list(a, [len(x) for x in cols], w)


def _check_kv_work_list(a, lengths, w):
    """The dK/dV work list: every unit's column list covered exactly once by
    its slices, and the slices, cuts and pool slots equal to the host mirror
    of the planner's rule (balance.kv_work_list) for this device's SMs."""
    from document_masked_gqa_gb300 import balance
    cp_ = a["col_ptr"].numpy()
    sl = a["kv_slices"].numpy()
    sp = a["kv_splits"].numpy()
    covered = {}
    for unit, first, n, seg, split, slot, z0, z1 in sl:
        assert z0 == 0 and z1 == 0
        covered.setdefault(int(unit), []).append((int(first) - int(cp_[unit]), int(n)))
    assert sorted(covered) == list(range(len(lengths)))
    for unit, parts in covered.items():
        parts.sort()
        pos = 0
        for first, n in parts:
            assert first == pos
            pos += n
        assert pos == lengths[unit]
    nqt = a["tile_class"].shape[1]
    assert a["kv_pool_slots"] == balance.kv_pool_slots(w.batch, w.seq_len, w.n_kv_heads, nqt)
    want = balance.kv_work_list(lengths, w.n_kv_heads, a["n_sms"], a["kv_pool_slots"])
    got = [(int(u), int(f) - int(cp_[u]), int(n), int(sg), int(spl), int(slot))
           for u, f, n, sg, spl, slot, _, _ in sl]
    assert got == want["slices"]
    assert [tuple(int(x) for x in row[:3]) for row in sp] == want["splits"]
    assert all(row[3] == 0 for row in sp)


@pytest.mark.parametrize("name", ["tiny", "70b", "sparse"])
def test_cp_gather_scatter_bit_exact(name):
    import document_masked_gqa_gb300 as dma
    w = wl.WORKLOADS[name]
    cu = wl.cu_doc_lens(w)
    x = wl.tensors(w, with_grad=False)["q"]
    for r in w.ranks:
        plan, _ = _plan(w, r, cu)
        loc = dma.dma_cp_gather(plan, x.cuda())
        want = ocp.gather_local(x.view(torch.int16).numpy(), w.seq_len, w.cp_size, r)
        assert np.array_equal(loc.cpu().view(torch.int16).numpy(), want)
        back = torch.zeros_like(x).cuda()
        dma.dma_cp_scatter(plan, loc, back)
        pos = ocp.local_positions(w.seq_len, w.cp_size, r)
        assert torch.equal(back.cpu()[:, pos], x[:, pos])


@pytest.mark.parametrize("cu", [[1, 100, 256], [0, 100, 100, 256], [0, 100, 255],
                                [0, 200, 300, 512]])
def test_bad_docs_reported(cu):
    import document_masked_gqa_gb300 as dma
    batch = 2 if cu[-1] == 512 else 1
    w = wl.custom("bad", 256, 2, batch, 4, 1, 64, "fixed", fixed_docs=[[256]] * batch)
    plan, _ = _plan(w, 0, cu)
    assert dma.dma_plan_check(plan) == dma.DMA_ERR_BAD_DOCS
    # kernels on a failed plan do nothing and return
    q = torch.zeros(batch, 128, 4, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(batch, 256, 1, 64, dtype=torch.bfloat16, device="cuda")
    o, lse = dma.dma_attn_fwd(plan, q, k, k)
    torch.cuda.synchronize()
    assert dma.dma_plan_check(plan) == dma.DMA_ERR_BAD_DOCS


def test_empty_batch_is_a_no_op():
    import document_masked_gqa_gb300 as dma
    plan = dma.dma_plan(None, 0, 256, 2, 1, 4, 1, 64)
    q = torch.zeros(0, 128, 4, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(0, 256, 1, 64, dtype=torch.bfloat16, device="cuda")
    o, lse = dma.dma_attn_fwd(plan, q, k, k)
    assert o.numel() == 0 and dma.dma_plan_check(plan) == 0


def test_bounded_wait_probe_reports_timeout():
    import document_masked_gqa_gb300 as dma
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert dma.dma_debug_wait_probe(2_000_000, st) == dma.DMA_ERR_TIMEOUT
    # the context is still usable afterwards
    x = torch.ones(1024, device="cuda")
    assert float(x.sum()) == 1024.0
