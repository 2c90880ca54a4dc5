"""The allocation-free forward (dma_attn_fwd_noalloc), for callers that may
not allocate device memory and so cannot hand the library a plan workspace.

Called straight through the C ABI, twice in a row on the same inputs, and
compared with the workspace-based dma_plan + dma_attn_fwd on the same inputs:
both run the same kernels on the same plan, so the results must be bitwise
equal (the forward's parity tolerances, O and LSE max-abs, are the looser
bound this implies).  A malformed document table must be reported through
status_dev with o and lse left untouched, and the status pointer may be
NULL.  Lives in a file pytest collects last, and also passes run alone in a
fresh process."""
import ctypes

import numpy as np
import pytest
import torch

from document_masked_gqa_gb300 import workloads as wl
from helpers import TOL_LSE, TOL_O

pytestmark = pytest.mark.gpu


def _noalloc(lib, w, rank, cu_d, q, k, v, o, lse, status):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return lib.dma_attn_fwd_noalloc(p(cu_d), cu_d.numel() - 1, w.batch, w.seq_len, w.cp_size,
                                    rank, w.n_heads, w.n_kv_heads, w.head_dim, 0.0, p(q), p(k),
                                    p(v), p(o), p(lse), p(status), stream)


@pytest.mark.parametrize("name", ["tiny", "70b", "8b"])
def test_noalloc_forward_matches_workspace_forward_twice(name):
    import document_masked_gqa_gb300 as dma
    lib = dma.lib()
    w = wl.WORKLOADS[name]
    cu = wl.cu_doc_lens(w)
    inp = wl.tensors(w, with_grad=False)
    cu_d = torch.from_numpy(cu).cuda()
    k = inp["k"].cuda()
    v = inp["v"].cuda()
    for rank in w.ranks:
        plan = dma.dma_plan(cu_d, w.batch, w.seq_len, w.cp_size, rank, w.n_heads, w.n_kv_heads,
                            w.head_dim)
        q = dma.dma_cp_gather(plan, inp["q"].cuda())
        o_ref, lse_ref = dma.dma_attn_fwd(plan, q, k, v)
        torch.cuda.synchronize()
        assert dma.dma_plan_check(plan) == 0
        for _ in range(2):  # the shared scratch keeps the last call's contents
            o = torch.full_like(o_ref, float("nan"))
            lse = torch.full_like(lse_ref, float("nan"))
            status = torch.full((1,), 77, dtype=torch.int32, device="cuda")
            assert _noalloc(lib, w, rank, cu_d, q, k, v, o, lse, status) == 0
            torch.cuda.synchronize()
            assert int(status.item()) == 0
            eo = float((o - o_ref).abs().max())
            el = float((lse - lse_ref).abs().max())
            assert np.isfinite(eo) and eo <= TOL_O, (name, rank, eo)
            assert np.isfinite(el) and el <= TOL_LSE, (name, rank, el)
            assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref), (name, rank)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    import document_masked_gqa_gb300 as dma
    lib = dma.lib()
    # 4 samples of 131072 tokens with 8 K/V heads of 128 need far more than 64 MiB
    w = wl.custom("big", 131072, 1, 4, 64, 8, 128, "single")
    need = dma.dma_plan_workspace_bytes(w.batch, w.seq_len, w.cp_size, w.n_heads, w.n_kv_heads,
                                        w.head_dim)
    assert need > (64 << 20)
    cu_d = torch.tensor([0, 131072, 262144, 393216, 524288], dtype=torch.int32, device="cuda")
    t = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    f = torch.zeros(16, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _noalloc(lib, w, 0, cu_d, t, t, t, f, f, st) == dma.DMA_ERR_WORKSPACE


def test_noalloc_bad_docs_reported_outputs_untouched_then_recovers():
    import document_masked_gqa_gb300 as dma
    lib = dma.lib()
    w = wl.WORKLOADS["tiny"]
    cu = wl.cu_doc_lens(w)
    inp = wl.tensors(w, with_grad=False)
    k = inp["k"].cuda()
    v = inp["v"].cuda()
    rank = 0
    bad = cu.copy()
    bad[2], bad[3] = cu[3], cu[2]  # no longer increasing
    bad_d = torch.from_numpy(bad).cuda()
    cu_d = torch.from_numpy(cu).cuda()
    plan = dma.dma_plan(cu_d, w.batch, w.seq_len, w.cp_size, rank, w.n_heads, w.n_kv_heads,
                        w.head_dim)
    q = dma.dma_cp_gather(plan, inp["q"].cuda())
    o_ref, lse_ref = dma.dma_attn_fwd(plan, q, k, v)
    o = torch.full_like(o_ref, float("nan"))
    lse = torch.full_like(lse_ref, float("nan"))
    status = torch.full((1,), 77, dtype=torch.int32, device="cuda")
    assert _noalloc(lib, w, rank, bad_d, q, k, v, o, lse, status) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == dma.DMA_ERR_BAD_DOCS
    assert torch.isnan(o).all() and torch.isnan(lse).all()
    # the next valid call starts from a clean status, with no status pointer
    assert _noalloc(lib, w, rank, cu_d, q, k, v, o, lse, None) == 0
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
    # and reports OK when asked
    assert _noalloc(lib, w, rank, cu_d, q, k, v, o, lse, status) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
