"""The context-parallel exchange (document_masked_gqa_gb300.cp_exchange) as
two gloo processes on CPU: the all-gather of the ranks' K/V rows gives the
whole sequence's K/V in natural order, and the fp32 reduce-scatter of the
ranks' partial dK/dV gives each rank the full gradient of its own rows,
against the oracle's CP re-assembly (tiny and 70B shapes).  The chunk
reorder is the oracle's here (the library's copy kernels are checked
bit-exact against it on the GPU)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from document_masked_gqa_gb300 import workloads as wl


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _oracle_unpermute(w):
    from oracle import cp as ocp

    def f(gathered):  # [CP, B, 2C, ...] -> [B, S, ...], moved as raw 16-bit words
        raw = gathered.view(torch.int16)
        full = ocp.assemble_full({r: raw[r].numpy() for r in range(raw.shape[0])}, w.seq_len,
                                 w.cp_size)
        return torch.from_numpy(np.ascontiguousarray(full)).view(gathered.dtype)
    return f


def _oracle_permute(w):
    from oracle import cp as ocp

    def f(full, cp):  # [B, S, ...] -> [CP, B, 2C, ...]
        return torch.stack([ocp.gather_local(full, w.seq_len, cp, r) for r in range(cp)])
    return f


def _worker(rank, world, port, name, out):
    import torch.distributed as dist
    from document_masked_gqa_gb300 import cp_exchange as cx
    from oracle import attention as oa
    from oracle import cp as ocp
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = wl.WORKLOADS[name]
    assert w.cp_size == world
    cu = wl.cu_doc_lens(w)
    inp = wl.tensors(w)
    # the rank holds its own rows of K and V ...
    k_loc = ocp.gather_local(inp["k"], w.seq_len, w.cp_size, rank)
    v_loc = ocp.gather_local(inp["v"], w.seq_len, w.cp_size, rank)
    k, v = cx.gather_kv(k_loc, v_loc, reorder=_oracle_unpermute(w))
    out[f"k_equal_{rank}"] = bool(torch.equal(k, inp["k"]) and torch.equal(v, inp["v"]))
    # the asynchronous form gives the same
    work, finish = cx.gather_kv(k_loc, v_loc, async_op=True, reorder=_oracle_unpermute(w))
    k2, v2 = finish()
    out[f"k_async_equal_{rank}"] = bool(torch.equal(k2, k) and torch.equal(v2, v))
    # ... and its queries' partial dK, dV, reduce-scattered in fp32
    res = oa.attention(ocp.gather_local(inp["q"], w.seq_len, w.cp_size, rank), k, v, cu,
                       w.cp_size, rank,
                       do_local=ocp.gather_local(inp["do"], w.seq_len, w.cp_size, rank),
                       threads=4)
    dk_p = torch.from_numpy(res["dk"]).float()
    dv_p = torch.from_numpy(res["dv"]).float()
    dk_mine, dv_mine = cx.reduce_scatter_kv_grads(dk_p, dv_p, reorder=_oracle_permute(w))
    out[f"dk_{rank}"] = dk_mine.double().numpy()
    out[f"dv_{rank}"] = dv_mine.double().numpy()
    dist.destroy_process_group()


@pytest.mark.parametrize("name", ["tiny", "70b"])
def test_gather_and_reduce_scatter_match_cp_reassembly(name):
    from oracle import attention as oa
    from oracle import cp as ocp
    w = wl.WORKLOADS[name]
    world = w.cp_size
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, name, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=600)
        assert p.exitcode == 0
    for r in range(world):
        assert out[f"k_equal_{r}"] and out[f"k_async_equal_{r}"], r
    # the whole sequence's gradients (CP = 1), cut into each rank's rows
    inp = wl.tensors(w)
    full = oa.attention(inp["q"], inp["k"], inp["v"], wl.cu_doc_lens(w), 1, 0,
                        do_local=inp["do"], threads=4)
    for r in range(world):
        for key in ("dk", "dv"):
            want = ocp.gather_local(full[key], w.seq_len, w.cp_size, r)
            got = out[f"{key}_{r}"]
            assert got.shape == want.shape
            # two fp32 partials summed in fp32 against the float64 whole
            err = np.abs(got - want).max() / max(np.abs(want).max(), 1e-30)
            assert err <= 1e-5, (name, r, key, err)
