"""Host-side logic of bench.py, on CPU: the FLOP convention's pair count
against the oracle's, and the multi-process path (weak scaling, max over
ranks) as two gloo ranks."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import bench
from document_masked_gqa_gb300 import workloads as wl
from oracle import flops as ofl


@pytest.mark.parametrize("name", ["tiny", "8b", "70b", "sparse", "405b-logu", "405b-1doc"])
def test_pair_count_matches_oracle(name):
    w = wl.WORKLOADS[name]
    cu = wl.cu_doc_lens(w)
    for r in w.ranks:
        got = bench.pairs_per_sample(cu, w.batch, w.seq_len, w.cp_size, r)
        want = ofl.pairs_per_head(cu, w.batch, w.seq_len, w.cp_size, r)
        assert np.array_equal(got, want)
    fl = bench.flops_of(w, cu, w.ranks)
    tot = sum(int(ofl.pairs_per_head(cu, w.batch, w.seq_len, w.cp_size, r).sum()) for r in w.ranks)
    assert fl == ofl.counted_flops(tot, w.n_heads, w.head_dim)


def test_rank_workloads_are_independent_problems():
    w = wl.WORKLOADS["8b"]
    seeds = {bench.rank_workload(w, r).seed for r in range(8)}
    assert len(seeds) == 8
    assert bench.rank_workload(w, 0) == w
    a = wl.cu_doc_lens(bench.rank_workload(w, 1))
    assert not np.array_equal(a, wl.cu_doc_lens(w))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, wsz, local = bench.dist_info()
    assert (r, wsz, local) == (rank, world, rank)
    bench.barrier(world)
    ms = bench.reduce_max(1.0 + rank * 2.5, world)
    out[rank] = ms
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_step_time():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] == out[1] == 3.5
