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


def test_kernels_per_step_follow_the_planner():
    # four planner kernels, V to fp16 + forward, Delta + dK/dV + dQ
    for name in ["tiny", "8b", "70b", "sparse", "405b-1doc"]:
        assert bench.kernels_per_rank_step(wl.WORKLOADS[name]) == 9
    # launch orders over 2048 units take one extra ranking kernel each: the
    # 128K single-rank workload has 16384 query tiles of 8 positions
    assert bench.kernels_per_rank_step(wl.WORKLOADS["causal-128k"]) == 10
    rows = wl.custom("rows", 32768, 1, 1, 16, 1, 64, "uniform", 64, 4096, seed=14)
    both = wl.custom("both", 16384, 1, 17, 2, 2, 64, "uniform", 64, 4096, seed=15)
    assert bench.kernels_per_rank_step(rows) == 10
    assert bench.kernels_per_rank_step(both) == 11


def test_source_hash_ignores_comments():
    a = "int f(int x) {  // one\n  return x + 1; /* two\n three */ }\n"
    b = "int f(int x) {\n\n  return x + 1;   }"
    c = "int f(int x) { return x + 2; }"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)


def test_hbm_byte_counts():
    w = wl.WORKLOADS["8b"]
    # O fp32 + dO bf16 in, Delta fp32 out: 2 x 8192 rows x 32 heads x (6*128 + 4)
    assert bench.delta_bytes(w) == 2 * 8192 * 32 * 772
    # a one-sample toy by hand: S = 256, CP = 1, Hq = Hkv = 1 (P = 128): 2 query
    # tiles, 2 key tiles; 3 non-skipped pairs; 2 documents
    t = wl.custom("toy", 256, 1, 1, 1, 1, 64, "fixed", fixed_docs=[[100, 156]])
    want = (4 * 3 + 4 * 256 + 4 * 256 + 4 * 256 + 4 * 2 + 4
            + 4 * 5 + 4 * 5 + 4 * 2 * 3 + 4 * 4)
    assert bench.plan_bytes(t, 2, 3) == want


def test_host_description_names_cpu_and_blas():
    d = bench.host_description()
    assert set(d) == {"cpu_model", "blas"}
    assert d["cpu_model"] is None or isinstance(d["cpu_model"], str)
