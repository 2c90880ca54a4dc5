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


def test_copies_are_independent_problems():
    w = wl.WORKLOADS["8b"]
    seeds = {bench.copy_workload(w, c).seed for c in range(8)}
    assert len(seeds) == 8
    assert bench.copy_workload(w, 0) == w
    a = wl.cu_doc_lens(bench.copy_workload(w, 1))
    assert not np.array_equal(a, wl.cu_doc_lens(w))


def test_units_split_the_emulated_ranks_then_add_copies():
    # N <= R: the emulated ranks of one workload, rank r to process r mod N
    shares, copies = bench.assign_units(4, (0, 1, 2, 3))
    assert copies == 1 and shares == [[(0, 0)], [(0, 1)], [(0, 2)], [(0, 3)]]
    assert bench.scaling_kind(4, copies) == "strong"
    shares, copies = bench.assign_units(3, (0, 7, 15))
    assert copies == 1 and shares == [[(0, 0)], [(0, 7)], [(0, 15)]]
    shares, copies = bench.assign_units(2, (0, 1, 2, 3))
    assert copies == 1 and shares == [[(0, 0), (0, 2)], [(0, 1), (0, 3)]]
    # one emulated rank: every process gets its own copy (weak scaling)
    shares, copies = bench.assign_units(8, (0,))
    assert copies == 8 and shares == [[(c, 0)] for c in range(8)]
    assert bench.scaling_kind(8, copies) == "weak"
    assert bench.scaling_kind(1, 1) == "weak"
    # every unit of the job is run exactly once
    for world, ranks in [(3, (0, 1)), (5, (0, 7, 15)), (8, (0, 1, 2, 3))]:
        shares, copies = bench.assign_units(world, ranks)
        units = sorted(u for sh in shares for u in sh)
        assert units == sorted((c, r) for c in range(copies) for r in ranks)
        assert max(map(len, shares)) - min(map(len, shares)) <= 1


def test_algorithmic_bytes_per_launch():
    w = wl.WORKLOADS["8b"]
    q = 2 * 8192 * 32 * 128 * 2          # bf16 q (or dO, dQ)
    kv = 2 * 8192 * 8 * 128 * 2          # bf16 k (or v)
    st = 2 * 32 * 8192 * 4               # fp32 LSE (or Delta)
    # dK/dV: q, dO, k, v, LSE, Delta in; dK, dV fp32 out: about 473 MB
    assert bench.algorithmic_bytes(w, "dkdv") == 2 * q + 2 * kv + 2 * st + 4 * kv
    assert 472e6 < bench.algorithmic_bytes(w, "dkdv") < 474e6
    # dQ with Delta: q, dO, k, v, LSE, O (fp32) in; dQ, Delta out
    assert bench.algorithmic_bytes(w, "dq") == 5 * q + 2 * kv + 2 * st
    assert bench.algorithmic_bytes(w, "fwd") == q + 2 * kv + 2 * q + st


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


def _split_worker(rank, world, port, out):
    """One process of a two-process run of the tiny workload: it takes the
    emulated CP ranks bench.assign_units gives it, computes their outputs
    (the oracle stands in for the kernels on CPU), and all processes gather
    every rank's outputs."""
    import torch.distributed as dist
    from oracle import attention as oa
    from oracle import cp as ocp
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = wl.WORKLOADS["tiny"]
    shares, copies = bench.assign_units(world, w.ranks)
    cu = wl.cu_doc_lens(w)
    inp = wl.tensors(w)
    mine = {}
    for c, r in shares[rank]:
        assert c == 0
        res = oa.attention(ocp.gather_local(inp["q"], w.seq_len, w.cp_size, r), inp["k"],
                           inp["v"], cu, w.cp_size, r,
                           do_local=ocp.gather_local(inp["do"], w.seq_len, w.cp_size, r))
        mine[r] = res
    gathered = [None] * world
    dist.all_gather_object(gathered, mine)
    if rank == 0:
        out["ranks"] = [sorted(part) for part in gathered]
        allr = {r: v for part in gathered for r, v in part.items()}
        out["o"] = ocp.assemble_full({r: allr[r]["o"] for r in allr}, w.seq_len, w.cp_size)
        out["dq"] = ocp.assemble_full({r: allr[r]["dq"] for r in allr}, w.seq_len, w.cp_size)
        out["dk"] = sum(allr[r]["dk"] for r in allr)
        out["dv"] = sum(allr[r]["dv"] for r in allr)
    dist.destroy_process_group()


def test_two_processes_split_the_emulated_ranks_and_reassemble():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_split_worker, args=(r, world, port, out))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    # rank r of the workload ran on process r
    assert out["ranks"] == [[0], [1]]
    # the processes' outputs, put back in sequence order, are the whole
    # sequence's attention (CP = 1), and the partial dK / dV sum to the full
    from oracle import attention as oa
    w = wl.WORKLOADS["tiny"]
    inp = wl.tensors(w)
    full = oa.attention(inp["q"], inp["k"], inp["v"], wl.cu_doc_lens(w), 1, 0,
                        do_local=inp["do"])
    for key in ("o", "dq", "dk", "dv"):
        assert np.allclose(out[key], full[key], rtol=1e-12, atol=1e-12), key


def test_kernels_per_step_follow_the_planner():
    # four planner kernels, V to fp16 + forward, dQ with Delta + dK/dV (cut
    # dK/dV lists are summed inside the dK/dV kernel)
    for name in ["tiny", "8b", "70b", "sparse", "405b-1doc", "405b-logu"]:
        assert bench.kernels_per_rank_step(wl.WORKLOADS[name]) == 8
    # launch orders over 2048 units take one extra ranking kernel each, and
    # over 2048 key tiles one more for the uncut dK/dV work list: the 128K
    # single-rank workload has 16384 query tiles of 8 positions (and 1024 key
    # tiles)
    assert bench.kernels_per_rank_step(wl.WORKLOADS["causal-128k"]) == 9
    rows = wl.custom("rows", 32768, 1, 1, 16, 1, 64, "uniform", 64, 4096, seed=14)
    both = wl.custom("both", 16384, 1, 17, 2, 2, 64, "uniform", 64, 4096, seed=15)
    assert bench.kernels_per_rank_step(rows) == 9
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
