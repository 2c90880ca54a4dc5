"""The chunk-order copies of the context-parallel exchange on the GPU,
bit-exact against the oracle's CP re-assembly: rank-major all-gather layout
-> natural order (dma_cp_unpermute) and back (dma_cp_permute), for bf16 K/V
rows and fp32 gradient rows, on the tiny, 70B, sparse and 405B shapes; and
the exchange module end to end on a one-process NCCL group."""
import os
import socket

import numpy as np
import pytest
import torch

from document_masked_gqa_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "70b", "sparse", "405b-logu"])
def test_chunk_order_copies_bit_exact(name):
    import document_masked_gqa_gb300 as dma
    from oracle import cp as ocp
    w = wl.WORKLOADS[name]
    g = torch.Generator().manual_seed(5)
    for dtype, heads in ((torch.bfloat16, w.n_kv_heads), (torch.float32, 2)):
        full = torch.randn(w.batch, w.seq_len, heads, 16, generator=g).to(dtype)
        # every rank's rows, stacked rank-major, as an all-gather leaves them
        gathered = torch.stack([ocp.gather_local(full, w.seq_len, w.cp_size, r)
                                for r in range(w.cp_size)]).contiguous()
        back = dma.dma_cp_unpermute(gathered.cuda())
        fwd = dma.dma_cp_permute(full.cuda(), w.cp_size)
        torch.cuda.synchronize()
        assert torch.equal(back.cpu(), full), (name, dtype)
        assert torch.equal(fwd.cpu(), gathered), (name, dtype)
    # the oracle's inverse agrees with the pages' pairing on the raw words
    raw = gathered.view(torch.int32) if gathered.dtype == torch.float32 else gathered
    re = ocp.assemble_full({r: raw[r].numpy() for r in range(w.cp_size)}, w.seq_len, w.cp_size)
    assert np.array_equal(re, full.view(torch.int32).numpy())


def test_exchange_module_on_one_process_group():
    import torch.distributed as dist

    from document_masked_gqa_gb300 import cp_exchange as cx
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("nccl", rank=0, world_size=1)
    try:
        k = torch.randn(1, 256, 1, 64, device="cuda").to(torch.bfloat16)
        v = torch.randn_like(k)
        k2, v2 = cx.gather_kv(k, v)  # CP = 1: the rank's rows are the sequence
        dk = torch.randn(1, 256, 1, 64, device="cuda")
        dv = torch.randn_like(dk)
        dk2, dv2 = cx.reduce_scatter_kv_grads(dk, dv)
        torch.cuda.synchronize()
        assert torch.equal(k2, k) and torch.equal(v2, v)
        assert torch.equal(dk2, dk) and torch.equal(dv2, dv)
    finally:
        dist.destroy_process_group()
