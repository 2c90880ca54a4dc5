"""Shared test plumbing: run one emulated CP rank through the C ABI, and the
oracle on the same seeded inputs."""
import numpy as np
import torch

from document_masked_gqa_gb300 import workloads as wl

# Parity tolerances for bf16 inputs with fp32 accumulation: O max-abs, LSE max-abs, gradients
# relative Frobenius per tensor per rank.
TOL_O = 1e-2
TOL_LSE = 1e-3
TOL_GRAD = 2e-2


def gpu_rank(w, rank, inputs, cu, backward=True, scale=0.0):
    """Plan + gather + fwd (+ bwd) for one rank on cuda:0. Returns CPU
    tensors and the plan."""
    import document_masked_gqa_gb300 as dma
    dev = torch.device("cuda:0")
    cu_d = torch.from_numpy(np.asarray(cu, dtype=np.int32)).to(dev)
    plan = dma.dma_plan(cu_d, w.batch, w.seq_len, w.cp_size, rank, w.n_heads,
                        w.n_kv_heads, w.head_dim, softmax_scale=scale)
    q_full = inputs["q"].to(dev)
    q = dma.dma_cp_gather(plan, q_full)
    k = inputs["k"].to(dev)
    v = inputs["v"].to(dev)
    o, lse = dma.dma_attn_fwd(plan, q, k, v)
    out = {"q_local": q, "o": o, "lse": lse}
    if backward:
        do = dma.dma_cp_gather(plan, inputs["do"].to(dev))
        dq, dk, dv = dma.dma_attn_bwd(plan, q, k, v, o, lse, do)
        out.update(dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    st = dma.dma_plan_check(plan)
    assert st == 0, f"plan status {st}: {dma.status_str(st)}"
    return {k_: v_.float().cpu() for k_, v_ in out.items()}, plan


def oracle_rank(w, rank, inputs, cu, backward=True, rows=None, threads=4, scale=None):
    from oracle import attention as oa
    from oracle import cp as ocp
    q_local = ocp.gather_local(inputs["q"], w.seq_len, w.cp_size, rank)
    do_local = None
    if backward:
        do_local = ocp.gather_local(inputs["do"], w.seq_len, w.cp_size, rank)
    return oa.attention(q_local, inputs["k"], inputs["v"], cu, w.cp_size, rank, scale=scale,
                        do_local=do_local, rows=rows, threads=threads)


def max_abs(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b))) if a.size else 0.0


def rel_fro(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / den) if den > 0 else float(np.linalg.norm(a - b))
