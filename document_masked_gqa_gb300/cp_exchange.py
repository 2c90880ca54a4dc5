"""The exchange steps around the attention of one context-parallel rank.

"The Llama 3 Herd of Models - part 3/16", 3.3.2 ("Context parallelism for
long sequences"): the sequence is cut into 2*CP chunks, rank r holds chunks
r and 2*CP-1-r, and K and V are all-gathered before the attention of the
rank's queries against the whole sequence; "Numerical stability": gradients
are accumulated and reduce-scattered in FP32.  The review of "Scaling Llama
3 Training with Efficient Parallelism Strategies" ("Context Parallelism
(CP)", implementation details) describes the same all-gather design.

Host orchestration over ``torch.distributed`` (NCCL between GPUs), with the
reordering done by the library's chunk-order copy kernels:

* ``gather_kv``: every rank contributes its local K and V rows ([B, 2C, H,
  D] in the plan's local order); an all-gather lands them rank-major
  ([CP, B, 2C, H, D]) and ``dma_cp_unpermute`` puts them in natural order
  ([B, S, H, D]), the layout ``dma_attn_fwd`` / ``dma_attn_bwd`` read.
* ``reduce_scatter_kv_grads``: every rank's partial dK, dV (fp32 [B, S, H,
  D], its own queries' contribution, as ``dma_attn_bwd`` returns them) are
  reordered rank-major by ``dma_cp_permute`` and reduce-scattered (sum, in
  fp32): each rank receives the full gradient of its own K and V rows,
  [B, 2C, H, D] in local order.

``async_op=True`` returns the collective's work handle with a function that
finishes the reorder once it has completed, so that a caller can run other
work (the previous layer, another micro-batch) while the collective is in
flight.  Not built here: starting the attention on the rank's local K/V
tiles before the gather completes, which needs the kernels to take the
remote tiles in a second pass.

``reorder`` exists for tests that run the collectives on CPU tensors (gloo):
the library's kernels take device memory only, and this module has no CPU
path of its own.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import _lib


def _unpermute_default(gathered):
    if not gathered.is_cuda:
        raise ValueError("gather_kv: CPU tensors need an explicit `reorder` "
                         "(the chunk-order kernels take device memory)")
    return _lib.dma_cp_unpermute(gathered)


def _permute_default(full, cp_size):
    if not full.is_cuda:
        raise ValueError("reduce_scatter_kv_grads: CPU tensors need an explicit `reorder` "
                         "(the chunk-order kernels take device memory)")
    return _lib.dma_cp_permute(full, cp_size)


def gather_kv(k_local, v_local, group=None, async_op: bool = False, reorder=None):
    """All-gather the ranks' local K and V rows and return them in natural
    sequence order, [B, S, H, D] each (S = CP * 2C).

    reorder: callable [CP, B, 2C, H, D] -> [B, S, H, D]; default: the
    library's dma_cp_unpermute (device tensors).  With async_op, returns
    (work, finish) where finish() waits for the collective and returns
    (k, v)."""
    cp = dist.get_world_size(group)
    unperm = reorder or _unpermute_default
    both = torch.stack([k_local, v_local])  # one collective for K and V: [2, B, 2C, H, D]
    # ranks' blocks concatenated along the first dimension: [CP * 2, B, 2C, H, D]
    out = torch.empty((cp * 2,) + tuple(both.shape[1:]), dtype=both.dtype, device=both.device)
    work = dist.all_gather_into_tensor(out, both, group=group, async_op=async_op)

    def finish():
        if work is not None and async_op:
            work.wait()
        per_rank = out.view((cp, 2) + tuple(both.shape[1:]))
        return unperm(per_rank[:, 0].contiguous()), unperm(per_rank[:, 1].contiguous())

    if async_op:
        return work, finish
    return finish()


def reduce_scatter_kv_grads(dk_partial, dv_partial, group=None, async_op: bool = False,
                            reorder=None):
    """Sum every rank's partial dK and dV (fp32, [B, S, H, D]) and give each
    rank the rows it holds, [B, 2C, H, D] in local order.

    reorder: callable ([B, S, H, D], cp) -> [CP, B, 2C, H, D]; default: the
    library's dma_cp_permute (device tensors).  With async_op, returns
    (work, finish) where finish() waits and returns (dk, dv)."""
    cp = dist.get_world_size(group)
    perm = reorder or _permute_default
    if dk_partial.dtype != torch.float32 or dv_partial.dtype != torch.float32:
        raise ValueError("reduce_scatter_kv_grads: the partial gradients are fp32")
    # block r (rows 2r, 2r + 1 of the first dimension) is rank r's dK and dV rows
    src = torch.stack([perm(dk_partial, cp), perm(dv_partial, cp)], dim=1)  # [CP, 2, B, 2C, H, D]
    src = src.reshape((cp * 2,) + tuple(src.shape[2:]))
    out = torch.empty((2,) + tuple(src.shape[1:]), dtype=src.dtype, device=src.device)
    work = dist.reduce_scatter_tensor(out, src, op=dist.ReduceOp.SUM, group=group,
                                      async_op=async_op)

    def finish():
        if work is not None and async_op:
            work.wait()
        return out[0], out[1]

    if async_op:
        return work, finish
    return finish()
