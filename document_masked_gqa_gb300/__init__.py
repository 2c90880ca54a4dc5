"""Causal + document-masked GQA attention for one context-parallel rank on
GB300 (sm_103a): a C-ABI CUDA library (``libdma.so``, ``include/dma.h``) and
this thin ctypes binding with the same entry-point names.

The shared library is loaded on first use; if it is missing the call raises
ImportError (build with ``document_masked_gqa_gb300/build.py``).
"""
from ._lib import (  # noqa: F401
    DMA_ERR_BAD_DOCS, DMA_ERR_CUDA, DMA_ERR_INVALID_ARG, DMA_ERR_TIMEOUT,
    DMA_ERR_UNSUPPORTED, DMA_ERR_WORKSPACE, DMA_OK, DMA_WARN_V_SATURATED, TILE_FULL, TILE_PARTIAL,
    TILE_SKIP, DmaError, Plan, dma_attn_bwd, dma_attn_bwd_delta, dma_attn_bwd_dkdv,
    dma_attn_bwd_dq, dma_attn_bwd_dq_delta, dma_attn_fwd, dma_cp_gather,
    dma_cp_permute, dma_cp_scatter, dma_cp_unpermute, dma_debug_wait_probe, dma_plan, dma_plan_check,
    dma_plan_set_wait_timeout, dma_plan_workspace_bytes, lib, plan_arrays,
    status_str,
)
