"""The C-ABI library loads (no GPU needed) and exports every entry point the
header declares; host-side argument checks answer without touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dma.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dma_[a-z_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from document_masked_gqa_gb300 import build as b
    b.build()
    import document_masked_gqa_gb300 as dma
    return dma.lib()


def test_header_declares_the_boundary():
    names = _declared()
    for must in ("dma_plan", "dma_attn_fwd", "dma_attn_bwd", "dma_plan_workspace_bytes",
                 "dma_plan_check", "dma_plan_destroy", "dma_status_str"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    import document_masked_gqa_gb300._lib as L
    assert sorted(L.EXPORTED) == _declared()


def test_status_strings(lib):
    import document_masked_gqa_gb300 as dma
    for s in range(8):
        assert dma.status_str(s) and dma.status_str(s) != "unknown status"
    assert dma.status_str(99) == "unknown status"


def test_workspace_bytes_and_shape_rules(lib):
    import document_masked_gqa_gb300 as dma
    assert dma.dma_plan_workspace_bytes(2, 8192, 1, 32, 8, 128) > 0
    assert dma.dma_plan_workspace_bytes(1, 131072, 16, 16, 1, 128) > 0
    assert dma.dma_plan_workspace_bytes(0, 256, 2, 4, 1, 64) > 0
    assert dma.dma_plan_workspace_bytes(1, 256, 2, 4, 1, 96) == 0      # head_dim
    assert dma.dma_plan_workspace_bytes(1, 256, 2, 12, 1, 64) == 0     # g = 12
    assert dma.dma_plan_workspace_bytes(1, 250, 2, 4, 1, 64) == 0      # S % 2CP
    assert dma.dma_plan_workspace_bytes(1, 192, 2, 4, 1, 64) == 0      # C % 64
    assert dma.dma_plan_workspace_bytes(1, 256, 2, 2, 2, 64) == 0      # C % (128/g)
    assert dma.dma_plan_workspace_bytes(1, 256, 0, 4, 1, 64) == 0      # cp_size


def test_plan_rejects_bad_arguments_on_the_host(lib):
    h = ctypes.c_void_p()
    ws = (ctypes.c_ubyte * 4096)()
    # rank out of range
    st = lib.dma_plan(None, 1, 1, 256, 2, 2, 4, 1, 64, 0.0, ctypes.cast(ws, ctypes.c_void_p),
                      4096, None, ctypes.byref(h))
    assert st == 1 and not h.value
    # unsupported head_dim
    st = lib.dma_plan(None, 1, 1, 256, 2, 0, 4, 1, 96, 0.0, ctypes.cast(ws, ctypes.c_void_p),
                      4096, None, ctypes.byref(h))
    assert st == 3
    # missing output handle / workspace
    assert lib.dma_plan(None, 1, 1, 256, 2, 0, 4, 1, 64, 0.0, None, 0, None, None) == 1
    assert lib.dma_plan(None, 1, 1, 256, 2, 0, 4, 1, 64, 0.0, None, 0, None,
                        ctypes.byref(h)) == 1
    # non-finite scale
    st = lib.dma_plan(None, 1, 1, 256, 2, 0, 4, 1, 64, float("nan"),
                      ctypes.cast(ws, ctypes.c_void_p), 4096, None, ctypes.byref(h))
    assert st == 1
    # calls on a null plan
    assert lib.dma_attn_fwd(None, None, None, None, None, None, None) == 1
    assert lib.dma_attn_bwd(None, *([None] * 10)) == 1
    assert lib.dma_plan_destroy(None) == 0


class _ShapeOnlyPlan:
    """Stands in for a plan: the binding checks tensors against plan.shape
    before it makes any library call."""
    handle = None
    shape = (1, 256, 2, 0, 4, 1, 64)  # batch, seq_len, cp_size, cp_rank, Hq, Hkv, D


def test_binding_checks_tensors_before_any_call():
    import torch
    import document_masked_gqa_gb300 as dma
    plan = _ShapeOnlyPlan()
    q = torch.zeros(1, 128, 4, 64, dtype=torch.bfloat16)        # right shape, but on the host
    kv = torch.zeros(1, 256, 1, 64, dtype=torch.bfloat16)
    o = torch.zeros(1, 128, 4, 64)
    lse = torch.zeros(1, 4, 128)
    dkv = torch.zeros(1, 256, 1, 64)
    calls = [
        lambda: dma.dma_attn_fwd(plan, q, kv, kv, o, lse),
        lambda: dma.dma_attn_bwd(plan, q, kv, kv, o, lse, q, q, dkv, dkv),
        lambda: dma.dma_attn_bwd_delta(plan, o, q),
        lambda: dma.dma_attn_bwd_dkdv(plan, q, kv, kv, lse, q, dkv, dkv),
        lambda: dma.dma_attn_bwd_dq(plan, q, kv, kv, lse, q, q),
        lambda: dma.dma_cp_gather(plan, kv, q),
        lambda: dma.dma_cp_scatter(plan, q, kv),
        lambda: dma.dma_plan(torch.zeros(2, dtype=torch.int32), 1, 256, 2, 0, 4, 1, 64,
                             workspace=torch.zeros(1 << 16, dtype=torch.uint8)),
    ]
    for call in calls:
        with pytest.raises(ValueError):
            call()


def test_binding_rejects_wrong_shapes_and_dtypes():
    import torch
    from document_masked_gqa_gb300 import _lib
    with pytest.raises(ValueError):
        _lib._expect(torch.zeros(1, 128, 4, 64), torch.bfloat16, (1, 128, 4, 64), "q")
    with pytest.raises(ValueError):
        _lib._expect(torch.zeros(1, 128, 4, 32, dtype=torch.bfloat16), torch.bfloat16,
                     (1, 128, 4, 64), "q")
    with pytest.raises(ValueError):
        _lib._expect(torch.zeros(1, 64, 128, 4, dtype=torch.bfloat16).transpose(1, 2),
                     torch.bfloat16, (1, 128, 64, 4), "q")
