"""ctypes binding of ``libdma.so`` (include/dma.h).

Argument marshalling only: torch tensors are checked for dtype, shape, device
and contiguity, and their data pointers and the current CUDA stream are
passed to the C entry points of the same names.  Every step of the attention
path runs in the library's kernels.  If the library has not been built, the
import fails loudly; there is no fallback.
"""
from __future__ import annotations

import ctypes
import math
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdma.so")

DMA_OK = 0
DMA_ERR_INVALID_ARG = 1
DMA_ERR_BAD_DOCS = 2
DMA_ERR_UNSUPPORTED = 3
DMA_ERR_CUDA = 4
DMA_ERR_TIMEOUT = 5
DMA_ERR_WORKSPACE = 6
DMA_WARN_V_SATURATED = 7

TILE_SKIP, TILE_FULL, TILE_PARTIAL = 0, 1, 2

EXPORTED = [
    "dma_plan_workspace_bytes", "dma_plan", "dma_attn_fwd", "dma_attn_bwd",
    "dma_plan_check", "dma_plan_destroy", "dma_status_str", "dma_cp_gather",
    "dma_cp_scatter", "dma_plan_get_view", "dma_plan_set_wait_timeout",
    "dma_debug_wait_probe", "dma_attn_bwd_delta", "dma_attn_bwd_dkdv", "dma_attn_bwd_dq",
    "dma_attn_fwd_noalloc", "dma_attn_bwd_dq_delta", "dma_cp_unpermute", "dma_cp_permute",
]


class DmaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_str(status)} ({status})")


class PlanView(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "batch", "seq_len", "cp_size", "cp_rank", "n_heads", "n_kv_heads", "head_dim",
        "chunk", "local_len", "group", "q_tile_positions", "n_qtiles", "n_ktiles")] + [
        ("softmax_scale", ctypes.c_float)] + [(n, ctypes.c_void_p) for n in (
            "qpos", "doc_lo", "chunk_order", "tile_class", "row_ptr", "row_idx", "col_ptr",
            "col_idx", "fwd_order", "bwd_order", "status", "kv_slices", "kv_splits",
            "counts")] + [(n, ctypes.c_int) for n in ("n_sms", "kv_pool_slots")]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` (or "
            "`python document_masked_gqa_gb300/build.py`)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, sz, f32, u64 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float,
                             ctypes.c_uint64)
    sigs = {
        "dma_plan_workspace_bytes": (sz, [i32] * 7),
        "dma_plan": (i32, [vp, i32, i32, i32, i32, i32, i32, i32, i32, f32, vp, sz, vp,
                           ctypes.POINTER(vp)]),
        "dma_attn_fwd": (i32, [vp] * 7),
        "dma_attn_bwd": (i32, [vp] * 11),
        "dma_plan_check": (i32, [vp, vp]),
        "dma_plan_destroy": (i32, [vp]),
        "dma_status_str": (ctypes.c_char_p, [i32]),
        "dma_cp_gather": (i32, [vp, vp, vp, sz, vp]),
        "dma_cp_scatter": (i32, [vp, vp, vp, sz, vp]),
        "dma_plan_get_view": (i32, [vp, ctypes.POINTER(PlanView)]),
        "dma_plan_set_wait_timeout": (i32, [vp, u64]),
        "dma_debug_wait_probe": (i32, [u64, vp, vp]),
        "dma_attn_bwd_delta": (i32, [vp] * 4),
        "dma_attn_bwd_dkdv": (i32, [vp] * 9),
        "dma_attn_bwd_dq": (i32, [vp] * 8),
        "dma_attn_bwd_dq_delta": (i32, [vp] * 9),
        "dma_cp_unpermute": (i32, [vp, vp, i32, i32, i32, sz, vp]),
        "dma_cp_permute": (i32, [vp, vp, i32, i32, i32, sz, vp]),
        "dma_attn_fwd_noalloc": (i32, [vp, i32, i32, i32, i32, i32, i32, i32, i32, f32] +
                                 [vp] * 7),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_LIB = None


def lib():
    global _LIB
    if _LIB is None:
        _LIB = _load()
    return _LIB


def status_str(status: int) -> str:
    return lib().dma_status_str(int(status)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status: int, what: str):
    if status != DMA_OK:
        raise DmaError(status, what)


def dma_plan_workspace_bytes(batch, seq_len, cp_size, n_heads, n_kv_heads, head_dim,
                             max_docs=0) -> int:
    return int(lib().dma_plan_workspace_bytes(batch, seq_len, cp_size, n_heads, n_kv_heads,
                                              head_dim, max_docs))


class Plan:
    """One rank's plan: wraps a ``dma_plan_t`` and the workspace it points
    into (a torch uint8 tensor, allocated here unless one is passed)."""

    def __init__(self, handle, workspace, shape, cu_doc_lens):
        self._h = handle
        self.workspace = workspace
        self.shape = shape
        self._cu = cu_doc_lens  # keep alive until the plan kernels have run

    @property
    def handle(self):
        return self._h

    def __del__(self):
        try:
            if self._h is not None and _LIB is not None:
                _LIB.dma_plan_destroy(self._h)
        except Exception:
            pass
        self._h = None

    def view(self) -> PlanView:
        v = PlanView()
        _check(lib().dma_plan_get_view(self._h, ctypes.byref(v)), "dma_plan_get_view")
        return v


def dma_plan(cu_doc_lens, batch, seq_len, cp_size, cp_rank, n_heads, n_kv_heads, head_dim,
             softmax_scale=0.0, workspace=None, stream=None) -> Plan:
    import torch
    need = dma_plan_workspace_bytes(batch, seq_len, cp_size, n_heads, n_kv_heads, head_dim)
    if workspace is None:
        if need == 0:
            # let the library report why the shape is rejected
            workspace = torch.empty(256, dtype=torch.uint8, device="cuda")
        else:
            workspace = torch.empty(need, dtype=torch.uint8, device="cuda")
    if cu_doc_lens is not None and (cu_doc_lens.dtype != torch.int32 or not cu_doc_lens.is_cuda
                                    or not cu_doc_lens.is_contiguous()
                                    or cu_doc_lens.dim() != 1):
        raise ValueError("cu_doc_lens: want a contiguous 1-D int32 cuda tensor")
    if not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace: want a contiguous cuda tensor")
    n_docs = 0 if cu_doc_lens is None else cu_doc_lens.numel() - 1
    h = ctypes.c_void_p()
    st = lib().dma_plan(_ptr(cu_doc_lens), n_docs, batch, seq_len, cp_size, cp_rank, n_heads,
                        n_kv_heads, head_dim, float(softmax_scale), _ptr(workspace),
                        workspace.numel() * workspace.element_size(), _stream(stream),
                        ctypes.byref(h))
    _check(st, "dma_plan")
    return Plan(h, workspace, (batch, seq_len, cp_size, cp_rank, n_heads, n_kv_heads, head_dim),
                cu_doc_lens)


def _expect(t, dtype, shape, name):
    import torch
    if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_cuda \
            or not t.is_contiguous():
        raise ValueError(f"{name}: want {dtype} {tuple(shape)} contiguous cuda, "
                         f"got {t.dtype} {tuple(t.shape)} cuda={t.is_cuda} "
                         f"contiguous={t.is_contiguous()}")


def dma_attn_fwd(plan: Plan, q, k, v, o=None, lse=None, stream=None):
    import torch
    B, S, cp, _, Hq, Hkv, D = plan.shape
    Lq = S // cp
    _expect(q, torch.bfloat16, (B, Lq, Hq, D), "q")
    _expect(k, torch.bfloat16, (B, S, Hkv, D), "k")
    _expect(v, torch.bfloat16, (B, S, Hkv, D), "v")
    if o is None:
        o = torch.empty(B, Lq, Hq, D, dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty(B, Hq, Lq, dtype=torch.float32, device=q.device)
    _expect(o, torch.float32, (B, Lq, Hq, D), "o")
    _expect(lse, torch.float32, (B, Hq, Lq), "lse")
    _check(lib().dma_attn_fwd(plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                              _stream(stream)), "dma_attn_fwd")
    return o, lse


def dma_attn_bwd(plan: Plan, q, k, v, o, lse, dout, dq=None, dk=None, dv=None, stream=None):
    import torch
    B, S, cp, _, Hq, Hkv, D = plan.shape
    Lq = S // cp
    _expect(q, torch.bfloat16, (B, Lq, Hq, D), "q")
    _expect(k, torch.bfloat16, (B, S, Hkv, D), "k")
    _expect(v, torch.bfloat16, (B, S, Hkv, D), "v")
    _expect(o, torch.float32, (B, Lq, Hq, D), "o")
    _expect(lse, torch.float32, (B, Hq, Lq), "lse")
    _expect(dout, torch.bfloat16, (B, Lq, Hq, D), "dout")
    if dq is None:
        dq = torch.empty_like(q)
    if dk is None:
        dk = torch.empty(B, S, Hkv, D, dtype=torch.float32, device=q.device)
    if dv is None:
        dv = torch.empty(B, S, Hkv, D, dtype=torch.float32, device=q.device)
    _expect(dq, torch.bfloat16, (B, Lq, Hq, D), "dq")
    _expect(dk, torch.float32, (B, S, Hkv, D), "dk")
    _expect(dv, torch.float32, (B, S, Hkv, D), "dv")
    _check(lib().dma_attn_bwd(plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                              _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _stream(stream)),
           "dma_attn_bwd")
    return dq, dk, dv


def dma_attn_bwd_delta(plan: Plan, o, dout, stream=None):
    import torch
    B, S, cp, _, Hq, Hkv, D = plan.shape
    Lq = S // cp
    _expect(o, torch.float32, (B, Lq, Hq, D), "o")
    _expect(dout, torch.bfloat16, (B, Lq, Hq, D), "dout")
    _check(lib().dma_attn_bwd_delta(plan.handle, _ptr(o), _ptr(dout), _stream(stream)),
           "dma_attn_bwd_delta")


def dma_attn_bwd_dkdv(plan: Plan, q, k, v, lse, dout, dk, dv, stream=None):
    import torch
    B, S, cp, _, Hq, Hkv, D = plan.shape
    Lq = S // cp
    _expect(q, torch.bfloat16, (B, Lq, Hq, D), "q")
    _expect(k, torch.bfloat16, (B, S, Hkv, D), "k")
    _expect(v, torch.bfloat16, (B, S, Hkv, D), "v")
    _expect(lse, torch.float32, (B, Hq, Lq), "lse")
    _expect(dout, torch.bfloat16, (B, Lq, Hq, D), "dout")
    _expect(dk, torch.float32, (B, S, Hkv, D), "dk")
    _expect(dv, torch.float32, (B, S, Hkv, D), "dv")
    _check(lib().dma_attn_bwd_dkdv(plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(lse),
                                   _ptr(dout), _ptr(dk), _ptr(dv), _stream(stream)),
           "dma_attn_bwd_dkdv")


def dma_attn_bwd_dq(plan: Plan, q, k, v, lse, dout, dq, stream=None):
    import torch
    B, S, cp, _, Hq, Hkv, D = plan.shape
    Lq = S // cp
    _expect(q, torch.bfloat16, (B, Lq, Hq, D), "q")
    _expect(k, torch.bfloat16, (B, S, Hkv, D), "k")
    _expect(v, torch.bfloat16, (B, S, Hkv, D), "v")
    _expect(lse, torch.float32, (B, Hq, Lq), "lse")
    _expect(dout, torch.bfloat16, (B, Lq, Hq, D), "dout")
    _expect(dq, torch.bfloat16, (B, Lq, Hq, D), "dq")
    _check(lib().dma_attn_bwd_dq(plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(lse),
                                 _ptr(dout), _ptr(dq), _stream(stream)), "dma_attn_bwd_dq")


def dma_attn_bwd_dq_delta(plan: Plan, q, k, v, o, lse, dout, dq, stream=None):
    import torch
    B, S, cp, _, Hq, Hkv, D = plan.shape
    Lq = S // cp
    _expect(q, torch.bfloat16, (B, Lq, Hq, D), "q")
    _expect(k, torch.bfloat16, (B, S, Hkv, D), "k")
    _expect(v, torch.bfloat16, (B, S, Hkv, D), "v")
    _expect(o, torch.float32, (B, Lq, Hq, D), "o")
    _expect(lse, torch.float32, (B, Hq, Lq), "lse")
    _expect(dout, torch.bfloat16, (B, Lq, Hq, D), "dout")
    _expect(dq, torch.bfloat16, (B, Lq, Hq, D), "dq")
    _check(lib().dma_attn_bwd_dq_delta(plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                       _ptr(lse), _ptr(dout), _ptr(dq), _stream(stream)),
           "dma_attn_bwd_dq_delta")


def dma_plan_check(plan: Plan, stream=None) -> int:
    return int(lib().dma_plan_check(plan.handle, _stream(stream)))


def dma_plan_set_wait_timeout(plan: Plan, timeout_ns: int):
    _check(lib().dma_plan_set_wait_timeout(plan.handle, int(timeout_ns)),
           "dma_plan_set_wait_timeout")


def dma_cp_gather(plan: Plan, full, local=None, stream=None):
    import torch
    B, S, cp, _, _, _, _ = plan.shape
    Lq = S // cp
    _expect(full, full.dtype, (B, S) + tuple(full.shape[2:]), "full")
    if local is None:
        local = torch.empty((B, Lq) + tuple(full.shape[2:]), dtype=full.dtype, device=full.device)
    _expect(local, full.dtype, (B, Lq) + tuple(full.shape[2:]), "local")
    row_bytes = math.prod(full.shape[2:]) * full.element_size()
    _check(lib().dma_cp_gather(plan.handle, _ptr(full), _ptr(local), row_bytes,
                               _stream(stream)), "dma_cp_gather")
    return local


def dma_cp_scatter(plan: Plan, local, full, stream=None):
    B, S, cp, _, _, _, _ = plan.shape
    Lq = S // cp
    _expect(full, full.dtype, (B, S) + tuple(full.shape[2:]), "full")
    _expect(local, full.dtype, (B, Lq) + tuple(full.shape[2:]), "local")
    row_bytes = math.prod(full.shape[2:]) * full.element_size()
    _check(lib().dma_cp_scatter(plan.handle, _ptr(local), _ptr(full), row_bytes,
                                _stream(stream)), "dma_cp_scatter")
    return full


def dma_cp_unpermute(gathered, full=None, stream=None):
    """[cp, B, 2C, ...] rank-major rows (an all-gather of every rank's local
    rows) -> [B, S, ...] natural order."""
    import torch
    cp, B, Lq = gathered.shape[:3]
    if full is None:
        full = torch.empty((B, cp * Lq) + tuple(gathered.shape[3:]), dtype=gathered.dtype,
                           device=gathered.device)
    _expect(gathered, gathered.dtype, tuple(gathered.shape), "gathered")
    _expect(full, gathered.dtype, (B, cp * Lq) + tuple(gathered.shape[3:]), "full")
    row_bytes = math.prod(gathered.shape[3:]) * gathered.element_size()
    _check(lib().dma_cp_unpermute(_ptr(gathered), _ptr(full), B, cp * Lq, cp, row_bytes,
                                  _stream(stream)), "dma_cp_unpermute")
    return full


def dma_cp_permute(full, cp_size, gathered=None, stream=None):
    """[B, S, ...] natural order -> [cp, B, 2C, ...] rank-major rows (the
    input of a reduce-scatter whose block r is rank r's rows)."""
    import torch
    B, S = full.shape[:2]
    Lq = S // cp_size
    if gathered is None:
        gathered = torch.empty((cp_size, B, Lq) + tuple(full.shape[2:]), dtype=full.dtype,
                               device=full.device)
    _expect(full, full.dtype, tuple(full.shape), "full")
    _expect(gathered, full.dtype, (cp_size, B, Lq) + tuple(full.shape[2:]), "gathered")
    row_bytes = math.prod(full.shape[2:]) * full.element_size()
    _check(lib().dma_cp_permute(_ptr(full), _ptr(gathered), B, S, cp_size, row_bytes,
                                _stream(stream)), "dma_cp_permute")
    return gathered


def dma_debug_wait_probe(timeout_ns: int, status_dev, stream=None) -> int:
    return int(lib().dma_debug_wait_probe(int(timeout_ns), _ptr(status_dev), _stream(stream)))


def plan_arrays(plan: Plan) -> dict:
    """Copies of the plan's device arrays as CPU tensors (for tests)."""
    import torch
    v = plan.view()
    B, nqt, nkt, Lq, cp = v.batch, v.n_qtiles, v.n_ktiles, v.local_len, v.cp_size
    torch.cuda.synchronize()

    ws = plan.workspace
    base = ws.data_ptr()

    def grab(ptr, n, dtype):
        # every view pointer lies inside the workspace tensor the plan owns
        esz = torch.empty(0, dtype=dtype).element_size()
        if n == 0:
            return torch.empty(0, dtype=dtype)
        off = int(ptr) - base
        assert 0 <= off and off + n * esz <= ws.numel()
        return ws[off:off + n * esz].cpu().view(dtype).clone()

    out = {"qpos": grab(v.qpos, Lq, torch.int32),
           "doc_lo": grab(v.doc_lo, B * Lq, torch.int32).reshape(B, Lq),
           "chunk_order": grab(v.chunk_order, 2 * cp, torch.int32),
           "tile_class": grab(v.tile_class, B * nqt * nkt, torch.uint8).reshape(B, nqt, nkt),
           "row_ptr": grab(v.row_ptr, B * nqt + 1, torch.int32),
           "col_ptr": grab(v.col_ptr, B * nkt + 1, torch.int32),
           "fwd_order": grab(v.fwd_order, B * nqt, torch.int32),
           "bwd_order": grab(v.bwd_order, B * nkt, torch.int32),
           "status": grab(v.status, 1, torch.int32)}
    nnz_r = int(out["row_ptr"][-1]) if B else 0
    nnz_c = int(out["col_ptr"][-1]) if B else 0
    out["row_idx"] = grab(v.row_idx, nnz_r, torch.int32)
    out["col_idx"] = grab(v.col_idx, nnz_c, torch.int32)
    counts = grab(v.counts, 2, torch.int32) if B else torch.zeros(2, dtype=torch.int32)
    n_sl, n_sp = int(counts[0]), int(counts[1])
    out["kv_slices"] = grab(v.kv_slices, 8 * n_sl, torch.int32).reshape(n_sl, 8)
    out["kv_splits"] = grab(v.kv_splits, 4 * n_sp, torch.int32).reshape(n_sp, 4)
    out["n_sms"] = int(v.n_sms)
    out["kv_pool_slots"] = int(v.kv_pool_slots)
    return out
