"""Batch-invariant paged prefill attention for GB300 (sm_103a).

Python binding of the C ABI in ``include/bip.h`` (libbip.so, loaded with
ctypes).  This layer only marshals arguments: every step of the attention
runs in the library's CUDA kernels, and there is no CPU or PyTorch fallback
(the library missing is an error).

    plan = Plan(qo_indptr, kv_indptr, kv_last_page_len, num_qo_heads=32,
                num_kv_heads=8, head_dim=128, page_size=16)
    out, lse = prefill(plan, q, k_pages, v_pages, kv_indices)

PyTorch supplies device memory and streams only.
"""

from __future__ import annotations

import ctypes
from typing import Optional

import numpy as np

from . import _lib

__all__ = ["BipError", "Plan", "prefill", "append_kv", "GraphPlan", "prefill_graph", "workspace_bound",
           "read_device_status", "pack_mask", "STATUS"]

STATUS = {
    0: "BIP_OK", 1: "BIP_ERR_INVALID_ARG", 2: "BIP_ERR_UNSUPPORTED", 3: "BIP_ERR_WORKSPACE_TOO_SMALL",
    4: "BIP_ERR_CUDA", 5: "BIP_ERR_DEVICE_TIMEOUT", 6: "BIP_ERR_OUT_OF_MEMORY", 7: "BIP_ERR_BAD_PAGE_INDEX",
}
_POLICY = {"auto": 0, "never": 1, "always": 2}
_KV = {"bf16": 0, "fp8_e4m3": 1}


class BipError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = int(code)
        super().__init__(f"{what}: {STATUS.get(self.code, self.code)}")


def _check(code: int, what: str) -> None:
    if code != 0:
        raise BipError(code, what)


def _i32_array(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def workspace_bound(max_batch: int, max_total_q: int, num_qo_heads: int, num_kv_heads: int, head_dim: int,
                    split_budget_bytes: int = 256 << 20) -> int:
    """Workspace bytes that suffice for any plan up to these sizes (0 if unsupported)."""
    return int(_lib.load().bip_workspace_bound(max_batch, max_total_q, num_qo_heads, num_kv_heads, head_dim,
                                               split_budget_bytes))


class Plan:
    """A batch's tile schedule and work list (host only; immutable).

    Closing (or dropping) a plan waits for the calls enqueued with it to
    finish; keep it alive while a CUDA graph that captured a call with it can
    still be replayed."""

    def __init__(self, qo_indptr, kv_indptr, kv_last_page_len, *, num_qo_heads: int, num_kv_heads: int,
                 head_dim: int, page_size: int = 16, kv_dtype: str = "bf16", split_policy: str = "auto",
                 split_budget_bytes: int = 256 << 20, num_sms: int = 0, wait_limit_ns: int = 0,
                 tiles_per_unit: int = 0, window_left: int = 0):
        self._lib = _lib.load()
        self._h = ctypes.c_void_p()
        qo, kv, last = _i32_array(qo_indptr), _i32_array(kv_indptr), _i32_array(kv_last_page_len)
        batch = len(qo) - 1
        if batch < 0 or len(kv) != batch + 1 or len(last) != batch:
            raise BipError(1, "indptr lengths disagree")
        opts = _lib.PlanOptions(_POLICY[split_policy], int(split_budget_bytes), int(num_sms), int(wait_limit_ns),
                                int(tiles_per_unit), int(window_left))
        ws = ctypes.c_size_t()
        _check(self._lib.bip_plan(ctypes.byref(self._h), _ptr(qo), _ptr(kv), _ptr(last) if batch else None,
                                  batch, num_qo_heads, num_kv_heads, head_dim, page_size, _KV[kv_dtype],
                                  ctypes.byref(opts), ctypes.byref(ws)), "bip_plan")
        self.workspace_bytes = int(ws.value)
        self.num_qo_heads, self.num_kv_heads, self.head_dim = num_qo_heads, num_kv_heads, head_dim
        self.page_size, self.kv_dtype = page_size, kv_dtype
        self.total_q = int(qo[-1]) if batch >= 0 else 0

    @property
    def info(self) -> dict:
        inf = _lib.PlanInfo()
        _check(self._lib.bip_plan_get_info(self._h, ctypes.byref(inf)), "bip_plan_get_info")
        return inf.as_dict()

    def items(self) -> np.ndarray:
        """Work items in launch order: request, kv_head, q_tile, seg_lo, seg_hi, split, kv_blocks, tile_mask."""
        n = ctypes.c_int32()
        _check(self._lib.bip_plan_get_items(self._h, None, 0, ctypes.byref(n)), "bip_plan_get_items")
        buf = np.zeros((max(n.value, 1), 8), dtype=np.int32)
        _check(self._lib.bip_plan_get_items(self._h, _ptr(buf), n.value, ctypes.byref(n)), "bip_plan_get_items")
        return buf[: n.value]

    def close(self) -> None:
        if self._h:
            self._lib.bip_plan_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _require_cuda(**tensors):
    """Every given tensor (None = to be allocated) must live on a CUDA device:
    there is no CPU path."""
    import torch
    for name, t in tensors.items():
        if t is not None and (not isinstance(t, torch.Tensor) or not t.is_cuda):
            raise BipError(1, f"{name} must be a CUDA tensor")


def _dev_ptr(t, name: str):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise BipError(1, f"{name} must be a CUDA tensor")
    return ctypes.c_void_p(t.data_ptr())


def pack_mask(masks, row_words: Optional[int] = None) -> np.ndarray:
    """Per-request boolean masks ``[q_len, kv_len]`` (in request order) as the
    words ``bip_prefill_masked`` reads: int32 ``[total_q, row_words]``, bit
    ``j % 32`` (least significant first) of word ``j // 32`` of a q row = key j
    visible.  ``row_words`` defaults to the fewest that hold the longest row.
    Host-side input preparation (numpy); copy the result to the device."""
    rows = [np.asarray(m, dtype=bool) for m in masks]
    if any(m.ndim != 2 for m in rows):
        raise BipError(1, "each mask must be a 2-d [q_len, kv_len] array")
    need = max([(m.shape[1] + 31) // 32 for m in rows], default=0)
    words = need if row_words is None else int(row_words)
    if words < need:
        raise BipError(1, f"row_words {words} < {need} needed for the longest mask row")
    total = sum(m.shape[0] for m in rows)
    out = np.zeros((total, words * 4), dtype=np.uint8)
    r = 0
    for m in rows:
        packed = np.packbits(m, axis=1, bitorder="little")  # byte b, bit i = key 8 b + i
        out[r:r + m.shape[0], :packed.shape[1]] = packed
        r += m.shape[0]
    return out.view("<u4").view(np.int32).reshape(total, words)


def prefill(plan: Plan, q, k_pages, v_pages, kv_indices, *, out=None, lse=None, workspace=None,
            k_scale: float = 1.0, v_scale: float = 1.0, stream=None, custom_mask=None):
    """Enqueue the attention on ``stream`` (default: torch's current stream).

    q [total_q, Hq, d] bf16; k_pages / v_pages [num_pages, page_size, Hkv, d]
    (a page stride other than page_size*Hkv*d is allowed, the same for K and V);
    kv_indices int32 on the device.  ``out``, ``lse`` and ``workspace`` are
    allocated on ``stream`` when not given; pass a workspace of your own to
    read the call's device status afterwards (``read_device_status``).  ``custom_mask``: None, or int32 words
    ``[total_q, row_words]`` on the device (see ``pack_mask``) that narrow each
    row's causal keys (``bip_prefill_masked``).  Returns (out bf16, lse fp32
    natural log).
    """
    import torch
    _require_cuda(q=q, k_pages=k_pages, v_pages=v_pages, kv_indices=kv_indices, out=out, lse=lse,
                  workspace=workspace, custom_mask=custom_mask)
    dev = q.device
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    # Buffers made here belong to the launch stream, so the caching allocator
    # reuses a temporary workspace only behind this call's kernels.
    with torch.cuda.stream(stream):
        if out is None:
            out = torch.empty_like(q)
        if lse is None:
            lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device=dev)
        if workspace is None:
            workspace = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device=dev)
    if q.dtype != torch.bfloat16 or out.dtype != torch.bfloat16 or lse.dtype != torch.float32:
        raise BipError(1, "q/out must be bf16 and lse fp32")
    if not (q.is_contiguous() and out.is_contiguous() and lse.is_contiguous()):
        raise BipError(1, "q, out and lse must be contiguous")
    if tuple(q.shape[1:]) != (plan.num_qo_heads, plan.head_dim) or out.shape != q.shape:
        raise BipError(1, "q/out shape does not match the plan")
    if kv_indices.dtype != torch.int32:
        raise BipError(1, "kv_indices must be int32")
    want = torch.bfloat16 if plan.kv_dtype == "bf16" else torch.uint8
    for name, pg in (("k_pages", k_pages), ("v_pages", v_pages)):
        if pg.dtype != want or pg.dim() != 4 or tuple(pg.shape[1:]) != (plan.page_size, plan.num_kv_heads,
                                                                        plan.head_dim):
            raise BipError(1, f"{name} must be [num_pages, page_size, Hkv, d] of {want}")
        if pg.stride()[1:] != (plan.num_kv_heads * plan.head_dim, plan.head_dim, 1):
            raise BipError(1, f"{name}: slots and heads must be contiguous inside a page")
    if k_pages.shape[0] != v_pages.shape[0] or k_pages.stride(0) != v_pages.stride(0):
        raise BipError(1, "k_pages and v_pages must share page count and stride")
    if custom_mask is not None:
        if custom_mask.dtype != torch.int32 or custom_mask.dim() != 2 or not custom_mask.is_contiguous():
            raise BipError(1, "custom_mask must be contiguous int32 [total_q, row_words]")
        if custom_mask.shape[0] != q.shape[0]:
            raise BipError(1, "custom_mask must have one row per q row")
    sptr = ctypes.c_void_p(stream.cuda_stream)
    args = (_dev_ptr(q, "q"), q.shape[0], _dev_ptr(k_pages, "k_pages"), _dev_ptr(v_pages, "v_pages"),
            k_pages.shape[0], k_pages.stride(0), _dev_ptr(kv_indices, "kv_indices"))
    tail = (float(k_scale), float(v_scale), _dev_ptr(out, "out"), _dev_ptr(lse, "lse"),
            _dev_ptr(workspace, "workspace"), workspace.numel() * workspace.element_size(), sptr)
    if custom_mask is None:
        _check(plan._lib.bip_prefill(plan._h, *args, *tail), "bip_prefill")
    else:
        _check(plan._lib.bip_prefill_masked(plan._h, *args, _dev_ptr(custom_mask, "custom_mask"),
                                            custom_mask.shape[1], *tail), "bip_prefill_masked")
    return out, lse


def append_kv(plan: Plan, k_new, v_new, k_pages, v_pages, kv_indices, *, workspace=None,
              k_scale: float = 1.0, v_scale: float = 1.0, stream=None):
    """Enqueue the paged KV append on ``stream`` (default: torch's current stream).

    k_new / v_new bf16 [total_q, Hkv, d]: request r's new rows, in the plan's
    row order, go to its positions kv_len - q_len .. kv_len - 1.  The pools
    (the same tensors ``prefill`` reads) are written in place: bf16 bits
    unchanged, or e4m3(x / scale) for uint8 (E4M3) pools.
    """
    import torch
    _require_cuda(k_new=k_new, v_new=v_new, k_pages=k_pages, v_pages=v_pages, kv_indices=kv_indices,
                  workspace=workspace)
    dev = k_new.device
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    if workspace is None:  # on the launch stream: reused only behind this call's kernel
        with torch.cuda.stream(stream):
            workspace = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device=dev)
    for name, t in (("k_new", k_new), ("v_new", v_new)):
        if t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise BipError(1, f"{name} must be contiguous bf16")
        if tuple(t.shape) != (plan.total_q, plan.num_kv_heads, plan.head_dim):
            raise BipError(1, f"{name} must be [total_q, Hkv, d] of the plan")
    if kv_indices.dtype != torch.int32:
        raise BipError(1, "kv_indices must be int32")
    want = torch.bfloat16 if plan.kv_dtype == "bf16" else torch.uint8
    for name, pg in (("k_pages", k_pages), ("v_pages", v_pages)):
        if pg.dtype != want or pg.dim() != 4 or tuple(pg.shape[1:]) != (plan.page_size, plan.num_kv_heads,
                                                                        plan.head_dim):
            raise BipError(1, f"{name} must be [num_pages, page_size, Hkv, d] of {want}")
        if pg.stride()[1:] != (plan.num_kv_heads * plan.head_dim, plan.head_dim, 1):
            raise BipError(1, f"{name}: slots and heads must be contiguous inside a page")
    if k_pages.shape[0] != v_pages.shape[0] or k_pages.stride(0) != v_pages.stride(0):
        raise BipError(1, "k_pages and v_pages must share page count and stride")
    _check(plan._lib.bip_append_kv(plan._h, _dev_ptr(k_new, "k_new"), _dev_ptr(v_new, "v_new"), k_new.shape[0],
                                   _dev_ptr(k_pages, "k_pages"), _dev_ptr(v_pages, "v_pages"), k_pages.shape[0],
                                   k_pages.stride(0), _dev_ptr(kv_indices, "kv_indices"), float(k_scale),
                                   float(v_scale), _dev_ptr(workspace, "workspace"),
                                   workspace.numel() * workspace.element_size(),
                                   ctypes.c_void_p(stream.cuda_stream)), "bip_append_kv")
    return k_pages, v_pages


class GraphPlan:
    """Capacities and shapes for device-planned, graph-replayable prefills."""

    def __init__(self, max_batch: int, max_total_q: int, *, num_qo_heads: int, num_kv_heads: int, head_dim: int,
                 page_size: int = 16, kv_dtype: str = "bf16", num_sms: int = 0, wait_limit_ns: int = 0,
                 tiles_per_unit: int = 0, window_left: int = 0, split_policy: str = "auto",
                 split_budget_bytes: int = 64 << 20):
        self._lib = _lib.load()
        self._h = ctypes.c_void_p()
        opts = _lib.PlanOptions(_POLICY[split_policy], int(split_budget_bytes), int(num_sms), int(wait_limit_ns),
                                int(tiles_per_unit), int(window_left))
        ws = ctypes.c_size_t()
        _check(self._lib.bip_graph_plan(ctypes.byref(self._h), int(max_batch), int(max_total_q), num_qo_heads,
                                        num_kv_heads, head_dim, page_size, _KV[kv_dtype], ctypes.byref(opts),
                                        ctypes.byref(ws)), "bip_graph_plan")
        self.workspace_bytes = int(ws.value)
        self.max_batch, self.max_total_q = int(max_batch), int(max_total_q)
        self.num_qo_heads, self.num_kv_heads, self.head_dim = num_qo_heads, num_kv_heads, head_dim
        self.page_size, self.kv_dtype = page_size, kv_dtype

    def close(self) -> None:
        if self._h:
            self._lib.bip_graph_plan_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def prefill_graph(plan: GraphPlan, batch: int, qo_indptr, kv_indptr, kv_last_page_len, q, k_pages, v_pages,
                  kv_indices, out, lse, workspace, *, k_scale: float = 1.0, v_scale: float = 1.0, stream=None,
                  custom_mask=None):
    """Enqueue a device-planned prefill (capturable in a CUDA graph).

    The indptr arrays are int32 device tensors read when the launch runs;
    q/out [max_total_q, Hq, d] bf16 and lse [max_total_q, Hq] fp32 are the
    graph's static buffers.  ``custom_mask``: None, or int32 words
    ``[max_total_q, row_words]`` on the device (``bip_prefill_graph_masked``).
    Results equal ``prefill`` on the same batch.
    """
    import torch
    _require_cuda(qo_indptr=qo_indptr, kv_indptr=kv_indptr, kv_last_page_len=kv_last_page_len, q=q,
                  k_pages=k_pages, v_pages=v_pages, kv_indices=kv_indices, out=out, lse=lse, workspace=workspace,
                  custom_mask=custom_mask)
    for name, t, n in (("qo_indptr", qo_indptr, batch + 1), ("kv_indptr", kv_indptr, batch + 1),
                       ("kv_last_page_len", kv_last_page_len, batch)):
        if t.dtype != torch.int32 or not t.is_contiguous() or t.numel() < n:
            raise BipError(1, f"{name} must be a contiguous int32 device tensor of at least {n} entries")
    rows = (plan.max_total_q, plan.num_qo_heads, plan.head_dim)
    if q.dtype != torch.bfloat16 or out.dtype != torch.bfloat16 or tuple(q.shape) != rows or out.shape != q.shape:
        raise BipError(1, "q and out must be bf16 [max_total_q, Hq, d]")
    if lse.dtype != torch.float32 or tuple(lse.shape) != rows[:2]:
        raise BipError(1, "lse must be fp32 [max_total_q, Hq]")
    if not (q.is_contiguous() and out.is_contiguous() and lse.is_contiguous()):
        raise BipError(1, "q, out and lse must be contiguous")
    if kv_indices.dtype != torch.int32:
        raise BipError(1, "kv_indices must be int32")
    want = torch.bfloat16 if plan.kv_dtype == "bf16" else torch.uint8
    for name, pg in (("k_pages", k_pages), ("v_pages", v_pages)):
        if pg.dtype != want or pg.dim() != 4 or tuple(pg.shape[1:]) != (plan.page_size, plan.num_kv_heads,
                                                                        plan.head_dim):
            raise BipError(1, f"{name} must be [num_pages, page_size, Hkv, d] of {want}")
        if pg.stride()[1:] != (plan.num_kv_heads * plan.head_dim, plan.head_dim, 1):
            raise BipError(1, f"{name}: slots and heads must be contiguous inside a page")
    if k_pages.shape[0] != v_pages.shape[0] or k_pages.stride(0) != v_pages.stride(0):
        raise BipError(1, "k_pages and v_pages must share page count and stride")
    if custom_mask is not None:
        if custom_mask.dtype != torch.int32 or custom_mask.dim() != 2 or not custom_mask.is_contiguous():
            raise BipError(1, "custom_mask must be contiguous int32 [max_total_q, row_words]")
        if custom_mask.shape[0] != plan.max_total_q:
            raise BipError(1, "custom_mask must have one row per q buffer row")
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    head = (_dev_ptr(qo_indptr, "qo_indptr"), _dev_ptr(kv_indptr, "kv_indptr"),
            _dev_ptr(kv_last_page_len, "kv_last_page_len"), _dev_ptr(q, "q"), _dev_ptr(k_pages, "k_pages"),
            _dev_ptr(v_pages, "v_pages"), k_pages.shape[0], k_pages.stride(0), _dev_ptr(kv_indices, "kv_indices"))
    tail = (float(k_scale), float(v_scale), _dev_ptr(out, "out"), _dev_ptr(lse, "lse"),
            _dev_ptr(workspace, "workspace"), workspace.numel() * workspace.element_size(),
            ctypes.c_void_p(stream.cuda_stream))
    if custom_mask is None:
        _check(plan._lib.bip_prefill_graph(plan._h, int(batch), *head, *tail), "bip_prefill_graph")
    else:
        _check(plan._lib.bip_prefill_graph_masked(plan._h, int(batch), *head, _dev_ptr(custom_mask, "custom_mask"),
                                                  custom_mask.shape[1], *tail), "bip_prefill_graph_masked")
    return out, lse


def read_device_status(workspace, stream=None) -> int:
    """Synchronise ``stream`` and return the status word of the last call on ``workspace``."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(workspace.device)
    return int(_lib.load().bip_read_device_status(_dev_ptr(workspace, "workspace"),
                                                  ctypes.c_void_p(stream.cuda_stream)))
