"""Shared helpers for the GPU tests: run the library, run the oracle, compare."""

from __future__ import annotations

import numpy as np
import torch

import invariant_paged_prefill_gb300 as bip
from invariant_paged_prefill_gb300 import workloads as W
from oracle import paged_attention as pa

# Tolerance for bf16 inputs with fp32 accumulation against the float64 oracle:
# |gpu - ref| <= ATOL + RTOL * |ref|, elementwise, for out and for lse.
ATOL, RTOL = 2e-2, 1e-2


def to_device(b: W.PagedBatch, device) -> W.PagedBatch:
    """Copy a batch to the device keeping the page pool's stride."""
    kflat = torch.as_strided(b.k_pages, (b.k_pages.untyped_storage().nbytes() // b.k_pages.element_size(),), (1,), 0)
    vflat = torch.as_strided(b.v_pages, (b.v_pages.untyped_storage().nbytes() // b.v_pages.element_size(),), (1,), 0)
    kd, vd = kflat.to(device), vflat.to(device)
    kp = kd.as_strided(b.k_pages.shape, b.k_pages.stride())
    vp = vd.as_strided(b.v_pages.shape, b.v_pages.stride())
    return W.PagedBatch(**{**b.__dict__, "q": b.q.to(device), "k_pages": kp, "v_pages": vp,
                           "kv_indices": b.kv_indices.to(device)})


def run_gpu(b: W.PagedBatch, device, *, policy: str = "auto", budget: int = 256 << 20, num_sms: int = 0,
            wait_limit_ns: int = 0, check_status: bool = True, k_scale: float = 1.0, v_scale: float = 1.0,
            tiles_per_unit: int = 0, window_left: int = 0, custom_mask=None, mask_row_words=None):
    """Plan + prefill on the device; returns (out, lse, plan) on the host.

    ``custom_mask``: one boolean ``[q_len, kv_len]`` array per request (packed
    with ``pack_mask`` and copied to the device), or None."""
    d = b if b.q.is_cuda else to_device(b, device)
    plan = bip.Plan(d.qo_indptr, d.kv_indptr, d.kv_last_page_len, num_qo_heads=d.num_qo_heads,
                    num_kv_heads=d.num_kv_heads, head_dim=d.head_dim, page_size=d.page_size, kv_dtype=d.kv_dtype,
                    split_policy=policy, split_budget_bytes=budget, num_sms=num_sms, wait_limit_ns=wait_limit_ns,
                    tiles_per_unit=tiles_per_unit, window_left=window_left)
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device=device)
    out = torch.full_like(d.q, float("nan"))
    lse = torch.full((d.q.shape[0], d.q.shape[1]), float("nan"), dtype=torch.float32, device=device)
    words = None
    if custom_mask is not None:
        words = torch.from_numpy(bip.pack_mask(custom_mask, mask_row_words)).to(device)
    bip.prefill(plan, d.q, d.k_pages, d.v_pages, d.kv_indices, out=out, lse=lse, workspace=ws,
                k_scale=k_scale, v_scale=v_scale, custom_mask=words)
    status = bip.read_device_status(ws)
    if check_status:
        where = int(ws[4:8].view(torch.int32).item())  # header: status, wait site, bad page count
        assert status == 0, f"{bip.STATUS.get(status, status)} (wait site {where})"
    return out.cpu(), lse.cpu(), plan


def oracle(b: W.PagedBatch, rows=None, window_left: int = 0, custom_mask=None):
    kind = "bf16" if b.kv_dtype == "bf16" else "e4m3"
    kp = b.k_pages.cpu() if b.k_pages.is_cuda else b.k_pages
    vp = b.v_pages.cpu() if b.v_pages.is_cuda else b.v_pages
    kview = kp.view(torch.int16) if kind == "bf16" else kp
    vview = vp.view(torch.int16) if kind == "bf16" else vp
    return pa.paged_prefill(b.q.cpu().view(torch.int16).numpy(), kview.numpy(), vview.numpy(),
                            b.qo_indptr.tolist(), b.kv_indptr.tolist(), b.kv_indices.cpu().tolist(),
                            b.kv_last_page_len.tolist(), b.num_qo_heads, b.num_kv_heads, b.page_size,
                            q_kind="bf16", kv_kind=kind, rows=rows, window_left=window_left,
                            custom_mask=custom_mask)


def assert_close_to_oracle(out, lse, ref_out, ref_lse, rows=None):
    o = out.float().numpy().astype(np.float64)
    l = lse.numpy().astype(np.float64)
    if rows is not None:
        o, l = o[rows], l[rows]
    assert np.isfinite(o).all() and np.isfinite(l).all(), "non-finite output"
    for name, got, ref in (("out", o, ref_out), ("lse", l, ref_lse)):
        err = np.abs(got - ref)
        bad = err > ATOL + RTOL * np.abs(ref)
        assert not bad.any(), f"{name}: {bad.sum()} elements outside tolerance, max abs err {err.max():.3e}"
    return float(np.abs(o - ref_out).max()), float(np.abs(l - ref_lse).max())


def assert_bitwise(a, b, what=""):
    """Bit-exact: equal values (+0 == -0), no NaN anywhere."""
    assert not torch.isnan(a).any() and not torch.isnan(b).any(), f"NaN in {what}"
    assert torch.equal(a, b), f"{what}: max |diff| = {(a.float() - b.float()).abs().max().item()}"


def sample_rows(b: W.PagedBatch, per_request: int = 24, seed: int = 0):
    """First/last rows, block and segment boundary rows, and random rows of every request."""
    rng = np.random.default_rng(seed)
    rows = []
    for r in range(b.batch):
        lo, hi = b.row_range(r)
        if hi == lo:
            continue
        ql, kl = hi - lo, b.kv_lens[r]
        cand = {lo, hi - 1}
        for pos in (63, 64, 127, 128, 4095, 4096, 8191, 8192):
            t = lo + pos - (kl - ql)
            if lo <= t < hi:
                cand.add(t)
        cand.update(int(x) for x in rng.integers(lo, hi, size=min(per_request, ql)))
        rows.extend(sorted(cand))
    return rows
