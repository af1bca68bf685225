"""bip_prefill_no_alloc, called through the C ABI.

Some callers cannot allocate device memory: a plugin inside an engine whose
memory pool owns the whole GPU, a serving loop that forbids allocation on the
request path.  bip_prefill_no_alloc serves them with a workspace that lives
in a fixed device array inside the library, so the caller passes only the
inputs and outputs.  This test checks that it gives the same results as
bip_prefill with a caller workspace, on two calls in a row and on calls
that alternate between a plan that splits units and one that folds them (the
array keeps the previous call's contents), and that a plan needing more
workspace than the array holds is refused.  It sits in a file that pytest collects last.
"""

import ctypes

import numpy as np
import pytest
import torch

import invariant_paged_prefill_gb300 as bip
from invariant_paged_prefill_gb300 import workloads as W

from gpu_helpers import ATOL, RTOL, to_device

pytestmark = pytest.mark.gpu

NO_ALLOC_BYTES = 32 << 20  # BIP_NO_ALLOC_WORKSPACE_BYTES in include/bip.h


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _call_no_alloc(lib, plan, b, out, lse):
    stream = torch.cuda.current_stream()
    return lib.bip_prefill_no_alloc(plan._h, _ptr(b.q), b.q.shape[0], _ptr(b.k_pages), _ptr(b.v_pages),
                                    b.k_pages.shape[0], b.k_pages.stride(0), _ptr(b.kv_indices), 1.0, 1.0,
                                    _ptr(out), _ptr(lse), ctypes.c_void_p(stream.cuda_stream))


def _within_tolerance(got, ref):
    g, r = got.float().cpu().numpy(), ref.float().cpu().numpy()
    return np.isfinite(g).all() and (np.abs(g - r) <= ATOL + RTOL * np.abs(r)).all()


def test_no_alloc_entry_matches_bip_prefill_twice(lib, cuda):
    prompts, q_lens = W.mixed_ragged_prompts()
    b = to_device(W.layout(prompts, q_lens, 16), cuda)
    plan = bip.Plan(b.qo_indptr, b.kv_indptr, b.kv_last_page_len, num_qo_heads=b.num_qo_heads,
                    num_kv_heads=b.num_kv_heads, head_dim=b.head_dim)
    assert plan.workspace_bytes <= NO_ALLOC_BYTES
    ref_out, ref_lse = bip.prefill(plan, b.q, b.k_pages, b.v_pages, b.kv_indices)
    torch.cuda.synchronize()
    for call in range(2):
        out = torch.full_like(b.q, float("nan"))
        lse = torch.full((b.q.shape[0], b.q.shape[1]), float("nan"), dtype=torch.float32, device=cuda)
        assert _call_no_alloc(lib, plan, b, out, lse) == 0
        torch.cuda.synchronize()
        assert _within_tolerance(out, ref_out), f"call {call}: out differs"
        assert _within_tolerance(lse, ref_lse), f"call {call}: lse differs"
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)


def test_no_alloc_entry_after_a_different_plan(lib, cuda):
    # The array keeps the previous call's contents.  A plan that splits units
    # (partials and merge units in the array) and one that folds them
    # alternate, so each call meets the other's bytes; every call must still
    # give bip_prefill's bits (it writes every region it reads, and the
    # upload rewrites the status word).  Two extends behind 9000 and 5000
    # keys (three and two segments) and a 700-token prefill.
    prompts = [W.make_prompt(n, *W.HEADS_A, seed=40 + i) for i, n in enumerate((9000, 5000, 700))]
    b = to_device(W.layout(prompts, [37, 5, 700], 16), cuda)
    kw = dict(num_qo_heads=b.num_qo_heads, num_kv_heads=b.num_kv_heads, head_dim=b.head_dim)
    fold = bip.Plan(b.qo_indptr, b.kv_indptr, b.kv_last_page_len, split_policy="never", **kw)
    split = bip.Plan(b.qo_indptr, b.kv_indptr, b.kv_last_page_len, split_policy="always", **kw)
    assert split.info["num_split_units"] > 0 and fold.info["num_split_units"] == 0
    assert fold.info["scratch_bytes"] > 0  # folded segments go through the array too
    assert max(fold.workspace_bytes, split.workspace_bytes) <= NO_ALLOC_BYTES
    refs = {}
    for name, plan in (("fold", fold), ("split", split)):
        refs[name] = bip.prefill(plan, b.q, b.k_pages, b.v_pages, b.kv_indices)
    torch.cuda.synchronize()
    assert torch.equal(refs["fold"][0], refs["split"][0])  # split and fold give the same bits
    for name in ("split", "fold", "split", "fold"):
        plan = split if name == "split" else fold
        out = torch.full_like(b.q, float("nan"))
        lse = torch.full((b.q.shape[0], b.q.shape[1]), float("nan"), dtype=torch.float32, device=cuda)
        assert _call_no_alloc(lib, plan, b, out, lse) == 0
        torch.cuda.synchronize()
        assert torch.equal(out, refs[name][0]) and torch.equal(lse, refs[name][1]), f"{name} after another plan"


def test_no_alloc_entry_refuses_a_plan_larger_than_its_array(lib, cuda):
    # Two 128-row extends behind 32768 keys, every unit split with a large
    # budget: the partial states alone far exceed the fixed array.  The size
    # check comes before any pointer is used.
    pages = 32768 // 16
    plan = bip.Plan([0, 128, 256], [0, pages, 2 * pages], [16, 16], num_qo_heads=32, num_kv_heads=8,
                    head_dim=128, split_policy="always", split_budget_bytes=1 << 30)
    assert plan.workspace_bytes > NO_ALLOC_BYTES
    dummy = torch.zeros(16, dtype=torch.uint8, device=cuda)
    p = _ptr(dummy)
    rc = lib.bip_prefill_no_alloc(plan._h, p, 256, p, p, 2 * pages, 16 * 8 * 128, p, 1.0, 1.0, p, p,
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 3  # BIP_ERR_WORKSPACE_TOO_SMALL
