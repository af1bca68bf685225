"""Device status word: bounded waits and page-id checks, with no GPU fault.

A plan whose wait limit is 1 ns makes the first wait that is not already
satisfied expire: the kernel records BIP_ERR_DEVICE_TIMEOUT, drains its own
copies and MMAs, frees tensor memory and returns.  The context stays usable:
the next ordinary call on the same workspace succeeds and is correct.
"""

import pytest
import torch

import invariant_paged_prefill_gb300 as bip
from invariant_paged_prefill_gb300 import workloads as W

from gpu_helpers import assert_bitwise, run_gpu, to_device

pytestmark = pytest.mark.gpu


def test_wait_limit_expiry_reports_timeout_and_context_survives(cuda):
    b = to_device(W.layout([W.make_prompt(3000, *W.HEADS_A, seed=3)], [3000], 16), cuda)
    ref_o, ref_l, _ = run_gpu(b, cuda)
    plan = bip.Plan(b.qo_indptr, b.kv_indptr, b.kv_last_page_len, num_qo_heads=32, num_kv_heads=8, head_dim=128,
                    wait_limit_ns=1)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=cuda)
    bip.prefill(plan, b.q, b.k_pages, b.v_pages, b.kv_indices, workspace=ws)
    assert bip.read_device_status(ws) == 5  # BIP_ERR_DEVICE_TIMEOUT
    # the next ordinary call on the same workspace is fine and exact
    good = bip.Plan(b.qo_indptr, b.kv_indptr, b.kv_last_page_len, num_qo_heads=32, num_kv_heads=8, head_dim=128)
    out, lse = bip.prefill(good, b.q, b.k_pages, b.v_pages, b.kv_indices, workspace=ws)
    assert bip.read_device_status(ws) == 0
    assert_bitwise(out.cpu(), ref_o)
    assert_bitwise(lse.cpu(), ref_l)


def test_out_of_range_page_id_is_reported(cuda):
    b = to_device(W.layout([W.make_prompt(100, *W.HEADS_A, seed=4)], [10], 16), cuda)
    bad = b.kv_indices.clone()
    bad[2] = b.k_pages.shape[0] + 5
    plan = bip.Plan(b.qo_indptr, b.kv_indptr, b.kv_last_page_len, num_qo_heads=32, num_kv_heads=8, head_dim=128)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=cuda)
    bip.prefill(plan, b.q, b.k_pages, b.v_pages, bad, workspace=ws)
    assert bip.read_device_status(ws) == 7  # BIP_ERR_BAD_PAGE_INDEX
    bip.prefill(plan, b.q, b.k_pages, b.v_pages, b.kv_indices, workspace=ws)
    assert bip.read_device_status(ws) == 0
