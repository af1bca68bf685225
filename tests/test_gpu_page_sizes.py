"""Token-granular and small pages (page_size 1, 2, 4) on the GPU.

Below 8 slots a page is gathered row by row instead of landing as a TMA box;
the operand tiles in shared memory, and therefore every result bit, must not
depend on how the pool is paged.  Checked: parity with the oracle, bit
equality across page sizes 1 .. 64 for the same tokens, the extend rows equal
to the full prefill's rows, the device-planned launch, the KV append and
page-id checking at page size 1."""

import numpy as np
import pytest
import torch

import invariant_paged_prefill_gb300 as bip
from invariant_paged_prefill_gb300 import workloads as W
from oracle.kv_append import append_paged_kv

from gpu_helpers import assert_bitwise, assert_close_to_oracle, oracle, run_gpu, sample_rows, to_device

pytestmark = pytest.mark.gpu


def _mixed(page_size, heads=W.HEADS_A, kv_dtype="bf16", seed_pages=3):
    # a 3700-token prefill and four extends behind 500..3000-token prefixes
    specs = W.mixed_ragged_specs()
    prompts = [W.make_prompt(kv, *heads, seed=10 * i, kv_dtype=kv_dtype) for i, (_, kv) in enumerate(specs)]
    return prompts, W.layout(prompts, [ql for ql, _ in specs], page_size, seed_pages=seed_pages, kv_dtype=kv_dtype,
                             poison=True)


@pytest.mark.parametrize("page_size", [1, 2, 4])
@pytest.mark.parametrize("heads,kv_dtype", [(W.HEADS_A, "bf16"), (W.HEADS_B, "bf16"), (W.HEADS_A, "fp8_e4m3"),
                                            (W.HEADS_B, "fp8_e4m3")])
def test_small_pages_match_oracle(cuda, page_size, heads, kv_dtype):
    _, b = _mixed(page_size, heads, kv_dtype)
    out, lse, _ = run_gpu(b, cuda)
    rows = sample_rows(b, per_request=16, seed=page_size)
    ro, rl = oracle(b, rows=rows)
    assert_close_to_oracle(out, lse, ro, rl, rows=rows)


@pytest.mark.parametrize("heads,kv_dtype", [(W.HEADS_A, "bf16"), (W.HEADS_B, "bf16"), (W.HEADS_A, "fp8_e4m3")])
def test_results_do_not_depend_on_the_page_size(cuda, heads, kv_dtype):
    ref = None
    for ps in (16, 1, 2, 4, 8, 64):
        _, b = _mixed(ps, heads, kv_dtype, seed_pages=ps)
        o, l, _ = run_gpu(b, cuda)
        if ref is None:
            ref = (o, l)
        else:
            assert_bitwise(o, ref[0], f"page size {ps} out")
            assert_bitwise(l, ref[1], f"page size {ps} lse")


def test_page_one_strided_pool_and_split_policies(cuda):
    specs = W.mixed_ragged_specs()
    prompts = [W.make_prompt(kv, *W.HEADS_A, seed=10 * i) for i, (_, kv) in enumerate(specs)]
    b = W.layout(prompts, [ql for ql, _ in specs], 1, seed_pages=5, poison=True, page_stride_pad=64)
    ref_o, ref_l, _ = run_gpu(b, cuda, policy="never")
    for kw in (dict(policy="always"), dict(tiles_per_unit=1), dict(window_left=900)):
        o, l, _ = run_gpu(b, cuda, **kw)
        if "window_left" in kw:
            rows = sample_rows(b, per_request=12, seed=1)
            ro, rl = oracle(b, rows=rows, window_left=900)
            assert_close_to_oracle(o, l, ro, rl, rows=rows)
        else:
            assert_bitwise(o, ref_o, f"page 1 {kw}")
            assert_bitwise(l, ref_l, f"page 1 {kw} lse")


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_page_one_radix_hit_equals_full_prefill(cuda, kv_dtype):
    # token-granular pools: the shared prefix (777 tokens) ends mid-block
    ext, cold = W.radix_burst(n_req=8, prefix=777, kv_dtype=kv_dtype, page_size=1)
    eo, el, _ = run_gpu(ext, cuda)
    co, cl, _ = run_gpu(cold, cuda)
    for r in range(len(ext.q_lens)):
        e0, c0 = int(ext.qo_indptr[r]), int(cold.qo_indptr[r])
        off = ext.kv_lens[r] - ext.q_lens[r]
        n = ext.q_lens[r]
        assert_bitwise(eo[e0:e0 + n], co[c0 + off:c0 + off + n], f"request {r} out")
        assert_bitwise(el[e0:e0 + n], cl[c0 + off:c0 + off + n], f"request {r} lse")
    ro, rl = oracle(ext)
    assert_close_to_oracle(eo, el, ro, rl)


def test_page_one_device_planned_launch_equals_host_planned(cuda):
    _, b = _mixed(1)
    d = to_device(b, cuda)
    want_o, want_l, _ = run_gpu(d, cuda)
    gp = bip.GraphPlan(8, b.q.shape[0] + 50, num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=1)
    i32 = dict(dtype=torch.int32, device=cuda)
    n = len(b.q_lens)
    qo = torch.full((9,), int(b.qo_indptr[-1]), **i32)
    kv = torch.full((9,), int(b.kv_indptr[-1]), **i32)
    last = torch.ones(8, **i32)
    qo[: n + 1] = torch.as_tensor(b.qo_indptr, dtype=torch.int32)
    kv[: n + 1] = torch.as_tensor(b.kv_indptr, dtype=torch.int32)
    last[:n] = torch.as_tensor(b.kv_last_page_len, dtype=torch.int32)
    q = torch.zeros(b.q.shape[0] + 50, 32, 128, dtype=torch.bfloat16, device=cuda)
    q[: b.q.shape[0]] = d.q
    out = torch.full_like(q, float("nan"))
    lse = torch.full((q.shape[0], 32), float("nan"), dtype=torch.float32, device=cuda)
    ws = torch.empty(gp.workspace_bytes, dtype=torch.uint8, device=cuda)
    bip.prefill_graph(gp, 8, qo, kv, last, q, d.k_pages, d.v_pages, d.kv_indices, out, lse, ws)
    assert bip.read_device_status(ws) == 0
    m = b.q.shape[0]
    assert_bitwise(out[:m].cpu(), want_o, "graph page 1 out")
    assert_bitwise(lse[:m].cpu(), want_l, "graph page 1 lse")


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_page_one_append_writes_exactly_the_oracle_pools(cuda, kv_dtype):
    prompts = [W.make_prompt(n, *W.HEADS_A, seed=60 + i, kv_dtype=kv_dtype) for i, n in enumerate((90, 33, 7))]
    b = W.layout(prompts, [41, 0, 7], 1, seed_pages=4, kv_dtype=kv_dtype, poison=True)
    g = torch.Generator().manual_seed(11)
    shape = (int(b.qo_indptr[-1]), 8, 128)
    k_new = torch.randn(shape, generator=g).to(torch.bfloat16)
    v_new = torch.randn(shape, generator=g).to(torch.bfloat16)
    scales = (0.5, 2.0) if kv_dtype == "fp8_e4m3" else (1.0, 1.0)
    d = to_device(b, cuda)
    plan = bip.Plan(d.qo_indptr, d.kv_indptr, d.kv_last_page_len, num_qo_heads=32, num_kv_heads=8, head_dim=128,
                    page_size=1, kv_dtype=kv_dtype)
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device=cuda)
    bip.append_kv(plan, k_new.to(cuda), v_new.to(cuda), d.k_pages, d.v_pages, d.kv_indices, workspace=ws,
                  k_scale=scales[0], v_scale=scales[1])
    assert bip.read_device_status(ws) == 0

    def bits(t):
        t = t.cpu()
        return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()

    kind = "bf16" if kv_dtype == "bf16" else "fp8"
    kw, vw = append_paged_kv(bits(k_new), bits(v_new), bits(b.k_pages), bits(b.v_pages), b.qo_indptr.tolist(),
                             b.kv_indptr.tolist(), b.kv_indices.tolist(), b.kv_last_page_len.tolist(), 1, kind,
                             *scales)
    assert np.array_equal(bits(d.k_pages), kw) and np.array_equal(bits(d.v_pages), vw)


def test_page_one_out_of_range_page_id_is_reported(cuda):
    b = to_device(W.layout([W.make_prompt(100, *W.HEADS_A, seed=4)], [10], 1), cuda)
    bad = b.kv_indices.clone()
    bad[37] = b.k_pages.shape[0] + 5
    plan = bip.Plan(b.qo_indptr, b.kv_indptr, b.kv_last_page_len, num_qo_heads=32, num_kv_heads=8, head_dim=128,
                    page_size=1)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=cuda)
    bip.prefill(plan, b.q, b.k_pages, b.v_pages, bad, workspace=ws)
    assert bip.read_device_status(ws) == 7  # BIP_ERR_BAD_PAGE_INDEX
    assert int(ws[8:12].view(torch.int32).item()) >= 1  # counted
    out, lse = bip.prefill(plan, b.q, b.k_pages, b.v_pages, b.kv_indices, workspace=ws)
    assert bip.read_device_status(ws) == 0
    want_o, want_l, _ = run_gpu(b, cuda)
    assert_bitwise(out.cpu(), want_o)
    assert_bitwise(lse.cpu(), want_l)
