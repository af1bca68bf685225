"""Sliding-window attention (each row sees keys position - W .. position) on the
GPU: parity with the oracle, and every bit-exactness property of the plain
causal path, under the window."""

import pytest
import torch

import invariant_paged_prefill_gb300 as bip
from invariant_paged_prefill_gb300 import workloads as W

from gpu_helpers import assert_bitwise, assert_close_to_oracle, oracle, run_gpu, sample_rows, to_device

pytestmark = pytest.mark.gpu


def _batch(heads, kv_dtype="bf16"):
    # a fresh prefill across two segments, extends behind long and short
    # prefixes, a request shorter than the window
    prompts = [W.make_prompt(n, *heads, seed=90 + i, kv_dtype=kv_dtype) for i, n in enumerate((5000, 4700, 1300, 60))]
    return W.layout(prompts, [5000, 37, 3, 60], 16, seed_pages=9, kv_dtype=kv_dtype, poison=True)


@pytest.mark.parametrize("window", [100, 1000, 4095, 4500])
def test_window_matches_oracle(cuda, window):
    b = _batch(W.HEADS_A)
    out, lse, _ = run_gpu(b, cuda, window_left=window)
    rows = sample_rows(b, per_request=16, seed=window)
    ro, rl = oracle(b, rows=rows, window_left=window)
    assert_close_to_oracle(out, lse, ro, rl, rows=rows)


@pytest.mark.parametrize("heads,kv_dtype", [(W.HEADS_B, "bf16"), (W.HEADS_A, "fp8_e4m3"), (W.HEADS_B, "fp8_e4m3")])
def test_window_matches_oracle_other_variants(cuda, heads, kv_dtype):
    b = _batch(heads, kv_dtype)
    out, lse, _ = run_gpu(b, cuda, window_left=700)
    rows = sample_rows(b, per_request=12, seed=3)
    ro, rl = oracle(b, rows=rows, window_left=700)
    assert_close_to_oracle(out, lse, ro, rl, rows=rows)


@pytest.mark.parametrize("window", [64, 777, 4096])
def test_window_extend_equals_full_prefill(cuda, window):
    # the extend rows of each prompt equal the same rows of its full prefill
    prompts = [W.make_prompt(n, *W.HEADS_A, seed=120 + i) for i, n in enumerate((4300, 900, 6100))]
    full = W.layout(prompts, [p.n for p in prompts], 16, seed_pages=2, poison=True)
    ext = W.layout(prompts, [5, 300, 1], 16, seed_pages=5, poison=True)
    fo, fl, _ = run_gpu(full, cuda, window_left=window)
    eo, el, _ = run_gpu(ext, cuda, window_left=window)
    for r in range(3):
        f0, e0 = int(full.qo_indptr[r]), int(ext.qo_indptr[r])
        n, off = ext.q_lens[r], full.q_lens[r] - ext.q_lens[r]
        assert_bitwise(eo[e0:e0 + n], fo[f0 + off:f0 + off + n], f"request {r} out")
        assert_bitwise(el[e0:e0 + n], fl[f0 + off:f0 + off + n], f"request {r} lse")


def test_window_split_fold_tiles_and_long_window_are_neutral(cuda):
    b = _batch(W.HEADS_A)
    ref_o, ref_l, _ = run_gpu(b, cuda, window_left=1500, policy="never")
    for kw in (dict(policy="always"), dict(policy="auto"), dict(tiles_per_unit=1), dict(tiles_per_unit=2)):
        o, l, _ = run_gpu(b, cuda, window_left=1500, **kw)
        assert_bitwise(o, ref_o, f"window 1500 {kw}")
        assert_bitwise(l, ref_l, f"window 1500 {kw} lse")
    # a window at least as long as every sequence is plain causal attention
    o, l, _ = run_gpu(b, cuda, window_left=5000)
    co, cl, _ = run_gpu(b, cuda)
    assert_bitwise(o, co, "window 5000 vs none")
    assert_bitwise(l, cl, "window 5000 vs none lse")


def test_window_skips_keys_outside(cuda):
    # the plan visits fewer KV blocks, and the graph-replayable launch agrees
    b = to_device(_batch(W.HEADS_A), cuda)
    plain = bip.Plan(b.qo_indptr, b.kv_indptr, b.kv_last_page_len, num_qo_heads=32, num_kv_heads=8, head_dim=128)
    win = bip.Plan(b.qo_indptr, b.kv_indptr, b.kv_last_page_len, num_qo_heads=32, num_kv_heads=8, head_dim=128,
                   window_left=256)
    assert win.info["kv_blocks"] < plain.info["kv_blocks"] / 4
    want_o, want_l, _ = run_gpu(b, cuda, window_left=256)
    gp = bip.GraphPlan(8, b.q.shape[0], num_qo_heads=32, num_kv_heads=8, head_dim=128, window_left=256)
    i32 = dict(dtype=torch.int32, device=cuda)
    n = len(b.q_lens)
    qo = torch.full((9,), int(b.qo_indptr[-1]), **i32)
    kv = torch.full((9,), int(b.kv_indptr[-1]), **i32)
    last = torch.ones(8, **i32)
    qo[: n + 1] = torch.as_tensor(b.qo_indptr, dtype=torch.int32)
    kv[: n + 1] = torch.as_tensor(b.kv_indptr, dtype=torch.int32)
    last[:n] = torch.as_tensor(b.kv_last_page_len, dtype=torch.int32)
    out = torch.empty_like(b.q)
    lse = torch.empty(b.q.shape[0], 32, dtype=torch.float32, device=cuda)
    ws = torch.empty(gp.workspace_bytes, dtype=torch.uint8, device=cuda)
    bip.prefill_graph(gp, 8, qo, kv, last, b.q, b.k_pages, b.v_pages, b.kv_indices, out, lse, ws)
    assert bip.read_device_status(ws) == 0
    assert_bitwise(out.cpu(), want_o, "graph window out")
    assert_bitwise(lse.cpu(), want_l, "graph window lse")
