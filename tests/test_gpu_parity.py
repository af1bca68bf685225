"""CUDA path against the float64 oracle, element by element (tolerance 2e-2 abs + 1e-2 rel).

Sizes span several q tiles, KV blocks, segments and ragged tails; full-size
workloads are checked on sampled rows that the oracle computes one by one.
"""

import numpy as np
import pytest
import torch

import invariant_paged_prefill_gb300 as bip
from invariant_paged_prefill_gb300 import workloads as W

from gpu_helpers import assert_bitwise, assert_close_to_oracle, oracle, run_gpu, sample_rows, to_device

pytestmark = pytest.mark.gpu


def test_tiny_full_and_extend_match_oracle_and_each_other(cuda):
    full, ext = W.tiny(64), W.tiny(3)
    fo, fl, _ = run_gpu(full, cuda)
    eo, el, _ = run_gpu(ext, cuda)
    ro, rl = oracle(full)
    assert_close_to_oracle(fo, fl, ro, rl)
    ro3, rl3 = oracle(ext)
    assert_close_to_oracle(eo, el, ro3, rl3)
    assert ext.q_lens[0] < ext.kv_lens[0]   # a real extend, not a vacuous one
    assert_bitwise(eo, fo[61:64], "extend out vs full rows 61..63")
    assert_bitwise(el, fl[61:64], "extend lse vs full rows 61..63")


@pytest.mark.parametrize("heads", [W.HEADS_A, W.HEADS_B, (8, 8, 128), (16, 1, 128), (12, 2, 256)])
@pytest.mark.parametrize("lens", [[(70, 70)], [(5, 300), (133, 133), (1, 1), (0, 17), (40, 290)]])
def test_small_batches_match_oracle(cuda, heads, lens):
    hq, hkv, d = heads
    prompts = [W.make_prompt(kv, hq, hkv, d, seed=31 + i) for i, (_, kv) in enumerate(lens)]
    b = W.layout(prompts, [q for q, _ in lens], 16, seed_pages=5)
    o, l, plan = run_gpu(b, cuda)
    ro, rl = oracle(b)
    assert_close_to_oracle(o, l, ro, rl)


@pytest.mark.parametrize("policy", ["never", "always"])
@pytest.mark.parametrize("heads", [W.HEADS_A, W.HEADS_B])
def test_multi_segment_rows_match_oracle(cuda, heads, policy):
    # kv 9000 > 2 segments of 4096; tile rows straddle a segment boundary for group 6
    hq, hkv, d = heads
    prompts = [W.make_prompt(9000, hq, hkv, d, seed=3), W.make_prompt(4200, hq, hkv, d, seed=4)]
    b = W.layout(prompts, [200, 150], 16, seed_pages=2)
    o, l, plan = run_gpu(b, cuda, policy=policy)
    if policy == "always":
        assert plan.info["num_split_units"] > 0
    ro, rl = oracle(b)
    assert_close_to_oracle(o, l, ro, rl)


def test_radix_burst_sampled_rows_match_oracle(cuda):
    ext, cold = W.radix_burst()
    eo, el, _ = run_gpu(ext, cuda)
    ro, rl = oracle(ext)
    assert_close_to_oracle(eo, el, ro, rl)
    co, cl, _ = run_gpu(cold, cuda)
    rows = sample_rows(cold, per_request=8)
    ro, rl = oracle(cold, rows=rows)
    assert_close_to_oracle(co, cl, ro, rl, rows=rows)


@pytest.mark.parametrize("n", [8192, 32768])
def test_large_head_prefill_sampled_rows(cuda, n):
    b = W.large_head(n, device=cuda)
    o, l, plan = run_gpu(b, cuda)
    assert plan.workspace_bytes <= bip.workspace_bound(1, n, 24, 4, 256)
    assert plan.workspace_bytes < 2 ** 31 // 64
    rows = sample_rows(b, per_request=12)
    ro, rl = oracle(b, rows=rows)
    assert_close_to_oracle(o, l, ro, rl, rows=rows)


def test_sweep_point_short_extend_long_kv(cuda):
    b = W.sweep_point(W.HEADS_A, 4, 32768, batch=4, device=cuda)
    o, l, plan = run_gpu(b, cuda)
    rows = sample_rows(b, per_request=4)
    ro, rl = oracle(b, rows=rows)
    assert_close_to_oracle(o, l, ro, rl, rows=rows)


@pytest.mark.parametrize("heads", [W.HEADS_A, W.HEADS_B])
def test_fp8_pages_match_oracle(cuda, heads):
    # E4M3 pages (N(0,1) clipped to +-448); the oracle decodes the stored codes itself.
    hq, hkv, d = heads
    lens = [(5, 300), (133, 133), (1, 1), (40, 4500)]
    prompts = [W.make_prompt(kv, hq, hkv, d, seed=41 + i, kv_dtype="fp8_e4m3") for i, (_, kv) in enumerate(lens)]
    b = W.layout(prompts, [q for q, _ in lens], 16, seed_pages=6, kv_dtype="fp8_e4m3")
    o, l, plan = run_gpu(b, cuda)
    assert plan.info["kv_dtype"] == 1
    ro, rl = oracle(b)
    assert_close_to_oracle(o, l, ro, rl)


def test_fp8_scales_match_oracle(cuda):
    # K scale multiplies the logits, V scale the output.
    from oracle import paged_attention as pa
    hq, hkv, d = W.HEADS_A
    prompts = [W.make_prompt(n, hq, hkv, d, seed=90 + n, kv_dtype="fp8_e4m3") for n in (70, 200)]
    b = W.layout(prompts, [70, 9], 16, kv_dtype="fp8_e4m3")
    o, l, _ = run_gpu(b, cuda, k_scale=0.5, v_scale=2.0)
    ro, rl = pa.paged_prefill(b.q.view(torch.int16).numpy(), b.k_pages.numpy(), b.v_pages.numpy(),
                              b.qo_indptr.tolist(), b.kv_indptr.tolist(), b.kv_indices.tolist(),
                              b.kv_last_page_len.tolist(), hq, hkv, 16, q_kind="bf16", kv_kind="e4m3",
                              k_scale=0.5, v_scale=2.0)
    assert_close_to_oracle(o, l, ro, rl)
