"""Bit-exactness of the CUDA path (torch.equal, max |diff| == 0.0, no NaN).

Each test checks that what it compares really differs in the way it claims
(q_len < kv_len, different batch make-up, different plans), so a pass is
never vacuous.
"""

import numpy as np
import pytest
import torch

from invariant_paged_prefill_gb300 import workloads as W

from gpu_helpers import assert_bitwise, run_gpu, to_device

pytestmark = pytest.mark.gpu


def test_radix_burst_extend_equals_cold_prefill(cuda):
    ext, cold = W.radix_burst()
    eo, el, ep = run_gpu(ext, cuda)
    co, cl, cp = run_gpu(cold, cuda)
    assert ep.info["num_units"] != cp.info["num_units"]
    for r in range(ext.batch):
        e0, e1 = ext.row_range(r)
        c0, c1 = cold.row_range(r)
        assert e1 - e0 < c1 - c0
        assert_bitwise(eo[e0:e1], co[c1 - (e1 - e0):c1], f"request {r} out")
        assert_bitwise(el[e0:e1], cl[c1 - (e1 - e0):c1], f"request {r} lse")


def test_mixed_ragged_batch_vs_alone_vs_full(cuda):
    prompts, q_lens = W.mixed_ragged_prompts()
    batch = W.layout(prompts, q_lens, 16, seed_pages=1)
    bo, bl, _ = run_gpu(batch, cuda)
    for r, (p, ql) in enumerate(zip(prompts, q_lens)):
        r0, r1 = batch.row_range(r)
        alone = W.layout([p], [ql], 16, seed_pages=11 + r)
        ao, al, _ = run_gpu(alone, cuda)
        assert_bitwise(bo[r0:r1], ao, f"request {r} batch vs alone")
        assert_bitwise(bl[r0:r1], al, f"request {r} lse batch vs alone")
        full = W.layout([p], [p.n], 16, seed_pages=21 + r)
        fo, fl, _ = run_gpu(full, cuda)
        assert_bitwise(ao, fo[p.n - ql:], f"request {r} extend vs full")
        assert_bitwise(al, fl[p.n - ql:], f"request {r} lse extend vs full")


def test_batch_mates_do_not_change_a_request(cuda):
    # A 512-token request alone versus beside 63 one-row batch-mates.
    hq, hkv, d = W.HEADS_A
    main = W.make_prompt(512, hq, hkv, d, seed=77)
    mates = [W.make_prompt(int(n), hq, hkv, d, seed=100 + i)
             for i, n in enumerate(np.random.default_rng(5).integers(1, 700, size=63))]
    alone = W.layout([main], [512], 16)
    crowd = W.layout([main] + mates, [512] + [1] * 63, 16, seed_pages=9)
    ao, al, _ = run_gpu(alone, cuda)
    co, cl, _ = run_gpu(crowd, cuda)
    assert_bitwise(ao, co[:512], "512-token request alone vs with 63 mates")
    assert_bitwise(al, cl[:512])


@pytest.mark.parametrize("heads", [W.HEADS_A, W.HEADS_B])
def test_split_fold_auto_identical(cuda, heads):
    hq, hkv, d = heads
    prompts = [W.make_prompt(9000, hq, hkv, d, seed=1), W.make_prompt(13000, hq, hkv, d, seed=2)]
    b = W.layout(prompts, [300, 47], 16)
    runs = {pol: run_gpu(b, cuda, policy=pol, num_sms=sms)
            for pol, sms in (("never", 0), ("always", 0), ("auto", 4))}
    assert runs["always"][2].info["num_split_units"] > 0
    assert runs["never"][2].info["num_split_units"] == 0
    for pol in ("always", "auto"):
        assert_bitwise(runs[pol][0], runs["never"][0], f"out {pol} vs never")
        assert_bitwise(runs[pol][1], runs["never"][1], f"lse {pol} vs never")


def test_repeated_runs_identical(cuda):
    b = W.layout([W.make_prompt(n, *W.HEADS_A, seed=n) for n in (1500, 37, 600)], [1500, 9, 600], 16)
    o1, l1, _ = run_gpu(b, cuda)
    o2, l2, _ = run_gpu(b, cuda)
    assert_bitwise(o1, o2)
    assert_bitwise(l1, l2)


def test_page_permutation_and_stride_invariance(cuda):
    p = W.make_prompt(777, *W.HEADS_A, seed=8)
    a = W.layout([p], [100], 16, seed_pages=1)
    b = W.layout([p], [100], 16, seed_pages=2, extra_pages=40)
    c = W.layout([p], [100], 16, seed_pages=3, page_stride_pad=64)
    assert not torch.equal(a.kv_indices, b.kv_indices)
    ao, al, _ = run_gpu(a, cuda)
    for other in (b, c):
        oo, ol, _ = run_gpu(other, cuda)
        assert_bitwise(ao, oo)
        assert_bitwise(al, ol)


def test_chunked_prefill_rows_equal_full_prefill(cuda):
    hq, hkv, d = W.HEADS_A
    p = W.make_prompt(1000, hq, hkv, d, seed=12)
    fo, fl, _ = run_gpu(W.layout([p], [1000], 16), cuda)
    for a, b in [(0, 1), (1, 77), (77, 300), (300, 301), (301, 1000)]:
        chunk = W.Prompt(p.q[:b], p.k[:b], p.v[:b])
        co, cl, _ = run_gpu(W.layout([chunk], [b - a], 16, seed_pages=b), cuda)
        assert_bitwise(co, fo[a:b], f"chunk [{a},{b})")
        assert_bitwise(cl, fl[a:b])


def test_nan_in_neighbour_rows_and_unused_slots_does_not_leak(cuda):
    hq, hkv, d = W.HEADS_A
    prompts = [W.make_prompt(n, hq, hkv, d, seed=50 + n) for n in (45, 300, 61)]
    clean = W.layout(prompts, [5, 300, 2], 16)
    dirty = W.layout(prompts, [5, 300, 2], 16)
    # rows of requests 0 and 2 sit in the same q tiles' neighbourhood of request 1
    dirty.q[0:5] = float("nan")
    dirty.q[305:307] = float("nan")
    co, cl, _ = run_gpu(clean, cuda)
    do, dl, _ = run_gpu(dirty, cuda, check_status=True)
    assert_bitwise(co[5:305], do[5:305], "request 1 beside NaN rows")
    assert_bitwise(cl[5:305], dl[5:305])
    # the pools are NaN-poisoned outside each request's kv_len, and no output is NaN
    assert not torch.isnan(co).any()


def test_zero_length_requests_and_single_token(cuda):
    hq, hkv, d = W.HEADS_A
    prompts = [W.make_prompt(n, hq, hkv, d, seed=n) for n in (20, 1, 33, 16)]
    b = W.layout(prompts, [0, 1, 0, 16], 16)
    o, l, plan = run_gpu(b, cuda)
    assert o.shape[0] == 17
    alone = W.layout([prompts[3]], [16], 16, seed_pages=4)
    ao, al, _ = run_gpu(alone, cuda)
    assert_bitwise(o[1:], ao)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_one_and_two_tiles_per_cta_identical(cuda, kv_dtype):
    # The memory-bound variant (one q tile per CTA, deeper KV ring) and the
    # ping-pong variant (two tiles per CTA) must give the same bits, with
    # bf16 and with E4M3 pages.
    hq, hkv, d = W.HEADS_A
    prompts = [W.make_prompt(n, hq, hkv, d, seed=60 + i, kv_dtype=kv_dtype) for i, n in enumerate((5000, 300, 4100, 77))]
    b = W.layout(prompts, [5000, 3, 900, 40], 16, kv_dtype=kv_dtype)
    r1 = run_gpu(b, cuda, tiles_per_unit=1)
    r2 = run_gpu(b, cuda, tiles_per_unit=2)
    assert r1[2].info["tiles_per_unit"] == 1 and r2[2].info["tiles_per_unit"] == 2
    assert_bitwise(r1[0], r2[0], "out 1 vs 2 tiles per CTA")
    assert_bitwise(r1[1], r2[1], "lse 1 vs 2 tiles per CTA")
    r3 = run_gpu(b, cuda, tiles_per_unit=2, policy="always")
    assert_bitwise(r3[0], r2[0], "out split vs fold, 2 tiles")


def test_fp8_extend_equals_full_and_split_equals_fold(cuda):
    hq, hkv, d = W.HEADS_A
    p = W.make_prompt(9000, hq, hkv, d, seed=70, kv_dtype="fp8_e4m3")
    full = W.layout([p], [9000], 16, kv_dtype="fp8_e4m3")
    ext = W.layout([p], [37], 16, seed_pages=4, kv_dtype="fp8_e4m3")
    fo, fl, _ = run_gpu(full, cuda)
    eo, el, _ = run_gpu(ext, cuda, policy="never")
    so, sl, sp = run_gpu(ext, cuda, policy="always")
    assert sp.info["num_split_units"] > 0
    assert_bitwise(eo, fo[9000 - 37:], "fp8 extend vs full")
    assert_bitwise(el, fl[9000 - 37:])
    assert_bitwise(so, eo, "fp8 split vs fold")
    assert_bitwise(sl, el)
