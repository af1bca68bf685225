"""The C ABI on the host (no GPU): exports, validation, workspace bound, schedule.

The planner is host-only, so everything here runs through libbip.so on a
machine without a GPU.
"""

import ctypes
import os
import re

import numpy as np
import pytest

import invariant_paged_prefill_gb300 as bip
from invariant_paged_prefill_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "bip.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bip_[a-z_0-9]+)\s*\(", text)))


def test_library_exports_every_declared_function(lib):
    names = declared_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(_lib.SIGNATURES), "binding and header disagree"


def test_status_strings(lib):
    for code, name in bip.STATUS.items():
        assert lib.bip_status_string(code).decode() == name


def plan_code(qo, kv, last, hq=32, hkv=8, d=128, ps=16, kv_dtype=0, opts=None):
    lib = _lib.load()
    h = ctypes.c_void_p()
    a = [np.ascontiguousarray(np.asarray(x, dtype=np.int32)) for x in (qo, kv, last)]
    ptrs = [x.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)) for x in a]
    ws = ctypes.c_size_t()
    rc = lib.bip_plan(ctypes.byref(h), ptrs[0], ptrs[1], ptrs[2], len(a[0]) - 1, hq, hkv, d, ps, kv_dtype,
                      opts, ctypes.byref(ws))
    if rc == 0:
        lib.bip_plan_destroy(h)
    return rc


@pytest.mark.parametrize("case,code", [
    (dict(qo=[0, 5], kv=[0, 1], last=[4]), 1),            # q_len 5 > kv_len 4
    (dict(qo=[0, 2, 1], kv=[0, 1, 2], last=[3, 3]), 1),   # decreasing qo_indptr
    (dict(qo=[1, 2], kv=[0, 1], last=[3]), 1),            # qo_indptr[0] != 0
    (dict(qo=[0, 1], kv=[0, 1], last=[17]), 1),           # last page overfull
    (dict(qo=[0, 1], kv=[0, 1], last=[0]), 1),            # empty last page
    (dict(qo=[0, 1], kv=[0, 1], last=[4], hq=30), 1),     # heads do not divide
    (dict(qo=[0, 1], kv=[0, 1], last=[4], d=64), 2),      # unsupported head_dim
    (dict(qo=[0, 1], kv=[0, 1], last=[4], ps=12), 2),     # page size not a power of two
    (dict(qo=[0, 1], kv=[0, 1], last=[3], ps=3), 2),      # nor below 8
    (dict(qo=[0, 1], kv=[0, 1], last=[4], ps=256), 2),    # page longer than a KV block
    (dict(qo=[0, 3], kv=[0, 3], last=[1], ps=1), 0),      # token-granular pool
    (dict(qo=[0, 3], kv=[0, 2], last=[2], ps=2), 0),
    (dict(qo=[0, 3], kv=[0, 1], last=[4], ps=4), 0),
    (dict(qo=[0, 1], kv=[0, 1], last=[2], ps=1), 1),      # last page overfull at page size 1
    (dict(qo=[0, 1], kv=[0, 1], last=[4], hkv=4, d=256, ps=64), 0),
    (dict(qo=[0, 1], kv=[0, 1], last=[4], hkv=4, d=256, ps=128), 2),  # d 256 runs 64-key blocks
    (dict(qo=[0, 1], kv=[0, 1], last=[4], kv_dtype=1), 0),  # FP8 E4M3 pages
    (dict(qo=[0, 1], kv=[0, 1], last=[4], kv_dtype=9), 1),
    (dict(qo=[0, 0, 3], kv=[0, 0, 1], last=[0, 3]), 0),   # zero-length request with no pages
    (dict(qo=[0, 0, 3], kv=[0, 2, 3], last=[16, 3]), 0),  # zero-length request behind a prefix
])
def test_plan_validation(lib, case, code):
    assert plan_code(**case) == code


def test_prefill_rejects_before_touching_memory(lib):
    plan = bip.Plan([0, 3], [0, 1], [5], num_qo_heads=32, num_kv_heads=8, head_dim=128)
    fake = ctypes.c_void_p(1 << 20)
    # q row count disagreeing with qo_indptr[-1] (the wrapper's shape check)
    rc = lib.bip_prefill(plan._h, fake, 4, fake, fake, 1, 16 * 8 * 128, fake, 1.0, 1.0, fake, fake, fake,
                         plan.workspace_bytes, None)
    assert rc == 1
    # too-small workspace
    rc = lib.bip_prefill(plan._h, fake, 3, fake, fake, 1, 16 * 8 * 128, fake, 1.0, 1.0, fake, fake, fake,
                         plan.workspace_bytes - 1, None)
    assert rc == 3
    # misaligned q
    rc = lib.bip_prefill(plan._h, ctypes.c_void_p((1 << 20) + 2), 3, fake, fake, 1, 16 * 8 * 128, fake, 1.0, 1.0,
                         fake, fake, fake, plan.workspace_bytes, None)
    assert rc == 1
    # page stride smaller than a page
    rc = lib.bip_prefill(plan._h, fake, 3, fake, fake, 1, 16 * 8 * 128 - 8, fake, 1.0, 1.0, fake, fake, fake,
                         plan.workspace_bytes, None)
    assert rc == 1
    # token-granular pools gather rows with 32-bit page offsets: a page stride
    # of 2^31 bytes or more is refused (before any launch)
    tok = bip.Plan([0, 3], [0, 3], [1], num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=1)
    rc = lib.bip_prefill(tok._h, fake, 3, fake, fake, 1, 1 << 30, fake, 1.0, 1.0, fake, fake, fake,
                         tok.workspace_bytes, None)
    assert rc == 2
    # scales must be finite
    for ks, vs in ((float("inf"), 1.0), (1.0, float("nan"))):
        rc = lib.bip_prefill(plan._h, fake, 3, fake, fake, 1, 16 * 8 * 128, fake, ks, vs, fake, fake, fake,
                             plan.workspace_bytes, None)
        assert rc == 1
    # a plan with only q_len = 0 requests has nothing to run
    empty = bip.Plan([0, 0], [0, 1], [5], num_qo_heads=32, num_kv_heads=8, head_dim=128)
    assert lib.bip_prefill(empty._h, None, 0, None, None, 0, 0, None, 1.0, 1.0, None, None, None, 0, None) == 0


def test_masked_prefill_rejects_before_touching_memory(lib):
    # kv_len 37 (pages 16, 16, 5): a mask row needs ceil(37 / 32) = 2 words
    plan = bip.Plan([0, 3], [0, 3], [5], num_qo_heads=32, num_kv_heads=8, head_dim=128)
    fake = ctypes.c_void_p(1 << 20)

    def call(mask, words):
        return lib.bip_prefill_masked(plan._h, fake, 3, fake, fake, 3, 16 * 8 * 128, fake, mask, words, 1.0, 1.0,
                                      fake, fake, fake, plan.workspace_bytes - 1, None)
    assert call(None, 2) == 1                                  # no mask
    assert call(ctypes.c_void_p((1 << 20) + 2), 2) == 1        # mask not 4-byte aligned
    assert call(fake, 1) == 1                                  # rows shorter than the longest kv_len
    assert call(fake, 2) == 3                                  # valid mask: on to the workspace check
    # the rule counts only requests with q rows: a long request without any
    # sets no minimum
    mixed = bip.Plan([0, 0, 2], [0, 40, 41], [16, 9], num_qo_heads=32, num_kv_heads=8, head_dim=128)
    rc = lib.bip_prefill_masked(mixed._h, fake, 2, fake, fake, 41, 16 * 8 * 128, fake, fake, 1, 1.0, 1.0, fake,
                                fake, fake, mixed.workspace_bytes - 1, None)
    assert rc == 3


def test_pack_mask_bit_layout():
    rng = np.random.default_rng(4)
    masks = [rng.random((3, 37)) < 0.5, rng.random((2, 70)) < 0.5, np.zeros((0, 5), dtype=bool)]
    words = bip.pack_mask(masks)
    assert words.dtype == np.int32 and words.shape == (5, 3)
    row = 0
    for m in masks:
        for i in range(m.shape[0]):
            for j in range(3 * 32):
                bit = (int(words[row, j // 32]) >> (j % 32)) & 1
                assert bit == (int(m[i, j]) if j < m.shape[1] else 0), (row, j)
            row += 1
    assert bip.pack_mask(masks, row_words=5).shape == (5, 5)
    assert np.array_equal(bip.pack_mask(masks, row_words=5)[:, :3], words)
    with pytest.raises(bip.BipError):
        bip.pack_mask(masks, row_words=2)


def test_append_rejects_before_touching_memory(lib):
    plan = bip.Plan([0, 3], [0, 1], [5], num_qo_heads=32, num_kv_heads=8, head_dim=128)
    fake = ctypes.c_void_p(1 << 20)
    args = lambda rows, stride=16 * 8 * 128, ks=1.0, vs=1.0, ws=plan.workspace_bytes, kn=fake: (
        plan._h, kn, fake, rows, fake, fake, 1, stride, fake, ks, vs, fake, ws, None)
    assert lib.bip_append_kv(*args(4)) == 1                      # row count != qo_indptr[-1]
    assert lib.bip_append_kv(*args(3, ks=0.5)) == 1              # bf16 pages take no scale
    assert lib.bip_append_kv(*args(3, stride=16 * 8 * 128 - 8)) == 1
    assert lib.bip_append_kv(*args(3, kn=ctypes.c_void_p((1 << 20) + 4))) == 1  # misaligned rows
    assert lib.bip_append_kv(*args(3, ws=64)) == 3               # workspace smaller than the upload
    f8 = bip.Plan([0, 3], [0, 1], [5], num_qo_heads=32, num_kv_heads=8, head_dim=128, kv_dtype="fp8_e4m3")
    for ks in (0.0, -1.0, float("inf"), float("nan")):
        assert lib.bip_append_kv(f8._h, fake, fake, 3, fake, fake, 1, 16 * 8 * 128, fake, ks, 1.0, fake,
                                 f8.workspace_bytes, None) == 1
    # nothing to append
    empty = bip.Plan([0, 0], [0, 1], [5], num_qo_heads=32, num_kv_heads=8, head_dim=128)
    assert lib.bip_append_kv(empty._h, None, None, 0, None, None, 0, 0, None, 1.0, 1.0, None, 0, None) == 0


def test_graph_plan_validation_and_sizes(lib):
    gp = bip.GraphPlan(8, 4096, num_qo_heads=32, num_kv_heads=8, head_dim=128)
    # the fixed workspace holds the worst-case work list and every CTA's fold state
    assert gp.workspace_bytes >= 256 + 8 * (4096 // 32 + 16) * 48
    fake = ctypes.c_void_p(1 << 20)
    args = lambda batch, ws=gp.workspace_bytes, q=fake: (gp._h, batch, fake, fake, fake, q, fake, fake, 1,
                                                         16 * 8 * 128, fake, 1.0, 1.0, fake, fake, fake, ws, None)
    assert lib.bip_prefill_graph(*args(9)) == 1                     # more requests than the capacity
    assert lib.bip_prefill_graph(*args(-1)) == 1
    assert lib.bip_prefill_graph(*args(8, ws=gp.workspace_bytes - 1)) == 3
    assert lib.bip_prefill_graph(*args(8, q=ctypes.c_void_p((1 << 20) + 2))) == 1
    with pytest.raises(bip.BipError):
        bip.GraphPlan(8, 4096, num_qo_heads=32, num_kv_heads=8, head_dim=96)
    # the masked launch takes the same checks, plus a non-null, 4-byte aligned mask of >= 1 word a row
    margs = lambda batch, mask=fake, words=4: (gp._h, batch, fake, fake, fake, fake, fake, fake, 1, 16 * 8 * 128,
                                               fake, mask, words, 1.0, 1.0, fake, fake, fake, gp.workspace_bytes,
                                               None)
    assert lib.bip_prefill_graph_masked(*margs(9)) == 1
    assert lib.bip_prefill_graph_masked(*margs(8, mask=None)) == 1
    assert lib.bip_prefill_graph_masked(*margs(8, mask=ctypes.c_void_p((1 << 20) + 2))) == 1
    assert lib.bip_prefill_graph_masked(*margs(8, words=0)) == 1
    # the split capacity follows the budget; NEVER reserves no partials
    never = bip.GraphPlan(8, 4096, num_qo_heads=32, num_kv_heads=8, head_dim=128, split_policy="never")
    small = bip.GraphPlan(8, 4096, num_qo_heads=32, num_kv_heads=8, head_dim=128, split_budget_bytes=1 << 20)
    assert never.workspace_bytes < small.workspace_bytes < gp.workspace_bytes
    assert gp.workspace_bytes - never.workspace_bytes >= 64 << 20
    opts = _lib.PlanOptions(2, 1 << 20, 0, 0, 0)   # BIP_SPLIT_ALWAYS: the batch decides on the device
    h = ctypes.c_void_p()
    assert lib.bip_graph_plan(ctypes.byref(h), 8, 4096, 32, 8, 128, 16, 0, ctypes.byref(opts), None) == 2
    opts = _lib.PlanOptions(0, 1 << 20, 0, 0, 2)   # FP8 pages have a two-tile variant at head_dim 128
    assert lib.bip_graph_plan(ctypes.byref(h), 8, 4096, 32, 8, 128, 16, 1, ctypes.byref(opts), None) == 0
    lib.bip_graph_plan_destroy(h)
    # so do token-granular pools (the row-gather warps take the second tile's room)
    assert lib.bip_graph_plan(ctypes.byref(h), 8, 4096, 32, 8, 128, 4, 0, ctypes.byref(opts), None) == 2
    assert lib.bip_graph_plan(ctypes.byref(h), 8, 4096, 32, 8, 128, 8, 0, ctypes.byref(opts), None) == 0
    lib.bip_graph_plan_destroy(h)


def test_token_granular_plans_run_one_tile_per_cta(lib):
    qo, kv, last = [0, 8192], [0, 8192], [1]   # one 8192-token fresh prefill, one slot a page
    p1 = bip.Plan(qo, kv, last, num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=1)
    p16 = bip.Plan(qo, [0, 512], [16], num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=16)
    assert p16.info["tiles_per_unit"] == 2 and p1.info["tiles_per_unit"] == 1
    assert plan_code(qo, kv, last, ps=1, opts=ctypes.byref(_lib.PlanOptions(0, 1 << 20, 0, 0, 2))) == 2
    assert plan_code(qo, kv, last, ps=1, opts=ctypes.byref(_lib.PlanOptions(0, 1 << 20, 0, 0, 1))) == 0


def test_window_plans_skip_keys_and_reject_negative_windows(lib):
    qo, kv, last = [0, 9000], [0, 563], [9000 - 16 * 562]  # one 9000-token fresh prefill
    plain = bip.Plan(qo, kv, last, num_qo_heads=32, num_kv_heads=8, head_dim=128, split_policy="never")
    win = bip.Plan(qo, kv, last, num_qo_heads=32, num_kv_heads=8, head_dim=128, split_policy="never",
                   window_left=1000)
    assert win.info["kv_blocks"] < plain.info["kv_blocks"] / 3
    items = win.items()
    # the last tile group's item starts in segment 1 (its rows see keys from ~8000 - 1000 on)
    assert items[:, 3].max() >= 1 and (items[:, 3] <= items[:, 4]).all()
    with pytest.raises(bip.BipError):
        bip.Plan(qo, kv, last, num_qo_heads=32, num_kv_heads=8, head_dim=128, window_left=-1)


def random_batch(rng, batch, max_kv, ps=16):
    kv_len = rng.integers(1, max_kv + 1, size=batch)
    q_len = np.minimum(kv_len, rng.integers(0, max_kv + 1, size=batch))
    npages = (kv_len + ps - 1) // ps
    qo = np.concatenate([[0], np.cumsum(q_len)])
    kv = np.concatenate([[0], np.cumsum(npages)])
    last = kv_len - (npages - 1) * ps
    return qo, kv, last


@pytest.mark.parametrize("heads", [(32, 8, 128), (24, 4, 256), (8, 8, 128), (16, 1, 256)])
def test_workspace_never_exceeds_bound(lib, heads):
    rng = np.random.default_rng(sum(heads))
    hq, hkv, d = heads
    for trial in range(25):
        batch = int(rng.integers(1, 12))
        qo, kv, last = random_batch(rng, batch, int(rng.choice([40, 900, 9000, 20000])))
        for policy in ("auto", "always", "never"):
            budget = int(rng.choice([0, 1 << 20, 64 << 20]))
            p = bip.Plan(qo, kv, last, num_qo_heads=hq, num_kv_heads=hkv, head_dim=d, split_policy=policy,
                         split_budget_bytes=budget, num_sms=int(rng.integers(1, 200)))
            bound = bip.workspace_bound(batch, int(qo[-1]), hq, hkv, d, budget)
            assert p.workspace_bytes <= bound
            assert p.info["partial_bytes"] <= budget


def test_large_head_workspace_is_small():
    # The pages' failure: one 8192-token 24/4/256 prefill needed 2,415,919,104
    # bytes of split buffers and overflowed a fixed 2 GiB workspace.
    for n in (8192, 32768):
        pages = n // 16
        p = bip.Plan([0, n], [0, pages], [16], num_qo_heads=24, num_kv_heads=4, head_dim=256)
        assert p.workspace_bytes < 64 << 20
        assert p.workspace_bytes <= bip.workspace_bound(1, n, 24, 4, 256)


def unit_geometry(plan, request):
    """(kv_head, q tile) pairs and item geometry of one request."""
    it = plan.items()
    mine = it[it[:, 0] == request]
    tiles = {(int(r[1]), int(r[2]) + t) for r in mine for t in range(2) if r[7] >> t & 1}
    return sorted(tiles), sorted(tuple(int(x) for x in list(r[1:6]) + [r[7]]) for r in mine)


def test_schedule_of_a_request_does_not_depend_on_its_batch_mates(lib):
    rng = np.random.default_rng(7)
    for trial in range(20):
        batch = int(rng.integers(2, 9))
        qo, kv, last = random_batch(rng, batch, 9000)
        together = bip.Plan(qo, kv, last, num_qo_heads=32, num_kv_heads=8, head_dim=128, split_policy="never")
        for r in range(batch):
            ql, np_ = qo[r + 1] - qo[r], kv[r + 1] - kv[r]
            alone = bip.Plan([0, ql], [0, np_], [last[r]], num_qo_heads=32, num_kv_heads=8, head_dim=128,
                             split_policy="never")
            t_units, t_items = unit_geometry(together, r)
            a_units, a_items = unit_geometry(alone, 0)
            assert t_units == a_units and t_items == a_items
            # tiles count from the request's first new row: tile t covers
            # positions kv_len - ql + [32 t, 32 t + 32), ceil(ql / 32) tiles
            if ql:
                tiles = sorted({t for _, t in a_units})
                assert tiles == list(range((ql + 31) // 32))


def test_split_policies_cover_the_same_units():
    qo, kv, last = [0, 40, 41], [0, 600, 1200], [7, 16]
    plans = {pol: bip.Plan(qo, kv, last, num_qo_heads=32, num_kv_heads=8, head_dim=128, split_policy=pol)
             for pol in ("never", "always", "auto")}
    assert plans["never"].info["num_split_units"] == 0
    assert plans["always"].info["num_split_units"] > 0
    ref = {(r[0], r[1], r[2]) for r in plans["never"].items()}
    for pol, p in plans.items():
        assert {(r[0], r[1], r[2]) for r in p.items()} == ref
        # every segment of every unit is covered exactly once
        seen = {}
        for r in p.items():
            for s in range(r[3], r[4] + 1):
                key = (r[0], r[1], r[2], s)
                assert key not in seen
                seen[key] = 1
        assert len(seen) == sum(r[4] - r[3] + 1 for r in plans["never"].items())


def test_tiles_per_unit_choice():
    # long requests pair q tiles; one-tile extends keep one tile per CTA
    assert bip.Plan([0, 8192], [0, 512], [16], num_qo_heads=32, num_kv_heads=8,
                    head_dim=128).info["tiles_per_unit"] == 2
    assert bip.Plan([0, 4], [0, 2048], [16], num_qo_heads=32, num_kv_heads=8,
                    head_dim=128).info["tiles_per_unit"] == 1
    assert bip.Plan([0, 8192], [0, 512], [16], num_qo_heads=24, num_kv_heads=4,
                    head_dim=256).info["tiles_per_unit"] == 1
    with pytest.raises(bip.BipError):
        bip.Plan([0, 8], [0, 1], [16], num_qo_heads=24, num_kv_heads=4, head_dim=256, tiles_per_unit=2)
    # FP8 pages follow the same rule (two tiles exist at head_dim 128), except token-granular pools
    assert bip.Plan([0, 8192], [0, 512], [16], num_qo_heads=32, num_kv_heads=8, head_dim=128,
                    kv_dtype="fp8_e4m3").info["tiles_per_unit"] == 2
    assert bip.Plan([0, 4], [0, 2048], [16], num_qo_heads=32, num_kv_heads=8, head_dim=128,
                    kv_dtype="fp8_e4m3").info["tiles_per_unit"] == 1
    with pytest.raises(bip.BipError):
        bip.Plan([0, 8], [0, 8], [1], num_qo_heads=32, num_kv_heads=8, head_dim=128, kv_dtype="fp8_e4m3",
                 page_size=1, tiles_per_unit=2)
    # forcing either variant covers the same tiles
    for tpu in (1, 2):
        p = bip.Plan([0, 100, 103], [0, 7, 70], [4, 16], num_qo_heads=32, num_kv_heads=8, head_dim=128,
                     tiles_per_unit=tpu)
        assert unit_geometry(p, 0)[0] == [(h, t) for h in range(8) for t in range(0, 4)]


def test_items_grouped_by_request_and_head_longest_first():
    qo, kv, last = [0, 3000, 3001], [0, 400, 800], [16, 16]
    it = bip.Plan(qo, kv, last, num_qo_heads=32, num_kv_heads=8, head_dim=128).items()
    keys = it[:, 0] * 65536 + it[:, 1]
    assert (np.diff(keys) >= 0).all()
    for k in np.unique(keys):
        assert (np.diff(it[keys == k, 6]) <= 0).all()


def test_work_list_does_not_depend_on_the_page_size(lib):
    # the same lengths in pools of 16-slot pages and of single slots: the plan
    # (units, segments, splits, order) is the same; only page offsets differ
    rng = np.random.default_rng(11)
    for trial in range(12):
        batch = int(rng.integers(1, 7))
        kv_lens = [int(x) for x in rng.integers(1, 9000, batch)]
        q_lens = [int(rng.integers(0, k + 1)) for k in kv_lens]
        qo = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
        plans = []
        for ps in (16, 1):
            pages = [(k + ps - 1) // ps for k in kv_lens]
            kv = np.concatenate([[0], np.cumsum(pages)]).astype(np.int32)
            last = [k - ps * (n - 1) for k, n in zip(kv_lens, pages)]
            for policy in ("never", "auto"):
                plans.append((ps, policy, bip.Plan(qo, kv, last, num_qo_heads=32, num_kv_heads=8, head_dim=128,
                                                   page_size=ps, split_policy=policy, tiles_per_unit=1)))
        by_policy = {}
        for ps, policy, plan in plans:
            by_policy.setdefault(policy, []).append(plan.items())
        for policy, (a, b) in by_policy.items():
            assert np.array_equal(a, b), f"trial {trial}, policy {policy}"


def test_entry_points_refuse_host_tensors_instead_of_computing_on_the_cpu(lib):
    # There is no CPU path: every compute entry point wants device tensors and
    # says so, before anything runs.
    import torch
    from invariant_paged_prefill_gb300 import workloads as W
    b = W.tiny(3)
    plan = bip.Plan(b.qo_indptr, b.kv_indptr, b.kv_last_page_len, num_qo_heads=32, num_kv_heads=8, head_dim=128)
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8)
    with pytest.raises(bip.BipError, match="CUDA tensor"):
        bip.prefill(plan, b.q, b.k_pages, b.v_pages, b.kv_indices, workspace=ws)
    k_new = torch.zeros(3, 8, 128, dtype=torch.bfloat16)
    with pytest.raises(bip.BipError, match="CUDA tensor"):
        bip.append_kv(plan, k_new, k_new, b.k_pages, b.v_pages, b.kv_indices, workspace=ws)
    gp = bip.GraphPlan(2, 8, num_qo_heads=32, num_kv_heads=8, head_dim=128)
    i32 = torch.zeros(3, dtype=torch.int32)
    out = torch.zeros(8, 32, 128, dtype=torch.bfloat16)
    lse = torch.zeros(8, 32, dtype=torch.float32)
    with pytest.raises(bip.BipError, match="CUDA tensor"):
        bip.prefill_graph(gp, 2, i32, i32, i32[:2], out, b.k_pages, b.v_pages, b.kv_indices, out, lse,
                          torch.empty(gp.workspace_bytes, dtype=torch.uint8))


def test_equal_length_items_keep_construction_order():
    # Inside a (request, kv head) group, items of equal length (the full
    # 4096-key segments of split units, fold units of equal reach) stay in
    # construction order: units by tile, a split unit's segments in order.
    qo, kv, last = [0, 70, 72, 700], [0, 1000, 1600, 2000], [16, 16, 16]
    for pol in ("always", "never", "auto"):
        it = bip.Plan(qo, kv, last, num_qo_heads=32, num_kv_heads=8, head_dim=128, split_policy=pol).items()
        keys = it[:, 0] * 65536 + it[:, 1]
        for k in np.unique(keys):
            g = it[keys == k]
            for b in np.unique(g[:, 6]):
                same = g[g[:, 6] == b]
                order = [(int(r[2]), int(r[3])) for r in same]
                assert order == sorted(order), (pol, order)
