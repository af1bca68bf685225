"""The device planner's work list, item by item.

Graph-replayable launches plan on the device.  These tests read the work
items and merge units it wrote into the workspace and compare them, field
for field and in order, with the list its rules define: one unit per
(request with new rows, kv head, group of tiles_per_unit q tiles counted from
the request's first new row), in (request, kv head, longest group first)
order; a batch with fewer units than 8 per CTA splits every unit with more
than one 4096-key segment into one item per segment, its partial rows and
merge units laid out in unit order, when the capacities hold them.  Cases
cover fold and split, empty requests, a sliding window, head_dim 256, page
size 1, and batches past the planner's one-unit-per-thread limit."""

import numpy as np
import pytest
import torch

import invariant_paged_prefill_gb300 as bip
from invariant_paged_prefill_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SPLIT_LEN = 4096
HEADER_BYTES = 256
ITEM = np.dtype([("kv_len", "<i4"), ("page_base", "<i4"), ("q_tok0", "<i4"), ("q_lo", "<i4"), ("tile", "<i4"),
                 ("kv_head", "<i2"), ("seg_lo", "<i2"), ("seg_hi", "<i2"), ("flags", "<i2"),
                 ("part_base", "<i4", (2,)), ("nseg", "<i2", (2,)), ("blk_min", "<i4"), ("pad", "<i4")])
MERGE = np.dtype([("q_tok0", "<i4"), ("q_lo", "<i4"), ("tile", "<i4"), ("part_base", "<i4"), ("rows", "<i4"),
                  ("kv_head", "<i2"), ("nseg", "<i2"), ("pad", "<i4", (2,))])
assert ITEM.itemsize == 48 and MERGE.itemsize == 32
GRID = 148          # num_sms given to the plan: the persistent grid
BUDGET = 64 << 20   # the graph plan's split budget


def _align(x, a):
    return (x + a - 1) // a * a


def _units(qo, kv, last, *, page_size, heads, nt, window):
    hq, hkv, d = heads
    group = hq // hkv
    T, bn = 128 // group, (128 if d == 128 else 64)
    units = []
    for r in range(len(qo) - 1):
        ql, npg = qo[r + 1] - qo[r], kv[r + 1] - kv[r]
        kl = (npg - 1) * page_size + last[r] if npg > 0 else 0
        if ql == 0:
            continue
        q_lo = kl - ql
        t1 = (ql - 1) // T
        for h in range(hkv):
            for gi in range(t1 // nt, -1, -1):
                nseg, rows, flags, firsts, ends = [0, 0], [0, 0], 0, [], []
                for t in range(nt):
                    tile = gi * nt + t
                    if tile > t1:
                        continue
                    first = q_lo + tile * T
                    end = min(first + T - 1, kl - 1)
                    nseg[t], rows[t] = end // SPLIT_LEN + 1, (end - first + 1) * group
                    flags |= 256 << t
                    firsts.append(first)
                    ends.append(end)
                key_lo = max(0, min(firsts) - window) if window > 0 else 0
                units.append(dict(kv_len=kl, page_base=kv[r], q_tok0=qo[r] - q_lo, q_lo=q_lo, tile=gi * nt,
                                  kv_head=h, seg_lo=key_lo // SPLIT_LEN, seg_hi=max(ends) // SPLIT_LEN,
                                  flags=flags, part_base=[0, 0], nseg=nseg, blk_min=key_lo // bn, pad=0,
                                  rows=rows))
    return units


def _work_list(qo, kv, last, *, page_size, heads, nt, window, max_batch, max_total_q):
    """(items, merge units, split) as the planner's rules define them."""
    hq, hkv, d = heads
    T = 128 // (hq // hkv)
    units = _units(qo, kv, last, page_size=page_size, heads=heads, nt=nt, window=window)
    cap = hkv * ((max_total_q + T - 1) // T + 2 * max_batch)
    item_cap, merge_cap, part_cap = cap + 65536, cap * nt, BUDGET // ((d + 4) * 4)
    items, merges, part = [], [], 0
    for u in units:
        if u["seg_hi"] == u["seg_lo"]:
            items.append(u)
            continue
        base = [0, 0]
        for t in range(2):
            if u["flags"] >> 8 >> t & 1:
                n = u["nseg"][t] - u["seg_lo"]
                merges.append(dict(q_tok0=u["q_tok0"], q_lo=u["q_lo"], tile=u["tile"] + t, part_base=part,
                                   rows=u["rows"][t], kv_head=u["kv_head"], nseg=n, pad=[0, 0]))
                base[t] = part
                part += n * u["rows"][t]
        for sg in range(u["seg_lo"], u["seg_hi"] + 1):
            items.append({**u, "seg_lo": sg, "seg_hi": sg, "flags": u["flags"] | 1,
                          "part_base": [base[t] + (sg - u["seg_lo"]) * u["rows"][t] for t in range(2)]})
    split = (len(units) < 8 * GRID and len(items) > len(units) and len(items) <= item_cap and part <= part_cap
             and len(merges) <= merge_cap)
    return (items, merges, True) if split else (units, [], False)


def _records(rows, dtype):
    a = np.zeros(len(rows), dtype=dtype)
    for i, row in enumerate(rows):
        for f in dtype.names:
            a[i][f] = row[f]
    return a


CASES = {
    # name: (heads, page_size, tiles_per_unit, window_left, [(q_len, kv_len), ...])
    "fold_many_units": (W.HEADS_A, 16, 2, 0, [(300, 5000 + 37 * i) for i in range(40)]),
    "split_with_empty_requests": (W.HEADS_A, 16, 2, 0,
                                  [(5, 9000), (0, 0), (37, 12300), (0, 50), (1, 4097), (64, 64), (0, 0)]),
    "split_one_tile_window": (W.HEADS_A, 16, 1, 1000, [(300, 9000), (4, 20000), (0, 0), (129, 129)]),
    "split_head_dim_256": (W.HEADS_B, 16, 1, 0, [(50, 10000), (700, 5000), (3, 4096)]),
    "split_page_size_1": (W.HEADS_A, 1, 1, 0, [(20, 5000), (3, 100), (0, 7)]),
    "fold_large_batch": (W.HEADS_A, 16, 2, 0, [(1 + i % 3, 8 + i % 40) for i in range(1600)]),
    "split_large_batch": (W.HEADS_A, 16, 2, 0,
                          [((3, 9000) if i % 300 == 7 else (0, 0)) for i in range(1600)]),
}


@pytest.mark.parametrize("name", list(CASES))
def test_device_work_list_is_the_planned_one(cuda, name):
    heads, page_size, nt, window, reqs = CASES[name]
    hq, hkv, d = heads
    q_lens = [q for q, _ in reqs]
    kv_lens = [k for _, k in reqs]
    pages = [(k + page_size - 1) // page_size for k in kv_lens]
    qo = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int64)
    kv = np.concatenate([[0], np.cumsum(pages)]).astype(np.int64)
    last = np.array([k - (p - 1) * page_size if p > 0 else 1 for k, p in zip(kv_lens, pages)], dtype=np.int64)
    batch, total_q = len(reqs), int(qo[-1])
    max_total_q = total_q + 8
    plan = bip.GraphPlan(batch, max_total_q, num_qo_heads=hq, num_kv_heads=hkv, head_dim=d, page_size=page_size,
                         num_sms=GRID, tiles_per_unit=nt, window_left=window)
    want_items, want_merges, want_split = _work_list(
        [int(x) for x in qo], [int(x) for x in kv], [int(x) for x in last], page_size=page_size, heads=heads,
        nt=nt, window=window, max_batch=batch, max_total_q=max_total_q)
    assert want_split == name.startswith("split")

    gen = torch.Generator().manual_seed(11)
    pool = 64
    k_pages = torch.randn(pool, page_size, hkv, d, generator=gen).to(torch.bfloat16).to(cuda)
    v_pages = torch.randn(pool, page_size, hkv, d, generator=gen).to(torch.bfloat16).to(cuda)
    idx = torch.randint(0, pool, (max(int(kv[-1]), 1),), generator=gen, dtype=torch.int32).to(cuda)
    q = torch.randn(max_total_q, hq, d, generator=gen).to(torch.bfloat16).to(cuda)
    out = torch.empty_like(q)
    lse = torch.empty(max_total_q, hq, dtype=torch.float32, device=cuda)
    ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device=cuda)
    i32 = dict(dtype=torch.int32, device=cuda)
    bip.prefill_graph(plan, batch, torch.as_tensor(qo, **i32), torch.as_tensor(kv, **i32),
                      torch.as_tensor(last, **i32), q, k_pages, v_pages, idx, out, lse, ws)
    torch.cuda.synchronize()
    assert bip.read_device_status(ws) == 0
    head = ws[:HEADER_BYTES].cpu().numpy().view(np.uint32)
    n_items, n_merges = int(head[3]), int(head[4])
    assert n_items == len(want_items) and n_merges == len(want_merges)

    T = 128 // (hq // hkv)
    cap = hkv * ((max_total_q + T - 1) // T + 2 * batch)
    off_merges = _align(HEADER_BYTES + (cap + 65536) * ITEM.itemsize, 256)
    got = ws[HEADER_BYTES: HEADER_BYTES + n_items * ITEM.itemsize].cpu().numpy().view(ITEM)
    want = _records(want_items, ITEM)
    bad = np.nonzero((got.view(np.uint8).reshape(-1, ITEM.itemsize) !=
                      want.view(np.uint8).reshape(-1, ITEM.itemsize)).any(axis=1))[0]
    assert bad.size == 0, f"{bad.size} items differ, first at {bad[0]}: {got[bad[0]]} vs {want[bad[0]]}"
    if n_merges:
        gm = ws[off_merges: off_merges + n_merges * MERGE.itemsize].cpu().numpy()
        assert np.array_equal(gm, _records(want_merges, MERGE).view(np.uint8))
