"""Custom masks on the GPU: each q row sees the keys that the causal (and
window) rule allows and its own mask row selects.  Parity with the oracle in
every kernel variant (both head dims, FP8 pages, token-granular pages, one or
two tiles per CTA), rows with no visible key written as zeros with lse -inf,
and the plain path's bit-exactness properties under a mask: extend rows equal
full-prefill rows, split / fold / tiles per CTA change no bit, an all-ones
mask equals no mask, a band mask equals the sliding window."""

import numpy as np
import pytest
import torch

import invariant_paged_prefill_gb300 as bip
from invariant_paged_prefill_gb300 import workloads as W

from gpu_helpers import ATOL, RTOL, assert_bitwise, oracle, run_gpu, sample_rows, to_device

pytestmark = pytest.mark.gpu

# a fresh prefill across two segments, extends behind long and short
# prefixes, a short fresh prefill
LENS, Q_LENS = (5000, 4700, 1300, 60), (5000, 37, 3, 60)


def _batch(heads, kv_dtype="bf16", page_size=16, lens=LENS, q_lens=Q_LENS, seed_pages=9):
    prompts = [W.make_prompt(n, *heads, seed=90 + i, kv_dtype=kv_dtype) for i, n in enumerate(lens)]
    return W.layout(prompts, list(q_lens), page_size, seed_pages=seed_pages, kv_dtype=kv_dtype, poison=True)


def _masks(b, seed=0):
    """Request r's rows of its prompt's mask (the prompt mask's tail rows)."""
    return [W.prompt_mask(n, seed + 31 * r)[n - ql:, :n] for r, (n, ql) in enumerate(zip(b.kv_lens, b.q_lens))]


def _rows(b, masks, seed, per_request=12):
    """Sampled rows plus up to six rows per request with no visible key."""
    rows = set(sample_rows(b, per_request=per_request, seed=seed))
    for r, m in enumerate(masks):
        lo, _ = b.row_range(r)
        ql, kl = b.q_lens[r], b.kv_lens[r]
        empty = [i for i in range(ql) if not m[i, :kl - ql + i + 1].any()]
        rows.update(lo + i for i in empty[:6])
    return sorted(rows)


def _check(out, lse, ref_out, ref_lse, rows):
    """Rows with no visible key: out exactly 0 and lse -inf; the rest within
    the tolerance.  Returns how many (row, head) pairs were empty."""
    o = out.float().numpy().astype(np.float64)[rows]
    l = lse.numpy().astype(np.float64)[rows]
    empty = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(l), empty), "the rows with no visible key differ"
    assert (o[empty] == 0).all(), "a row with no visible key has a nonzero output"
    full = ~empty
    assert np.isfinite(o[full]).all() and np.isfinite(l[full]).all(), "non-finite output"
    for name, got, ref in (("out", o[full], ref_out[full]), ("lse", l[full], ref_lse[full])):
        err = np.abs(got - ref)
        bad = err > ATOL + RTOL * np.abs(ref)
        assert not bad.any(), f"{name}: {bad.sum()} elements outside tolerance, max abs err {err.max():.3e}"
    return int(empty.sum())


VARIANTS = [
    (W.HEADS_A, "bf16", 16, 2), (W.HEADS_A, "bf16", 16, 1), (W.HEADS_B, "bf16", 16, 1),
    (W.HEADS_A, "fp8_e4m3", 16, 1), (W.HEADS_B, "fp8_e4m3", 16, 1),
    (W.HEADS_A, "bf16", 1, 1), (W.HEADS_B, "bf16", 2, 1), (W.HEADS_A, "fp8_e4m3", 1, 1), (W.HEADS_B, "fp8_e4m3", 4, 1),
]


@pytest.mark.parametrize("heads,kv_dtype,page_size,tiles", VARIANTS)
def test_mask_matches_oracle(cuda, heads, kv_dtype, page_size, tiles):
    b = _batch(heads, kv_dtype, page_size)
    masks = _masks(b, seed=page_size)
    out, lse, _ = run_gpu(b, cuda, custom_mask=masks, tiles_per_unit=tiles)
    rows = _rows(b, masks, seed=page_size)
    ro, rl = oracle(b, rows=rows, custom_mask=masks)
    assert _check(out, lse, ro, rl, rows) > 0  # rows with no visible key were covered


@pytest.mark.parametrize("page_size", [16, 1])
def test_mask_with_window_matches_oracle(cuda, page_size):
    b = _batch(W.HEADS_A, page_size=page_size)
    masks = _masks(b, seed=5)
    out, lse, _ = run_gpu(b, cuda, custom_mask=masks, window_left=700)
    rows = _rows(b, masks, seed=5)
    ro, rl = oracle(b, rows=rows, custom_mask=masks, window_left=700)
    _check(out, lse, ro, rl, rows)


@pytest.mark.parametrize("window", [0, 777])
def test_mask_extend_equals_full_prefill(cuda, window):
    # the extend rows of each prompt, with their rows of the prompt's mask,
    # equal the same rows of its full prefill
    prompts = [W.make_prompt(n, *W.HEADS_A, seed=120 + i) for i, n in enumerate((4300, 900, 6100))]
    full = W.layout(prompts, [p.n for p in prompts], 16, seed_pages=2, poison=True)
    ext = W.layout(prompts, [5, 300, 1], 16, seed_pages=5, poison=True)
    fo, fl, _ = run_gpu(full, cuda, custom_mask=_masks(full, seed=7), window_left=window)
    eo, el, _ = run_gpu(ext, cuda, custom_mask=_masks(ext, seed=7), window_left=window)
    for r in range(3):
        f0, e0 = int(full.qo_indptr[r]), int(ext.qo_indptr[r])
        n, off = ext.q_lens[r], full.q_lens[r] - ext.q_lens[r]
        assert_bitwise(eo[e0:e0 + n], fo[f0 + off:f0 + off + n], f"request {r} out")
        assert torch.equal(el[e0:e0 + n], fl[f0 + off:f0 + off + n]), f"request {r} lse"


def test_mask_split_fold_tiles_and_row_words_are_neutral(cuda):
    b = _batch(W.HEADS_A)
    masks = _masks(b, seed=11)
    ref_o, ref_l, _ = run_gpu(b, cuda, custom_mask=masks, policy="never")
    assert torch.isneginf(ref_l).any()  # empty rows take part, also in the merge kernel below
    for kw in (dict(policy="always"), dict(policy="auto"), dict(tiles_per_unit=1), dict(tiles_per_unit=2),
               dict(mask_row_words=170)):
        o, l, _ = run_gpu(b, cuda, custom_mask=masks, **kw)
        assert_bitwise(o, ref_o, f"mask {kw}")
        assert torch.equal(l, ref_l), f"mask {kw} lse"


@pytest.mark.parametrize("heads,kv_dtype,page_size", [(W.HEADS_A, "bf16", 16), (W.HEADS_B, "fp8_e4m3", 16),
                                                      (W.HEADS_A, "bf16", 1)])
def test_all_ones_mask_is_no_mask(cuda, heads, kv_dtype, page_size):
    b = _batch(heads, kv_dtype, page_size)
    ones = [np.ones((ql, n), dtype=bool) for n, ql in zip(b.kv_lens, b.q_lens)]
    mo, ml, _ = run_gpu(b, cuda, custom_mask=ones)
    po, pl, _ = run_gpu(b, cuda)
    assert_bitwise(mo, po, "all-ones mask vs none")
    assert_bitwise(ml, pl, "all-ones mask vs none lse")


@pytest.mark.parametrize("window", [100, 4500])
def test_band_mask_equals_window(cuda, window):
    # keys position - window .. position of every row, as a mask and as the
    # plan's sliding window: the mask visits the blocks the window skips,
    # which contribute exact zeros
    b = _batch(W.HEADS_A)
    bands = []
    for n, ql in zip(b.kv_lens, b.q_lens):
        pos = np.arange(n - ql, n)[:, None]
        cols = np.arange(n)[None, :]
        bands.append((cols >= pos - window) & (cols <= pos))
    mo, ml, _ = run_gpu(b, cuda, custom_mask=bands)
    wo, wl, _ = run_gpu(b, cuda, window_left=window)
    assert_bitwise(mo, wo, f"band {window} vs window")
    assert_bitwise(ml, wl, f"band {window} vs window lse")


def test_mask_rows_too_short_are_rejected(cuda):
    b = to_device(_batch(W.HEADS_A, lens=(100, 40), q_lens=(100, 40)), cuda)
    plan = bip.Plan(b.qo_indptr, b.kv_indptr, b.kv_last_page_len, num_qo_heads=32, num_kv_heads=8, head_dim=128)
    short = torch.zeros(b.q.shape[0], 3, dtype=torch.int32, device=cuda)  # 100 keys need 4 words
    with pytest.raises(bip.BipError):
        bip.prefill(plan, b.q, b.k_pages, b.v_pages, b.kv_indices, custom_mask=short)
    with pytest.raises(bip.BipError):
        bip.prefill(plan, b.q, b.k_pages, b.v_pages, b.kv_indices, custom_mask=short[:-1, :].contiguous())


def _doc_masks(b, seed, lo=300, hi=1500, dead=()):
    """Per request, its rows of a document mask over the prompt: the prompt is
    cut into documents of lo..hi tokens and a row sees only its own document's
    keys.  Requests in `dead` see keys only from the last document on, and the
    rows before it see nothing (whole items with no visible key)."""
    rng = np.random.default_rng(seed)
    out = []
    for r, (n, ql) in enumerate(zip(b.kv_lens, b.q_lens)):
        doc = np.zeros(n, dtype=np.int64)
        cut = 0
        while cut < n:
            step = int(rng.integers(lo, hi + 1))
            doc[cut:cut + step] = doc[cut - 1] + 1 if cut else 0
            cut += step
        m = doc[:, None] == doc[None, :]
        if r in dead:
            m &= doc[None, :] == doc[-1]
        out.append(m[n - ql:, :n])
    return out


def test_document_masks_skip_blocks_and_keep_the_bits(cuda):
    # Items start at the first block one of their rows sees: under document
    # masks most blocks before the diagonal are skipped.  Rows match the
    # oracle (rows with no visible key: zeros, lse -inf), extend rows equal
    # full-prefill rows bit for bit, split / fold / tiles per CTA change no
    # bit, and making key 0 visible to the last row of each request (so that
    # the items holding it cannot skip) changes no bit of any other row.
    prompts = [W.make_prompt(n, *W.HEADS_A, seed=140 + i) for i, n in enumerate((6000, 4500, 2100))]
    full = W.layout(prompts, [p.n for p in prompts], 16, seed_pages=3, poison=True)
    ext = W.layout(prompts, [700, 33, 2], 16, seed_pages=6, poison=True)
    fm, em = _doc_masks(full, 5, dead=(1,)), _doc_masks(ext, 5, dead=(1,))
    fo, fl, _ = run_gpu(full, cuda, custom_mask=fm, policy="never")
    rows = _rows(full, fm, seed=3)
    ro, rl = oracle(full, rows=rows, custom_mask=fm)
    assert _check(fo, fl, ro, rl, rows) > 0
    eo, el, _ = run_gpu(ext, cuda, custom_mask=em)
    for r in range(3):
        f0, e0 = int(full.qo_indptr[r]), int(ext.qo_indptr[r])
        n, off = ext.q_lens[r], full.q_lens[r] - ext.q_lens[r]
        assert_bitwise(eo[e0:e0 + n], fo[f0 + off:f0 + off + n], f"request {r} out")
        assert torch.equal(el[e0:e0 + n], fl[f0 + off:f0 + off + n]), f"request {r} lse"
    for kw in (dict(policy="always"), dict(policy="auto"), dict(tiles_per_unit=1), dict(tiles_per_unit=2)):
        o, l, _ = run_gpu(full, cuda, custom_mask=fm, **kw)
        assert_bitwise(o, fo, f"documents {kw}")
        assert torch.equal(l, fl), f"documents {kw} lse"
    opened = [m.copy() for m in fm]
    moved = []
    for r, m in enumerate(opened):
        i = m.shape[0] - 1          # the request's last row
        m[i, 0] = True
        moved.append(int(full.qo_indptr[r]) + i)
    oo, ol, _ = run_gpu(full, cuda, custom_mask=opened, policy="never")
    keep = torch.ones(fo.shape[0], dtype=torch.bool)
    keep[moved] = False
    assert_bitwise(oo[keep], fo[keep], "rows of items that can no longer skip")
    assert torch.equal(ol[keep], fl[keep])


@pytest.mark.parametrize("window", [0, 1500])
def test_document_masks_in_graph_launches_and_with_windows(cuda, window):
    # The skip passes in device-planned launches (split on the device for a
    # short batch) and under a sliding window (rows scan from position -
    # window): bits equal the host-planned masked launch, extend rows equal
    # full-prefill rows, and sampled rows match the oracle.
    prompts = [W.make_prompt(n, *W.HEADS_A, seed=160 + i) for i, n in enumerate((9000, 5100))]
    full = W.layout(prompts, [p.n for p in prompts], 16, seed_pages=4, poison=True)
    ext = W.layout(prompts, [40, 3], 16, seed_pages=8, poison=True)
    fm, em = _doc_masks(full, 9, lo=400, hi=2500), _doc_masks(ext, 9, lo=400, hi=2500)
    fo, fl, _ = run_gpu(full, cuda, custom_mask=fm, window_left=window)
    eo, el, _ = run_gpu(ext, cuda, custom_mask=em, window_left=window)
    for r in range(2):
        f0, e0 = int(full.qo_indptr[r]), int(ext.qo_indptr[r])
        n, off = ext.q_lens[r], full.q_lens[r] - ext.q_lens[r]
        assert_bitwise(eo[e0:e0 + n], fo[f0 + off:f0 + off + n], f"request {r} out")
        assert torch.equal(el[e0:e0 + n], fl[f0 + off:f0 + off + n]), f"request {r} lse"
    rows = _rows(full, fm, seed=4)
    ro, rl = oracle(full, rows=rows, custom_mask=fm, window_left=window)
    _check(fo, fl, ro, rl, rows)
    # the extend through the graph-replayable launch (device planner, device-side split)
    d = to_device(ext, cuda)
    words = (max(ext.kv_lens) + 31) // 32
    gp = bip.GraphPlan(4, 64, num_qo_heads=32, num_kv_heads=8, head_dim=128, window_left=window)
    i32 = dict(dtype=torch.int32, device=cuda)
    qo = torch.zeros(5, **i32)
    kv = torch.zeros(5, **i32)
    last = torch.ones(4, **i32)
    qo[:3] = torch.as_tensor(np.asarray(ext.qo_indptr), dtype=torch.int32)
    kv[:3] = torch.as_tensor(np.asarray(ext.kv_indptr), dtype=torch.int32)
    qo[3:] = int(ext.qo_indptr[-1])
    kv[3:] = int(ext.kv_indptr[-1])
    last[:2] = torch.as_tensor(np.asarray(ext.kv_last_page_len), dtype=torch.int32)
    q = torch.zeros(64, 32, 128, dtype=torch.bfloat16, device=cuda)
    n = ext.q.shape[0]
    q[:n].copy_(d.q)
    mask_buf = torch.zeros(64, words, dtype=torch.int32, device=cuda)
    mask_buf[:n].copy_(torch.from_numpy(bip.pack_mask(em, words)))
    out = torch.full_like(q, float("nan"))
    lse = torch.full((64, 32), float("nan"), dtype=torch.float32, device=cuda)
    ws = torch.empty(gp.workspace_bytes, dtype=torch.uint8, device=cuda)
    bip.prefill_graph(gp, 4, qo, kv, last, q, d.k_pages, d.v_pages, d.kv_indices, out, lse, ws, custom_mask=mask_buf)
    torch.cuda.synchronize()
    assert bip.read_device_status(ws) == 0
    assert_bitwise(out[:n].cpu(), eo, "graph launch out")
    assert torch.equal(lse[:n].cpu(), el), "graph launch lse"
