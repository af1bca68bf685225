"""Pins for the float64 oracle, against things other than itself.

* A library routine: ``torch.nn.functional.scaled_dot_product_attention`` in
  float64 on CPU (its own softmax and its own GQA head mapping,
  ``enable_gqa``), with a boolean tail-aligned mask built by ``torch.tril``;
  lse against ``torch.logsumexp``.
* Closed forms: one key; q = 0 (uniform weights); all keys equal; all
  values equal; a dominant key; two keys by scalar ``math``; a positional
  value channel that exposes the row -> position map.
* Invariants: extend rows equal full-prefill rows, page permutation, batch
  composition and chunked prefill change nothing.
* Planted mistakes: each plausible error in one of the oracle's pieces makes
  at least one of the pins above fail.
"""

import math

import numpy as np
import pytest
import torch

import oracle.paged_attention as pa
from invariant_paged_prefill_gb300 import workloads as W


# --------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------

def paged_from_dense(qs, ks, vs, page_size=4, seed=0):
    """Pack per-request dense float64 q/k/v into a shuffled, NaN-poisoned page pool."""
    rng = np.random.default_rng(seed)
    hkv, d = ks[0].shape[1], ks[0].shape[2]
    npages = [(k.shape[0] + page_size - 1) // page_size for k in ks]
    total = sum(npages) + 2
    perm = rng.permutation(total)
    kp = np.full((total, page_size, hkv, d), np.nan)
    vp = np.full((total, page_size, hkv, d), np.nan)
    kv_indices, kv_indptr, last, qo = [], [0], [], [0]
    cur = 0
    for k, v, n in zip(ks, vs, npages):
        ids = perm[cur:cur + n]
        cur += n
        for j in range(k.shape[0]):
            kp[ids[j // page_size], j % page_size] = k[j]
            vp[ids[j // page_size], j % page_size] = v[j]
        kv_indices.extend(int(x) for x in ids)
        kv_indptr.append(kv_indptr[-1] + n)
        last.append(k.shape[0] - (n - 1) * page_size)
    for q in qs:
        qo.append(qo[-1] + q.shape[0])
    return dict(q=np.concatenate(qs), k_pages=kp, v_pages=vp, qo_indptr=qo, kv_indptr=kv_indptr,
                kv_indices=kv_indices, kv_last_page_len=last, num_qo_heads=qs[0].shape[1],
                num_kv_heads=hkv, page_size=page_size)


def oracle_on_batch(b: W.PagedBatch, mod=pa, rows=None):
    kind = "bf16" if b.kv_dtype == "bf16" else "e4m3"
    kview = b.k_pages.view(torch.int16) if kind == "bf16" else b.k_pages
    vview = b.v_pages.view(torch.int16) if kind == "bf16" else b.v_pages
    return mod.paged_prefill(b.q.view(torch.int16).numpy(), kview.numpy(), vview.numpy(),
                             b.qo_indptr.tolist(), b.kv_indptr.tolist(), b.kv_indices.tolist(),
                             b.kv_last_page_len.tolist(), b.num_qo_heads, b.num_kv_heads, b.page_size,
                             q_kind="bf16", kv_kind=kind, rows=rows)


def sdpa_reference(q, k, v, q_len):
    """Library attention for one request: q [q_len,Hq,d], k/v [kv_len,Hkv,d] float64."""
    kv_len = k.shape[0]
    mask = torch.ones(q_len, kv_len, dtype=torch.bool).tril(diagonal=kv_len - q_len)
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]
    kt = torch.from_numpy(k).permute(1, 0, 2)[None]
    vt = torch.from_numpy(v).permute(1, 0, 2)[None]
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, enable_gqa=True)
    g = q.shape[1] // k.shape[1]
    kr = kt.repeat_interleave(g, dim=1)
    scores = (qt @ kr.transpose(-1, -2)) / math.sqrt(q.shape[2])
    lse = torch.logsumexp(scores.masked_fill(~mask, float("-inf")), dim=-1)
    return out[0].permute(1, 0, 2).numpy(), lse[0].permute(1, 0).numpy()


def random_requests(specs, hq, hkv, d, seed):
    rng = np.random.default_rng(seed)
    qs, ks, vs = [], [], []
    for q_len, kv_len in specs:
        qs.append(rng.standard_normal((q_len, hq, d)))
        ks.append(rng.standard_normal((kv_len, hkv, d)))
        vs.append(rng.standard_normal((kv_len, hkv, d)))
    return qs, ks, vs


def _err(x) -> float:
    """Largest |x|, with any NaN or infinity counted as an infinite error."""
    x = np.asarray(x, dtype=np.float64)
    return float("inf") if not np.isfinite(x).all() else float(np.abs(x).max(initial=0.0))


# --------------------------------------------------------------------------
# pin checks, returning the worst error so the planted-mistake tests can reuse them
# --------------------------------------------------------------------------

SDPA_CASES = [
    # (specs [(q_len, kv_len)], hq, hkv, d, page_size)
    ([(7, 7), (3, 11), (1, 5), (0, 4), (5, 9)], 8, 2, 16, 4),
    ([(4, 13), (13, 13)], 6, 1, 8, 16),
    ([(2, 2), (6, 21)], 12, 2, 32, 4),
    ([(3, 9), (9, 9)], 4, 2, 16, 1),     # token-granular pools
    ([(5, 10), (1, 7)], 4, 1, 8, 2),
]


def sdpa_error(mod=pa):
    worst = 0.0
    for i, (specs, hq, hkv, d, ps) in enumerate(SDPA_CASES):
        qs, ks, vs = random_requests(specs, hq, hkv, d, seed=10 + i)
        args = paged_from_dense(qs, ks, vs, page_size=ps, seed=i)
        out, lse = mod.paged_prefill(**args)
        row = 0
        for q, k, v, (ql, kl) in zip(qs, ks, vs, specs):
            if ql:
                ro, rl = sdpa_reference(q, k, v, ql)
                worst = max(worst, _err(out[row:row + ql] - ro), _err(lse[row:row + ql] - rl))
            row += ql
    return worst


def closed_form_errors(mod=pa):
    """Worst error of each closed form (dict name -> error)."""
    rng = np.random.default_rng(3)
    hq, hkv, d = 8, 2, 16
    g = hq // hkv
    errs = {}

    # one key: out = v0, lse = q.k0/sqrt(d)
    q = rng.standard_normal((1, hq, d)); k = rng.standard_normal((1, hkv, d)); v = rng.standard_normal((1, hkv, d))
    out, lse = mod.paged_prefill(**paged_from_dense([q], [k], [v], page_size=4))
    want_lse = np.array([q[0, h] @ k[0, h // g] / math.sqrt(d) for h in range(hq)])
    errs["one_key"] = max(_err(out[0] - v[0][np.arange(hq) // g]), _err(lse[0] - want_lse))

    # q = 0 behind a prefix: uniform weights, out = mean(V[0..pos]), lse = ln(pos+1)
    kv_len, q_len = 11, 4
    q = np.zeros((q_len, hq, d)); k = rng.standard_normal((kv_len, hkv, d)); v = rng.standard_normal((kv_len, hkv, d))
    out, lse = mod.paged_prefill(**paged_from_dense([q], [k], [v], page_size=4))
    e = 0.0
    for i in range(q_len):
        pos = i + kv_len - q_len
        for h in range(hq):
            e = max(e, _err(out[i, h] - v[:pos + 1, h // g].mean(axis=0)), _err(lse[i, h] - math.log(pos + 1)))
    errs["q_zero"] = e

    # all keys equal: out = mean V[0..pos], lse = s + ln(pos+1)
    q = rng.standard_normal((q_len, hq, d)); k1 = rng.standard_normal((1, hkv, d))
    k = np.repeat(k1, kv_len, axis=0)
    out, lse = mod.paged_prefill(**paged_from_dense([q], [k], [v], page_size=4))
    e = 0.0
    for i in range(q_len):
        pos = i + kv_len - q_len
        for h in range(hq):
            s = q[i, h] @ k1[0, h // g] / math.sqrt(d)
            e = max(e, _err(out[i, h] - v[:pos + 1, h // g].mean(axis=0)), _err(lse[i, h] - (s + math.log(pos + 1))))
    errs["keys_equal"] = e

    # all values of a KV head equal to c_hk: out = c_{h // g}
    c = rng.standard_normal((hkv, d))
    vc = np.repeat(c[None], kv_len, axis=0)
    q = rng.standard_normal((q_len, hq, d)); k = rng.standard_normal((kv_len, hkv, d))
    out, _ = mod.paged_prefill(**paged_from_dense([q], [k], [vc], page_size=4))
    errs["values_equal"] = max(_err(out[:, h] - c[h // g]) for h in range(hq))

    # positional value channel, q = 0: out[..., 0] = pos / 2 exactly
    vpos = rng.standard_normal((kv_len, hkv, d)); vpos[:, :, 0] = np.arange(kv_len)[:, None]
    q = np.zeros((q_len, hq, d))
    out, _ = mod.paged_prefill(**paged_from_dense([q], [k], [vpos], page_size=4))
    errs["positions"] = max(_err(out[i, h, 0] - (i + kv_len - q_len) / 2) for i in range(q_len) for h in range(hq))

    # a dominant key: q_h = 80 sqrt(d) k_j / |k_j| for j = pos - 2 -> out = v_j up to exp(-gap)
    k = rng.standard_normal((kv_len, hkv, d)); v = rng.standard_normal((kv_len, hkv, d))
    q = np.zeros((1, hq, d))
    j = kv_len - 3
    for h in range(hq):
        q[0, h] = 80.0 * math.sqrt(d) * k[j, h // g] / np.linalg.norm(k[j, h // g])
    out, _ = mod.paged_prefill(**paged_from_dense([q], [k], [v], page_size=4))
    errs["dominant"] = max(_err(out[0, h] - v[j, h // g]) for h in range(hq))

    # two keys by scalar math
    q = rng.standard_normal((1, hq, d)); k = rng.standard_normal((2, hkv, d)); v = rng.standard_normal((2, hkv, d))
    out, lse = mod.paged_prefill(**paged_from_dense([q], [k], [v], page_size=4))
    e = 0.0
    for h in range(hq):
        a = float(q[0, h] @ k[0, h // g]) / math.sqrt(d)
        b = float(q[0, h] @ k[1, h // g]) / math.sqrt(d)
        z = math.exp(a) + math.exp(b)
        want = (math.exp(a) * v[0, h // g] + math.exp(b) * v[1, h // g]) / z
        e = max(e, _err(out[0, h] - want), _err(lse[0, h] - math.log(z)))
    errs["two_keys"] = e
    return errs


TOL = 1e-10


# --------------------------------------------------------------------------
# the pins
# --------------------------------------------------------------------------

def test_oracle_matches_library_sdpa():
    assert sdpa_error() < TOL


@pytest.mark.parametrize("name", ["one_key", "q_zero", "keys_equal", "values_equal", "positions",
                                  "dominant", "two_keys"])
def test_oracle_closed_forms(name):
    assert closed_form_errors()[name] < TOL


def test_extend_rows_equal_full_prefill_rows():
    full = W.tiny(64)
    ext = W.tiny(3)
    fo, fl = oracle_on_batch(full)
    eo, el = oracle_on_batch(ext)
    assert _err(eo - fo[61:64]) < 1e-12 and _err(el - fl[61:64]) < 1e-12


def test_page_permutation_invariance():
    a = W.layout([W.make_prompt(40, 8, 2, 32, seed=4)], [9], 16, seed_pages=1)
    b = W.layout([W.make_prompt(40, 8, 2, 32, seed=4)], [9], 16, seed_pages=7, extra_pages=11)
    assert not torch.equal(a.kv_indices, b.kv_indices)
    (ao, al), (bo, bl) = oracle_on_batch(a), oracle_on_batch(b)
    assert _err(ao - bo) < 1e-12 and _err(al - bl) < 1e-12


def test_batch_composition_invariance():
    prompts = [W.make_prompt(n, 8, 2, 32, seed=20 + n) for n in (33, 17, 50)]
    qls = [5, 17, 1]
    together = oracle_on_batch(W.layout(prompts, qls, 16))
    row = 0
    for p, ql in zip(prompts, qls):
        alone = oracle_on_batch(W.layout([p], [ql], 16, seed_pages=3))
        assert _err(alone[0] - together[0][row:row + ql]) < 1e-12
        assert _err(alone[1] - together[1][row:row + ql]) < 1e-12
        row += ql


def test_chunked_prefill_invariance():
    p = W.make_prompt(70, 8, 2, 32, seed=9)
    full = oracle_on_batch(W.layout([p], [70], 16))
    for a, b in [(0, 23), (23, 41), (41, 70)]:
        chunk = W.Prompt(p.q[:b], p.k[:b], p.v[:b])
        co, cl = oracle_on_batch(W.layout([chunk], [b - a], 16, seed_pages=b))
        assert _err(co - full[0][a:b]) < 1e-12 and _err(cl - full[1][a:b]) < 1e-12


def test_rows_subset_equals_full_computation():
    b = W.layout([W.make_prompt(n, 8, 2, 32, seed=n) for n in (20, 31)], [20, 7], 16)
    fo, fl = oracle_on_batch(b)
    rows = [26, 0, 19, 21]
    so, sl = oracle_on_batch(b, rows=rows)
    assert np.array_equal(so, fo[rows]) and np.array_equal(sl, fl[rows])


def test_unused_slots_are_never_read():
    # The pools are NaN-poisoned outside each request's kv_len: any read would show.
    e, c = W.radix_burst(n_req=3, prefix=32)
    for b in (e, c):
        o, l = oracle_on_batch(b)
        assert np.isfinite(o).all() and np.isfinite(l).all()


def test_q_len_greater_than_kv_len_rejected():
    qs, ks, vs = random_requests([(3, 2)], 4, 1, 8, seed=0)
    with pytest.raises(ValueError):
        pa.paged_prefill(**paged_from_dense(qs, ks, vs))


# --------------------------------------------------------------------------
# planted mistakes: each must make some pin fail
# --------------------------------------------------------------------------

MUTATIONS = {
    "position_off_by_one": ("row_position", lambda i, ql, kl: i + kl - ql - 1),
    "head_aligned_not_tail": ("row_position", lambda i, ql, kl: i),
    "diagonal_excluded": ("visible_keys", lambda p: max(p, 1)),
    "kv_head_interleaved": ("kv_head_of", lambda h, hq, hkv: h % hkv),
    "kv_len_full_pages": ("kv_lengths", lambda ind, last, ps: [(ind[r + 1] - ind[r]) * ps for r in range(len(ind) - 1)]),
}


def _wrong_gather(pages, kv_indices, page_lo, kv_len, page_size):
    pages = np.asarray(pages)
    return np.stack([pages[int(kv_indices[page_lo + j // page_size]), (j + 1) % page_size] for j in range(kv_len)])


@pytest.mark.parametrize("name", sorted(MUTATIONS) + ["slot_shift", "scale_squared"])
def test_planted_mistake_is_caught(name, monkeypatch):
    if name == "slot_shift":
        monkeypatch.setattr(pa, "gather_request_kv", _wrong_gather)
    elif name == "scale_squared":
        real = pa.attend_rows
        monkeypatch.setattr(pa, "attend_rows", lambda q, k, v, p, s, *rest: real(q, k, v, p, s * s, *rest))
    else:
        attr, fn = MUTATIONS[name]
        monkeypatch.setattr(pa, attr, fn)
    try:
        caught = sdpa_error() > TOL or max(closed_form_errors().values()) > TOL
    except (ValueError, IndexError):
        caught = True  # a mistake that breaks the shapes is caught as well
    assert caught, f"planted mistake {name} went unnoticed"


# --------------------------------------------------------------------------
# sliding window
# --------------------------------------------------------------------------

def sdpa_window_reference(q, k, v, q_len, window_left):
    """Library attention with a banded mask: row at position p sees keys p - W .. p."""
    kv_len = k.shape[0]
    pos = torch.arange(q_len)[:, None] + (kv_len - q_len)
    key = torch.arange(kv_len)[None, :]
    mask = (key <= pos) & (key >= pos - window_left)
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]
    kt = torch.from_numpy(k).permute(1, 0, 2)[None]
    vt = torch.from_numpy(v).permute(1, 0, 2)[None]
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, enable_gqa=True)
    g = q.shape[1] // k.shape[1]
    kr = kt.repeat_interleave(g, dim=1)
    scores = (qt @ kr.transpose(-1, -2)) / math.sqrt(q.shape[2])
    lse = torch.logsumexp(scores.masked_fill(~mask, float("-inf")), dim=-1)
    return out[0].permute(1, 0, 2).numpy(), lse[0].permute(1, 0).numpy()


@pytest.mark.parametrize("window", [1, 3, 8, 40])
def test_oracle_window_matches_library_banded_mask(window):
    specs, hq, hkv, d, ps = [(7, 7), (3, 11), (1, 5), (5, 30), (12, 50)], 8, 2, 16, 4
    qs, ks, vs = random_requests(specs, hq, hkv, d, seed=77)
    args = paged_from_dense(qs, ks, vs, page_size=ps, seed=5)
    out, lse = pa.paged_prefill(**args, window_left=window)
    row = 0
    for q, k, v, (ql, kl) in zip(qs, ks, vs, specs):
        ro, rl = sdpa_window_reference(q, k, v, ql, window)
        assert _err(out[row:row + ql] - ro) < TOL and _err(lse[row:row + ql] - rl) < TOL
        row += ql


def test_oracle_window_closed_forms():
    # window 1 over keys of one value channel: a row sees exactly keys p-1 and p;
    # with q = 0 the output is their mean and lse = ln 2 (one key at p = 0: lse 0).
    hq, hkv, d, n = 4, 1, 8, 9
    q = np.zeros((n, hq, d))
    k = np.random.default_rng(1).standard_normal((n, hkv, d))
    v = np.zeros((n, hkv, d))
    v[:, 0, 0] = np.arange(n, dtype=np.float64)
    args = paged_from_dense([q], [k], [v], page_size=4, seed=2)
    out, lse = pa.paged_prefill(**args, window_left=1)
    want = np.array([0.0] + [p - 0.5 for p in range(1, n)])
    assert _err(out[:, 0, 0] - want) < TOL
    assert _err(lse[0]) < TOL and _err(lse[1:] - math.log(2)) < TOL
    # a window at least as long as the sequence is plain causal attention
    o2, l2 = pa.paged_prefill(**args, window_left=n)
    o3, l3 = pa.paged_prefill(**args)
    assert np.array_equal(o2, o3) and np.array_equal(l2, l3)


def test_oracle_window_extend_rows_equal_full_rows():
    specs, hq, hkv, d = [(40, 40)], 4, 2, 8
    qs, ks, vs = random_requests(specs, hq, hkv, d, seed=9)
    full = paged_from_dense(qs, ks, vs, page_size=4, seed=1)
    ext = paged_from_dense([qs[0][30:]], ks, vs, page_size=4, seed=1)
    fo, fl = pa.paged_prefill(**full, window_left=6)
    eo, el = pa.paged_prefill(**ext, window_left=6)
    assert np.array_equal(eo, fo[30:]) and np.array_equal(el, fl[30:])


def window_sdpa_error(window: int) -> float:
    specs, hq, hkv, d, ps = [(7, 7), (3, 11), (5, 30), (12, 50)], 8, 2, 16, 4
    qs, ks, vs = random_requests(specs, hq, hkv, d, seed=78)
    args = paged_from_dense(qs, ks, vs, page_size=ps, seed=6)
    out, lse = pa.paged_prefill(**args, window_left=window)
    worst, row = 0.0, 0
    for q, k, v, (ql, kl) in zip(qs, ks, vs, specs):
        ro, rl = sdpa_window_reference(q, k, v, ql, window)
        worst = max(worst, _err(out[row:row + ql] - ro), _err(lse[row:row + ql] - rl))
        row += ql
    return worst


@pytest.mark.parametrize("mistake", ["one_short", "one_long", "ignored"])
def test_planted_window_mistake_is_caught(mistake, monkeypatch):
    real = pa.first_visible_key
    wrong = {"one_short": lambda p, w=0: real(p, w) + (1 if w > 0 and p - w >= 0 else 0),
             "one_long": lambda p, w=0: max(0, real(p, w) - 1),
             "ignored": lambda p, w=0: 0}[mistake]
    monkeypatch.setattr(pa, "first_visible_key", wrong)
    assert window_sdpa_error(5) > TOL, f"planted window mistake {mistake} went unnoticed"
