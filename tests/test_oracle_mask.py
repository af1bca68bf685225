"""Pins for the oracle's custom-mask reading (CPU).

The mask narrows the causal rule: key j is visible to row i when the causal
(and window) rule allows it and mask[i, j] is set.  Pinned against the
library attention with an explicit boolean mask, closed forms, the window
rule it must reproduce, and planted mistakes the pins must catch.
"""

import math

import numpy as np
import pytest
import torch

from oracle import paged_attention as pa

from test_oracle_pins import paged_from_dense, random_requests

SPECS = [(7, 7), (3, 11), (5, 9), (1, 5)]
HQ, HKV, D = 8, 2, 16


def _masks(specs, seed, density=0.6, keep_diagonal=True):
    rng = np.random.default_rng(seed)
    out = []
    for ql, kl in specs:
        m = rng.random((ql, kl)) < density
        if keep_diagonal:  # every row keeps its own position, so no row is empty
            for i in range(ql):
                m[i, kl - ql + i] = True
        out.append(m)
    return out


def _run(qs, ks, vs, masks=None, window_left=0, ps=4, mod=pa):
    args = paged_from_dense(qs, ks, vs, page_size=ps, seed=3)
    return mod.paged_prefill(**args, custom_mask=masks, window_left=window_left)


def _library(q, k, v, mask):
    """torch SDPA in float64 with mask = causal AND custom, and its logsumexp."""
    ql, kl = mask.shape
    causal = torch.ones(ql, kl, dtype=torch.bool).tril(diagonal=kl - ql)
    m = causal & torch.from_numpy(mask)
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]
    kt = torch.from_numpy(k).permute(1, 0, 2)[None]
    vt = torch.from_numpy(v).permute(1, 0, 2)[None]
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=m, enable_gqa=True)
    kr = kt.repeat_interleave(q.shape[1] // k.shape[1], dim=1)
    scores = (qt @ kr.transpose(-1, -2)) / math.sqrt(q.shape[2])
    lse = torch.logsumexp(scores.masked_fill(~m, float("-inf")), dim=-1)
    return out[0].permute(1, 0, 2).numpy(), lse[0].permute(1, 0).numpy()


def library_error(mod=pa, seed=0):
    qs, ks, vs = random_requests(SPECS, HQ, HKV, D, seed=seed)
    masks = _masks(SPECS, seed + 1)
    out, lse = _run(qs, ks, vs, masks, mod=mod)
    worst, row = 0.0, 0
    for q, k, v, m in zip(qs, ks, vs, masks):
        ro, rl = _library(q, k, v, m)
        n = q.shape[0]
        worst = max(worst, float(np.abs(out[row:row + n] - ro).max()), float(np.abs(lse[row:row + n] - rl).max()))
        row += n
    return worst


def single_key_error(mod=pa):
    # each row sees exactly one key j_i <= its position: out = v[j_i], lse = q . k[j_i] / sqrt(d)
    qs, ks, vs = random_requests([(6, 10)], HQ, HKV, D, seed=5)
    rng = np.random.default_rng(6)
    mask = np.zeros((6, 10), dtype=bool)
    picks = [int(rng.integers(0, 4 + i + 1)) for i in range(6)]
    for i, j in enumerate(picks):
        mask[i, j] = True
    out, lse = _run(qs, ks, vs, [mask], mod=mod)
    g = HQ // HKV
    worst = 0.0
    for i, j in enumerate(picks):
        for h in range(HQ):
            worst = max(worst, float(np.abs(out[i, h] - vs[0][j, h // g]).max()))
            want = float(qs[0][i, h] @ ks[0][j, h // g]) / math.sqrt(D)
            worst = max(worst, abs(float(lse[i, h]) - want))
    return worst


TOL = 1e-12


def test_mask_matches_library_attention_with_a_boolean_mask():
    assert library_error() < TOL


def test_single_visible_key_closed_form():
    assert single_key_error() < TOL


def test_all_true_mask_is_no_mask():
    qs, ks, vs = random_requests(SPECS, HQ, HKV, D, seed=9)
    ones = [np.ones(s, dtype=bool) for s in SPECS]
    a, la = _run(qs, ks, vs, ones)
    b, lb = _run(qs, ks, vs, None)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


@pytest.mark.parametrize("window", [0, 1, 3])
def test_band_mask_reproduces_the_window_rule(window):
    # a mask that keeps positions p - window .. p of each row equals window_left = window
    specs = [(6, 13), (4, 4)]
    qs, ks, vs = random_requests(specs, HQ, HKV, D, seed=10 + window)
    masks = []
    for ql, kl in specs:
        m = np.zeros((ql, kl), dtype=bool)
        for i in range(ql):
            p = kl - ql + i
            m[i, max(0, p - window):p + 1] = True
        masks.append(m)
    a, la = _run(qs, ks, vs, masks)
    b, lb = _run(qs, ks, vs, None, window_left=window) if window else _run(qs, ks, vs, None, window_left=10 ** 6)
    if window == 0:  # window_left 0 means no window: compare with the diagonal-only closed form instead
        g = HQ // HKV
        row = 0
        for q, k, v, (ql, kl) in zip(qs, ks, vs, specs):
            for i in range(ql):
                p = kl - ql + i
                assert np.allclose(a[row + i], v[p][np.arange(HQ) // g], rtol=0, atol=TOL)
            row += ql
    else:
        assert np.abs(a - b).max() < TOL and np.abs(la - lb).max() < TOL


def test_empty_row_gives_zero_output_and_minus_infinity_lse():
    qs, ks, vs = random_requests([(3, 5)], HQ, HKV, D, seed=12)
    mask = np.ones((3, 5), dtype=bool)
    mask[1, :] = False
    out, lse = _run(qs, ks, vs, [mask])
    assert np.all(out[1] == 0.0) and np.all(np.isneginf(lse[1]))
    assert np.isfinite(out[[0, 2]]).all() and np.isfinite(lse[[0, 2]]).all()


def test_extend_rows_with_their_mask_rows_equal_the_full_prefill_rows():
    specs_full, tail = [(11, 11)], 4
    qs, ks, vs = random_requests(specs_full, HQ, HKV, D, seed=13)
    mask = _masks(specs_full, 14)[0]
    fo, fl = _run(qs, ks, vs, [mask])
    eo, el = _run([qs[0][-tail:]], ks, vs, [mask[-tail:]])
    assert np.array_equal(eo, fo[-tail:]) and np.array_equal(el, fl[-tail:])


def test_mask_shape_is_checked():
    qs, ks, vs = random_requests([(3, 5)], HQ, HKV, D, seed=15)
    with pytest.raises(ValueError):
        _run(qs, ks, vs, [np.ones((3, 4), dtype=bool)])


# planted mistakes: each plausible slip in applying the mask must fail a pin
def _planted(kind):
    real = pa.attend_rows

    def wrong(q_rows, keys, values, positions, sm_scale, window_left=0, mask_rows=None):
        if mask_rows is not None:
            m = np.asarray(mask_rows, dtype=bool)
            if kind == "ignored":
                m = None
            elif kind == "shifted":
                m = np.roll(m, 1, axis=1)
            elif kind == "or_with_causal":
                # visible = causal OR mask: every key is causally allowed here
                # (positions moved to the last key) and the mask is widened
                n_keys = keys.shape[0]
                pos = np.asarray(positions)
                causal = np.arange(n_keys)[None, :] <= pos[:, None]
                widened = causal | m[:, :n_keys]
                return real(q_rows, keys, values, np.full_like(pos, n_keys - 1), sm_scale, window_left, widened)
            mask_rows = m
        return real(q_rows, keys, values, positions, sm_scale, window_left, mask_rows)
    return wrong


@pytest.mark.parametrize("kind", ["ignored", "shifted", "or_with_causal"])
def test_planted_mask_mistake_is_caught(kind, monkeypatch):
    monkeypatch.setattr(pa, "attend_rows", _planted(kind))
    # the full-density mask past the diagonal exercises the OR slip
    errs = [library_error(seed=s) for s in (0, 20)] + [single_key_error()]
    assert max(errs) > 1e-6
