"""Pins for the oracle's paged KV append (CPU).

The expected pools never come from the oracle itself: they are the pools the
input generator lays out for the whole prompts (sglang PR 46351, "Root
cause": an extend sends the prompt's tail rows, q_len = seq_len -
prefix_len).  A batch whose tail rows hold junk gets the prompts' true tail
rows appended; afterwards the pools must equal the whole prompts' layout byte
for byte (so nothing else was touched), and every request's gathered keys and
values must end with its own tail rows.  Planted slips in the slot rule must
fail those pins.  FP8 quantisation is pinned against a library cast."""

import numpy as np
import pytest
import torch

from invariant_paged_prefill_gb300 import workloads as W
from oracle import kv_append as ka
from oracle.formats import e4m3_bits_to_f64
from oracle.kv_append import append_paged_kv, quantize_e4m3
from oracle.paged_attention import gather_request_kv, kv_lengths, q_lengths

LENS, Q_LENS = (45, 16, 70, 33), (5, 16, 1, 20)


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()


def _prompts(kv_dtype="bf16"):
    return [W.make_prompt(n, 4, 2, 128, seed=31 + i, kv_dtype=kv_dtype) for i, n in enumerate(LENS)]


def _with_tails(prompts, tails_k, tails_v):
    """The prompts with their last q_len K/V rows replaced."""
    out = []
    for p, ql, tk, tv in zip(prompts, Q_LENS, tails_k, tails_v):
        k, v = p.k.clone(), p.v.clone()
        k[p.n - ql:], v[p.n - ql:] = tk, tv
        out.append(W.Prompt(p.q, k, v))
    return out


def _append_case(kv_dtype, new_rows="prompt"):
    """(expected pools, pools after the oracle's append, tail rows, batch).

    Pools start as the layout of the prompts with junk tail rows; the rows
    appended are the prompts' tails ("prompt") or random rows ("random",
    expected = the layout of the prompts carrying those rows)."""
    prompts = _prompts(kv_dtype)
    junk = 0x7F if kv_dtype != "bf16" else float("nan")
    junk_k = [torch.full((ql,) + tuple(p.k.shape[1:]), junk, dtype=p.k.dtype) for p, ql in zip(prompts, Q_LENS)]
    holey = W.layout(_with_tails(prompts, junk_k, junk_k), Q_LENS, 16, seed_pages=3, kv_dtype=kv_dtype)
    if new_rows == "prompt":
        tails_k = [p.k[p.n - ql:] for p, ql in zip(prompts, Q_LENS)]
        tails_v = [p.v[p.n - ql:] for p, ql in zip(prompts, Q_LENS)]
        want = W.layout(prompts, Q_LENS, 16, seed_pages=3, kv_dtype=kv_dtype)
    else:
        g = torch.Generator().manual_seed(2)
        tails_k = [torch.randn((ql,) + tuple(p.k.shape[1:]), generator=g).to(torch.bfloat16) for p, ql in
                   zip(prompts, Q_LENS)]
        tails_v = [torch.randn((ql,) + tuple(p.k.shape[1:]), generator=g).to(torch.bfloat16) for p, ql in
                   zip(prompts, Q_LENS)]
        want = W.layout(_with_tails(prompts, tails_k, tails_v), Q_LENS, 16, seed_pages=3, kv_dtype=kv_dtype)
    # rows to append are bf16; E4M3 tails are their decoded values (which re-encode to the same codes)
    as_bf16 = (lambda t: t) if kv_dtype == "bf16" else (lambda t: t.view(torch.float8_e4m3fn).to(torch.bfloat16))
    k_new = _bits(torch.cat([as_bf16(t) for t in tails_k]))
    v_new = _bits(torch.cat([as_bf16(t) for t in tails_v]))
    kind = "bf16" if kv_dtype == "bf16" else "fp8"
    got_k, got_v = append_paged_kv(k_new, v_new, _bits(holey.k_pages), _bits(holey.v_pages), holey.qo_indptr,
                                   holey.kv_indptr, holey.kv_indices.tolist(), holey.kv_last_page_len, 16, kind)
    return (_bits(want.k_pages), _bits(want.v_pages)), (got_k, got_v), (tails_k, tails_v), holey


def _pins_hold(kv_dtype="bf16", new_rows="prompt") -> bool:
    (wk, wv), (gk, gv), (tk, tv), b = _append_case(kv_dtype, new_rows)
    ok = np.array_equal(gk, wk) and np.array_equal(gv, wv)
    kl = kv_lengths(b.kv_indptr, b.kv_last_page_len, 16)
    ql = q_lengths(b.qo_indptr)
    for r in range(len(ql)):
        keys = gather_request_kv(gk, b.kv_indices.tolist(), b.kv_indptr[r], kl[r], 16)
        vals = gather_request_kv(gv, b.kv_indices.tolist(), b.kv_indptr[r], kl[r], 16)
        ok &= np.array_equal(keys[kl[r] - ql[r]:], _bits(tk[r])) and np.array_equal(vals[kl[r] - ql[r]:], _bits(tv[r]))
    return bool(ok)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_append_of_the_prompt_tails_rebuilds_the_whole_prompt_pools(kv_dtype):
    assert _pins_hold(kv_dtype, "prompt")


def test_append_of_random_rows_lands_at_every_request_tail_and_nowhere_else():
    assert _pins_hold("bf16", "random")


def _slots_with(mistake):
    def wrong(qo_indptr, kv_indptr, kv_indices, kv_last_page_len, page_size):
        ql = q_lengths(qo_indptr)
        kl = kv_lengths(kv_indptr, kv_last_page_len, page_size)
        slots = []
        for r in range(len(ql)):
            for i in range(ql[r]):
                pos = kl[r] - ql[r] + i
                if mistake == "head_aligned":
                    pos = i
                elif mistake == "off_by_one":
                    pos = min(pos + 1, kl[r] - 1)
                base = 0 if mistake == "page_offset_dropped" else kv_indptr[r]
                if mistake == "slot_of_page_size_mod":
                    slot = (pos + 1) % page_size
                else:
                    slot = pos % page_size
                slots.append((int(kv_indices[base + pos // page_size]), slot))
        return slots
    return wrong


@pytest.mark.parametrize("mistake", ["page_offset_dropped", "head_aligned", "off_by_one", "slot_of_page_size_mod"])
def test_planted_append_mistake_is_caught(mistake, monkeypatch):
    monkeypatch.setattr(ka, "new_row_slots", _slots_with(mistake))
    assert not _pins_hold("bf16", "prompt"), f"planted append mistake {mistake} went unnoticed"


def test_fp8_quantisation_matches_library_cast():
    g = torch.Generator().manual_seed(4)
    x = (torch.randn(4096, generator=g) * 3).to(torch.bfloat16)
    bits = _bits(x)
    for scale in (1.0, 0.5, 2.3):
        want = (x.float() / torch.tensor(scale, dtype=torch.float32)).clamp(-448, 448)
        want = want.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(quantize_e4m3(bits, scale), want)


def test_fp8_append_decodes_close_to_the_values():
    prompts = _prompts()
    b = W.layout(prompts, Q_LENS, 16, seed_pages=3)
    total = b.qo_indptr[-1]
    g = torch.Generator().manual_seed(9)
    k_new = torch.randn(total, 2, 128, generator=g).to(torch.bfloat16)
    pool = np.zeros((b.k_pages.shape[0], 16, 2, 128), dtype=np.uint8)
    k_got, _ = append_paged_kv(_bits(k_new), _bits(k_new), pool, pool, b.qo_indptr, b.kv_indptr,
                               b.kv_indices.tolist(), b.kv_last_page_len, 16, "fp8", 0.5, 0.5)
    kl = kv_lengths(b.kv_indptr, b.kv_last_page_len, 16)
    rows = []
    for r, ql in enumerate(Q_LENS):
        keys = gather_request_kv(k_got, b.kv_indices.tolist(), b.kv_indptr[r], kl[r], 16)
        rows.append(keys[kl[r] - ql:])
    dec = e4m3_bits_to_f64(np.concatenate(rows)) * 0.5
    ref = k_new.double().numpy()
    assert np.all(np.abs(dec - ref) <= 2.0 ** -4 * np.abs(ref) + 2.0 ** -10)  # E4M3: 3 mantissa bits
