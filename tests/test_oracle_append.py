"""Pins for the oracle's paged KV append (CPU): positions, untouched slots,
agreement with pools laid out from the whole prompt, and FP8 quantisation
against a library cast."""

import numpy as np
import torch

from invariant_paged_prefill_gb300 import workloads as W
from oracle.formats import e4m3_bits_to_f64
from oracle.kv_append import append_paged_kv, new_row_slots, quantize_e4m3
from oracle.paged_attention import gather_request_kv, kv_lengths


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()


def _batch(kv_dtype="bf16"):
    prompts = [W.make_prompt(n, 4, 2, 128, seed=31 + i, kv_dtype=kv_dtype) for i, n in enumerate((45, 16, 70))]
    return prompts, W.layout(prompts, [5, 16, 1], 16, seed_pages=3, kv_dtype=kv_dtype, poison=True)


def test_new_rows_land_at_the_tail_positions():
    prompts, b = _batch()
    kl = kv_lengths(b.kv_indptr, b.kv_last_page_len, 16)
    slots = new_row_slots(b.qo_indptr, b.kv_indptr, b.kv_indices.tolist(), b.kv_last_page_len, 16)
    row = 0
    for r, n_new in enumerate((5, 16, 1)):
        for i in range(n_new):
            pos = kl[r] - n_new + i
            page = b.kv_indices.tolist()[b.kv_indptr[r] + pos // 16]
            assert slots[row] == (page, pos % 16)
            row += 1
    assert len(set(slots)) == len(slots)  # no two new rows share a slot


def test_append_rebuilds_the_pools_of_the_whole_prompt():
    # Pools laid out from the whole prompt, with the new rows' slots
    # overwritten by junk, get every new row back from the append.
    prompts, b = _batch()
    k_pool, v_pool = _bits(b.k_pages), _bits(b.v_pages)
    slots = new_row_slots(b.qo_indptr, b.kv_indptr, b.kv_indices.tolist(), b.kv_last_page_len, 16)
    k_new = np.stack([k_pool[p, s] for p, s in slots])
    v_new = np.stack([v_pool[p, s] for p, s in slots])
    k_hole, v_hole = k_pool.copy(), v_pool.copy()
    for p, s in slots:
        k_hole[p, s] = 0x7FC0
        v_hole[p, s] = 0x1234
    k_got, v_got = append_paged_kv(k_new, v_new, k_hole, v_hole, b.qo_indptr, b.kv_indptr,
                                   b.kv_indices.tolist(), b.kv_last_page_len, 16)
    assert np.array_equal(k_got, k_pool) and np.array_equal(v_got, v_pool)
    # and the request's gathered keys end with the new rows
    kl = kv_lengths(b.kv_indptr, b.kv_last_page_len, 16)
    keys = gather_request_kv(k_got, b.kv_indices.tolist(), b.kv_indptr[0], kl[0], 16)
    assert np.array_equal(keys[kl[0] - 5:], k_new[:5])


def test_append_touches_nothing_else():
    prompts, b = _batch()
    k_pool, v_pool = _bits(b.k_pages), _bits(b.v_pages)
    rng = np.random.default_rng(2)
    total = b.qo_indptr[-1]
    k_new = rng.integers(0, 1 << 15, (total, 2, 128)).astype(np.uint16)
    v_new = rng.integers(0, 1 << 15, (total, 2, 128)).astype(np.uint16)
    k_got, v_got = append_paged_kv(k_new, v_new, k_pool, v_pool, b.qo_indptr, b.kv_indptr,
                                   b.kv_indices.tolist(), b.kv_last_page_len, 16)
    mask = np.ones(k_pool.shape[:2], dtype=bool)
    for p, s in new_row_slots(b.qo_indptr, b.kv_indptr, b.kv_indices.tolist(), b.kv_last_page_len, 16):
        mask[p, s] = False
    assert np.array_equal(k_got[mask], k_pool[mask], equal_nan=False)
    assert np.array_equal(v_got[mask], v_pool[mask])


def test_fp8_quantisation_matches_library_cast():
    g = torch.Generator().manual_seed(4)
    x = (torch.randn(4096, generator=g) * 3).to(torch.bfloat16)
    bits = _bits(x)
    for scale in (1.0, 0.5, 2.3):
        want = (x.float() / torch.tensor(scale, dtype=torch.float32)).clamp(-448, 448)
        want = want.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(quantize_e4m3(bits, scale), want)


def test_fp8_append_decodes_close_to_the_values():
    prompts, b = _batch()
    total = b.qo_indptr[-1]
    g = torch.Generator().manual_seed(9)
    k_new = torch.randn(total, 2, 128, generator=g).to(torch.bfloat16)
    pool = np.zeros((b.k_pages.shape[0], 16, 2, 128), dtype=np.uint8)
    k_got, _ = append_paged_kv(_bits(k_new), _bits(k_new), pool, pool, b.qo_indptr, b.kv_indptr,
                               b.kv_indices.tolist(), b.kv_last_page_len, 16, "fp8", 0.5, 0.5)
    slots = new_row_slots(b.qo_indptr, b.kv_indptr, b.kv_indices.tolist(), b.kv_last_page_len, 16)
    dec = np.stack([e4m3_bits_to_f64(k_got[p, s]) for p, s in slots]) * 0.5
    ref = k_new.double().numpy()
    assert np.all(np.abs(dec - ref) <= 2.0 ** -4 * np.abs(ref) + 2.0 ** -10)  # E4M3: 3 mantissa bits
