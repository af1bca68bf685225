"""Writing new K/V rows into a paged cache: the step before attention.

TEST INFRASTRUCTURE ONLY (see the package docstring).

A request's new rows (its q_len newest tokens, one K row and one V row per
kv head) belong at sequence positions kv_len - q_len .. kv_len - 1, the same
tail alignment the attention uses (model-serving-minefield, "the tail rows of
the extend").  Position p of request r lives in page
``kv_indices[kv_indptr[r] + p // page_size]``, slot ``p % page_size`` (the
paged layout of the radix cache's page table).  An FP8 E4M3 cache stores
e4m3(x / scale): the bf16 value is widened to float32, divided by the scale
in float32 (IEEE round to nearest), then encoded by ``f64_to_e4m3_bits``
(nearest, ties to even, saturating at 448).  A bf16 cache stores the bf16
bits unchanged (scale 1).
"""

from __future__ import annotations

from typing import Sequence

import numpy as np

from .formats import f64_to_e4m3_bits
from .paged_attention import kv_lengths, q_lengths


def new_row_slots(qo_indptr: Sequence[int], kv_indptr: Sequence[int], kv_indices: Sequence[int],
                  kv_last_page_len: Sequence[int], page_size: int) -> list[tuple[int, int]]:
    """(page, slot) of every new row, in row order."""
    ql = q_lengths(qo_indptr)
    kl = kv_lengths(kv_indptr, kv_last_page_len, page_size)
    slots = []
    for r in range(len(ql)):
        for i in range(ql[r]):
            pos = kl[r] - ql[r] + i
            slots.append((int(kv_indices[kv_indptr[r] + pos // page_size]), pos % page_size))
    return slots


def quantize_e4m3(bf16_bits: np.ndarray, scale: float) -> np.ndarray:
    """e4m3(float32(x) / float32(scale)) for bf16 storage bits x."""
    word = (np.asarray(bf16_bits).astype(np.uint32) & 0xFFFF) << 16
    x = word.view(np.float32)
    with np.errstate(invalid="ignore", over="ignore"):
        y = x / np.float32(scale)
    return f64_to_e4m3_bits(y.astype(np.float64))


def append_paged_kv(k_new: np.ndarray, v_new: np.ndarray, k_pool: np.ndarray, v_pool: np.ndarray,
                    qo_indptr: Sequence[int], kv_indptr: Sequence[int], kv_indices: Sequence[int],
                    kv_last_page_len: Sequence[int], page_size: int, kv_dtype: str = "bf16",
                    k_scale: float = 1.0, v_scale: float = 1.0) -> tuple[np.ndarray, np.ndarray]:
    """Copies of the pools with the new rows written.

    k_new, v_new: bf16 storage bits (uint16) [total_q, Hkv, d].
    k_pool, v_pool: [num_pages, page_size, Hkv, d] of uint16 (bf16) or uint8 (e4m3).
    """
    k_out, v_out = k_pool.copy(), v_pool.copy()
    for row, (page, slot) in enumerate(new_row_slots(qo_indptr, kv_indptr, kv_indices, kv_last_page_len,
                                                     page_size)):
        if kv_dtype == "bf16":
            k_out[page, slot] = k_new[row]
            v_out[page, slot] = v_new[row]
        else:
            k_out[page, slot] = quantize_e4m3(k_new[row], k_scale)
            v_out[page, slot] = quantize_e4m3(v_new[row], v_scale)
    return k_out, v_out
