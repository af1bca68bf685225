"""Float64 definition of tail-aligned causal GQA prefill attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY (see the package docstring).  No kernel, header,
helper or constant is shared with the CUDA library.

What is computed, and where the pages fix it
--------------------------------------------
The method reaches ordinary causal attention exactly (up to rounding order),
so this module is that definition written out; it restates no algorithm.

* Paged KV layout and request lengths.  A request's keys/values live in pages
  named by ``kv_indices[kv_indptr[r]:kv_indptr[r+1]]``; the last page holds
  ``kv_last_page_len[r]`` valid slots (the paged-prefill wrapper of sglang
  PR 46351, "Validation"; array names as used there).  Hence
  ``kv_len = (num_pages - 1) * page_size + last_page_len`` (0 pages => 0).
  ``q_len = qo_indptr[r+1] - qo_indptr[r]``; the q tensor is
  ``[total_tokens, num_qo_heads, head_dim]`` with
  ``total_tokens = qo_indptr[-1]`` (the ValueError quoted in sglang PR 46351,
  Woody-Hu's A100 report).
* Tail alignment.  A request served from a radix-cache hit sends only its
  uncached tail, ``q_len = seq_len - prefix_len`` (sglang PR 46351,
  "Root cause"); q row ``i`` sits at sequence position
  ``i + kv_len - q_len`` and key ``j`` is masked when ``j > position``
  (sglang PR 46351, jbymy2000's reply, "Tail alignment").  The diagonal is
  included, so every row sees at least one key.
* GQA grouping.  Query heads are packed ``gqa_group = num_qo_heads /
  num_kv_heads`` to a KV head (sglang PR 46351, "Root cause": the packed q
  length is ``q_len * gqa_group``).  The pages do not say which query heads
  share a KV head; the reading taken is contiguous groups, ``h // group``.
* Scores, softmax, output.  ``s_j = q . k_j / sqrt(head_dim)``;
  ``out = sum_j softmax(s)_j v_j``; ``lse = log(sum_j exp(s_j))`` in natural
  log (the pages name "LSE" without a base; natural log is the reading).
* FP8 pages.  Codes are decoded with the E4M3 definition and multiplied by
  ``k_scale`` / ``v_scale`` (the pages give no scale semantics; scaling the
  decoded values is the reading, and equals folding ``k_scale`` into the
  logit scale and ``v_scale`` into the output).
* Slots at or beyond ``kv_len`` are never read.
* Custom masks.  The pages list "custom KV indices/masks" among the cases
  the padding skipped (sglang PR 46351, "Fix") without defining them.  The
  reading taken: an optional boolean mask per request, one row per q row and
  one column per key, that narrows the causal (and window) rule -- key j is
  visible to row i when the causal rule allows it and ``mask[i, j]`` is set.
  A row left with no visible key has no softmax; it is defined as out = 0,
  lse = -inf.

Structure: the small helpers below are the definition's pieces; the tests
replace one at a time with a plausible mistake to show the pins catch it.
"""

from __future__ import annotations

import math
from typing import Iterable, Sequence

import numpy as np

from .formats import bf16_bits_to_f64, e4m3_bits_to_f64


def q_lengths(qo_indptr: Sequence[int]) -> list[int]:
    """q rows per request: consecutive differences of ``qo_indptr``."""
    ind = [int(x) for x in qo_indptr]
    return [ind[r + 1] - ind[r] for r in range(len(ind) - 1)]


def kv_lengths(kv_indptr: Sequence[int], kv_last_page_len: Sequence[int], page_size: int) -> list[int]:
    """KV length per request from its page count and last-page fill."""
    ind = [int(x) for x in kv_indptr]
    out = []
    for r in range(len(ind) - 1):
        npages = ind[r + 1] - ind[r]
        out.append(0 if npages == 0 else (npages - 1) * page_size + int(kv_last_page_len[r]))
    return out


def row_position(i: int, q_len: int, kv_len: int) -> int:
    """Sequence position of local q row ``i`` (tail alignment)."""
    return i + kv_len - q_len


def kv_head_of(h: int, num_qo_heads: int, num_kv_heads: int) -> int:
    """KV head read by query head ``h`` (contiguous GQA groups)."""
    return h // (num_qo_heads // num_kv_heads)


def visible_keys(position: int) -> int:
    """Number of keys a row at ``position`` attends to (keys 0..position)."""
    return position + 1


def first_visible_key(position: int, window_left: int = 0) -> int:
    """First key a row at ``position`` attends to.

    Without a window (``window_left`` 0) every earlier key is visible.  With
    a sliding window of ``window_left`` keys to the left of the diagonal,
    the row sees keys ``position - window_left .. position`` (sliding-window
    KV pools are among the cases the padding skips, sglang PR 46351, "Fix"),
    clipped at 0.
    """
    return 0 if window_left <= 0 else max(0, position - window_left)


def gather_request_kv(pages: np.ndarray, kv_indices: Sequence[int], page_lo: int, kv_len: int,
                      page_size: int) -> np.ndarray:
    """Keys (or values) ``[kv_len, num_kv_heads, head_dim]`` of one request, token order.

    Token ``j`` lives in page ``kv_indices[page_lo + j // page_size]`` at slot
    ``j % page_size``.
    """
    pages = np.asarray(pages)
    if kv_len == 0:
        return np.zeros((0,) + pages.shape[2:], dtype=pages.dtype)
    toks = []
    for j in range(kv_len):
        page = int(kv_indices[page_lo + j // page_size])
        toks.append(pages[page, j % page_size])
    return np.stack(toks, axis=0)


def attend_rows(q_rows: np.ndarray, keys: np.ndarray, values: np.ndarray, positions: np.ndarray,
                sm_scale: float, window_left: int = 0,
                mask_rows: np.ndarray | None = None) -> tuple[np.ndarray, np.ndarray]:
    """Causal (optionally sliding-window, optionally custom-masked) softmax
    attention of some rows against one head's keys.

    q_rows ``[n, d]``, keys/values ``[kv_len, d]``, positions ``[n]``;
    mask_rows ``[n, >= kv_len]`` booleans (columns past kv_len ignored).
    Returns out ``[n, d]`` and natural-log lse ``[n]`` in float64; a row with
    no visible key gets out = 0 and lse = -inf.
    """
    scores = (q_rows @ keys.T) * sm_scale                       # [n, kv_len]
    kv_idx = np.arange(keys.shape[0])[None, :]
    visible = kv_idx < np.array([visible_keys(int(p)) for p in positions])[:, None]
    visible &= kv_idx >= np.array([first_visible_key(int(p), window_left) for p in positions])[:, None]
    if mask_rows is not None:
        visible &= np.asarray(mask_rows, dtype=bool)[:, :keys.shape[0]]
    scores = np.where(visible, scores, -np.inf)
    empty = ~visible.any(axis=1)
    m = np.where(empty[:, None], 0.0, scores.max(axis=1, keepdims=True))
    w = np.exp(scores - m)                                       # masked entries -> 0
    denom = w.sum(axis=1, keepdims=True)
    out = (w @ values) / np.where(empty[:, None], 1.0, denom)
    lse = np.where(empty, -np.inf, (m + np.log(np.where(empty[:, None], 1.0, denom)))[:, 0])
    return out, lse


def _as_f64(x, kind: str) -> np.ndarray:
    """Values as float64; ``kind`` is 'f64' (already numeric), 'bf16' or 'e4m3' (raw bits)."""
    if kind == "f64":
        return np.asarray(x, dtype=np.float64)
    if kind == "bf16":
        return bf16_bits_to_f64(x)
    if kind == "e4m3":
        return e4m3_bits_to_f64(x)
    raise ValueError(f"unknown storage kind {kind!r}")


def paged_prefill(q, k_pages, v_pages, qo_indptr, kv_indptr, kv_indices, kv_last_page_len,
                  num_qo_heads: int, num_kv_heads: int, page_size: int, *,
                  q_kind: str = "f64", kv_kind: str = "f64", k_scale: float = 1.0,
                  v_scale: float = 1.0, sm_scale: float | None = None,
                  rows: Iterable[int] | None = None, row_chunk: int = 512, window_left: int = 0,
                  custom_mask: Sequence[np.ndarray | None] | None = None):
    """Reference output and lse of paged causal GQA prefill.

    q ``[total_tokens, num_qo_heads, head_dim]``; k_pages/v_pages
    ``[num_pages, page_size, num_kv_heads, head_dim]``; storage kinds select
    how raw arrays are decoded ('f64', 'bf16' bits, 'e4m3' bits).

    ``rows`` restricts the computation to the listed token rows (all rows when
    None); the returned arrays then hold those rows in the order given.
    ``window_left`` > 0 restricts each row to its last window_left + 1 keys.
    ``custom_mask`` (one entry per request: a boolean ``[q_len, kv_len]``
    array, or None) further narrows which keys each q row sees.
    Returns ``(out [n, num_qo_heads, head_dim], lse [n, num_qo_heads])``.
    """
    q_raw = np.asarray(q)
    total, hq, d = q_raw.shape
    if hq != num_qo_heads or num_qo_heads % num_kv_heads != 0:
        raise ValueError("head counts do not match q or do not divide")
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(d)
    qo = [int(x) for x in qo_indptr]
    if qo[-1] != total:
        raise ValueError(f"q has {total} rows but qo_indptr[-1] = {qo[-1]}")
    qlens = q_lengths(qo)
    kvlens = kv_lengths(kv_indptr, kv_last_page_len, page_size)
    kv_ind = [int(x) for x in kv_indptr]

    wanted = np.arange(total) if rows is None else np.asarray(list(rows), dtype=np.int64)
    out = np.zeros((len(wanted), hq, d), dtype=np.float64)
    lse = np.zeros((len(wanted), hq), dtype=np.float64)
    order = {int(t): n for n, t in enumerate(wanted)}

    for r in range(len(qlens)):
        ql, kl = qlens[r], kvlens[r]
        if ql > kl:
            raise ValueError(f"request {r}: q_len {ql} > kv_len {kl}")
        mine = [t for t in range(qo[r], qo[r] + ql) if t in order]
        if not mine:
            continue
        # Gather the request's raw slots first, then decode only those.
        keys = _as_f64(gather_request_kv(k_pages, kv_indices, kv_ind[r], kl, page_size), kv_kind) * float(k_scale)
        vals = _as_f64(gather_request_kv(v_pages, kv_indices, kv_ind[r], kl, page_size), kv_kind) * float(v_scale)
        for c0 in range(0, len(mine), row_chunk):
            toks = mine[c0:c0 + row_chunk]
            pos = np.array([row_position(t - qo[r], ql, kl) for t in toks])
            last = int(pos.max()) + 1              # keys beyond the last position are never visible
            q_rows = _as_f64(q_raw[toks], q_kind)          # decode only the rows used
            for h in range(hq):
                hk = kv_head_of(h, num_qo_heads, num_kv_heads)
                mrows = None
                if custom_mask is not None and custom_mask[r] is not None:
                    mask_r = np.asarray(custom_mask[r], dtype=bool)
                    if mask_r.shape != (ql, kl):
                        raise ValueError(f"request {r}: custom mask must be [{ql}, {kl}]")
                    mrows = mask_r[[t - qo[r] for t in toks], :last]
                o, s = attend_rows(q_rows[:, h, :], keys[:last, hk, :], vals[:last, hk, :], pos, sm_scale,
                                   window_left, mrows)
                idx = [order[t] for t in toks]
                out[idx, h, :] = o
                lse[idx, h] = s
    return out, lse
