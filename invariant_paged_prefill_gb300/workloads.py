"""Seeded synthetic inputs for paged prefill attention.

This module only draws random numbers and lays tokens out in page pools; it
holds none of the attention arithmetic.  Both the CUDA-path tests and the
oracle tests take their inputs from here.

Value recipe (the pages' model shapes with synthetic values):
* q, k, v ~ N(0, 1) in float32, rounded to bf16.
* FP8 pages: N(0, 1) clipped to +-448, cast to ``float8_e4m3fn`` and stored
  as raw uint8 codes.
* Page ids: a seeded random permutation of the pool; pool pages and slots
  that no request owns are poisoned (NaN) so that any read of them shows up.
* Seeds: data 0, pages 1, lengths 2 unless a caller passes others.
* Custom masks (``prompt_mask``): one boolean ``[n, n]`` mask per prompt, a
  row pattern drawn per row (all keys, a random half, a contiguous range of
  keys ending at the row, or none); an extend takes the prompt mask's tail
  rows, so its rows carry the same mask rows as the full prefill.

A request is a *prompt* (per-token q, k, v for ``kv_len`` tokens) plus the
number of tail rows ``q_len`` sent to attention.  The q rows of a request
are the prompt's last ``q_len`` rows, so an extend and a full prefill of the
same prompt see identical data.  Radix-cache prefix hits are modelled by
letting requests that share a prompt prefix also share its pages.
"""

from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import numpy as np
import torch

BF16_NAN_BITS = 0x7FC0
E4M3_NAN_CODE = 0x7F
KV_DTYPES = ("bf16", "fp8_e4m3")


@dataclasses.dataclass
class Prompt:
    q: torch.Tensor  # [n, Hq, d] bf16
    k: torch.Tensor  # [n, Hkv, d] bf16, or uint8 E4M3 codes
    v: torch.Tensor

    @property
    def n(self) -> int:
        return int(self.q.shape[0])


@dataclasses.dataclass
class PagedBatch:
    q: torch.Tensor                # [total_q, Hq, d] bf16
    k_pages: torch.Tensor          # [num_pages, page_size, Hkv, d] bf16 or uint8
    v_pages: torch.Tensor
    qo_indptr: torch.Tensor        # int32 [B+1] (host)
    kv_indptr: torch.Tensor        # int32 [B+1] (host)
    kv_indices: torch.Tensor       # int32 [kv_indptr[-1]] (same device as the pages)
    kv_last_page_len: torch.Tensor  # int32 [B] (host)
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    kv_dtype: str
    q_lens: list
    kv_lens: list

    @property
    def batch(self) -> int:
        return len(self.q_lens)

    @property
    def total_q(self) -> int:
        return int(self.qo_indptr[-1])

    def to(self, device) -> "PagedBatch":
        return dataclasses.replace(
            self, q=self.q.to(device), k_pages=self.k_pages.to(device),
            v_pages=self.v_pages.to(device), kv_indices=self.kv_indices.to(device))

    def row_range(self, r: int) -> tuple[int, int]:
        return int(self.qo_indptr[r]), int(self.qo_indptr[r + 1])


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal(shape, gen, device) -> torch.Tensor:
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32)


def _kv_store(x: torch.Tensor, kv_dtype: str) -> torch.Tensor:
    if kv_dtype == "bf16":
        return x.to(torch.bfloat16)
    if kv_dtype == "fp8_e4m3":
        return x.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    raise ValueError(f"kv_dtype must be one of {KV_DTYPES}")


def make_prompt(n: int, num_qo_heads: int, num_kv_heads: int, head_dim: int, seed: int,
                kv_dtype: str = "bf16", device="cpu") -> Prompt:
    """``n`` tokens of q/k/v drawn from N(0,1) with one generator seeded ``seed``."""
    g = _gen(seed, device)
    q = _normal((n, num_qo_heads, head_dim), g, device).to(torch.bfloat16)
    k = _kv_store(_normal((n, num_kv_heads, head_dim), g, device), kv_dtype)
    v = _kv_store(_normal((n, num_kv_heads, head_dim), g, device), kv_dtype)
    return Prompt(q, k, v)


def concat_prompts(*parts: Prompt) -> Prompt:
    return Prompt(torch.cat([p.q for p in parts]), torch.cat([p.k for p in parts]),
                  torch.cat([p.v for p in parts]))


def layout(prompts: Sequence[Prompt], q_lens: Sequence[int], page_size: int, *, seed_pages: int = 1,
           share_prefix_tokens: int = 0, kv_dtype: str = "bf16", extra_pages: int = 3,
           poison: bool = True, page_stride_pad: int = 0) -> PagedBatch:
    """Place prompts in a shuffled page pool and select each request's tail q rows.

    ``share_prefix_tokens`` (a multiple of ``page_size``): every request's
    first that-many tokens are identical and stored once, in pages that all
    requests' page lists name (a radix-cache hit).  ``extra_pages`` unused
    pool pages are added and poisoned.  ``page_stride_pad`` adds that many
    elements of padding after each page (a strided pool).
    """
    assert len(prompts) == len(q_lens)
    p0 = prompts[0]
    device = p0.q.device
    hq, hkv, d = p0.q.shape[1], p0.k.shape[1], p0.q.shape[2]
    if share_prefix_tokens:
        assert share_prefix_tokens % page_size == 0
        for p in prompts[1:]:
            assert torch.equal(p.k[:share_prefix_tokens], p0.k[:share_prefix_tokens])
            assert torch.equal(p.v[:share_prefix_tokens], p0.v[:share_prefix_tokens])
    shared_pages = share_prefix_tokens // page_size
    npages = [(p.n + page_size - 1) // page_size for p in prompts]
    total_pages = shared_pages + sum(n - shared_pages if shared_pages else n for n in npages) + extra_pages
    perm = torch.randperm(total_pages, generator=_gen(seed_pages, "cpu")).to(torch.int32)

    elem_dtype = torch.bfloat16 if kv_dtype == "bf16" else torch.uint8
    page_elems = page_size * hkv * d + page_stride_pad
    kflat = torch.empty(total_pages * page_elems, dtype=elem_dtype, device=device)
    vflat = torch.empty_like(kflat)
    if poison:
        bits = BF16_NAN_BITS if kv_dtype == "bf16" else E4M3_NAN_CODE
        view_dt = torch.int16 if kv_dtype == "bf16" else torch.uint8
        kflat.view(view_dt).fill_(bits)
        vflat.view(view_dt).fill_(bits)
    else:
        kflat.zero_()
        vflat.zero_()
    kp = kflat.as_strided((total_pages, page_size, hkv, d), (page_elems, hkv * d, d, 1))
    vp = vflat.as_strided((total_pages, page_size, hkv, d), (page_elems, hkv * d, d, 1))

    cursor = 0
    shared_ids = perm[:shared_pages]
    cursor = shared_pages
    kv_indices, kv_indptr, last = [], [0], []
    for r, p in enumerate(prompts):
        if shared_pages:
            own = perm[cursor:cursor + npages[r] - shared_pages]
            cursor += npages[r] - shared_pages
            ids = torch.cat([shared_ids, own])
        else:
            ids = perm[cursor:cursor + npages[r]]
            cursor += npages[r]
        # Token j goes to page ids[j // page_size], slot j % page_size; shared
        # prefix tokens are written once, by request 0.
        j0 = share_prefix_tokens if (shared_pages and r > 0) else 0
        j = torch.arange(j0, p.n, device=device)
        page_of = ids.to(device=device, dtype=torch.long)[j // page_size]
        kp[page_of, j % page_size] = p.k[j0:]
        vp[page_of, j % page_size] = p.v[j0:]
        kv_indices.append(ids)
        kv_indptr.append(kv_indptr[-1] + npages[r])
        last.append(p.n - (npages[r] - 1) * page_size if npages[r] else 0)

    q_rows = [p.q[p.n - ql:] for p, ql in zip(prompts, q_lens)]
    qo = [0]
    for ql in q_lens:
        qo.append(qo[-1] + int(ql))
    idx = torch.cat(kv_indices) if kv_indices else torch.zeros(0, dtype=torch.int32)
    return PagedBatch(
        q=torch.cat(q_rows).contiguous() if q_rows else torch.zeros((0, hq, d), dtype=torch.bfloat16, device=device),
        k_pages=kp, v_pages=vp,
        qo_indptr=torch.tensor(qo, dtype=torch.int32),
        kv_indptr=torch.tensor(kv_indptr, dtype=torch.int32),
        kv_indices=idx.to(torch.int32).to(device),
        kv_last_page_len=torch.tensor(last, dtype=torch.int32),
        num_qo_heads=hq, num_kv_heads=hkv, head_dim=d, page_size=page_size, kv_dtype=kv_dtype,
        q_lens=[int(x) for x in q_lens], kv_lens=[p.n for p in prompts])


# ---------------------------------------------------------------------------
# The five workloads, by their shapes.
# ---------------------------------------------------------------------------

HEADS_A = (32, 8, 128)   # num_qo_heads, num_kv_heads, head_dim
HEADS_B = (24, 4, 256)
PAGE_SIZE = 16


def tiny(q_len: int, *, seed_data: int = 0, seed_pages: int = 1, kv_dtype: str = "bf16",
         device="cpu") -> PagedBatch:
    """One request, 32/8/128, kv_len 64 on 4 shuffled pages, the last ``q_len`` rows sent."""
    p = make_prompt(64, *HEADS_A, seed=seed_data, kv_dtype=kv_dtype, device=device)
    return layout([p], [q_len], PAGE_SIZE, seed_pages=seed_pages, kv_dtype=kv_dtype)


def radix_burst(*, n_req: int = 16, prefix: int = 1024, seed_data: int = 0, seed_pages: int = 1,
                seed_lengths: int = 2, kv_dtype: str = "bf16", device="cpu", page_size: int = PAGE_SIZE):
    """16 requests behind a shared 1024-token prefix, tails of 1-4 tokens.

    Returns ``(extend, cold)``: the extend batch sends only the tails and
    shares the prefix pages; the cold batch prefills the same prompts in
    full on private pages (different page ids, same values).
    """
    hq, hkv, d = HEADS_A
    tails = torch.randint(1, 5, (n_req,), generator=_gen(seed_lengths, "cpu")).tolist()
    pre = make_prompt(prefix, hq, hkv, d, seed=seed_data, kv_dtype=kv_dtype, device=device)
    prompts = [concat_prompts(pre, make_prompt(t, hq, hkv, d, seed=seed_data + 1000 + i,
                                               kv_dtype=kv_dtype, device=device))
               for i, t in enumerate(tails)]
    extend = layout(prompts, tails, page_size, seed_pages=seed_pages, share_prefix_tokens=prefix,
                    kv_dtype=kv_dtype)
    cold = layout(prompts, [p.n for p in prompts], page_size, seed_pages=seed_pages + 100,
                  kv_dtype=kv_dtype)
    return extend, cold


def mixed_ragged_specs(seed_lengths: int = 2):
    """(q_len, kv_len) of the mixed batch: a 3700-token prefill and four extends."""
    g = _gen(seed_lengths, "cpu")
    specs = [(3700, 3700)]
    for ql in (2, 4, 6, 37):
        prefix = int(torch.randint(500, 3001, (1,), generator=g))
        specs.append((ql, prefix + ql))
    return specs


def mixed_ragged_prompts(*, seed_data: int = 0, kv_dtype: str = "bf16", device="cpu"):
    hq, hkv, d = HEADS_A
    specs = mixed_ragged_specs()
    prompts = [make_prompt(kv, hq, hkv, d, seed=seed_data + 10 * i, kv_dtype=kv_dtype, device=device)
               for i, (_, kv) in enumerate(specs)]
    return prompts, [ql for ql, _ in specs]


def large_head(n_tokens: int, *, seed_data: int = 0, seed_pages: int = 1, kv_dtype: str = "bf16",
               device="cpu") -> PagedBatch:
    """A single fresh 24/4/256 prefill of ``n_tokens`` (8192 or 32768)."""
    p = make_prompt(n_tokens, *HEADS_B, seed=seed_data, kv_dtype=kv_dtype, device=device)
    return layout([p], [n_tokens], PAGE_SIZE, seed_pages=seed_pages, kv_dtype=kv_dtype)


def sweep_point(heads: Sequence[int], q_len: int, kv_len: int, *, batch: int = 16, kv_dtype: str = "bf16",
                seed_data: int = 0, seed_pages: int = 1, device="cpu", poison: bool = True,
                page_size: int = PAGE_SIZE) -> PagedBatch:
    """Batch of ``batch`` requests with private pages, each ``q_len`` rows behind ``kv_len`` keys."""
    hq, hkv, d = heads
    assert kv_len >= q_len
    prompts = [make_prompt(kv_len, hq, hkv, d, seed=seed_data + 7 * i, kv_dtype=kv_dtype, device=device)
               for i in range(batch)]
    return layout(prompts, [q_len] * batch, page_size, seed_pages=seed_pages, kv_dtype=kv_dtype,
                  poison=poison)


SWEEP_Q = (1, 4, 32, 128, 1028, 8192)
SWEEP_KV = (1028, 8192, 32768)


def sweep_grid():
    """(heads, q_len, kv_len) points of the throughput sweep with kv_len >= q_len."""
    pts = []
    for heads in (HEADS_A, HEADS_B):
        for ql in SWEEP_Q:
            for kv in SWEEP_KV:
                kv_eff = max(kv, ql)
                if (heads, ql, kv_eff) not in pts:
                    pts.append((heads, ql, kv_eff))
    return pts


MASK_ROW_KINDS = ("all", "half", "range", "none")


def prompt_mask(n: int, seed: int, probs: Sequence[float] = (0.4, 0.4, 0.15, 0.05)) -> np.ndarray:
    """Seeded boolean custom mask ``[n, n]`` for the full prefill of an n-token prompt.

    Row i (sequence position i) follows one of ``MASK_ROW_KINDS``, drawn with
    ``probs``: every key; each key with probability 1/2; keys s .. n - 1 for a
    uniform s in [0, i]; no key.  Bits past a row's own position are drawn too
    (attention ignores them).  Row i of an extend is row kv_len - q_len + i.
    """
    rng = np.random.default_rng(seed)
    kind = rng.choice(len(MASK_ROW_KINDS), size=n, p=np.asarray(probs, dtype=np.float64))
    m = rng.random((n, n)) < 0.5
    start = (rng.random(n) * (np.arange(n) + 1)).astype(np.int64)
    cols = np.arange(n)[None, :]
    m[kind == 0] = True
    m[kind == 2] = cols >= start[kind == 2][:, None]
    m[kind == 3] = False
    return m
