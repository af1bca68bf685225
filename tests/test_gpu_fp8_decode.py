"""E4M3 pages are decoded exactly, code by code, on the GPU.

With one key per request the softmax weight is exactly 1, so each output row
is the decoded V row (v_scale 1, exact in bf16), and with a one-hot q row the
lse is the selected K entry times 1/sqrt(d).  Every finite E4M3 code, the
subnormals and both zeros included, is placed in V and probed in K; the
expected values come from the oracle's decoder (the OCP E4M3 definition).
Both head dims run (their kernels convert with different dequant warpgroup
layouts).
"""

import math

import numpy as np
import pytest
import torch

from invariant_paged_prefill_gb300 import workloads as W
from oracle.formats import e4m3_bits_to_f64

from gpu_helpers import run_gpu

pytestmark = pytest.mark.gpu

HEADS = [W.HEADS_A, W.HEADS_B]  # (num_qo_heads, num_kv_heads, head_dim)
CODES = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)  # 254 finite codes


def _one_key_batch(k_codes: np.ndarray, v_codes: np.ndarray, q: torch.Tensor, heads) -> W.PagedBatch:
    """len(q) requests, each one key (one page of 16 slots, slot 0 used)."""
    HQ, HKV, D = heads
    n = q.shape[0]
    k_pages = torch.full((n, 16, HKV, D), 0x7F, dtype=torch.uint8)  # unused slots: NaN codes
    v_pages = torch.full((n, 16, HKV, D), 0x7F, dtype=torch.uint8)
    k_pages[:, 0] = torch.from_numpy(k_codes)
    v_pages[:, 0] = torch.from_numpy(v_codes)
    ar = torch.arange(n + 1, dtype=torch.int32)
    return W.PagedBatch(q=q, k_pages=k_pages, v_pages=v_pages, qo_indptr=ar, kv_indptr=ar.clone(),
                        kv_indices=torch.arange(n, dtype=torch.int32).flip(0).contiguous(),
                        kv_last_page_len=torch.ones(n, dtype=torch.int32), num_qo_heads=HQ,
                        num_kv_heads=HKV, head_dim=D, page_size=16, kv_dtype="fp8_e4m3",
                        q_lens=[1] * n, kv_lens=[1] * n)


@pytest.mark.parametrize("heads", HEADS, ids=lambda h: f"d{h[2]}")
def test_v_codes_decode_exactly(cuda, heads):
    # request r's V row holds every finite code (tiled); out row r = decoded V row
    HQ, HKV, D = heads
    n = 4
    rng = np.random.default_rng(0)
    v = np.stack([rng.permutation(np.resize(CODES, HKV * D)).reshape(HKV, D) for _ in range(n)]).astype(np.uint8)
    k = np.zeros((n, HKV, D), dtype=np.uint8)
    q = torch.randn(n, HQ, D, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    b = _one_key_batch(k, v, q, heads)
    out, lse, _ = run_gpu(b, cuda)
    # the kernel's pages are indexed through kv_indices (reversed): request r reads page n - 1 - r
    want = e4m3_bits_to_f64(v[::-1].copy())                                    # [n, Hkv, D]
    want = np.repeat(want, HQ // HKV, axis=1)                                   # q head h reads kv head h // 4
    got = out.float().numpy().astype(np.float64)
    assert np.array_equal(got, want), f"{np.sum(got != want)} decoded V values differ"
    assert torch.equal(lse, torch.zeros_like(lse))  # all-zero keys: one weight of exactly 1


@pytest.mark.parametrize("heads", HEADS, ids=lambda h: f"d{h[2]}")
def test_k_codes_decode_exactly(cuda, heads):
    # every q head is one-hot on its own column: lse = k[kv head, column] / sqrt(d)
    HQ, HKV, D = heads
    n = math.ceil(len(CODES) / HQ)
    k = np.zeros((n, HKV, D), dtype=np.uint8)
    q = torch.zeros(n, HQ, D, dtype=torch.bfloat16)
    probes = []
    for i, code in enumerate(CODES):
        r, h = divmod(i, HQ)
        col = (7 * h + 3) % D
        k[n - 1 - r, h // (HQ // HKV), col] = code   # request r reads page n - 1 - r
        q[r, h, col] = 1.0
        probes.append((r, h, code))
    v = np.zeros((n, HKV, D), dtype=np.uint8)
    b = _one_key_batch(k, v, q, heads)  # the q heads of a kv head probe 4 different columns
    out, lse, _ = run_gpu(b, cuda)
    for r, h, code in probes:
        want = float(e4m3_bits_to_f64(np.array([code], dtype=np.uint8))[0]) / math.sqrt(D)
        got = float(lse[r, h])
        assert abs(got - want) <= 1e-6 * max(1.0, abs(want)), f"code {code:#04x}: lse {got} vs {want}"


@pytest.mark.parametrize("heads", HEADS, ids=lambda h: f"d{h[2]}")
def test_nan_codes_inside_kv_len(cuda, heads):
    # The NaN codes 0x7F / 0xFF in a V row the softmax weights by exactly 1
    # give NaN outputs in their columns and touch no other column.
    HQ, HKV, D = heads
    v = np.zeros((1, HKV, D), dtype=np.uint8)
    v[0, :, 0], v[0, :, 1] = 0x7F, 0xFF
    k = np.zeros((1, HKV, D), dtype=np.uint8)
    q = torch.randn(1, HQ, D, generator=torch.Generator().manual_seed(2)).to(torch.bfloat16)
    out, _, _ = run_gpu(_one_key_batch(k, v, q, heads), cuda)
    got = out.float()[0]
    assert torch.isnan(got[:, :2]).all()
    assert torch.equal(got[:, 2:], torch.zeros_like(got[:, 2:]))
