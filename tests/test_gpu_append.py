"""Paged KV append on the GPU against the oracle: whole pools compared byte for
byte (bf16 bits, E4M3 codes), then the append composed with the attention of
an extend."""

import numpy as np
import pytest
import torch

import invariant_paged_prefill_gb300 as bip
from invariant_paged_prefill_gb300 import workloads as W
from oracle.kv_append import append_paged_kv

from gpu_helpers import assert_bitwise, oracle, assert_close_to_oracle, run_gpu, to_device

pytestmark = pytest.mark.gpu


def _np_bits(t: torch.Tensor) -> np.ndarray:
    t = t.cpu()
    return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()


def _pool_bits(pages: torch.Tensor) -> np.ndarray:
    """The whole pool storage (every page, padding included) as raw bits."""
    n = pages.untyped_storage().nbytes() // pages.element_size()
    return _np_bits(torch.as_strided(pages, (n,), (1,), 0))


def _batch(heads, lens, q_lens, kv_dtype, stride_pad=0, seed=0):
    prompts = [W.make_prompt(n, *heads, seed=seed + 13 * i, kv_dtype=kv_dtype) for i, n in enumerate(lens)]
    return W.layout(prompts, q_lens, 16, seed_pages=seed + 1, kv_dtype=kv_dtype, poison=True,
                    page_stride_pad=stride_pad)


def _append_gpu(b, cuda, k_new, v_new, k_scale=1.0, v_scale=1.0):
    d = to_device(b, cuda)
    plan = bip.Plan(d.qo_indptr, d.kv_indptr, d.kv_last_page_len, num_qo_heads=d.num_qo_heads,
                    num_kv_heads=d.num_kv_heads, head_dim=d.head_dim, page_size=d.page_size, kv_dtype=d.kv_dtype)
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device=cuda)
    bip.append_kv(plan, k_new.to(cuda), v_new.to(cuda), d.k_pages, d.v_pages, d.kv_indices, workspace=ws,
                  k_scale=k_scale, v_scale=v_scale)
    status = bip.read_device_status(ws)
    return d, status


def _oracle_append(b, k_new, v_new, k_scale=1.0, v_scale=1.0):
    kv = "bf16" if b.kv_dtype == "bf16" else "fp8"
    # the oracle works on [pages, slots, heads, d] views of the raw storage
    k_pool = _pool_bits(b.k_pages)
    v_pool = _pool_bits(b.v_pages)
    stride = b.k_pages.stride(0)
    page_elems = int(np.prod(b.k_pages.shape[1:]))
    k_pages = np.lib.stride_tricks.as_strided(k_pool, (b.k_pages.shape[0],) + tuple(b.k_pages.shape[1:]),
                                              (stride * k_pool.itemsize,) + tuple(
                                                  s * k_pool.itemsize for s in b.k_pages.stride()[1:]))
    v_pages = np.lib.stride_tricks.as_strided(v_pool, k_pages.shape, k_pages.strides)
    kw, vw = append_paged_kv(_np_bits(k_new), _np_bits(v_new), np.ascontiguousarray(k_pages),
                             np.ascontiguousarray(v_pages), b.qo_indptr.tolist(), b.kv_indptr.tolist(),
                             b.kv_indices.tolist(), b.kv_last_page_len.tolist(), b.page_size, kv, k_scale, v_scale)
    # written pools back into full storage images (padding untouched)
    k_img, v_img = k_pool.copy(), v_pool.copy()
    for p in range(b.k_pages.shape[0]):
        k_img[p * stride:p * stride + page_elems] = kw[p].reshape(-1)
        v_img[p * stride:p * stride + page_elems] = vw[p].reshape(-1)
    return k_img, v_img


def _new_rows(b, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    shape = (int(b.qo_indptr[-1]), b.num_kv_heads, b.head_dim)
    k = (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)
    v = (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)
    return k, v


@pytest.mark.parametrize("heads", [W.HEADS_A, W.HEADS_B])
@pytest.mark.parametrize("stride_pad", [0, 64])
def test_bf16_append_writes_exactly_the_oracle_pools(cuda, heads, stride_pad):
    # ragged: a tail crossing page boundaries, a whole-page tail, a one-row
    # tail, a request with no new rows, a fresh prompt
    b = _batch(heads, [200, 48, 33, 70, 17], [37, 16, 1, 0, 17], "bf16", stride_pad=stride_pad)
    k_new, v_new = _new_rows(b, 5)
    d, status = _append_gpu(b, cuda, k_new, v_new)
    assert status == 0
    want_k, want_v = _oracle_append(b, k_new, v_new)
    got_k, got_v = _pool_bits(d.k_pages), _pool_bits(d.v_pages)
    assert np.array_equal(got_k, want_k) and np.array_equal(got_v, want_v)


@pytest.mark.parametrize("heads", [W.HEADS_A, W.HEADS_B])
@pytest.mark.parametrize("scales", [(1.0, 1.0), (0.5, 2.3), (0.01, 0.01)])
def test_fp8_append_writes_exactly_the_oracle_codes(cuda, heads, scales):
    # scale 0.01 drives many values past 448: saturation; small values hit subnormals
    b = _batch(heads, [130, 40, 9], [61, 40, 2], "fp8_e4m3")
    k_new, v_new = _new_rows(b, 8, scale=3.0)
    d, status = _append_gpu(b, cuda, k_new, v_new, *scales)
    assert status == 0
    want_k, want_v = _oracle_append(b, k_new, v_new, *scales)
    assert np.array_equal(_pool_bits(d.k_pages), want_k)
    assert np.array_equal(_pool_bits(d.v_pages), want_v)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_append_then_extend_equals_the_full_prefill(cuda, kv_dtype):
    # Six prompts behind a shared 304-token prefix.  Pools laid out from the
    # prompts with junk tail rows get each prompt's own tail rows appended
    # (sglang PR 46351, "Root cause": the extend sends q_len = seq_len -
    # prefix_len tail rows): the pools must equal the whole prompts' layout
    # byte for byte, and the extend's attention on them equals the extend on
    # the laid-out pools and the oracle.
    hq, hkv, d = W.HEADS_A
    tails = [1, 4, 2, 3, 4, 1]
    pre = W.make_prompt(304, hq, hkv, d, seed=0, kv_dtype=kv_dtype)
    prompts = [W.concat_prompts(pre, W.make_prompt(t, hq, hkv, d, seed=1000 + i, kv_dtype=kv_dtype))
               for i, t in enumerate(tails)]
    junk = 0x7F if kv_dtype == "fp8_e4m3" else float("nan")
    holes = []
    for p, t in zip(prompts, tails):
        k, v = p.k.clone(), p.v.clone()
        k[p.n - t:] = junk
        v[p.n - t:] = junk
        holes.append(W.Prompt(p.q, k, v))
    kw = dict(seed_pages=1, share_prefix_tokens=304, kv_dtype=kv_dtype)
    b = W.layout(prompts, tails, 16, **kw)
    holey = W.layout(holes, tails, 16, **kw)
    k_new = torch.cat([p.k[p.n - t:] for p, t in zip(prompts, tails)])
    v_new = torch.cat([p.v[p.n - t:] for p, t in zip(prompts, tails)])
    if kv_dtype == "fp8_e4m3":  # rows to append are bf16: the decoded E4M3 values re-encode to the same codes
        k_new = k_new.view(torch.float8_e4m3fn).to(torch.bfloat16)
        v_new = v_new.view(torch.float8_e4m3fn).to(torch.bfloat16)
    d_, status = _append_gpu(holey, cuda, k_new, v_new)
    assert status == 0
    assert np.array_equal(_pool_bits(d_.k_pages), _pool_bits(b.k_pages))
    assert np.array_equal(_pool_bits(d_.v_pages), _pool_bits(b.v_pages))
    out_a, lse_a, _ = run_gpu(d_, cuda)
    out_b, lse_b, _ = run_gpu(b, cuda)
    assert_bitwise(out_a, out_b, "extend after append vs extend on the laid-out pools")
    assert_bitwise(lse_a, lse_b, "lse")
    ro, rl = oracle(b)
    assert_close_to_oracle(out_a, lse_a, ro, rl)


def test_out_of_range_page_id_is_counted_and_skipped(cuda):
    b = _batch(W.HEADS_A, [40], [20], "bf16")
    k_new, v_new = _new_rows(b, 3)
    bad = b.kv_indices.clone()
    bad[1] = b.k_pages.shape[0] + 7          # the page holding positions 16..31
    bb = W.PagedBatch(**{**b.__dict__, "kv_indices": bad})
    d, status = _append_gpu(bb, cuda, k_new, v_new)
    assert status == 7  # BIP_ERR_BAD_PAGE_INDEX
    # rows bound for valid pages were written, the others nowhere
    want_k, _ = _oracle_append(b, k_new, v_new)
    got_k = _pool_bits(d.k_pages)
    stride = b.k_pages.stride(0)
    page_elems = int(np.prod(b.k_pages.shape[1:]))
    p_ok = int(b.kv_indices[2])
    assert np.array_equal(got_k[p_ok * stride:p_ok * stride + page_elems],
                          want_k[p_ok * stride:p_ok * stride + page_elems])
