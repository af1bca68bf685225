"""Device-planned, graph-replayable prefill: the same bits as the host-planned
launch for the same batch, eagerly, under CUDA graph replay with new batches
in the captured buffers, and across captured buckets (a radix hit and the
full recompute of the same prompts); short batches split by segment on the
device; custom masks through the graph launch."""

import numpy as np
import pytest
import torch

import invariant_paged_prefill_gb300 as bip
from invariant_paged_prefill_gb300 import workloads as W

from gpu_helpers import assert_bitwise, assert_close_to_oracle, oracle, run_gpu, to_device

pytestmark = pytest.mark.gpu


class Bucket:
    """Static device buffers of one captured bucket (batch and row capacity)."""

    def __init__(self, cuda, max_batch, max_total_q, heads, num_pages, kv_dtype="bf16", max_pages_idx=None):
        hq, hkv, d = heads
        self.cuda, self.max_batch, self.max_total_q, self.heads = cuda, max_batch, max_total_q, heads
        self.plan = bip.GraphPlan(max_batch, max_total_q, num_qo_heads=hq, num_kv_heads=hkv, head_dim=d,
                                  kv_dtype=kv_dtype)
        i32 = dict(dtype=torch.int32, device=cuda)
        self.qo = torch.zeros(max_batch + 1, **i32)
        self.kv = torch.zeros(max_batch + 1, **i32)
        self.last = torch.ones(max_batch, **i32)
        self.q = torch.zeros(max_total_q, hq, d, dtype=torch.bfloat16, device=cuda)
        self.out = torch.zeros_like(self.q)
        self.lse = torch.zeros(max_total_q, hq, dtype=torch.float32, device=cuda)
        self.ws = torch.empty(self.plan.workspace_bytes, dtype=torch.uint8, device=cuda)
        self.idx = torch.zeros(max_pages_idx or num_pages, **i32)

    def load(self, b: W.PagedBatch):
        """Copy a batch into the buffers, padding with empty requests."""
        n = len(b.q_lens)
        assert n <= self.max_batch and b.q.shape[0] <= self.max_total_q
        qo = torch.full((self.max_batch + 1,), int(b.qo_indptr[-1]), dtype=torch.int32)
        kv = torch.full((self.max_batch + 1,), int(b.kv_indptr[-1]), dtype=torch.int32)
        qo[: n + 1] = torch.as_tensor(np.asarray(b.qo_indptr), dtype=torch.int32)
        kv[: n + 1] = torch.as_tensor(np.asarray(b.kv_indptr), dtype=torch.int32)
        last = torch.ones(self.max_batch, dtype=torch.int32)
        last[:n] = torch.as_tensor(np.asarray(b.kv_last_page_len), dtype=torch.int32)
        self.qo.copy_(qo)
        self.kv.copy_(kv)
        self.last.copy_(last)
        self.q.zero_()
        self.q[: b.q.shape[0]].copy_(b.q)
        self.idx.zero_()
        self.idx[: b.kv_indices.numel()].copy_(b.kv_indices)
        self.out.fill_(float("nan"))
        self.lse.fill_(float("nan"))

    def launch(self, k_pages, v_pages, custom_mask=None):
        bip.prefill_graph(self.plan, self.max_batch, self.qo, self.kv, self.last, self.q, k_pages, v_pages,
                          self.idx, self.out, self.lse, self.ws, custom_mask=custom_mask)


def _merges_written(ws) -> int:
    """Merge units the device planner wrote (workspace header word 4)."""
    return int(ws[16:20].view(torch.int32).item())


def _capture(fn):
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    return graph


def test_device_planned_launch_equals_host_planned(cuda):
    prompts, q_lens = W.mixed_ragged_prompts()
    mixed = W.layout(prompts, q_lens, 16, seed_pages=1, poison=True)
    for b in (mixed, W.tiny(3), W.tiny(64), W.large_head(8192)):
        d = to_device(b, cuda)
        want_o, want_l, _ = run_gpu(d, cuda)
        heads = (b.num_qo_heads, b.num_kv_heads, b.head_dim)
        bk = Bucket(cuda, len(b.q_lens) + 3, b.q.shape[0] + 100, heads, d.k_pages.shape[0],
                    max_pages_idx=d.kv_indices.numel() + 8)
        bk.load(d)
        bk.launch(d.k_pages, d.v_pages)
        assert bip.read_device_status(bk.ws) == 0
        n = b.q.shape[0]
        assert_bitwise(bk.out[:n].cpu(), want_o, "device-planned out")
        assert_bitwise(bk.lse[:n].cpu(), want_l, "device-planned lse")
        assert torch.isnan(bk.out[n:].float()).all(), "rows past qo_indptr[batch] were written"


@pytest.mark.parametrize("heads,kv_dtype", [(W.HEADS_A, "bf16"), (W.HEADS_B, "bf16"), (W.HEADS_A, "fp8_e4m3")])
def test_graph_replay_with_new_batches_matches_eager(cuda, heads, kv_dtype):
    # One pool, one capture; a full prefill and an extend replayed through it.
    prompts = [W.make_prompt(n, *heads, seed=70 + i, kv_dtype=kv_dtype) for i, n in enumerate((700, 140, 1029, 18))]
    # the same prompts and page layout (one pool), full prefill and extends
    batches = [W.layout(prompts, [p.n for p in prompts], 16, seed_pages=7, kv_dtype=kv_dtype, poison=True),
               W.layout(prompts, [3, 1, 64, 18], 16, seed_pages=7, kv_dtype=kv_dtype, poison=True)]
    dev = [to_device(b, cuda) for b in batches]
    assert torch.equal(dev[0].k_pages.view(torch.uint8), dev[1].k_pages.view(torch.uint8))
    eager = [run_gpu(d, cuda) for d in dev]
    max_rows = max(b.q.shape[0] for b in batches) + 64
    max_idx = max(b.kv_indices.numel() for b in batches) + 16
    bk = Bucket(cuda, 6, max_rows, heads, dev[0].k_pages.shape[0], kv_dtype, max_pages_idx=max_idx)
    # warm up once eagerly (sets kernel attributes), then capture
    bk.load(dev[0])
    bk.launch(dev[0].k_pages, dev[0].v_pages)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            bk.launch(dev[0].k_pages, dev[0].v_pages)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    for i in (0, 1):  # both use the captured pool
        bk.load(dev[i])
        graph.replay()
        torch.cuda.synchronize()
        assert bip.read_device_status(bk.ws) == 0
        n = batches[i].q.shape[0]
        assert_bitwise(bk.out[:n].cpu(), eager[i][0], f"replay {i} out")
        assert_bitwise(bk.lse[:n].cpu(), eager[i][1], f"replay {i} lse")


def test_radix_hit_and_full_recompute_in_different_buckets(cuda):
    # The extend (a few rows behind a cached prefix) and the cold prefill of
    # the same prompts, each through its own captured bucket: extend rows
    # equal the matching rows of the full prefill, bit for bit.
    ext, cold = W.radix_burst(n_req=8, prefix=512)
    de, dc = to_device(ext, cuda), to_device(cold, cuda)
    outs = []
    for d, rows in ((de, 64), (dc, cold.q.shape[0] + 32)):
        bk = Bucket(cuda, 16 if d is de else 8, rows, W.HEADS_A, d.k_pages.shape[0],
                    max_pages_idx=d.kv_indices.numel() + 4)
        bk.load(d)
        bk.launch(d.k_pages, d.v_pages)   # warm-up
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(graph, stream=s):
                bk.launch(d.k_pages, d.v_pages)
        torch.cuda.current_stream().wait_stream(s)
        bk.load(d)
        graph.replay()
        torch.cuda.synchronize()
        assert bip.read_device_status(bk.ws) == 0
        n = d.q.shape[0]
        outs.append((bk.out[:n].cpu(), bk.lse[:n].cpu()))
    (eo, el), (co, cl) = outs
    # row i of request r in the extend = row (kv_len - q_len + i) of request r in the cold batch
    for r in range(len(ext.q_lens)):
        e0, c0 = int(ext.qo_indptr[r]), int(cold.qo_indptr[r])
        off = ext.kv_lens[r] - ext.q_lens[r]
        for i in range(ext.q_lens[r]):
            assert torch.equal(eo[e0 + i], co[c0 + off + i]), f"request {r} row {i}"
            assert torch.equal(el[e0 + i], cl[c0 + off + i]), f"request {r} row {i} lse"
    ro, rl = oracle(ext)
    assert_close_to_oracle(eo, el, ro, rl)


def test_invalid_batch_on_the_device_reports_and_computes_nothing(cuda):
    b = to_device(W.tiny(64), cuda)
    bk = Bucket(cuda, 2, 128, W.HEADS_A, b.k_pages.shape[0], max_pages_idx=b.kv_indices.numel())
    bk.load(b)
    bk.qo[1] = 65  # q_len 65 > kv_len 64
    bk.qo[2] = 65
    bk.launch(b.k_pages, b.v_pages)
    assert bip.read_device_status(bk.ws) == 1  # BIP_ERR_INVALID_ARG
    assert torch.isnan(bk.out.float()).all()
    # and the next valid launch on the same workspace is fine
    bk.load(b)
    bk.launch(b.k_pages, b.v_pages)
    assert bip.read_device_status(bk.ws) == 0


@pytest.mark.parametrize("heads,kv_dtype", [(W.HEADS_A, "bf16"), (W.HEADS_B, "bf16"), (W.HEADS_A, "fp8_e4m3")])
def test_short_batch_splits_on_the_device_and_keeps_the_bits(cuda, heads, kv_dtype):
    # Few units, each behind several 4096-key segments: the device planner
    # splits them by segment (merge units written), and the results equal the
    # host-planned launch bit for bit and the oracle within the tolerance,
    # eagerly and replayed from a captured graph; a plan that never splits
    # gives the same bits.
    prompts = [W.make_prompt(n, *heads, seed=80 + i, kv_dtype=kv_dtype) for i, n in enumerate((9000, 5000, 12300))]
    b = W.layout(prompts, [4, 1, 37], 16, seed_pages=8, kv_dtype=kv_dtype, poison=True)
    d = to_device(b, cuda)
    want_o, want_l, _ = run_gpu(d, cuda)
    n = b.q.shape[0]
    bk = Bucket(cuda, 4, 64, heads, d.k_pages.shape[0], kv_dtype, max_pages_idx=d.kv_indices.numel() + 8)
    bk.load(d)
    bk.launch(d.k_pages, d.v_pages)
    torch.cuda.synchronize()
    assert bip.read_device_status(bk.ws) == 0
    assert _merges_written(bk.ws) > 0, "the short batch was not split"
    assert_bitwise(bk.out[:n].cpu(), want_o, "split device-planned out")
    assert_bitwise(bk.lse[:n].cpu(), want_l, "split device-planned lse")
    graph = _capture(lambda: bk.launch(d.k_pages, d.v_pages))
    bk.load(d)
    graph.replay()
    torch.cuda.synchronize()
    assert bip.read_device_status(bk.ws) == 0
    assert_bitwise(bk.out[:n].cpu(), want_o, "split replay out")
    assert_bitwise(bk.lse[:n].cpu(), want_l, "split replay lse")
    ro, rl = oracle(b)
    assert_close_to_oracle(bk.out[:n].cpu(), bk.lse[:n].cpu(), ro, rl)
    hq, hkv, dd = heads
    fold = bip.GraphPlan(4, 64, num_qo_heads=hq, num_kv_heads=hkv, head_dim=dd, kv_dtype=kv_dtype,
                         split_policy="never")
    ws = torch.empty(fold.workspace_bytes, dtype=torch.uint8, device=cuda)
    bk.load(d)
    bip.prefill_graph(fold, bk.max_batch, bk.qo, bk.kv, bk.last, bk.q, d.k_pages, d.v_pages, bk.idx, bk.out,
                      bk.lse, ws)
    torch.cuda.synchronize()
    assert bip.read_device_status(ws) == 0 and _merges_written(ws) == 0
    assert_bitwise(bk.out[:n].cpu(), want_o, "folded device-planned out")


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_masked_graph_replay_matches_host_planned_and_oracle(cuda, kv_dtype):
    # Custom masks through the graph-replayable launch: an extend behind two
    # segments (split on the device) and a short fresh prefill, each row
    # narrowed by its prompt mask's row.  Bits equal the host-planned masked
    # launch, eagerly and under replay; rows with no visible key are 0 / -inf;
    # the rest is within the tolerance of the oracle.
    lens, q_lens = (5000, 300), (37, 300)
    prompts = [W.make_prompt(n, *W.HEADS_A, seed=60 + i, kv_dtype=kv_dtype) for i, n in enumerate(lens)]
    b = W.layout(prompts, list(q_lens), 16, seed_pages=4, kv_dtype=kv_dtype, poison=True)
    d = to_device(b, cuda)
    masks = [W.prompt_mask(n, 7 + r)[n - ql:, :n] for r, (n, ql) in enumerate(zip(lens, q_lens))]
    words = (max(lens) + 31) // 32
    want_o, want_l, _ = run_gpu(d, cuda, custom_mask=masks, mask_row_words=words)
    n = b.q.shape[0]
    bk = Bucket(cuda, 3, n + 40, W.HEADS_A, d.k_pages.shape[0], kv_dtype, max_pages_idx=d.kv_indices.numel() + 8)
    mask_buf = torch.zeros(bk.max_total_q, words, dtype=torch.int32, device=cuda)
    mask_buf[:n].copy_(torch.from_numpy(bip.pack_mask(masks, words)))
    bk.load(d)
    bk.launch(d.k_pages, d.v_pages, custom_mask=mask_buf)
    torch.cuda.synchronize()
    assert bip.read_device_status(bk.ws) == 0
    assert_bitwise(bk.out[:n].cpu(), want_o, "masked device-planned out")
    assert_bitwise(bk.lse[:n].cpu(), want_l, "masked device-planned lse")
    graph = _capture(lambda: bk.launch(d.k_pages, d.v_pages, custom_mask=mask_buf))
    bk.load(d)
    graph.replay()
    torch.cuda.synchronize()
    assert bip.read_device_status(bk.ws) == 0
    out, lse = bk.out[:n].cpu(), bk.lse[:n].cpu()
    assert_bitwise(out, want_o, "masked replay out")
    assert_bitwise(lse, want_l, "masked replay lse")
    ro, rl = oracle(b, custom_mask=masks)
    o = out.float().numpy().astype(np.float64)
    l = lse.numpy().astype(np.float64)
    empty = np.isneginf(rl)
    assert empty.any() and np.array_equal(np.isneginf(l), empty) and (o[empty] == 0).all()
    full = ~empty
    err_o = np.abs(o[full] - ro[full])
    assert (err_o <= 2e-2 + 1e-2 * np.abs(ro[full])).all()
    err_l = np.abs(l[full] - rl[full])
    assert (err_l <= 2e-2 + 1e-2 * np.abs(rl[full])).all()


def test_masked_graph_launch_rejects_a_mask_row_shorter_than_the_keys(cuda):
    b = to_device(W.tiny(64), cuda)
    bk = Bucket(cuda, 2, 128, W.HEADS_A, b.k_pages.shape[0], max_pages_idx=b.kv_indices.numel())
    bk.load(b)
    short = torch.full((128, 1), -1, dtype=torch.int32, device=cuda)   # 32 keys a row < kv_len 64
    bk.launch(b.k_pages, b.v_pages, custom_mask=short)
    assert bip.read_device_status(bk.ws) == 1  # BIP_ERR_INVALID_ARG
    assert torch.isnan(bk.out.float()).all()
