"""Benchmark: batch-invariant paged prefill attention on GB300.

Default workload (the throughput sweep's long-q point): heads 32/8/128, 16
requests, q_len = kv_len = 8192 (fresh causal prefill), bf16 pages of 16
tokens, synthetic N(0,1) data.  `value` = algorithmic causal TFLOP/s
(4 * head_dim * num_qo_heads * sum of unmasked (row, key) pairs) with inputs
resident in HBM.  The same JSON line carries the sweep's short-extend point
(16 requests, q_len 4 behind kv_len 32768) as KV-read GB/s, the roofline of
each against MEASURED_PEAKS.json, an end-to-end number through the public
API with host buffers, and the float64 oracle timed on host cores.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
    python bench.py --sweep        # every sweep point, one JSON line each

Multi-GPU (torchrun): requests are independent, so every rank runs its own
16-request batch (weak scaling) with no collective on the data path.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged prefill attn TFLOP/s (long q) & KV-read GB/s (short extends), bit-exact"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = ["bip_host.cpp", "bip_attn.cu", "bip_attn_gather.cu", "bip_attn_mask.cu", "bip_attn_impl.cuh",
                  "bip_merge.cu", "bip_append.cu", "bip_plan_dev.cu", "bip_mask_skip.cu", "bip_internal.h",
                  "bip_numerics.cuh", "bip_ptx.cuh"]


# ----------------------------------------------------------------- helpers

def pairs(q_len: int, kv_len: int) -> int:
    """Unmasked (row, key) pairs of one head: sum over rows of (position + 1)."""
    return q_len * (kv_len - q_len) + q_len * (q_len + 1) // 2


def flops_of(heads, q_lens, kv_lens) -> float:
    hq, _, d = heads
    return float(sum(4 * d * hq * pairs(q, k) for q, k in zip(q_lens, kv_lens)))


def kv_bytes_of(heads, kv_lens, elem=2) -> float:
    _, hkv, d = heads
    return float(sum(k * 2 * hkv * d * elem for k in kv_lens))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_hash() -> str:
    h = hashlib.sha256()
    for s in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "invariant_paged_prefill_gb300", "csrc", s), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it matches these sources."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    ent = rec.get(workload)
    if not ent or ent.get("source_hash") != source_hash():
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.3)
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------- workloads

WORKLOADS = {
    # name: (heads, batch, q_len, kv_len)
    "long_q": ((32, 8, 128), 16, 8192, 8192),
    "short_extend": ((32, 8, 128), 16, 4, 32768),
    # the large-head shape, for --profile
    "long_q_d256": ((24, 4, 256), 16, 8192, 8192),
    "short_extend_d256": ((24, 4, 256), 16, 4, 32768),
    # sweep points below their targets, for --profile
    "extend32_d256": ((24, 4, 256), 16, 32, 32768),
    "ridge_q128": ((32, 8, 128), 16, 128, 32768),
    "prefill_1028": ((32, 8, 128), 16, 1028, 1028),
}


def make_batch(heads, batch, q_len, kv_len, device, kv_dtype="bf16", seed=0, page_size=16):
    from invariant_paged_prefill_gb300 import workloads as W
    return W.sweep_point(heads, q_len, kv_len, batch=batch, kv_dtype=kv_dtype, device=device, seed_data=seed,
                         page_size=page_size)


class Runner:
    """One workload resident on the device, with its plan and buffers."""

    def __init__(self, b, device, window_left: int = 0, mask=None, tiles_per_unit: int = 0):
        import invariant_paged_prefill_gb300 as bip
        self.bip, self.b, self.device = bip, b, device
        self.mask = mask  # packed custom mask words on the device, or None
        self.plan = bip.Plan(b.qo_indptr, b.kv_indptr, b.kv_last_page_len, num_qo_heads=b.num_qo_heads,
                             num_kv_heads=b.num_kv_heads, head_dim=b.head_dim, page_size=b.page_size,
                             kv_dtype=b.kv_dtype, window_left=window_left, tiles_per_unit=tiles_per_unit)
        self.ws = torch.empty(max(self.plan.workspace_bytes, 256), dtype=torch.uint8, device=device)
        self.out = torch.empty_like(b.q)
        self.lse = torch.empty(b.q.shape[0], b.q.shape[1], dtype=torch.float32, device=device)
        # work-list upload kernel + attention (+ merge when units are split)
        self.launches_per_step = 2 + (1 if self.plan.info["num_split_units"] else 0)

    def step(self, q=None, kp=None, vp=None, idx=None):
        b = self.b
        self.bip.prefill(self.plan, b.q if q is None else q, b.k_pages if kp is None else kp,
                         b.v_pages if vp is None else vp, b.kv_indices if idx is None else idx,
                         out=self.out, lse=self.lse, workspace=self.ws, custom_mask=self.mask)

    def timed(self, steps, warmup, barrier=lambda: None):
        for _ in range(warmup):
            self.step()
        torch.cuda.synchronize()
        stream = torch.cuda.current_stream()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        barrier()
        torch.cuda.synchronize()
        ev[0].record(stream)
        for i in range(steps):
            self.step()
            ev[i + 1].record(stream)
        torch.cuda.synchronize()
        barrier()
        per = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
        return ev[0].elapsed_time(ev[-1]), per

    def timed_e2e(self, steps, warmup):
        """Public API with host buffers, pipelined over two buffer slots.

        Every step copies its own inputs from pinned host memory (q, K and V
        pages, page table), runs the prefill through the C ABI, and copies
        out and lse back to pinned host memory.  Host-to-device copies run on
        one stream, prefills on another, device-to-host copies on a third, so
        step i+1's inputs and step i-1's outputs move while step i computes;
        a slot is reused only after its previous prefill and read-back are
        done (events).  The timed region spans the first copy-in to the last
        copy-out.
        """
        b = self.b
        hq = b.q.cpu().pin_memory()
        nbytes = b.k_pages.untyped_storage().nbytes()

        def host_bytes(t):
            flat = torch.as_strided(t.view(torch.uint8) if t.dtype == torch.uint8 else t.view(torch.int16),
                                    (nbytes // t.element_size(),), (1,), 0)
            return flat.cpu().view(torch.uint8).pin_memory()

        hk, hv = host_bytes(b.k_pages), host_bytes(b.v_pages)
        hidx = b.kv_indices.cpu().pin_memory()
        slots = []
        for _ in range(2):
            dk = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
            dv = torch.empty_like(dk)
            slots.append({
                "q": torch.empty_like(b.q), "k": dk, "v": dv, "idx": torch.empty_like(b.kv_indices),
                "kview": dk.view(b.k_pages.dtype).as_strided(b.k_pages.shape, b.k_pages.stride()),
                "vview": dv.view(b.v_pages.dtype).as_strided(b.v_pages.shape, b.v_pages.stride()),
                "out": torch.empty_like(self.out), "lse": torch.empty_like(self.lse),
                "ws": torch.empty_like(self.ws),
                "ho": torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory(),
                "hl": torch.empty(self.lse.shape, dtype=self.lse.dtype).pin_memory(),
                "in_ready": torch.cuda.Event(), "computed": torch.cuda.Event(), "read_back": torch.cuda.Event(),
                "used": False,
            })
        s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

        def one(i):
            sl = slots[i % 2]
            with torch.cuda.stream(s_in):
                if sl["used"]:
                    s_in.wait_event(sl["computed"])  # the slot's previous prefill has read its inputs
                sl["q"].copy_(hq, non_blocking=True)
                sl["k"].copy_(hk, non_blocking=True)
                sl["v"].copy_(hv, non_blocking=True)
                sl["idx"].copy_(hidx, non_blocking=True)
                sl["in_ready"].record(s_in)
            s_comp.wait_event(sl["in_ready"])
            if sl["used"]:
                s_comp.wait_event(sl["read_back"])  # its previous output has been copied out
            self.bip.prefill(self.plan, sl["q"], sl["kview"], sl["vview"], sl["idx"], out=sl["out"],
                             lse=sl["lse"], workspace=sl["ws"], stream=s_comp)
            sl["computed"].record(s_comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(sl["computed"])
                sl["ho"].copy_(sl["out"], non_blocking=True)
                sl["hl"].copy_(sl["lse"], non_blocking=True)
                sl["read_back"].record(s_out)
            sl["used"] = True

        for i in range(warmup):
            one(i)
        torch.cuda.synchronize()
        # The host link is shared with the node's other GPUs: a loop now and
        # then stalls for tens of milliseconds.  Three timed loops, median.
        runs = []
        for _ in range(3):
            t0 = time.perf_counter()
            for i in range(steps):
                one(i)
            torch.cuda.synchronize()
            runs.append((time.perf_counter() - t0) / steps)
        dt = statistics.median(runs)
        self.e2e_runs_ms = [r * 1e3 for r in runs]
        h2d = hq.numel() * hq.element_size() + hk.numel() + hv.numel() + hidx.numel() * 4
        d2h = self.out.numel() * self.out.element_size() + self.lse.numel() * self.lse.element_size()
        ref = self.out.cpu()
        for sl in slots:
            assert torch.equal(sl["ho"], ref), "end-to-end output differs from the device-resident run"
        return dt, h2d, d2h


# ------------------------------------------------------------ oracle (CPU)

def oracle_sample(b, rows):
    from oracle import paged_attention as pa
    kind = "bf16" if b.kv_dtype == "bf16" else "e4m3"
    q = b.q.cpu()
    kp, vp = b.k_pages.cpu(), b.v_pages.cpu()
    kview = kp.view(torch.int16) if kind == "bf16" else kp
    vview = vp.view(torch.int16) if kind == "bf16" else vp
    t0 = time.perf_counter()
    out, lse = pa.paged_prefill(q.view(torch.int16).numpy(), kview.numpy(), vview.numpy(), b.qo_indptr.tolist(),
                                b.kv_indptr.tolist(), b.kv_indices.cpu().tolist(), b.kv_last_page_len.tolist(),
                                b.num_qo_heads, b.num_kv_heads, b.page_size, q_kind="bf16", kv_kind=kind, rows=rows)
    return out, lse, time.perf_counter() - t0


def sample_rows_for(b, n_rows, seed=0):
    """Rows of request 0 spread over its positions (first, last, evenly spaced)."""
    lo, hi = b.row_range(0)
    rng = np.random.default_rng(seed)
    rows = sorted(set([lo, hi - 1] + [int(x) for x in rng.integers(lo, hi, size=max(n_rows - 2, 0))]))
    return rows


def sample_flops(b, heads, rows):
    hq, _, d = heads
    lo, hi = b.row_range(0)
    ql, kl = hi - lo, b.kv_lens[0]
    return float(sum(4 * d * hq * (t - lo + kl - ql + 1) for t in rows))


def cores_used() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ------------------------------------------------------------------- arms

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def rank_seed(rank: int, base: int = 0) -> int:
    """Data seed of a rank's batch: every rank prefills its own 16 requests (weak scaling)."""
    return base + 1000 * rank


def max_over_ranks(x: float, device="cpu") -> float:
    """The slowest rank's time (identity with one process)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_value(units_per_rank: float, world: int, ms_max: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest rank's time (per second)."""
    return world * units_per_rank / (ms_max * 1e-3)


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    name = args.workload
    heads, batch, q_len, kv_len = WORKLOADS[name]
    b = make_batch(heads, batch, q_len, kv_len, "cpu")
    rows = sample_rows_for(b, args.ref_rows)
    fl = sample_flops(b, heads, rows)
    for _ in range(args.warmup):
        oracle_sample(b, rows[:2])
    times = []
    for _ in range(args.steps):
        _, _, dt = oracle_sample(b, rows)
        times.append(dt)
    tot = sum(times)
    value = fl * args.steps / tot / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(name),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores_used(), "kind": "oracle",
                             "sample": f"{len(rows)} q rows of request 0 (all 32 heads) per step"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_config(name):
    heads, batch, q_len, kv_len = WORKLOADS[name]
    return {"workload": f"{name}: {batch} requests x q_len {q_len} behind kv_len {kv_len}, heads "
                        f"{heads[0]}/{heads[1]}/{heads[2]}, bf16 pages of 16",
            "heads": list(heads), "batch": batch, "q_len": q_len, "kv_len": kv_len, "page_size": 16,
            "l2": "inputs larger than L2 (129 MB) between timed iterations"}


def time_append(b, device, steps: int, warmup: int):
    """Paged KV append of every q row's K/V into b's pools (overwrites them):
    (ms per call, bytes moved per call).  Bytes: the bf16 rows read plus the
    pool slots written."""
    import invariant_paged_prefill_gb300 as bip
    plan = bip.Plan(b.qo_indptr, b.kv_indptr, b.kv_last_page_len, num_qo_heads=b.num_qo_heads,
                    num_kv_heads=b.num_kv_heads, head_dim=b.head_dim, page_size=b.page_size, kv_dtype=b.kv_dtype)
    g = torch.Generator(device=device).manual_seed(77)
    shape = (plan.total_q, b.num_kv_heads, b.head_dim)
    k_new = torch.randn(shape, generator=g, device=device).to(torch.bfloat16)
    v_new = torch.randn(shape, generator=g, device=device).to(torch.bfloat16)
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device=device)
    for _ in range(warmup):
        bip.append_kv(plan, k_new, v_new, b.k_pages, b.v_pages, b.kv_indices, workspace=ws)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        bip.append_kv(plan, k_new, v_new, b.k_pages, b.v_pages, b.kv_indices, workspace=ws)
    e1.record(stream)
    torch.cuda.synchronize()
    elem = 2 if b.kv_dtype == "bf16" else 1
    moved = 2 * k_new.numel() * (2 + elem)
    return e0.elapsed_time(e1) / steps, moved


def windowed_work(heads, q_lens, kv_lens, window: int):
    """(FLOP, KV bytes) of sliding-window attention: row at position p sees
    min(p + 1, window + 1) keys; a request with rows reads its last q + window
    keys (one with none reads nothing)."""
    hq, hkv, d = heads
    pairs, keys = 0, 0
    for q, kv in zip(q_lens, kv_lens):
        for p in range(kv - q, kv):
            pairs += min(p + 1, window + 1)
        keys += min(kv, q + window) if q > 0 else 0
    return 4 * d * hq * pairs, keys * 2 * hkv * d * 2


def measure_host_planning(reps: int = 5) -> dict:
    """Host planning time (bip_plan: validation, units, split choice, launch
    order, the upload image) for the long_q and short_extend batches, median
    of ``reps`` plans; no device work and outside every timed region."""
    import invariant_paged_prefill_gb300 as bip
    out = {}
    for name in ("long_q", "short_extend"):
        heads, batch, q_len, kv_len = WORKLOADS[name]
        pages = (kv_len + 15) // 16
        qo = np.arange(batch + 1, dtype=np.int32) * q_len
        kv = np.arange(batch + 1, dtype=np.int32) * pages
        last = np.full(batch, kv_len - (pages - 1) * 16, dtype=np.int32)
        ts, items = [], 0
        for _ in range(reps):
            t0 = time.perf_counter()
            p = bip.Plan(qo, kv, last, num_qo_heads=heads[0], num_kv_heads=heads[1], head_dim=heads[2])
            ts.append((time.perf_counter() - t0) * 1e3)
            items = p.info["num_items"]
            p.close()
        out[name] = {"ms": statistics.median(ts), "items": items}
    return out


def measure_configs(device, reps: int = 20):
    """The smaller configurations of the benchmark's list: bit-exactness checks
    and latencies (median of ``reps`` CUDA-event timings per call, inputs
    resident; these are latency figures, not L2-flushed throughput)."""
    from invariant_paged_prefill_gb300 import workloads as W
    import invariant_paged_prefill_gb300 as bip

    def timed_run(b):
        r = Runner(b, device)
        r.step()
        torch.cuda.synchronize()
        st = bip.read_device_status(r.ws)
        s = torch.cuda.current_stream()
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            r.step()
            e1.record(s)
            e1.synchronize()
            ts.append(e0.elapsed_time(e1))
        return r.out.cpu(), r.lse.cpu(), statistics.median(ts), st, r

    def rows_equal(o1, l1, a, o2, l2, b2, n):
        return bool(torch.equal(o1[a:a + n], o2[b2:b2 + n]) and torch.equal(l1[a:a + n], l2[b2:b2 + n]))

    res = {}
    # tiny: a 64-token prefill and the 3-row extend behind its 61-token prefix
    fo, fl, f_ms, f_st, _ = timed_run(W.tiny(64, device=device))
    eo, el, e_ms, e_st, _ = timed_run(W.tiny(3, device=device))
    res["tiny"] = {"extend_rows_bit_exact": rows_equal(eo, el, 0, fo, fl, 61, 3) and f_st == 0 and e_st == 0,
                   "prefill_us": f_ms * 1e3, "extend_us": e_ms * 1e3}
    # radix-hit burst: 16 extends behind a shared 1024-token prefix vs the cold prefill
    ext, cold = W.radix_burst(device=device)
    xo, xl, x_ms, x_st, _ = timed_run(ext)
    co, cl, c_ms, c_st, _ = timed_run(cold)
    ok = x_st == 0 and c_st == 0
    for r in range(len(ext.q_lens)):
        ok &= rows_equal(xo, xl, int(ext.qo_indptr[r]), co, cl,
                         int(cold.qo_indptr[r]) + ext.kv_lens[r] - ext.q_lens[r], ext.q_lens[r])
    res["radix_burst"] = {"extend_rows_bit_exact_vs_cold": bool(ok), "extend_latency_us": x_ms * 1e3,
                          "extend_rows": int(ext.q.shape[0]), "cold_ms": c_ms,
                          "cold_tflops": flops_of(W.HEADS_A, cold.q_lens, cold.kv_lens) / (c_ms * 1e-3) / 1e12}
    # mixed ragged batch: each request against itself alone and against its own full prefill
    prompts, q_lens = W.mixed_ragged_prompts(device=device)
    mixed = W.layout(prompts, q_lens, 16, seed_pages=1)
    mo, ml, m_ms, m_st, _ = timed_run(mixed)
    ok = m_st == 0
    for r, (p, ql) in enumerate(zip(prompts, q_lens)):
        ao, al, _, a_st, _ = timed_run(W.layout([p], [ql], 16, seed_pages=5 + r))
        po, pl, _, p_st, _ = timed_run(W.layout([p], [p.n], 16, seed_pages=9 + r))
        m0 = int(mixed.qo_indptr[r])
        ok &= a_st == 0 and p_st == 0 and rows_equal(mo, ml, m0, ao, al, 0, ql)
        ok &= rows_equal(mo, ml, m0, po, pl, p.n - ql, ql)
    res["mixed_ragged"] = {"bit_exact_vs_alone_and_full_prefill": bool(ok), "ms": m_ms,
                           "tflops": flops_of(W.HEADS_A, mixed.q_lens, mixed.kv_lens) / (m_ms * 1e-3) / 1e12}
    # large-head GQA: single fresh prefills of 8192 and 32768 tokens, 24/4/256
    for n in (8192, 32768):
        lb = W.large_head(n, device=device)
        _, _, l_ms, l_st, r = timed_run(lb)
        bound = bip.workspace_bound(1, n, 24, 4, 256)
        tf = flops_of(W.HEADS_B, lb.q_lens, lb.kv_lens) / (l_ms * 1e-3) / 1e12
        res[f"large_head_{n}"] = {"ms": l_ms, "tflops": tf,
                                  "status": l_st, "workspace_bytes": r.plan.workspace_bytes,
                                  "workspace_bound_bytes": bound,
                                  "within_bound": r.plan.workspace_bytes <= bound}
        del r, lb
    return res


# Sweep points timed inside the default run, each reported with its own
# CUDA-event time per step and roofline: the largest long-q points of both
# head shapes, and the E4M3 pages.  (heads, q_len, kv_len, kv_dtype)
SWEEP_EXTRAS = [
    ((32, 8, 128), 8192, 32768, "bf16"),
    ((24, 4, 256), 8192, 8192, "bf16"),
    ((24, 4, 256), 8192, 32768, "bf16"),
    ((24, 4, 256), 4, 8192, "bf16"),
    ((24, 4, 256), 32, 32768, "bf16"),
    ((32, 8, 128), 8192, 8192, "fp8_e4m3"),
    ((32, 8, 128), 4, 32768, "fp8_e4m3"),
    ((24, 4, 256), 8192, 8192, "fp8_e4m3"),
    ((24, 4, 256), 1, 32768, "fp8_e4m3"),
]


def measure_point(heads, q_len, kv_len, kv_dtype, device, steps, warmup, peaks, peak_kind):
    """One 16-request sweep point: CUDA-event ms per step (mean over ``steps``
    launches after ``warmup``), TFLOP/s and KV GB/s, and the roofline of the
    bound that applies (tensor for q_len >= 1028, HBM for q_len <= 32)."""
    b = make_batch(heads, 16, q_len, kv_len, device, kv_dtype=kv_dtype)
    run = Runner(b, device)
    _, per = run.timed(steps, warmup)
    ms = statistics.mean(per)
    fl = flops_of(heads, b.q_lens, b.kv_lens)
    kvb = kv_bytes_of(heads, b.kv_lens, elem=2 if kv_dtype == "bf16" else 1)
    tflops, gbs = fl / ms / 1e9, kvb / ms / 1e6
    if q_len >= 1028:
        peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
        roof = {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s", "frac": tflops / peak,
                "peak_source": f"bf16_tflops (burst) of {peak_kind}"}
    else:
        peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        roof = {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                "peak_source": f"hbm_gbs of {peak_kind}"}
    st = run.bip.read_device_status(run.ws)
    res = {"workload": f"{16} requests x q_len {q_len} behind kv_len {kv_len}, heads "
                       f"{heads[0]}/{heads[1]}/{heads[2]}, {kv_dtype} pages of 16",
           "heads": list(heads), "q_len": q_len, "kv_len": kv_len, "kv_dtype": kv_dtype, "steps": steps,
           "ms_per_step": ms, "tflops": tflops, "kv_gbs": gbs, "roofline": roof, "status": st,
           "items": run.plan.info["num_items"], "split_units": run.plan.info["num_split_units"]}
    del run, b
    torch.cuda.empty_cache()
    return res


def time_graph(b, device, steps: int, warmup: int):
    """Device-planned prefill captured in a CUDA graph (buffers sized to b):
    ms per replay, and whether the replay matches the host-planned result."""
    import invariant_paged_prefill_gb300 as bip
    plan = bip.GraphPlan(len(b.q_lens), b.q.shape[0], num_qo_heads=b.num_qo_heads, num_kv_heads=b.num_kv_heads,
                         head_dim=b.head_dim, page_size=b.page_size, kv_dtype=b.kv_dtype)
    i32 = dict(dtype=torch.int32, device=device)
    qo = torch.as_tensor(np.asarray(b.qo_indptr), **i32)
    kv = torch.as_tensor(np.asarray(b.kv_indptr), **i32)
    last = torch.as_tensor(np.asarray(b.kv_last_page_len), **i32)
    out = torch.empty_like(b.q)
    lse = torch.empty(b.q.shape[0], b.q.shape[1], dtype=torch.float32, device=device)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=device)

    def launch():
        bip.prefill_graph(plan, len(b.q_lens), qo, kv, last, b.q, b.k_pages, b.v_pages, b.kv_indices, out, lse, ws)

    launch()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            launch()
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps, out, lse


def run_ours(args):
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
        barrier = lambda: dist.barrier()
    else:
        barrier = lambda: None
    torch.cuda.set_device(local)
    device = torch.device(f"cuda:{local}")
    from invariant_paged_prefill_gb300 import build as B
    B.ensure_built()
    peaks, peak_kind = load_peaks()

    name = args.workload
    heads, batch, q_len, kv_len = WORKLOADS[name]
    b = make_batch(heads, batch, q_len, kv_len, device, seed=rank_seed(rank))
    run = Runner(b, device)
    fl = flops_of(heads, b.q_lens, b.kv_lens)
    with ClockSampler(local) as clk:
        total_ms, per = run.timed(args.steps, args.warmup, barrier)
    ms = max_over_ranks(total_ms / args.steps, device)
    value = aggregate_value(fl, world, ms) / 1e12
    kernel_ms = statistics.mean(per)
    achieved = fl / (kernel_ms * 1e-3) / 1e12
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
            "peak_source": f"bf16_tflops (burst) of {peak_kind}", "traffic": recorded_traffic(name),
            "kernel": "bip_attn_kernel<128>", "note": "launch duration from CUDA events around each bip_prefill"}

    # bit-exactness across repeated runs of the timed step
    o1 = run.out.clone(); l1 = run.lse.clone()
    run.step(); torch.cuda.synchronize()
    repeat_exact = bool(torch.equal(o1, run.out) and torch.equal(l1, run.lse))

    # short-extend point: KV-read GB/s
    sheads, sbatch, sq, skv = WORKLOADS["short_extend"]
    sb = make_batch(sheads, sbatch, sq, skv, device, seed=rank_seed(rank, 100))
    srun = Runner(sb, device)
    s_total, s_per = srun.timed(args.steps, args.warmup, barrier)
    s_total = max_over_ranks(s_total, device)
    s_ms = statistics.mean(s_per)
    kvb = kv_bytes_of(sheads, sb.kv_lens)
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    s_gbs = kvb / (s_ms * 1e-3) / 1e9
    kv_read = {"workload": f"short_extend: {sbatch} requests x q_len {sq} behind kv_len {skv}",
               "value": aggregate_value(kvb, world, s_total / args.steps) / 1e9, "unit": "GB/s",
               "ms_per_step": s_total / args.steps,
               "roofline": {"bound": "hbm", "achieved": s_gbs, "peak": hbm, "unit": "GB/s", "frac": s_gbs / hbm,
                            "peak_source": f"hbm_gbs of {peak_kind}", "traffic": recorded_traffic("short_extend")},
               "split_units": srun.plan.info["num_split_units"], "items": srun.plan.info["num_items"]}
    launches = args.steps * run.launches_per_step

    line = None
    if rank == 0:
        e2e_s, h2d, d2h = run.timed_e2e(max(6, args.steps), 2)
        # parity and the CPU baseline from the same oracle sample
        rows = sample_rows_for(b, args.ref_rows)
        ro, rl, odt = oracle_sample(b, rows)
        got = run.out.cpu()[rows].float().numpy().astype(np.float64)
        gl = run.lse.cpu()[rows].numpy().astype(np.float64)
        parity_ok = bool((np.abs(got - ro) <= 2e-2 + 1e-2 * np.abs(ro)).all() and
                         (np.abs(gl - rl) <= 2e-2 + 1e-2 * np.abs(rl)).all())
        cpu_val = sample_flops(b, heads, rows) / odt / 1e12
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": workload_config(name),
                "roofline": roof,
                "cpu_baseline": {"value": cpu_val, "unit": "TFLOP/s", "cores": cores_used(), "kind": "oracle",
                                 "sample": f"{len(rows)} q rows of request 0, all heads, float64",
                                 "seconds": odt},
                "e2e": {"value": world * fl / e2e_s / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3,
                        "runs_ms_per_step": run.e2e_runs_ms,
                        "note": "median of three timed loops of pipelined steps (copies in, prefill, copies out)"},
                "gpu_launches": launches, "clocks": clk.summary(), "kv_read": kv_read,
                "parity": {"rows": len(rows), "within_tolerance": parity_ok,
                           "max_abs_out": float(np.abs(got - ro).max()), "max_abs_lse": float(np.abs(gl - rl).max())},
                "bit_exact_repeat": repeat_exact, "workspace_bytes": run.plan.workspace_bytes,
                "source_hash": source_hash()}
        # sliding window: long_q with a 1024-key window, the short extend with 4096
        wl = Runner(b, device, window_left=1024)
        wl_total, _ = wl.timed(args.steps, args.warmup)
        ws_ = Runner(sb, device, window_left=4096)
        ws_total, _ = ws_.timed(args.steps, args.warmup)
        wfl, _ = windowed_work(heads, b.q_lens, b.kv_lens, 1024)
        _, wkvb = windowed_work(sheads, sb.q_lens, sb.kv_lens, 4096)
        line["window"] = {
            "long_q_window_1024_tflops": wfl / (wl_total / args.steps * 1e-3) / 1e12,
            "short_extend_window_4096_kv_gbs": wkvb / (ws_total / args.steps * 1e-3) / 1e9,
            "short_extend_window_4096_ms": ws_total / args.steps,
            "note": "algorithmic work of the window only (pairs within the window, keys the window reads)"}
        del wl, ws_
        # token-granular pools (page size 1, every row of a block gathered on
        # its own): the same prompts, so the same bits as the 16-slot pages
        b1 = make_batch(heads, batch, q_len, kv_len, device, seed=rank_seed(rank), page_size=1)
        sb1 = make_batch(sheads, sbatch, sq, skv, device, seed=rank_seed(rank, 100), page_size=1)
        r1, sr1 = Runner(b1, device), Runner(sb1, device)
        p1_total, _ = r1.timed(args.steps, args.warmup)
        sp1_total, _ = sr1.timed(args.steps, args.warmup)
        p1_gbs = kvb / (sp1_total / args.steps * 1e-3) / 1e9
        line["page_size_1"] = {
            "what": "token-granular pools: K and V rows gathered by cp.async warps (one q tile per CTA)",
            "long_q_tflops": fl / (p1_total / args.steps * 1e-3) / 1e12,
            "short_extend_kv_gbs": p1_gbs,
            "short_extend_ms": sp1_total / args.steps,
            "short_extend_roofline": {"bound": "hbm", "achieved": p1_gbs, "peak": hbm, "unit": "GB/s",
                                      "frac": p1_gbs / hbm, "peak_source": f"hbm_gbs of {peak_kind}",
                                      "traffic": recorded_traffic("short_extend_page1")},
            "bit_exact_vs_page_16": bool(torch.equal(r1.out, run.out) and torch.equal(r1.lse, run.lse) and
                                         torch.equal(sr1.out, srun.out) and torch.equal(sr1.lse, srun.lse))}
        del r1, sr1, b1, sb1
        # device-planned launches replayed from a CUDA graph (fold only, no split)
        g_ms, g_out, g_lse = time_graph(b, device, args.steps, args.warmup)
        sg_ms, sg_out, sg_lse = time_graph(sb, device, args.steps, args.warmup)
        line["graph"] = {
            "what": "device-planned prefill replayed from a captured CUDA graph (a batch of few units is split "
                    "by segment on the device; tiles per CTA from the bucket's capacities)",
            "long_q_tflops": fl / (g_ms * 1e-3) / 1e12,
            "short_extend_kv_gbs": kvb / (sg_ms * 1e-3) / 1e9,
            "bit_exact_vs_host_planned": bool(torch.equal(g_out, run.out) and torch.equal(g_lse, run.lse) and
                                              torch.equal(sg_out, srun.out) and torch.equal(sg_lse, srun.lse))}
        # the paged KV append (the step before attention), timed last: it
        # overwrites the pools of both batches
        a_ms, a_bytes = time_append(b, device, args.steps, args.warmup)
        sa_ms, _ = time_append(sb, device, args.steps, args.warmup)
        a_gbs = a_bytes / (a_ms * 1e-3) / 1e9
        line["append"] = {
            "workload": f"paged KV append of {batch} x {q_len} new rows (bf16 K and V, heads "
                        f"{heads[1]} x {heads[2]}) into the long_q pools",
            "value": a_gbs, "unit": "GB/s", "ms_per_step": a_ms,
            "roofline": {"bound": "hbm", "achieved": a_gbs, "peak": hbm, "unit": "GB/s", "frac": a_gbs / hbm,
                         "peak_source": f"hbm_gbs of {peak_kind}", "traffic": recorded_traffic("append")},
            "short_extend_us": sa_ms * 1e3}
        # custom masks over the long_q and short_extend batches (FLOPs over
        # the causal pairs: a mask narrows what is visible, not the work)
        masked = {}
        for wname, bb, mkind in (("long_q", b, "half"), ("long_q", b, "documents"), ("short_extend", sb, "half")):
            words, density = profile_mask(bb, mkind)
            mr = Runner(bb, device, mask=torch.from_numpy(words).to(device))
            _, mper = mr.timed(args.steps, args.warmup)
            mms = statistics.mean(mper)
            hh = heads if wname == "long_q" else sheads
            ent = {"ms_per_step": mms, "visible_fraction": density,
                   "tflops": flops_of(hh, bb.q_lens, bb.kv_lens) / mms / 1e9,
                   "kv_gbs": kv_bytes_of(hh, bb.kv_lens) / mms / 1e6}
            ent["visible_tflops"] = ent["tflops"] * density  # FLOPs of the visible pairs only
            ent["roofline_frac"] = (ent["tflops"] / float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
                                    if wname == "long_q" else
                                    ent["kv_gbs"] / float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])))
            masked[f"{wname}_{mkind}"] = ent
            del mr
        masked["note"] = ("half: each key visible with probability 1/2; documents: 512-4096-token documents, each "
                          "row seeing its own; tflops, kv_gbs and roofline_frac count the FLOPs and bytes of the "
                          "unmasked causal work (blocks no row of a work item sees are skipped, so under documents "
                          "they can exceed the dense peak); visible_tflops counts the visible pairs only")
        line["custom_mask"] = masked
        line["configs"] = measure_configs(device)
        line["host_plan_ms"] = measure_host_planning()
        line["sweep_points"] = [measure_point(h, q, kv, dt, device, args.steps, args.warmup, peaks, peak_kind)
                                for h, q, kv, dt in SWEEP_EXTRAS]
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


def profile_mask(b, kind: str, seed: int = 0):
    """Packed custom mask words ([total_q, words] int32) for a profile run, and
    the fraction of causal (row, key) pairs it leaves visible.  'half': every
    key visible with probability 1/2 (no block has all bits set, so every block
    takes the masked softmax path); 'documents': each request cut into
    documents of 512 to 4096 tokens, a row seeing only its own document's keys
    (packed sequences; blocks are wholly in, wholly out or cut once)."""
    rng = np.random.default_rng(seed)
    words = (max(b.kv_lens) + 31) // 32
    out = np.zeros((b.total_q, words), dtype=np.uint32)
    visible = causal = 0
    col = np.arange(words, dtype=np.int64)[None, :] * 32
    for r in range(b.batch):
        lo, hi = b.row_range(r)
        ql, kl = b.q_lens[r], b.kv_lens[r]
        if ql == 0:
            continue
        pos = np.arange(kl - ql, kl, dtype=np.int64)
        causal += int((pos + 1).sum())
        if kind == "half":
            out[lo:hi] = rng.integers(0, 1 << 32, size=(ql, words), dtype=np.uint32)
            bits = np.unpackbits(out[lo:hi].view(np.uint8), axis=1, bitorder="little").reshape(ql, words, 32)
            rows, wp = np.arange(ql), pos // 32   # the word holding each row's own position
            before = np.cumsum(bits.sum(axis=2, dtype=np.int64), axis=1)[rows, wp] - bits[rows, wp].sum(axis=1)
            upto = np.cumsum(bits[rows, wp], axis=1, dtype=np.int64)[rows, pos % 32]
            visible += int((before + upto).sum())
        else:
            cuts = [0]
            while cuts[-1] < kl:
                cuts.append(cuts[-1] + int(rng.integers(512, 4097)))
            start = np.asarray(cuts, dtype=np.int64)[np.searchsorted(cuts, pos, side="right") - 1][:, None]
            full = col >= start
            part = (col < start) & (col + 32 > start)
            shift = np.clip(start - col, 0, 31).astype(np.uint64)
            w = np.where(full, np.uint64(0xFFFFFFFF),
                         np.where(part, (np.uint64(0xFFFFFFFF) << shift) & np.uint64(0xFFFFFFFF), np.uint64(0)))
            out[lo:hi] = w.astype(np.uint32)
            visible += int((pos[:, None] - start + 1).sum())
    return out.view(np.int32), visible / max(causal, 1)


def run_profile(args):
    """The timed step alone (no extras), for ncu: --workload, --batch override."""
    from invariant_paged_prefill_gb300 import build as B
    B.ensure_built()
    device = torch.device("cuda:0")
    if args.workload == "append":  # the paged KV append of every long_q row
        heads, batch, q_len, kv_len = WORKLOADS["long_q"]
        batch = args.batch or batch
        b = make_batch(heads, batch, q_len, kv_len, device)
        ms, moved = time_append(b, device, args.steps, args.warmup)
        print(json.dumps({"profile": "append", "batch": batch, "ms": ms, "gbs": moved / ms / 1e6,
                          "source_hash": source_hash()}), flush=True)
        return
    heads, batch, q_len, kv_len = WORKLOADS[args.workload]
    batch = args.batch or batch
    b = make_batch(heads, batch, q_len, kv_len, device, kv_dtype=args.kv_dtype, page_size=args.page_size)
    mask, density = None, 1.0
    if args.mask != "none":
        words, density = profile_mask(b, args.mask)
        mask = torch.from_numpy(words).to(device)
    if args.graph:  # the device-planned launch replayed from a captured graph
        ms, _, _ = time_graph(b, device, args.steps, args.warmup)
        fl = flops_of(heads, b.q_lens, b.kv_lens)
        kvb = kv_bytes_of(heads, b.kv_lens, elem=2 if args.kv_dtype == "bf16" else 1)
        print(json.dumps({"profile": args.workload, "graph": True, "kv_dtype": args.kv_dtype, "batch": batch,
                          "ms": ms, "tflops": fl / ms / 1e9, "kv_gbs": kvb / ms / 1e6,
                          "source_hash": source_hash()}), flush=True)
        return
    run = Runner(b, device, mask=mask)
    total, per = run.timed(args.steps, args.warmup)
    ms = statistics.mean(per)
    # causal pairs: a custom mask narrows what is visible, not what is computed
    fl = flops_of(heads, b.q_lens, b.kv_lens)
    kvb = kv_bytes_of(heads, b.kv_lens, elem=2 if args.kv_dtype == "bf16" else 1)
    print(json.dumps({"profile": args.workload, "page_size": args.page_size, "kv_dtype": args.kv_dtype,
                      "mask": args.mask, "mask_density": density, "batch": batch, "ms": ms,
                      "tflops": fl / ms / 1e9,
                      "kv_gbs": kvb / ms / 1e6, "launches_per_step": run.launches_per_step,
                      "items": run.plan.info["num_items"], "grid": run.plan.info["grid"],
                      "source_hash": source_hash()}), flush=True)


def run_sweep(args):
    from invariant_paged_prefill_gb300 import workloads as W
    from invariant_paged_prefill_gb300 import build as B
    B.ensure_built()
    device = torch.device("cuda:0")
    peaks, kind = load_peaks()
    for heads, q_len, kv_len in W.sweep_grid():
        if args.q_lens and q_len not in args.q_lens:
            continue
        b = make_batch(heads, 16, q_len, kv_len, device, kv_dtype=args.kv_dtype, page_size=args.page_size)
        try:
            run = Runner(b, device, tiles_per_unit=args.tiles)
        except Exception as e:  # unsupported shapes are reported, not fatal
            print(json.dumps({"heads": heads, "q_len": q_len, "kv_len": kv_len, "error": str(e)}), flush=True)
            continue
        total, per = run.timed(args.steps, args.warmup)
        ms = statistics.mean(per)
        fl = flops_of(heads, b.q_lens, b.kv_lens)
        kvb = kv_bytes_of(heads, b.kv_lens, elem=2 if args.kv_dtype == "bf16" else 1)
        print(json.dumps({"heads": list(heads), "batch": 16, "page_size": args.page_size,
                          "kv_dtype": args.kv_dtype, "q_len": q_len,
                          "kv_len": kv_len, "ms": ms,
                          "tflops": fl / ms / 1e9, "tensor_frac": fl / ms / 1e9 / peaks["bf16_tflops"],
                          "kv_gbs": kvb / ms / 1e6, "hbm_frac": kvb / ms / 1e6 / peaks["hbm_gbs"],
                          "items": run.plan.info["num_items"], "split_units": run.plan.info["num_split_units"],
                          "tiles_per_unit": run.plan.info["tiles_per_unit"]}),
              flush=True)
        del run, b
        torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS) + ["append"], default="long_q",
                    help="append: with --profile only, the paged KV append of the long_q rows")
    ap.add_argument("--ref-rows", type=int, default=48)
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--profile", action="store_true", help="time only the main step (for ncu captures)")
    ap.add_argument("--batch", type=int, default=0, help="with --profile: requests per batch")
    ap.add_argument("--page-size", type=int, default=16, help="with --profile or --sweep: slots per KV page")
    ap.add_argument("--kv-dtype", choices=["bf16", "fp8_e4m3"], default="bf16", help="with --sweep or --profile: KV page type")
    ap.add_argument("--graph", action="store_true", help="with --profile: the device-planned launch, replayed")
    ap.add_argument("--tiles", type=int, default=0, help="with --sweep: force q tiles per CTA (0 = the plan's)")
    ap.add_argument("--q-lens", type=int, nargs="*", default=None, help="with --sweep: only these q lengths")
    ap.add_argument("--mask", choices=["none", "half", "documents"], default="none",
                    help="with --profile: a custom mask (random half of the keys, or per-document causal)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.sweep:
        run_sweep(args)
    elif args.profile:
        run_profile(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
