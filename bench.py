#!/usr/bin/env python3
"""Benchmark of the paged MXFP4 index-K scorer on GB300.

Metric: microseconds per scorer call (lower is better), with the achieved HBM
bandwidth (decode) or block-scaled MMA rate (prefill) against the GB300 peak.

Headline workload: decode, B=64 requests x 1 query row, 131,072-token contexts
(1024 pages each) scattered by a seeded block table over a 70,000-page pool
with split data/scale views.  One step = one call over the whole batch; the K
timed steps are one replay of a CUDA graph holding K calls (device time, no
host launch gaps), bracketed by CUDA events on the launching stream.
The pool (623 MB, 570 MB read per call) is larger than L2, so no flush is
needed between calls.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--config decode|prefill-tiny|prefill-long|mtp|chunked]
                  [--no-secondary]

For N > 1 run under torchrun: every rank scores its own replica of the
workload (the calls are independent; there is no exchange step).
``--impl reference`` times the fp64 CPU oracle on the machine's host cores on a
bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import signal
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
# nominal dense ratios on GB300: fp8 = 2 x bf16, fp4 = 6 x bf16
FP8_OVER_BF16 = 2.0
FP4_OVER_BF16 = 6.0


# ------------------------------------------------------------------ helpers --
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, world_size: int, device="cpu") -> float:
    """Largest per-rank value over the job (the slowest rank sets the step
    time); identity on one rank."""
    if world_size <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            hbm = d.get("hbm_gbs")
            bf16 = d.get("bf16_tflops")
            bf16s = d.get("bf16_tflops_sustained", bf16)
            if hbm and bf16:
                return {"hbm_gbs": float(hbm), "bf16_tflops": float(bf16),
                        "bf16_tflops_sustained": float(bf16s), "source": "measured"}
        except Exception:
            pass
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
            "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"mx4_clocks_bench_{os.getpid()}.csv")

    def _lines(self) -> int:
        try:
            with open(self.path) as f:
                return sum(1 for ln in f if ln.count(",") >= 8)
        except OSError:
            return 0

    def _wait_for_lines(self, n: int, timeout_s: float):
        t0 = time.time()
        while self._lines() < n and time.time() - t0 < timeout_s and self.proc.poll() is None:
            time.sleep(0.005)

    def start(self):
        """Start sampling and return once the first sample is written
        (nvidia-smi takes a moment to start; a short timed region would
        otherwise pass before it)."""
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "20"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        self._wait_for_lines(1, 15.0)

    def stop(self):
        if self.proc is None:
            return None
        # one more sample taken after the timed region ended
        self._wait_for_lines(self._lines() + 1, 2.0)
        self.proc.send_signal(signal.SIGTERM)
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "samples": 0, "reasons": [],
                    "note": "no nvidia-smi sample fell inside the sampling window (warm-up and timed region)"}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons),
                "window": "every 20 ms from just before the warm-up calls to the first sample after the timed "
                          "replay (a timed region shorter than 20 ms may fall between two samples)"}


def library_source_hash():
    """Hash of the CUDA sources' code (comments and blank lines removed), so a
    committed ncu summary stays matched to the code it measured."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_attention_mxfp4_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        text = open(os.path.join(csrc, name)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        lines = [ln.rstrip() for ln in text.splitlines() if ln.strip()]
        h.update(name.encode() + b"\0" + "\n".join(lines).encode())
    return h.hexdigest()[:16]


def profile_traffic(kernel_tag: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel and
    workload, or None when the summary is missing or was taken on other
    kernel source."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    src = re.search(r"source_hash:\s*([0-9a-f]+)", text)
    if not m or not src or src.group(1) != library_source_hash():
        return None
    return int(m.group(1))


def workload_work(w):
    """Algorithmic bytes and flops of one call (each live page read once)."""
    import numpy as np
    from sparse_attention_mxfp4_gb300 import workloads as W
    seq = w.seq_lens.numpy().astype(np.int64)
    if w.decode:
        L_last = np.minimum(seq, w.max_seq_len)
        live_pairs = int(L_last.sum())
        rows_L = L_last
    else:
        cu = w.cu_seqlens_q.numpy().astype(np.int64)
        pl = w.prefix_lens.numpy().astype(np.int64)
        rows_L = []
        L_last = np.zeros_like(seq)
        for b in range(w.num_seqs):
            ql = cu[b + 1] - cu[b]
            if ql <= 0:
                continue
            Ls = np.minimum(seq[b], pl[b] + np.arange(ql) + 1).clip(0, w.max_seq_len)
            rows_L.append(Ls)
            L_last[b] = Ls.max()
        rows_L = np.concatenate(rows_L) if rows_L else np.zeros(0, np.int64)
        live_pairs = int(rows_L.sum())
    pages_read = int(((L_last + W.PAGE - 1) // W.PAGE).sum())
    q_bytes = w.q.numel() * w.q.element_size()
    out_bytes = w.total_rows * W.HEADS * w.num_out_pages * 4
    k_bytes = pages_read * (W.FP8_PAGE_BYTES if w.cache == "fp8" else W.PAGE_BYTES)
    bt_bytes = pages_read * 4
    flops = live_pairs * W.HEADS * W.DIM * 2
    return {"k_bytes": k_bytes, "q_bytes": q_bytes, "out_bytes": out_bytes, "bt_bytes": bt_bytes,
            "bytes": k_bytes + q_bytes + out_bytes + bt_bytes, "flops": flops, "live_pairs": live_pairs,
            "pages_read": pages_read}


# ------------------------------------------------------------------ our arm --
def capture_calls(case, out, n, stream):
    """A CUDA graph of n back-to-back scorer calls on ``stream`` (the calls
    a serving step would replay); returns the graph."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(n):
            case.run(out=out, stream=stream)
    return g


def time_calls(case, out, steps, warmup, stream):
    """Device time per call: ``warmup`` eager calls, then one untimed and one
    timed replay of a graph of ``steps`` calls (CUDA events on the stream)."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            case.run(out=out, stream=stream)
        torch.cuda.synchronize()
        g = capture_calls(case, out, steps, stream)
        g.replay()
        torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        g.replay()
        end.record(stream)
        torch.cuda.synchronize()
    return start.elapsed_time(end) / steps


def measure_e2e(case, steps, stream):
    """Same call through the public API with host-resident inputs: every step
    copies the inputs from pinned host memory, scores, and reads the scores
    back into pinned host memory."""
    import torch
    from sparse_attention_mxfp4_gb300.harness import DeviceCase
    dev_bufs = [case.q, case.block_table, case.seq_lens] + list(case.buffers)
    if case.cu_seqlens_q is not None:
        dev_bufs += [case.cu_seqlens_q, case.prefix_lens]
    host_bufs = [b.cpu().pin_memory() for b in dev_bufs]
    out = torch.empty(case.out_shape_scores, dtype=torch.float32, device=case.q.device)
    host_out = torch.empty(out.shape, dtype=torch.float32).pin_memory()
    h2d = sum(b.numel() * b.element_size() for b in host_bufs)
    d2h = out.numel() * 4

    def step():
        for d, h in zip(dev_bufs, host_bufs):
            d.copy_(h, non_blocking=True)
        case.run(out=out, stream=stream)
        host_out.copy_(out, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(2):
            step()
        torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for _ in range(steps):
            step()
        end.record(stream)
        torch.cuda.synchronize()
    return start.elapsed_time(end) / steps, h2d, d2h


# Configurations whose CPU baseline runs the oracle on a seeded sample of
# query rows (the full call would take minutes), extrapolated by live pairs.
CPU_SAMPLED_ROWS = {"prefill-long": 256, "chunked": 256, "prefill-long-fp8": 256}


def cpu_baseline_config(w):
    """The oracle, as it stands, on every host core: the full call for
    prefill-tiny, decode, MTP and decode-fp8; 256 seeded sampled rows for
    prefill-long, chunked and prefill-long-fp8, extrapolated to the full call
    by live (row, token) pairs.  A single-core figure beside it for
    prefill-tiny (the full call) and decode (4 rows, scaled by rows)."""
    import numpy as np
    import oracle
    from sparse_attention_mxfp4_gb300 import workloads as W
    kd, ks, sd, ss, bt, n = W.compact_host(w)
    cores = os.cpu_count() or 1
    n_sample = CPU_SAMPLED_ROWS.get(w.name)
    rows = W.sample_rows(w, n_sample, 0) if n_sample else np.arange(w.total_rows)
    lp = dict(decode=w.decode, seq_lens=w.seq_lens.numpy(), max_seq_len=w.max_seq_len,
              cu_seqlens_q=None if w.decode else w.cu_seqlens_q.numpy(),
              prefix_lens=None if w.decode else w.prefix_lens.numpy())
    all_pairs = oracle.live_pairs(rows=np.arange(w.total_rows), **lp)
    common = dict(decode=w.decode, q=W.q_numpy(w), q_is_e4m3=w.q_is_e4m3, block_table=bt,
                  block_table_stride=w.block_table_stride, seq_lens=w.seq_lens.numpy(),
                  cu_seqlens_q=None if w.decode else w.cu_seqlens_q.numpy(),
                  prefix_lens=None if w.decode else w.prefix_lens.numpy(), max_seq_len=w.max_seq_len,
                  sm_scale=w.sm_scale, rows=rows, num_pool_pages=n, num_threads=cores)

    def run(**kw):
        t0 = time.perf_counter()
        if w.cache == "fp8":
            oracle.score_fp8(k_fp8=kd, k_page_stride=sd, **kw)
        else:
            oracle.score(k_data=kd, k_scale=ks, k_data_page_stride=sd, k_scale_page_stride=ss, **kw)
        return time.perf_counter() - t0

    dt = run(**common)
    if n_sample:
        pairs = oracle.live_pairs(rows=rows, **lp)
        dt *= all_pairs / max(1, pairs)
        sample = (f"{len(rows)} seeded sampled query rows of the {w.name} workload ({pairs} of {all_pairs} live "
                  f"row-token pairs), fp64, OpenMP over rows; time extrapolated by live pairs")
    else:
        sample = (f"full call: all {len(rows)} query rows of the {w.name} workload, fp64, OpenMP over rows, "
                  f"1 repetition (not extrapolated)")
    res = {"value": round(dt * 1e6, 1), "unit": "us/call", "cores": cores, "kind": "oracle", "sample": sample,
           "extrapolated": bool(n_sample)}
    if w.name in ("prefill-tiny", "decode"):
        # one core: the whole tiny call; the first 4 decode rows (the rows all
        # have the same length) scaled to the full call by rows
        one_rows = rows if w.name == "prefill-tiny" else rows[:4]
        dt1 = run(**dict(common, rows=one_rows, num_threads=1)) * len(rows) / len(one_rows)
        res["single_core"] = {"value": round(dt1 * 1e6, 1), "unit": "us/call", "cores": 1,
                              "sample": "the full call on one thread" if w.name == "prefill-tiny" else
                              f"rows 0..3 of the {w.name} workload on one thread, scaled by rows "
                              f"({len(rows)} / 4)"}
    return res


L2_BYTES = 129 * 1024 * 1024   # GB300 L2 (nominal)


def time_calls_rotating(cases, outs, steps, warmup, stream, call=None):
    """Device time per call with a cold L2: one replay of a graph of ``steps``
    calls that cycle over ``len(cases)`` disjoint copies of the inputs and
    outputs (together larger than L2, so no call finds its pages in L2)."""
    import torch
    call = call or (lambda c, o: c.run(out=o, stream=stream))
    with torch.cuda.stream(stream):
        for i in range(warmup):
            call(cases[i % len(cases)], outs[i % len(outs)])
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(steps):
                call(cases[i % len(cases)], outs[i % len(outs)])
        g.replay()
        torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        g.replay()
        end.record(stream)
        torch.cuda.synchronize()
    del g
    return start.elapsed_time(end) / steps


# Configurations whose index cache fits in L2: timed warm (the same inputs
# every call) and cold (rotating over disjoint copies larger than L2).
COLD_L2_CONFIGS = ("prefill-tiny", "prefill-long", "chunked")


def secondary_configs(names, peaks, stream, cpu=True):
    import torch
    from sparse_attention_mxfp4_gb300 import harness
    from sparse_attention_mxfp4_gb300 import workloads as W
    res = {}
    fp8_peak = peaks["bf16_tflops"] * FP8_OVER_BF16
    fp4_peak = peaks["bf16_tflops"] * FP4_OVER_BF16
    for name in names:
        w = W.make_config(name)
        case = harness.to_device(w)
        out = torch.empty(case.out_shape_scores, dtype=torch.float32, device="cuda")
        work = workload_work(w)
        steps = 200 if name == "prefill-tiny" else (5 if name == "chunked" else 20)
        ms = time_calls(case, out, steps, 3, stream)
        tf = work["flops"] / (ms * 1e-3) / 1e12
        r = {"us_per_call": round(ms * 1e3, 3), "steps": steps, "cache": w.cache,
             "l2": "inputs larger than L2" if work["k_bytes"] > L2_BYTES else "warm: the same inputs every call",
             "mma_tflops": round(tf, 1),
             "frac_of_fp8_dense_peak": round(tf / fp8_peak, 4),
             "frac_of_fp4_dense_peak": round(tf / fp4_peak, 4),
             "hbm_gbs_algorithmic": round(work["bytes"] / (ms * 1e-3) / 1e9, 1),
             "frac_of_hbm_peak": round(work["bytes"] / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
             "flops_per_call": work["flops"], "bytes_per_call": work["bytes"]}
        if name == "prefill-tiny":
            # eager calls back to back (no graph): the host's launch path,
            # tensor-map lookups included, sets the pace of a small call
            n_eager = 200
            with torch.cuda.stream(stream):
                for _ in range(10):
                    case.run(out=out, stream=stream)
                torch.cuda.synchronize()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                t0 = time.perf_counter()
                e0.record(stream)
                for _ in range(n_eager):
                    case.run(out=out, stream=stream)
                e1.record(stream)
                host_s = time.perf_counter() - t0
                torch.cuda.synchronize()
            r["eager"] = {"us_per_call": round(e0.elapsed_time(e1) / n_eager * 1e3, 3), "calls": n_eager,
                          "host_us_per_call": round(host_s / n_eager * 1e6, 3),
                          "timing": "CUDA events around eager calls enqueued back to back through the Python "
                                    "binding (host launch path included)"}
        if name in COLD_L2_CONFIGS:
            # disjoint copies of the pool, query and output, rotated so that
            # together they exceed twice the L2 (at least 2 copies)
            region = sum(b.numel() for b in case.buffers) + case.q.numel() * case.q.element_size() \
                + out.numel() * 4
            n_reg = max(2, -(-2 * L2_BYTES // region))
            cases = [case] + [harness.to_device(w) for _ in range(n_reg - 1)]
            outs = [out] + [torch.empty_like(out) for _ in range(n_reg - 1)]
            csteps = max(n_reg, steps if name != "prefill-tiny" else 2 * n_reg)
            cms = time_calls_rotating(cases, outs, csteps, n_reg, stream)
            ctf = work["flops"] / (cms * 1e-3) / 1e12
            r["cold"] = {"us_per_call": round(cms * 1e3, 3), "steps": csteps, "regions": n_reg,
                         "region_bytes": region,
                         "l2": f"cold: {n_reg} disjoint copies of pool, query and output rotated",
                         "mma_tflops": round(ctf, 1), "frac_of_fp8_dense_peak": round(ctf / fp8_peak, 4),
                         "frac_of_fp4_dense_peak": round(ctf / fp4_peak, 4)}
            del cases, outs
        if cpu:
            r["cpu_baseline"] = cpu_baseline_config(w)
        res[name] = r
        del case, out
        torch.cuda.empty_cache()
    return res


DECODE_SWEEP_BATCHES = (1, 4, 16, 64)
DECODE_SWEEP_CONTEXTS = (8192, 131072)


def secondary_decode_sweep(peaks, stream, steps=20):
    """Decode block scores over B requests x ctx tokens for B in 1, 4, 16, 64
    and ctx in 8K, 128K (the pages' decode auto-CTA table spans the same
    range): the pages of the decode workload's 70,000-page pool (split views),
    block tables drawn by a seeded permutation of its pages, bf16 N(0,1)
    queries.  When one call's pages fit in L2, the calls rotate over disjoint
    groups of B requests (distinct pages) covering more than twice the L2."""
    import torch
    import sparse_attention_mxfp4_gb300 as mx4
    from sparse_attention_mxfp4_gb300 import harness
    from sparse_attention_mxfp4_gb300 import workloads as W
    w = W.make_config("decode")
    case = harness.to_device(w)
    ids = w.page_ids.to(torch.int32)
    g = torch.Generator().manual_seed(4242)
    res = {}
    for ctx in DECODE_SWEEP_CONTEXTS:
        P = ctx // W.PAGE
        for B in DECODE_SWEEP_BATCHES:
            per_call = B * P * W.PAGE_BYTES
            n_reg = max(1, min(ids.numel() // (B * P), -(-2 * L2_BYTES // per_call)))
            rows = n_reg * B
            perm = ids[torch.randperm(ids.numel(), generator=g)[: rows * P]]
            bt = perm.view(rows, P).contiguous().cuda()
            q = torch.randn((rows, W.HEADS, W.DIM), generator=g).to(torch.bfloat16).cuda()
            sl = torch.full((rows,), ctx, dtype=torch.int32, device="cuda")
            out = torch.empty((rows, W.HEADS, P), dtype=torch.float32, device="cuda")
            regions = [slice(r * B, (r + 1) * B) for r in range(n_reg)]

            def call(rg, _o):
                mx4.mx4_index_score_decode(q[rg], case.k_data, case.k_scale, w.k_data_page_stride,
                                           w.k_scale_page_stride, bt[rg], sl[rg], ctx, w.sm_scale, out[rg],
                                           num_pool_pages=w.num_pool_pages, stream=stream)
            n_steps = max(steps, n_reg)
            ms = time_calls_rotating(regions, regions, n_steps, min(n_reg, 8), stream, call=call)
            nbytes = per_call + B * W.HEADS * W.DIM * 2 + B * W.HEADS * P * 4 + B * P * 4
            gbs = nbytes / (ms * 1e-3) / 1e9
            res[f"B{B}_ctx{ctx // 1024}K"] = {
                "us_per_call": round(ms * 1e3, 3), "requests": B, "context": ctx, "steps": n_steps,
                "regions": n_reg, "bytes_per_call": nbytes, "hbm_gbs_algorithmic": round(gbs, 1),
                "frac_of_hbm_peak": round(gbs / peaks["hbm_gbs"], 4),
                "l2": "inputs larger than L2" if n_reg == 1 else f"cold: {n_reg} disjoint request groups rotated"}
            del bt, q, sl, out
    res["device_status"] = mx4.mx4_index_get_device_status()
    del case
    torch.cuda.empty_cache()
    return res


def writer_work(case):
    """Algorithmic bytes of one index-K write: per written token 256 B of bf16
    key read, 64 + 4 B of page bytes written, 8 B of slot read."""
    n = int((case.slot_mapping >= 0).sum())
    return {"tokens": n, "bytes": n * (2 * 128 + 64 + 4 + 8)}


def secondary_writer(peaks, stream, steps=20):
    """The index-K page writer on its measured workloads, each call timed
    alone with CUDA events after a 256 MiB L2 flush (the keys and pages of one
    call fit in L2)."""
    import torch
    import sparse_attention_mxfp4_gb300 as mx4
    from sparse_attention_mxfp4_gb300 import workloads as W
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    res = {}
    for name in W.WRITE_CONFIG_NAMES:
        case = W.make_write_config(name)
        bufs, (dbuf, doff), (sbuf, soff) = W.write_pool(case, device="cuda")
        k = case.k.cuda()
        sm = case.slot_mapping.cuda()

        def call():
            mx4.mx4_index_k_write(k, sm, dbuf[doff:], sbuf[soff:], case.k_data_page_stride,
                                  case.k_scale_page_stride, num_pool_pages=case.num_pool_pages, stream=stream)
        with torch.cuda.stream(stream):
            for _ in range(3):
                call()
            evs = []
            for _ in range(steps):
                flush.zero_()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                call()
                e1.record(stream)
                evs.append((e0, e1))
            torch.cuda.synchronize()
        us = statistics.median(a.elapsed_time(b) for a, b in evs) * 1e3
        work = writer_work(case)
        gbs = work["bytes"] / (us * 1e-6) / 1e9
        res[name] = {"us_per_call": round(us, 3), "steps": steps, "tokens": work["tokens"],
                     "bytes_per_call": work["bytes"], "hbm_gbs_algorithmic": round(gbs, 1),
                     "frac_of_hbm_peak": round(gbs / peaks["hbm_gbs"], 4),
                     "l2": "flushed before each call (256 MiB write)",
                     "description": case.description}
        del bufs, dbuf, sbuf, k, sm
    del flush
    torch.cuda.empty_cache()
    return res


def secondary_topk(peaks, stream, topk=16, steps=50):
    """Top-k page selection (topk pages, the last page forced, one head
    group) on the block scores of the decode and prefill-long workloads,
    timed as one replay of a graph of `steps` calls.  Algorithmic bytes: the
    scores read (rows x 64 x P x 4) plus the selection written."""
    import torch
    import sparse_attention_mxfp4_gb300 as mx4
    from sparse_attention_mxfp4_gb300 import harness
    from sparse_attention_mxfp4_gb300 import workloads as W
    res = {}
    for name in ("decode", "prefill-long"):
        w = W.make_config(name)
        case = harness.to_device(w)
        with torch.cuda.stream(stream):
            scores = case.run(stream=stream)
            torch.cuda.synchronize()
            sel = torch.empty((w.total_rows, 1, topk), dtype=torch.int32, device="cuda")
            cnt = torch.empty((w.total_rows, 1), dtype=torch.int32, device="cuda")

            def call():
                if w.decode:
                    mx4.mx4_index_topk_decode(scores, case.block_table, case.seq_lens, w.max_seq_len, topk,
                                              sel=sel, count=cnt, stream=stream)
                else:
                    mx4.mx4_index_topk_prefill(scores, case.block_table, case.cu_seqlens_q, case.seq_lens,
                                               case.prefix_lens, w.max_query_len, w.max_seq_len, topk, sel=sel,
                                               count=cnt, stream=stream)
            for _ in range(3):
                call()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(steps):
                    call()
            g.replay()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
        us = e0.elapsed_time(e1) / steps * 1e3
        nbytes = scores.numel() * 4 + sel.numel() * 4 + cnt.numel() * 4
        gbs = nbytes / (us * 1e-6) / 1e9
        res[name] = {"us_per_call": round(us, 3), "steps": steps, "topk": topk, "local_pages": 1, "kv_groups": 1,
                     "bytes_per_call": nbytes, "hbm_gbs_algorithmic": round(gbs, 1),
                     "frac_of_hbm_peak": round(gbs / peaks["hbm_gbs"], 4),
                     "l2": "scores larger than L2" if scores.numel() * 4 > 129e6 else "scores fit in L2 (warm)"}
        del case, scores, sel, cnt, g
        torch.cuda.empty_cache()
    return res


def secondary_attn(peaks, stream, steps=50, name="pa-decode"):
    """Sparse paged-attention decode on the pa-decode workload (64 rows x 16
    query heads over 16 selected MXFP4 pages of K and V), timed as one replay
    of a graph of `steps` calls.  Algorithmic bytes: the listed K and V pages
    (8704 B each per KV head) + Q + the bf16 output."""
    import torch
    import sparse_attention_mxfp4_gb300 as mx4
    from sparse_attention_mxfp4_gb300 import workloads as W
    c = W.make_attn_config(name)
    q, kp, vp = c.q.cuda(), c.k_pool.cuda(), c.v_pool.cuda()
    bt, cl = c.block_table.cuda(), c.context_lens.cuda()
    out = torch.empty((c.rows, c.kv_heads, c.groups, W.DIM), dtype=torch.bfloat16, device="cuda")
    with torch.cuda.stream(stream):
        for _ in range(3):
            mx4.mx4_sparse_pa_decode(q, kp, vp, bt, cl, c.softmax_scale, out, stream=stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(steps):
                mx4.mx4_sparse_pa_decode(q, kp, vp, bt, cl, c.softmax_scale, out, stream=stream)
        g.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
    us = e0.elapsed_time(e1) / steps * 1e3
    ctx = c.context_lens.to(torch.int64)
    pages = int(((ctx + 127) // 128).sum())
    nbytes = pages * 2 * W.PAGE_BYTES + q.numel() + out.numel() * 2
    flops = int(ctx.sum()) * c.groups * W.DIM * 2 * 2
    res = {"us_per_call": round(us, 3), "steps": steps, "rows": c.rows, "kv_heads": c.kv_heads,
           "groups": c.groups, "pages_per_row": int(c.block_table.shape[2]), "bytes_per_call": nbytes,
           "hbm_gbs_algorithmic": round(nbytes / (us * 1e-6) / 1e9, 1),
           "frac_of_hbm_peak": round(nbytes / (us * 1e-6) / 1e9 / peaks["hbm_gbs"], 4),
           "tflops": round(flops / (us * 1e-6) / 1e12, 2), "description": c.description}
    del q, kp, vp, bt, cl, out, g
    torch.cuda.empty_cache()
    return res


def secondary_decode_step(peaks, stream, topk=16, steps=20):
    """One decode step of the whole sparse-attention path on the decode
    workload (64 requests x 131,072 tokens): the new token's index key and
    its K and V quantised into their caches (three writer calls), the block
    scores, the top-k pages (the last page forced), and attention of 16 query
    heads over the selected pages of an MXFP4 K/V cache (one KV head).  The
    row context for the attention is derived from the selection count on the
    device.  Timed as one replay of a graph of ``steps`` steps."""
    import torch
    import sparse_attention_mxfp4_gb300 as mx4
    from sparse_attention_mxfp4_gb300 import harness
    from sparse_attention_mxfp4_gb300 import workloads as W
    w = W.make_config("decode")
    case = harness.to_device(w)
    B, npool = w.total_rows, w.num_pool_pages
    g = torch.Generator().manual_seed(77)
    with torch.cuda.stream(stream):
        keys = torch.randn((3, B, W.DIM), generator=g).to(torch.bfloat16).cuda()
        lens = w.seq_lens.to(torch.int64)
        last = torch.tensor([int(w.block_table[b, (int(lens[b]) - 1) // W.PAGE]) for b in range(B)],
                            dtype=torch.int64)
        slots = (last * W.PAGE + (lens - 1) % W.PAGE).cuda()
        # main K and V caches: [pages, 1 KV head, 8704], codes then scales
        kv = torch.empty((2, npool, 1, W.PAGE_BYTES), dtype=torch.uint8, device="cuda")
        kv[..., :W.DATA_BYTES].random_(0, 256)
        kv[..., W.DATA_BYTES:].random_(122, 128)
        q_att = torch.randn((B, 1, 16, W.DIM), generator=g).to(torch.float8_e4m3fn).view(torch.uint8).cuda()
        scores = torch.empty(case.out_shape_scores, dtype=torch.float32, device="cuda")
        sel = torch.empty((B, 1, topk), dtype=torch.int32, device="cuda")
        cnt = torch.empty((B, 1), dtype=torch.int32, device="cuda")
        out = torch.empty((B, 1, 16, W.DIM), dtype=torch.bfloat16, device="cuda")
        ctx = torch.empty((B, 1), dtype=torch.int32, device="cuda")
        kflat = kv[0].view(-1)
        vflat = kv[1].view(-1)

        def step():
            mx4.mx4_index_k_write(keys[0], slots, case.k_data, case.k_scale, w.k_data_page_stride,
                                  w.k_scale_page_stride, num_pool_pages=npool, stream=stream)
            mx4.mx4_index_k_write(keys[1], slots, kflat, kflat[W.DATA_BYTES:], W.PAGE_BYTES, W.PAGE_BYTES,
                                  num_pool_pages=npool, stream=stream)
            mx4.mx4_index_k_write(keys[2], slots, vflat, vflat[W.DATA_BYTES:], W.PAGE_BYTES, W.PAGE_BYTES,
                                  num_pool_pages=npool, stream=stream)
            case.run(out=scores, stream=stream)
            # the selection also emits each row's context: the live tokens of
            # its selected pages
            mx4.mx4_index_topk_decode(scores, case.block_table, case.seq_lens, w.max_seq_len, topk, sel=sel,
                                      count=cnt, tokens=ctx, stream=stream)
            mx4.mx4_sparse_pa_decode(q_att, kv[0], kv[1], sel, ctx, w.sm_scale, out, stream=stream)

        for _ in range(3):
            step()
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            for _ in range(steps):
                step()
        gr.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        gr.replay()
        e1.record(stream)
        torch.cuda.synchronize()
    us = e0.elapsed_time(e1) / steps * 1e3
    res = {"us_per_step": round(us, 3), "steps": steps, "rows": B, "context_tokens": int(w.max_seq_len),
           "topk": topk, "kernels_per_step": 6,
           "description": "3 writer calls (index K, K, V) + block scorer + top-k (which also emits each row's "
                          "attention context) + sparse attention (16 query heads, 1 KV head) over the selected "
                          "pages; no other kernel",
           "device_status": mx4.mx4_index_get_device_status()}
    del case, kv, scores, sel, cnt, out, gr
    torch.cuda.empty_cache()
    return res


def run_ours(args):
    import torch
    import torch.distributed as dist
    import sparse_attention_mxfp4_gb300 as mx4
    from sparse_attention_mxfp4_gb300 import harness
    from sparse_attention_mxfp4_gb300 import workloads as W

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    mx4.build()
    mx4.load_library()
    peaks = load_peaks()
    stream = torch.cuda.Stream()

    w = W.make_config(args.config)
    case = harness.to_device(w)
    out = torch.empty(case.out_shape_scores, dtype=torch.float32, device="cuda")
    work = workload_work(w)

    # W eager warm-up calls, then the K timed steps as one replay of a CUDA
    # graph holding K calls (captured and replayed once untimed first), so
    # the number is device time without host launch gaps.  The clock samples
    # cover the warm-up and the timed replay (a short timed region alone may
    # fall between two samples).
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            case.run(out=out, stream=stream)
        torch.cuda.synchronize()
        graph = capture_calls(case, out, args.steps, stream)
        graph.replay()
        torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):        # a graph replays on the current stream
        start.record(stream)
        graph.replay()
        end.record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    ms_rank = start.elapsed_time(end) / args.steps
    clocks = sampler.stop() if sampler else None
    status = mx4.mx4_index_get_device_status()
    ms = max_over_ranks(ms_rank, ws, "cuda")

    e2e_ms, h2d, d2h = measure_e2e(case, max(3, min(args.steps, 20)), stream)

    line = None
    if rank == 0:
        us_per_call = ms * 1e3 / ws          # N independent calls per step across the job
        if w.decode:
            achieved = work["bytes"] / (ms * 1e-3) / 1e9
            roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                    "traffic": profile_traffic("mx4_score_kernel", w.name),
                    "peak_source": peaks["source"],
                    "algorithmic_bytes_per_launch": work["bytes"],
                    "index_cache_bytes_per_launch": work["k_bytes"],
                    "index_cache_gbs": round(work["k_bytes"] / (ms * 1e-3) / 1e9, 1)}
        else:
            fp8_peak = peaks["bf16_tflops"] * FP8_OVER_BF16
            achieved = work["flops"] / (ms * 1e-3) / 1e12
            roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": fp8_peak, "unit": "TFLOP/s",
                    "frac": round(achieved / fp8_peak, 4),
                    "traffic": profile_traffic("mx4_score_kernel", w.name),
                    "peak_source": peaks["source"] + " bf16 x 2 (nominal fp8/bf16 ratio)",
                    "algorithmic_flops_per_launch": work["flops"]}
        line = {
            "metric": "MXFP4 index-score us/call (decode B=64, ctx 131072)" if w.name == "decode"
            else f"index-score us/call ({w.name})",
            "value": round(us_per_call, 3), "unit": "us/call", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 6), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 x e2m1 -> f32",
            "data": "synthetic (seeded; no dataset or weights)",
            "config": {"workload": w.name, "description": w.description, "heads": W.HEADS, "head_dim": W.DIM,
                       "page_tokens": W.PAGE, "rows": w.total_rows, "requests": w.num_seqs,
                       "max_seq_len": w.max_seq_len, "q_dtype": "e4m3" if w.q_is_e4m3 else "bf16",
                       "layout": w.layout, "l2": "inputs larger than L2 (no flush)" if work["k_bytes"] > 129e6
                       else "K fits in L2: warm-L2 number",
                       "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                       "timing": "CUDA events around one replay of a CUDA graph of K back-to-back calls"},
            "roofline": roof,
            "e2e": {"value": round(e2e_ms * 1e3 / ws, 3), "unit": "us/call", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": args.steps,
            "clocks": clocks,
            "device_status": status,
        }
        if ws == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline_config(w)
        if ws == 1 and not args.no_secondary:
            del case, out
            torch.cuda.empty_cache()
            names = [n for n in W.CONFIG_NAMES + W.FP8_CONFIG_NAMES if n != w.name]
            line["secondary"] = secondary_configs(names, peaks, stream, cpu=not args.no_cpu_baseline)
            line["secondary"]["decode_sweep"] = secondary_decode_sweep(peaks, stream)
            line["secondary"]["index_k_write"] = secondary_writer(peaks, stream)
            line["secondary"]["topk"] = secondary_topk(peaks, stream)
            line["secondary"]["sparse_pa_decode"] = secondary_attn(peaks, stream)
            line["secondary"]["sparse_pa_decode_4kvh"] = secondary_attn(peaks, stream, name="pa-decode-4kvh")
            line["secondary"]["decode_step"] = secondary_decode_step(peaks, stream)
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


# ------------------------------------------------------------ reference arm --
def run_reference(args):
    """The fp64 oracle timed on the host cores, on a bounded sample of the
    same workload per step: every request's first T tokens (all 64 heads),
    T chosen so the whole run takes about two minutes; the per-call time is
    extrapolated by live (row, token) pairs."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import dataclasses
    import numpy as np
    import torch
    import oracle
    from sparse_attention_mxfp4_gb300 import workloads as W

    oracle.build()
    w = W.make_config(args.config)
    cores = os.cpu_count() or 1
    work = workload_work(w)
    budget_s = 120.0 / max(1, args.steps + args.warmup)
    rows = np.arange(min(w.total_rows, cores), dtype=np.int64)
    # ~1e9 multiply-adds per second per core for the oracle
    tokens = int(budget_s * 1e9 / (W.HEADS * W.DIM))
    tokens = max(W.PAGE, min(w.max_seq_len, tokens // W.PAGE * W.PAGE))
    sub = dataclasses.replace(w, seq_lens=torch.clamp(w.seq_lens, max=tokens),
                              max_seq_len=min(w.max_seq_len, tokens))
    if not sub.decode:
        sub = dataclasses.replace(sub, prefix_lens=torch.clamp(sub.prefix_lens, max=tokens))
    kd, ks, sd, ss, bt, n = W.compact_host(sub)
    sample_pairs = oracle.live_pairs(decode=sub.decode, seq_lens=sub.seq_lens.numpy(),
                                     max_seq_len=sub.max_seq_len,
                                     cu_seqlens_q=None if sub.decode else sub.cu_seqlens_q.numpy(),
                                     prefix_lens=None if sub.decode else sub.prefix_lens.numpy(), rows=rows)

    def step():
        oracle.score(decode=sub.decode, q=W.q_numpy(sub), q_is_e4m3=sub.q_is_e4m3, k_data=kd, k_scale=ks,
                     k_data_page_stride=sd, k_scale_page_stride=ss, block_table=bt,
                     block_table_stride=sub.block_table_stride, seq_lens=sub.seq_lens.numpy(),
                     cu_seqlens_q=None if sub.decode else sub.cu_seqlens_q.numpy(),
                     prefix_lens=None if sub.decode else sub.prefix_lens.numpy(),
                     max_seq_len=sub.max_seq_len, sm_scale=sub.sm_scale, rows=rows, num_pool_pages=n,
                     num_threads=cores)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    scale = work["live_pairs"] / max(1, sample_pairs)
    us = dt * scale * 1e6
    sample = (f"per step: query rows 0..{len(rows) - 1} of the {w.name} workload, first {tokens} tokens "
              f"of each context ({sample_pairs} live row-token pairs of {work['live_pairs']}); "
              f"time extrapolated by live pairs")
    line = {"impl": "reference",
            "metric": "MXFP4 index-score us/call (decode B=64, ctx 131072)" if w.name == "decode"
            else f"index-score us/call ({w.name})",
            "value": round(us, 1), "unit": "us/call", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": {"workload": w.name, "description": w.description},
            "cpu_baseline": {"value": round(us, 1), "unit": "us/call", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(us, 1), "unit": "us/call", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--config", default="decode",
                    choices=("decode", "prefill-tiny", "prefill-long", "mtp", "chunked", "decode-fp8",
                             "prefill-long-fp8"))
    ap.add_argument("--no-secondary", action="store_true", help="skip the other configurations")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
