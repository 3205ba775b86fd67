"""Host-side arithmetic of bench.py (no GPU): the algorithmic work per call
that the roofline divides by, and the source hash that ties a committed ncu
summary to the code it measured."""
import os
import shutil
import types

import torch

import bench
from sparse_attention_mxfp4_gb300 import workloads as W

ROOT = os.path.abspath(os.path.join(os.path.dirname(__file__), ".."))


def _decode_like(B, L, cache="mxfp4"):
    seq = torch.full((B,), L, dtype=torch.int32)
    return types.SimpleNamespace(decode=True, seq_lens=seq, max_seq_len=L, cache=cache, num_seqs=B,
                                 q=torch.zeros((B, W.HEADS, W.DIM), dtype=torch.bfloat16), total_rows=B,
                                 num_out_pages=(L + W.PAGE - 1) // W.PAGE)


def test_decode_algorithmic_bytes_closed_form():
    """64 requests x 131,072 tokens: 1024 pages each read once (8704 B), Q
    (bf16), one fp32 cell per (row, head, page) and one 4-byte block-table
    entry per page."""
    w = _decode_like(64, 131072)
    work = bench.workload_work(w)
    pages = 64 * 1024
    assert work["pages_read"] == pages
    assert work["k_bytes"] == pages * 8704 == 570_425_344
    assert work["q_bytes"] == 64 * 64 * 128 * 2
    assert work["out_bytes"] == 64 * 64 * 1024 * 4
    assert work["bt_bytes"] == pages * 4
    assert work["bytes"] == 588_513_280
    assert work["flops"] == 64 * 131072 * 64 * 128 * 2


def test_fp8_cache_pages_are_16_kib():
    w = _decode_like(3, 1000, cache="fp8")
    work = bench.workload_work(w)
    assert work["pages_read"] == 3 * 8
    assert work["k_bytes"] == 3 * 8 * 16384


def test_prefill_live_pairs_closed_form():
    """One request, 4096 rows after a 126,976-token prefix: row i sees
    126,976 + i + 1 tokens; the live pairs are sum_i (126,977 + i)."""
    rows, prefix = 4096, 126976
    w = types.SimpleNamespace(decode=False, seq_lens=torch.tensor([prefix + rows], dtype=torch.int32),
                              max_seq_len=prefix + rows, cache="mxfp4", num_seqs=1,
                              cu_seqlens_q=torch.tensor([0, rows], dtype=torch.int32),
                              prefix_lens=torch.tensor([prefix], dtype=torch.int32),
                              q=torch.zeros((rows, W.HEADS, W.DIM), dtype=torch.bfloat16), total_rows=rows,
                              num_out_pages=(prefix + rows) // W.PAGE)
    work = bench.workload_work(w)
    pairs = rows * prefix + rows * (rows + 1) // 2
    assert work["live_pairs"] == pairs == 528_484_352
    assert work["flops"] == pairs * 2 * 64 * 128
    assert work["pages_read"] == 1024


def test_prefill_ragged_rows_use_their_own_limits():
    """Three requests, one without query rows (it contributes nothing); a row's limit is
    min(seq_len, prefix + position + 1) capped at max_seq_len."""
    w = types.SimpleNamespace(decode=False, seq_lens=torch.tensor([10, 300, 50], dtype=torch.int32),
                              max_seq_len=300, cache="mxfp4", num_seqs=3,
                              cu_seqlens_q=torch.tensor([0, 3, 3, 5], dtype=torch.int32),
                              prefix_lens=torch.tensor([8, 0, 40], dtype=torch.int32),
                              q=torch.zeros((5, W.HEADS, W.DIM), dtype=torch.bfloat16), total_rows=5,
                              num_out_pages=3)
    work = bench.workload_work(w)
    expect = [min(10, 8 + i + 1) for i in range(3)] + [min(50, 40 + i + 1) for i in range(2)]
    assert work["live_pairs"] == sum(expect)
    assert work["pages_read"] == 1 + 0 + 1


def _copy_tree(tmp_path):
    root = tmp_path / "repo"
    shutil.copytree(os.path.join(ROOT, "sparse_attention_mxfp4_gb300", "csrc"),
                    root / "sparse_attention_mxfp4_gb300" / "csrc")
    shutil.copytree(os.path.join(ROOT, "profiles"), root / "profiles")
    return root


def test_source_hash_ignores_comments_not_code(tmp_path, monkeypatch):
    root = _copy_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    h0 = bench.library_source_hash()
    f = root / "sparse_attention_mxfp4_gb300" / "csrc" / "writer_kernel.cuh"
    text = f.read_text()
    f.write_text(text.replace("namespace mx4 {", "// a new comment line\nnamespace mx4 {  /* and a block */", 1))
    assert bench.library_source_hash() == h0
    f.write_text(text.replace("namespace mx4 {", "namespace mx4 {\nconstexpr int kUnusedForTheTest = 1;", 1))
    assert bench.library_source_hash() != h0


def test_profile_traffic_only_for_matching_source(tmp_path, monkeypatch):
    root = _copy_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    prof = root / "profiles" / "mx4_score_kernel_decode.md"
    text = prof.read_text()
    want = int(text.split("traffic_bytes_per_launch:")[1].split()[0])
    prof.write_text(text.replace(text.split("source_hash:")[1].split()[0], bench.library_source_hash(), 1))
    assert bench.profile_traffic("mx4_score_kernel", "decode") == want
    prof.write_text(text.replace(text.split("source_hash:")[1].split()[0], "0123456789abcdef", 1))
    assert bench.profile_traffic("mx4_score_kernel", "decode") is None
    assert bench.profile_traffic("mx4_score_kernel", "no-such-workload") is None



def test_cpu_baseline_full_and_sampled(monkeypatch):
    """The CPU baseline runs the oracle on the whole call, or on sampled rows
    extrapolated by live pairs, and says which."""
    from sparse_attention_mxfp4_gb300 import workloads as W
    w = W.make_config("prefill-tiny")
    full = bench.cpu_baseline_config(w)
    assert full["kind"] == "oracle" and full["cores"] >= 1 and full["value"] > 0
    assert not full["extrapolated"] and "full call" in full["sample"]
    assert full["single_core"]["cores"] == 1
    monkeypatch.setitem(bench.CPU_SAMPLED_ROWS, "prefill-tiny", 8)
    part = bench.cpu_baseline_config(w)
    assert part["extrapolated"] and "8 seeded sampled query rows" in part["sample"]
    assert part["value"] > 0


def test_clock_sampler_waits_for_samples(tmp_path, monkeypatch):
    """The sampler returns from start() only once nvidia-smi has written a
    sample, and stop() waits for one sample after the timed region, so a
    region of a few milliseconds still has samples on both sides (a fake
    nvidia-smi on PATH that starts slowly and then prints every 20 ms)."""
    fake = tmp_path / "nvidia-smi"
    fake.write_text("#!/bin/sh\nsleep 0.3\n"
                    "while true; do echo '0, 1965, 2070, 700.5, 0x4, Not Active, Not Active, Not Active, Active'; "
                    "sleep 0.02; done\n")
    fake.chmod(0o755)
    monkeypatch.setenv("PATH", f"{tmp_path}{os.pathsep}{os.environ['PATH']}")
    s = bench.ClockSampler(0)
    s.path = str(tmp_path / "clocks.csv")
    s.start()
    assert s._lines() >= 1
    n = s._lines()
    res = s.stop()
    assert res["samples"] >= n + 1
    assert res["sm_mhz"] == 1965.0 and res["sm_max_mhz"] == 2070.0
    assert res["reasons"] == ["sw_power_cap"]
