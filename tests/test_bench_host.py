"""bench.py's host-side arithmetic and parsing, without a GPU.

The reported numbers rest on a few pure functions: the algorithmic work of a
call (flops, the key and query bytes read once, the outputs), the choice of
roofline (tensor for query chunks, HBM for decode), the kernel classes read
from an ncu CSV, the DRAM-traffic record and its source check, and the clock
summary of the timed region. Expected values are worked out by hand below.
"""
import hashlib
import json
import os
import shutil
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from sparse_attention_key_gb300 import workloads as wl  # noqa: E402

PEAKS = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1800.0,
         "source": "test"}


def _batch(q_pos, q_counts, k_lens, topk=2048):
    """A Workload with hand-set query positions (zero q/k/w: only shapes matter)."""
    T = len(q_pos)
    cu_q = np.concatenate([[0], np.cumsum(q_counts)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(k_lens)]).astype(np.int32)
    return wl.Workload("hand", np.zeros((T, 32, 128), np.uint16), np.zeros((T, 32), np.float32),
                       np.asarray(q_pos, np.int32), cu_q, cu_k,
                       np.zeros((int(cu_k[-1]), 128), np.uint16), topk=topk)


def test_algorithmic_work_of_a_ragged_batch():
    # sequence 0: queries at positions 10 and 700 of 1,000 keys (keys 0..700
    # are read); sequence 1: one query at position 5 of 50 keys (keys 0..5)
    w = _batch([10, 700, 5], [2, 1], [1000, 50])
    a = bench.algorithmic(w)
    assert a["unique_keys"] == 701 + 6
    assert a["score_bytes"] == 707 * 256 + 3 * (8192 + 128)      # keys once, q and w per query
    assert a["topk_bytes"] == 3 * (2048 * 4 + 4)                 # idx rows and counts
    assert a["call_bytes"] == a["score_bytes"] + a["topk_bytes"]
    assert a["flops"] == 8192.0 * (11 + 701 + 6)                 # 2 x 32 heads x 128 dims per pair
    assert a["staged_bytes"] == 4 * (11 + 701 + 6)
    assert a["ln_bytes"] == 0                                    # no raw keys in this batch


def test_algorithmic_work_of_the_decode_batch():
    # eight decode queries at the end of 8..64 Ki keys: every key read once,
    # 249,856 x 256 B + 8 x (8 KB q + 128 B w) = 64,029,696 B; the LayerNorm
    # reads and writes each raw key row (512 B) plus its bf16 weight and bias
    w = wl.by_index(2)
    a = bench.algorithmic(w)
    assert a["unique_keys"] == 249_856
    assert a["score_bytes"] == 64_029_696
    assert a["ln_bytes"] == 249_856 * 512 + 512
    assert not bench.tensor_bound(w)


def test_roofline_choice_and_arithmetic():
    chunk = _batch(list(range(100, 120)), [20], [120])           # 20 queries, one sequence
    assert bench.tensor_bound(chunk)                             # T > 4 B: the contraction dominates
    per_call, call = bench.rooflines(chunk, {"plan": 0.01, "score": 0.5, "topk": 0.2}, 0.75, PEAKS)
    flops = 8192.0 * sum(range(101, 121))
    assert per_call["score"]["bound"] == "tensor"
    assert per_call["score"]["achieved"] == pytest.approx(flops / 0.5e-3 / 1e12)
    assert per_call["score"]["frac"] == pytest.approx(flops / 0.5e-3 / 1e12 / 2000.0)
    assert call["bound"] == "tensor" and call["ms"] == 0.75
    # the selection is priced at its outputs; its staged-score reads are overhead
    topk = per_call["topk"]
    assert topk["bound"] == "hbm" and topk["bytes"] == 20 * (2048 * 4 + 4)
    assert topk["overhead_bytes"] == 4 * sum(range(101, 121))
    assert per_call["plan"] == {"bound": "latency", "ms": 0.01}

    decode = _batch([999, 49], [1, 1], [1000, 50])
    assert not bench.tensor_bound(decode)                        # T <= 4 B: the key bytes dominate
    per_call, call = bench.rooflines(decode, {"score": 0.002}, 0.004, PEAKS)
    score_bytes = (1000 + 50) * 256 + 2 * (8192 + 128)
    assert per_call["score"]["bound"] == "hbm"
    assert per_call["score"]["achieved"] == pytest.approx(score_bytes / 2e-6 / 1e9)
    assert call["bytes"] == score_bytes + 2 * (2048 * 4 + 4)
    assert bench.rooflines(decode, {"score": 0.0}, 0.0, PEAKS) == ({"score": None}, None)


@pytest.mark.parametrize("name, cls", [
    ("void lidx::score_tc_kernel<lidx::TcCfg<8, 2, 2, 3, 16>>(CUtensorMap_st, CUtensorMap_st)", "score"),
    ("void lidx::score_tc_dyn_kernel<lidx::TcCfg<1, 1, 4, 6, 4>>(CUtensorMap_st)", "score"),
    ("void lidx::<unnamed>::topk_stream_kernel<512>(const float *, long)", "topk"),
    ("lidx::<unnamed>::topk_cluster_kernel(const float *, long)", "topk"),
    ("void lidx::key_layernorm_kernel<0, 0>(const unsigned short *)", "key_layernorm"),
    ("void lidx::tc_plan_fast_kernel<16>(const int *, const int *)", None),
    ("void lidx::sparse_mla_kernel<96, false>(CUtensorMap_st)", None),
    ("void at::vectorized_elementwise_kernel<4, at::FillFunctor<int>>(int, T2, T3)", None),
])
def test_kernel_classes_of_ncu_names(name, cls):
    assert bench._kernel_class(name) == cls


def _ncu_csv(path, launches):
    """A CSV in ncu's --csv layout: launches = [(kernel name, read bytes, write bytes)]."""
    cols = ["ID", "Process ID", "Process Name", "Host Name", "Kernel Name", "Context", "Stream",
            "Block Size", "Grid Size", "Device", "CC", "Section Name", "Metric Name", "Metric Unit",
            "Metric Value"]
    lines = ["==PROF== Connected to process 1", ",".join(f'"{c}"' for c in cols)]
    for i, (name, rd, wr) in enumerate(launches):
        for metric, unit, val in (("dram__bytes_read.sum", "Mbyte", f"{rd / 1e6:,.6f}"),
                                  ("dram__bytes_write.sum", "byte", f"{wr:,}"),
                                  ("gpu__time_duration.sum", "ns", "1000")):
            row = [str(i), "1", "python3", "host", name, "1", "7", "(128, 1, 1)", "(1, 1, 1)", "0",
                   "10.3", "Command line profiler metrics", metric, unit, val]
            lines.append(",".join(f'"{x}"' for x in row))
    open(path, "w").write("\n".join(lines) + "\n")


def test_traffic_record_round_trip_and_source_check(tmp_path, monkeypatch):
    # a private copy of the sources and profiles/, so the test writes nothing in the repo
    csrc = tmp_path / "sparse_attention_key_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    for src in bench.KERNEL_SOURCES.values():
        shutil.copy(os.path.join(ROOT, "sparse_attention_key_gb300", "csrc", src), csrc / src)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    plan, score = "void lidx::tc_plan_fast_kernel<16>(int)", "void lidx::score_tc_kernel<X>(int)"
    topk = "void lidx::<unnamed>::topk_stream_kernel<512>(int)"
    # two fused calls: plan, scorer and selection each; a torch fill in between
    csv_path = tmp_path / "dram.csv"
    _ncu_csv(csv_path, [(plan, 1_000, 0), (score, 240e6, 600_000_000), (topk, 645e6, 25_000_000),
                        ("void at::vectorized_elementwise_kernel<4>(int)", 5e6, 200_000_000),
                        (plan, 1_000, 0), (score, 260e6, 604_000_000), (topk, 647e6, 25_000_000)])
    bench.record_traffic(4, str(csv_path))
    rec = json.load(open(tmp_path / "profiles" / "dram_traffic.json"))["agentic_chunk"]
    assert set(rec) == {"score", "topk"}                          # the plan and torch are not classes
    assert rec["score"]["bytes_per_launch"] == (240e6 + 600e6 + 260e6 + 604e6) / 2
    assert rec["topk"]["bytes_per_launch"] == (645e6 + 25e6 + 647e6 + 25e6) / 2
    assert rec["score"]["sha256"] == hashlib.sha256((csrc / "score_tc.cu").read_bytes()).hexdigest()
    assert bench.dram_traffic(4, "score") == 852_000_000
    assert bench.dram_traffic(2, "score") is None                 # no record for that workload
    # a changed source invalidates its record, and only its record
    with open(csrc / "topk.cu", "a") as f:
        f.write("\n// changed\n")
    assert bench.dram_traffic(4, "topk") is None
    assert bench.dram_traffic(4, "score") == 852_000_000


def test_clock_summary_of_the_timed_region():
    cs = bench.ClockSampler("0")
    row = "0, {mhz}, 2070, 900.5, 0x0, {hw}, Not Active, Not Active, {cap}"
    cs.samples = [(1.0, row.format(mhz=1500, hw="Not Active", cap="Not Active")),   # before t0
                  (2.0, row.format(mhz=2070, hw="Not Active", cap="Active")),
                  (2.5, row.format(mhz=2040, hw="Not Active", cap="Not Active")),
                  (3.0, row.format(mhz=1980, hw="Not Active", cap="Active")),
                  (3.5, "[N/A], [N/A]"),                                          # unreadable
                  (9.0, row.format(mhz=900, hw="Active", cap="Not Active"))]     # after t1
    s = cs.summary(2.0, 3.5)
    assert s == {"sm_mhz": 2040.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    # no sample inside the window: every sample counts
    s = cs.summary(100.0, 101.0)
    assert s["samples"] == 5 and s["reasons"] == ["hw_slowdown", "sw_power_cap"]
