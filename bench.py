"""Benchmark of the GB300 Lightning Indexer: query-key pairs/s of score + exact top-2048.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload I] [--impl ours|reference]

One step = one idx_score_topk call over one batch of the named workload (the
agentic chunk by default, the largest single-GPU workload): head scores with
the relu / head-weighted epilogue and the exact top-2048 with the tie/order
rule. The key LayerNorm runs once per key at cache fill and is timed on its
own where the workload chains it (decode batch). Inputs are resident in HBM
when the timed region starts; between timed steps L2 is flushed by writing a
256 MB buffer and then reading another 256 MB buffer (so that every step
starts with a cold L2 that holds no dirty lines of the flush). Rank 0 prints
one JSON line. Per-kernel times come from the same fused call: the library
records CUDA events between its launches (idx_set_kernel_events). The line
also carries a by_workload block with the fused-call time, per-kernel times
and rooflines of the decode batch, prefill ties, long decode and speculative
verification workloads. The e2e figure runs the same public call with the
inputs copied from pinned host memory and the indices and counts copied back
inside the timed region, the batch cut into up to four groups of whole
sequences whose copies overlap the earlier groups' calls.

--impl reference times the CPU oracle (the plain fp64 definition) on the host's
cores on a bounded row sample of the same workload, as the reference arm.

Multi-GPU (torchrun): each rank runs an independent replica of the workload
(the indexer has no exchange step); value = all ranks' pairs / max rank time.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_attention_key_gb300 import workloads as wl  # noqa: E402

METRIC = "indexer query-key pairs/s (score+exact top-2048); % of HBM / tensor roofline"
UNIT = "pairs/s"
DEFAULT_WORKLOAD = 4   # the agentic chunk: 4 x (50,000 cached keys + 800 new queries)


E2E_CHUNKS = 4   # groups of sequences (and copy streams) pipelined in the e2e step


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: str):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.marks = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self):
        self.marks.append(time.time())

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [s for (ts, s) in self.samples if t0 <= ts <= t1] or [s for _, s in self.samples]
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 9:
                continue
            try:
                mhz.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": float(np.median(mhz)) if mhz else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(mhz)}


def dram_traffic(workload: int, kernel: str):
    """DRAM bytes per launch of `kernel` from the ncu capture recorded in
    profiles/dram_traffic.json, or None when there is none or when the kernel's
    source file changed since the capture (sha256 recorded with it)."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get(wl.NAMES[workload], {}).get(kernel)
    if not rec:
        return None
    src = os.path.join(ROOT, "sparse_attention_key_gb300", "csrc", rec["source"])
    if not os.path.exists(src) or hashlib.sha256(open(src, "rb").read()).hexdigest() != rec["sha256"]:
        return None
    return rec["bytes_per_launch"]


KERNEL_SOURCES = {"key_layernorm": "layernorm.cu", "score": "score_tc.cu", "topk": "topk.cu"}


def _kernel_class(name: str):
    if "key_layernorm" in name:
        return "key_layernorm"
    if "score_tc_kernel" in name or "score_tc_dyn_kernel" in name:
        return "score"
    if "topk" in name:
        return "topk"
    return None


def record_traffic(workload: int, csv_path: str):
    """Average DRAM bytes per call of each kernel class in an ncu CSV of a
    --fused-only run, stored with the sha256 of the class's source file."""
    import csv
    import hashlib
    rows = list(csv.reader(open(csv_path)))
    hdr = next(i for i, r in enumerate(rows) if "Kernel Name" in r and "Metric Name" in r)
    h = rows[hdr]
    ki, mi, vi, ui, ii = (h.index("Kernel Name"), h.index("Metric Name"), h.index("Metric Value"),
                          h.index("Metric Unit"), h.index("ID"))
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "KB": 1e3, "MB": 1e6, "GB": 1e9}
    launches = {}
    for r in rows[hdr + 1:]:
        if len(r) <= vi or r[mi] not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            continue
        cls = _kernel_class(r[ki])
        if cls is None:
            continue
        launches.setdefault((r[ii], cls), 0.0)
        launches[(r[ii], cls)] += float(r[vi].replace(",", "")) * scale.get(r[ui], 1)
    calls = sum(1 for (_, c) in launches if c == "score")
    if calls == 0:
        raise SystemExit("no scorer launch in " + csv_path)
    out_path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    data = json.load(open(out_path)) if os.path.exists(out_path) else {}
    entry = {}
    for cls, src in KERNEL_SOURCES.items():
        total = sum(v for (_, c), v in launches.items() if c == cls)
        n = sum(1 for (_, c) in launches if c == cls)
        if n == 0:
            continue
        path = os.path.join(ROOT, "sparse_attention_key_gb300", "csrc", src)
        entry[cls] = {"source": src,
                      "sha256": hashlib.sha256(open(path, "rb").read()).hexdigest(),
                      "bytes_per_launch": int(round(total / calls))}
    data[wl.NAMES[workload]] = entry
    data["_note"] = ("DRAM bytes per fused call of each kernel class (dram__bytes_read.sum + "
                     "dram__bytes_write.sum, ncu --clock-control none, default cache control) "
                     "from a `bench.py --fused-only` capture, recorded by `bench.py "
                     "--record-traffic`; topk sums the selection kernels of one call. bench.py "
                     "reports a value only while the source file's sha256 matches.")
    json.dump(data, open(out_path, "w"), indent=1, sort_keys=True)
    print(json.dumps({wl.NAMES[workload]: entry}))


# ---------------------------------------------------------------------------
# replicas over ranks (the indexer has no exchange step: each rank runs an
# independent replica of the workload)
# ---------------------------------------------------------------------------

def max_over_ranks(values, world: int, device):
    """Element-wise maximum of per-rank timings over all ranks (a MAX
    all-reduce of one float64 vector on `device`; the identity for world 1)."""
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def whole_job_value(pairs_per_step: int, world: int, steps: int, max_ms: float) -> float:
    """Pairs per second of the whole job: every rank's pairs over the slowest
    rank's time."""
    return pairs_per_step * world * steps / (max_ms / 1e3)


# ---------------------------------------------------------------------------
# algorithmic work per call (the scorer's contraction, its key/query bytes, the
# selection's outputs; staged fp32 scores are overhead of the two-kernel design)
# ---------------------------------------------------------------------------

def algorithmic(w: wl.Workload):
    """Per-call algorithmic work of idx_score_topk and of the key LayerNorm."""
    unique_keys = 0
    for b in range(w.B):
        q0, q1 = int(w.cu_q[b]), int(w.cu_q[b + 1])
        if q1 > q0:
            unique_keys += int(w.q_pos[q0:q1].max()) + 1
    score_bytes = unique_keys * 256 + w.T * (32 * 128 * 2 + 32 * 4)
    topk_bytes = w.T * (w.topk * 4 + 4)                 # idx and cnt written
    staged_bytes = 4 * w.pairs                          # fp32 scores: written once, read back
    ln_bytes = (w.k_raw.shape[0] * 512 + 2 * 128 * 2) if w.k_raw is not None else 0
    return {"flops": 8192.0 * w.pairs, "score_bytes": score_bytes, "topk_bytes": topk_bytes,
            "call_bytes": score_bytes + topk_bytes, "staged_bytes": staged_bytes,
            "ln_bytes": ln_bytes, "unique_keys": unique_keys}


def tensor_bound(w: wl.Workload) -> bool:
    """Many queries per sequence share each key tile: the contraction dominates
    (8,192 flop per pair against 256 B per key, shared by the sequence's queries)."""
    return w.T > 4 * w.B


def _roof(bound, amount, ms, pk):
    if ms is None or ms <= 0:
        return None
    if bound == "tensor":
        ach = amount / (ms / 1e3) / 1e12
        return {"bound": "tensor", "achieved": ach, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": ach / pk["bf16_tflops"], "flops": amount, "ms": ms}
    ach = amount / (ms / 1e3) / 1e9
    return {"bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": ach / pk["hbm_gbs"], "bytes": amount, "ms": ms}


def rooflines(w: wl.Workload, kernels_ms: dict, fused_ms: float, pk: dict):
    """Per-kernel and whole-call rooflines of one idx_score_topk call."""
    alg = algorithmic(w)
    tb = tensor_bound(w)
    out = {}
    if "score" in kernels_ms:
        out["score"] = (_roof("tensor", alg["flops"], kernels_ms["score"], pk) if tb else
                        _roof("hbm", alg["score_bytes"], kernels_ms["score"], pk))
    if "topk" in kernels_ms:
        r = _roof("hbm", alg["topk_bytes"], kernels_ms["topk"], pk)
        if r is not None:
            # its read of the staged scores is overhead of the two-kernel design
            r["overhead_bytes"] = alg["staged_bytes"]
            r["overhead_gbs"] = alg["staged_bytes"] / (kernels_ms["topk"] / 1e3) / 1e9
        out["topk"] = r
    if "plan" in kernels_ms:
        out["plan"] = {"bound": "latency", "ms": kernels_ms["plan"]}
    call = (_roof("tensor", alg["flops"], fused_ms, pk) if tb else
            _roof("hbm", alg["call_bytes"], fused_ms, pk))
    return out, call


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

PHASES = ("plan", "score", "topk")   # kernels of one fused call, in launch order


class Bench:
    """Device state shared by the timed loops of one process."""

    def __init__(self, dev):
        import torch
        self.torch = torch
        self.dev = dev
        self.flush_w = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.int32, device=dev)
        self.flush_r = torch.ones(256 * 1024 * 1024 // 4, dtype=torch.int32, device=dev)
        self.stream = torch.cuda.current_stream()

    def flush_l2(self):
        self.flush_w.zero_()        # evicts everything the step could reuse
        self.flush_r.max()          # writes the flush's dirty lines back before the step

    def up(self, a, dt=None):
        x = self.torch.from_numpy(np.ascontiguousarray(a))
        return (x.view(dt) if dt is not None else x).to(self.dev)

    def event(self):
        return self.torch.cuda.Event(enable_timing=True)


class FusedCase:
    """One workload resident in HBM with its outputs and workspace."""

    def __init__(self, bn: Bench, w: wl.Workload):
        import torch
        from sparse_attention_key_gb300 import binding as B
        self.B, self.w, self.bn = B, w, bn
        self.q, self.wt, self.q_pos = bn.up(w.q, torch.int16), bn.up(w.w), bn.up(w.q_pos)
        self.cu_q, self.cu_k = bn.up(w.cu_q), bn.up(w.cu_k)
        self.chained_ln = w.k is None
        if self.chained_ln:
            self.k_raw = bn.up(w.k_raw, torch.int16)
            self.ln_w, self.ln_b = bn.up(w.ln_w, torch.int16), bn.up(w.ln_b, torch.int16)
            self.k = torch.empty_like(self.k_raw)
            B.key_layernorm(self.k_raw, self.ln_w, self.ln_b, w.eps, out=self.k)
        else:
            self.k = bn.up(w.k, torch.int16)
        T, K = w.T, w.topk
        self.idx = torch.empty((T, K), dtype=torch.int32, device=bn.dev)
        self.cnt = torch.empty((T,), dtype=torch.int32, device=bn.dev)
        self.ws = B.workspace(B.score_topk_workspace_size(w.B, T, w.max_len, K), bn.dev)

    def call(self):
        w = self.w
        self.B.score_topk(self.q, self.k, self.wt, self.q_pos, self.cu_q, self.cu_k, w.max_len,
                          w.topk, idx=self.idx, cnt=self.cnt, ws=self.ws)

    def ln(self):
        self.B.key_layernorm(self.k_raw, self.ln_w, self.ln_b, self.w.eps, out=self.k)

    def warm(self, n):
        for _ in range(max(n, 3)):
            self.call()
        self.bn.torch.cuda.synchronize()
        code, detail = self.B.get_status(self.ws)
        if code != 0:
            raise RuntimeError(f"device status {code} (detail {detail}) after warm-up")

    def time_calls(self, steps):
        """Per-step ms of the fused call, L2 flushed before each."""
        bn = self.bn
        st = [bn.event() for _ in range(steps)]
        en = [bn.event() for _ in range(steps)]
        for i in range(steps):
            bn.flush_l2()
            st[i].record(bn.stream)
            self.call()
            en[i].record(bn.stream)
        bn.torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in zip(st, en)]

    def time_kernels(self, steps):
        """Mean ms of each kernel of the fused call, from events the library
        records between its launches (idx_set_kernel_events)."""
        bn, B = self.bn, self.B
        n0 = B.kernel_launches()
        self.call()
        bn.torch.cuda.synchronize()
        per_call = B.kernel_launches() - n0
        rows = []
        for _ in range(steps):
            ev = [bn.event() for _ in range(per_call + 1)]
            for e in ev:                 # creates the CUDA events
                e.record(bn.stream)
            bn.flush_l2()
            ev[0].record(bn.stream)
            B.set_kernel_events(ev[1:])
            self.call()
            B.set_kernel_events([])
            rows.append(ev)
        bn.torch.cuda.synchronize()
        gaps = np.array([[ev[i].elapsed_time(ev[i + 1]) for i in range(per_call)] for ev in rows])
        mean = gaps.mean(axis=0)
        out = {"plan": float(mean[0]), "score": float(mean[1]), "topk": float(mean[2:].sum())}
        self.launch_ms = [float(x) for x in mean]   # every launch of the call, in order
        return out, int(per_call)

    def time_ln(self, steps):
        bn = self.bn
        ms = []
        for _ in range(steps):
            bn.flush_l2()
            a, e = bn.event(), bn.event()
            a.record(bn.stream)
            self.ln()
            e.record(bn.stream)
            ms.append((a, e))
        bn.torch.cuda.synchronize()
        return float(np.mean([a.elapsed_time(e) for a, e in ms]))


def workload_block(bn: Bench, w: wl.Workload, steps: int, warmup: int, pk: dict):
    """Fused-call time, per-kernel times and rooflines of one workload."""
    fc = FusedCase(bn, w)
    fc.warm(warmup)
    ms = fc.time_calls(steps)
    kern, per_call = fc.time_kernels(steps)
    fused_ms = float(np.mean(ms))
    per_kernel, call = rooflines(w, kern, fused_ms, pk)
    block = {"B": w.B, "T": w.T, "pairs": w.pairs, "max_len": w.max_len,
             "fused_ms": fused_ms, "fused_ms_median": float(np.median(ms)),
             "pairs_per_s": w.pairs / (fused_ms / 1e3), "kernels_per_call": per_call,
             "kernels_ms": kern, "launch_ms": fc.launch_ms, "kernel_rooflines": per_kernel,
             "call_roofline": call,
             "bound": "tensor" if tensor_bound(w) else "hbm", "steps": steps}
    if fc.chained_ln:
        ln_ms = fc.time_ln(steps)
        alg = algorithmic(w)
        block["key_layernorm"] = _roof("hbm", alg["ln_bytes"], ln_ms, pk)
    del fc
    bn.torch.cuda.empty_cache()
    return block


def run_ours(args, rank, world, local_rank):
    import torch
    from sparse_attention_key_gb300 import build as lib_build
    if rank == 0:
        lib_build.build()
    if world > 1:
        torch.distributed.barrier()
    from sparse_attention_key_gb300 import binding as B

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    bn = Bench(dev)
    w = wl.by_index(args.workload)
    T, K = w.T, w.topk
    fc = FusedCase(bn, w)
    fc.warm(args.warmup)

    cvd = [x for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x]
    clocks = ClockSampler(cvd[local_rank] if local_rank < len(cvd) else str(local_rank))
    clocks.start()
    time.sleep(0.3)

    # ---- timed region: K steps of the fused call
    starts = [bn.event() for _ in range(args.steps)]
    ends = [bn.event() for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    launches0 = B.kernel_launches()
    t_wall0 = time.time()
    for i in range(args.steps):
        bn.flush_l2()
        starts[i].record(bn.stream)
        fc.call()
        ends[i].record(bn.stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    launches = B.kernel_launches() - launches0
    if world > 1:
        torch.distributed.barrier()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = float(sum(step_ms))
    if args.fused_only:   # profiling runs: the timed fused steps only
        clocks.stop()
        if rank == 0:
            print(json.dumps({"mode": "fused-only", "workload": wl.NAMES[args.workload],
                              "steps": args.steps, "ms_per_step": total_ms / args.steps,
                              "value": w.pairs * args.steps / (total_ms / 1e3), "unit": UNIT}),
                  flush=True)
        return

    # ---- per-kernel durations inside the same fused call (events between its launches)
    kern, per_call = fc.time_kernels(args.steps)
    launch_ms = fc.launch_ms
    ln_ms = fc.time_ln(args.steps) if fc.chained_ln else None
    t_wall2 = time.time()
    clocks.stop()

    ref_idx, ref_cnt = fc.idx.cpu().numpy(), fc.cnt.cpu().numpy()   # the resident call's result

    # ---- end to end through the public API with host buffers
    # The batch is cut into up to E2E_CHUNKS groups of whole sequences
    # (contiguous, balanced by pairs). Each group's inputs are copied from
    # pinned host memory on a stream of their own (its keys LayerNormed there
    # as they land, when the workload chains the LayerNorm); the main stream
    # runs one fused call per group as soon as that group has landed, and a
    # copy stream reads each group's indices and counts back once its call is
    # done. So the copies of later groups overlap the calls of earlier ones.
    # Every byte and every kernel of the step stays inside the timed region.
    def pinned(a):
        return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    chained_ln = fc.chained_ln
    big = "k_raw" if chained_ln else "k"
    seq_pairs = np.array([int((w.q_pos[w.cu_q[b]:w.cu_q[b + 1]].astype(np.int64) + 1).sum())
                          for b in range(w.B)])
    cum = np.concatenate([[0], np.cumsum(seq_pairs)])
    n_groups = min(E2E_CHUNKS, w.B)
    cuts = [0] + [int(np.searchsorted(cum, cum[-1] * g / n_groups)) for g in range(1, n_groups)] + [w.B]
    cuts = sorted(set(min(max(c, 0), w.B) for c in cuts))
    groups = []
    for b0, b1 in zip(cuts[:-1], cuts[1:]):
        q0, q1 = int(w.cu_q[b0]), int(w.cu_q[b1])
        k0, k1 = int(w.cu_k[b0]), int(w.cu_k[b1])
        if q1 == q0:
            continue
        src = w.k_raw if chained_ln else w.k
        h = {"q": pinned(w.q[q0:q1].view(np.int16)), "w": pinned(w.w[q0:q1]),
             "q_pos": pinned(w.q_pos[q0:q1]),
             "cu_q": pinned((w.cu_q[b0:b1 + 1] - q0).astype(np.int32)),
             "cu_k": pinned((w.cu_k[b0:b1 + 1] - k0).astype(np.int32)),
             big: pinned(src[k0:k1].view(np.int16))}
        d = {n: torch.empty(t.shape, dtype=t.dtype, device=dev) for n, t in h.items()}
        kd = torch.empty_like(d[big]) if chained_ln else d[big]
        groups.append({"q0": q0, "q1": q1, "B": b1 - b0, "h": h, "d": d, "k": kd,
                       "max_len": int(w.max_len), "s": torch.cuda.Stream(device=dev),
                       "ready": torch.cuda.Event(), "done": torch.cuda.Event()})
    h_idx = torch.empty((T, K), dtype=torch.int32).pin_memory()
    h_cnt = torch.empty((T,), dtype=torch.int32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for g in groups for t in g["h"].values())
    d2h = h_idx.numel() * 4 + h_cnt.numel() * 4
    go = torch.cuda.Event()
    back = torch.cuda.Stream(device=dev)
    back_done = torch.cuda.Event()
    stream = bn.stream

    def e2e_step():
        go.record(stream)
        for g in groups:
            with torch.cuda.stream(g["s"]):
                g["s"].wait_event(go)
                for n, t in g["h"].items():
                    g["d"][n].copy_(t, non_blocking=True)
                if chained_ln:
                    B.key_layernorm(g["d"]["k_raw"], fc.ln_w, fc.ln_b, w.eps, out=g["k"])
                g["ready"].record(g["s"])
        for g in groups:
            stream.wait_event(g["ready"])
            q0, q1 = g["q0"], g["q1"]
            B.score_topk(g["d"]["q"], g["k"], g["d"]["w"], g["d"]["q_pos"], g["d"]["cu_q"],
                         g["d"]["cu_k"], g["max_len"], K, idx=fc.idx[q0:q1], cnt=fc.cnt[q0:q1],
                         ws=fc.ws)
            g["done"].record(stream)
            with torch.cuda.stream(back):
                back.wait_event(g["done"])
                h_idx[q0:q1].copy_(fc.idx[q0:q1], non_blocking=True)
                h_cnt[q0:q1].copy_(fc.cnt[q0:q1], non_blocking=True)
        back_done.record(back)
        stream.wait_event(back_done)

    fc.idx.fill_(-7)
    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e_start = [bn.event() for _ in range(args.steps)]
    e_end = [bn.event() for _ in range(args.steps)]
    for i in range(args.steps):
        bn.flush_l2()
        e_start[i].record(stream)
        e2e_step()
        e_end[i].record(stream)
    torch.cuda.synchronize()
    e2e_ms = float(sum(s.elapsed_time(e) for s, e in zip(e_start, e_end)))
    ok = np.array_equal(h_idx.numpy(), ref_idx) and np.array_equal(h_cnt.numpy(), ref_cnt)
    n_e2e_groups = len(groups)
    del fc, groups
    torch.cuda.empty_cache()

    # ---- the other full-size workloads, each with its own fused-call rooflines
    pk = peaks()
    by_workload = {}
    if args.by_workload and world == 1:
        for i in [x for x in (2, 3, 5, 6) if x != args.workload]:
            by_workload[wl.NAMES[i]] = workload_block(bn, wl.by_index(i), args.other_steps,
                                                      args.warmup, pk)

    total_ms, e2e_ms = max_over_ranks([total_ms, e2e_ms], world, dev)
    if rank != 0:
        return

    pairs = w.pairs
    value = whole_job_value(pairs, world, args.steps, total_ms)
    e2e_value = whole_job_value(pairs, world, args.steps, e2e_ms)
    fused_ms = total_ms / args.steps
    per_kernel, call_roof = rooflines(w, kern, fused_ms, pk)
    timed = {k_: v for k_, v in per_kernel.items() if v is not None and "frac" in v}
    dominant = max(timed, key=lambda k_: timed[k_]["ms"])
    roof = {k_: v for k_, v in timed[dominant].items() if k_ in ("bound", "achieved", "peak", "unit", "frac")}
    roof.update({"kernel": dominant, "ms": timed[dominant]["ms"],
                 "traffic": dram_traffic(args.workload, dominant),
                 "peak_source": pk["source"],
                 "units": ("8,192 flop per (query, causal key) pair" if roof["bound"] == "tensor"
                           else "bytes: 256 per (sequence, key) read + 8,320 per query (q, w)")})
    if ln_ms is not None:
        per_kernel["key_layernorm"] = _roof("hbm", algorithmic(w)["ln_bytes"], ln_ms, pk)

    ck = clocks.summary(t_wall0, t_wall2)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": fused_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": wl.NAMES[args.workload], "B": w.B, "T": T, "L": w.L,
                   "pairs_per_step": pairs, "topk": K, "max_len": w.max_len,
                   "step": "one idx_score_topk call (score + exact top-2048); the key "
                           "LayerNorm is timed on its own",
                   "l2": "flushed between steps: 256 MB written, then 256 MB read (cold, clean)",
                   "parallelism": f"replicas{world}" if world > 1 else "single"},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "matches_device_result": bool(ok),
                "copies": (f"pinned host buffers; {n_e2e_groups} groups of whole sequences, each copied "
                           "on its own stream while earlier groups compute (one fused call per group), "
                           "indices and counts read back per group on a copy stream")
                          + (", each LayerNormed as it lands" if chained_ln else "")},
        "gpu_launches": int(launches),
        "kernels_per_call": per_call,
        "kernels_ms": kern,
        "launch_ms": launch_ms,
        "kernels_source": "events recorded by the library between the kernels of the fused "
                          "call (idx_set_kernel_events), mean over the steps",
        "roofline": roof,
        "call_roofline": call_roof,
        "kernel_rooflines": per_kernel,
        "clocks": ck,
    }
    if by_workload:
        line["by_workload"] = by_workload
    if args.cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args)
    print(json.dumps(line), flush=True)


def run_ln_append(args):
    """Key-cache append with the LayerNorm fused in, on one GPU."""
    import torch
    from sparse_attention_key_gb300 import build as lib_build
    lib_build.build()
    from sparse_attention_key_gb300 import binding as B
    dev = torch.device("cuda", 0)
    n = args.ln_append
    rng = np.random.default_rng(2024)
    x = torch.from_numpy(wl.f32_to_bf16_bits(rng.standard_normal((n, 128), dtype=np.float32))
                         .view(np.int16)).to(dev)
    g = torch.from_numpy(wl.f32_to_bf16_bits((1 + 0.1 * rng.standard_normal(128)).astype(np.float32))
                         .view(np.int16)).to(dev)
    b = torch.from_numpy(wl.f32_to_bf16_bits((0.1 * rng.standard_normal(128)).astype(np.float32))
                         .view(np.int16)).to(dev)
    rows = 4 * n
    cache = torch.zeros((rows, 128), dtype=torch.int16, device=dev)
    slot = torch.from_numpy(rng.permutation(rows)[:n].astype(np.int64)).to(dev)
    staging = torch.empty_like(x)
    flush_w = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.int32, device=dev)
    flush_r = torch.ones(256 * 1024 * 1024 // 4, dtype=torch.int32, device=dev)

    def timed(fn):
        for _ in range(max(args.warmup, 3)):
            fn()
        torch.cuda.synchronize()
        ms = []
        for _ in range(args.steps):
            flush_w.zero_()
            flush_r.max()
            a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            e.record()
            torch.cuda.synchronize()
            ms.append(a.elapsed_time(e))
        return float(np.median(ms)) * 1e3

    fused_us = timed(lambda: B.key_layernorm_append(x, g, b, 1e-6, cache, slot))
    unfused_us = timed(lambda: cache.index_copy_(0, slot, B.key_layernorm(x, g, b, 1e-6, out=staging)))
    pk = peaks()
    alg = n * (256 + 256 + 8)
    ach = alg / (fused_us * 1e-6) / 1e9
    print(json.dumps({"mode": "ln-append", "rows": n, "cache_rows": rows, "steps": args.steps,
                      "us_per_call": fused_us, "unfused_us_per_call": unfused_us,
                      "roofline": {"bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"],
                                   "unit": "GB/s", "frac": ach / pk["hbm_gbs"],
                                   "bytes_per_call": alg},
                      "l2": "flushed between calls: 256 MB written, then 256 MB read"}), flush=True)


def run_project(args):
    """Indexer projections of T tokens (random weights), on one GPU."""
    import torch
    from sparse_attention_key_gb300 import build as lib_build
    lib_build.build()
    from sparse_attention_key_gb300 import binding as B
    dev = torch.device("cuda", 0)
    T, H, R = args.project, args.hidden, args.q_rank
    gen = torch.Generator(device="cpu").manual_seed(7)
    mk = lambda *shape, s=1.0: (torch.randn(*shape, generator=gen) * s).to(torch.bfloat16).to(dev)
    x, ql = mk(T, H), mk(T, R)
    wq, wk, ww = mk(4096, R, s=R ** -0.5), mk(128, H, s=H ** -0.5), mk(32, H, s=0.01)
    g, b = mk(128, s=0.1) + 1, mk(128, s=0.1)
    cache = torch.zeros((2 * T, 128), dtype=torch.bfloat16, device=dev)
    slot = torch.randperm(2 * T, generator=gen)[:T].to(dev)
    q = torch.empty((T, 32, 128), dtype=torch.bfloat16, device=dev)
    w = torch.empty((T, 32), dtype=torch.float32, device=dev)
    ws = B.workspace(B.indexer_project_workspace_size(T), dev)
    flush_w = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.int32, device=dev)
    flush_r = torch.ones(256 * 1024 * 1024 // 4, dtype=torch.int32, device=dev)
    call = lambda: B.indexer_project(x, ql, wq, wk, ww, g, b, 1e-6, cache, slot, q=q, w=w, ws=ws)
    for _ in range(max(args.warmup, 3)):
        call()
    torch.cuda.synchronize()
    ms = []
    for _ in range(args.steps):
        flush_w.zero_()
        flush_r.max()
        a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        call()
        e.record()
        torch.cuda.synchronize()
        ms.append(a.elapsed_time(e))
    us = float(np.median(ms)) * 1e3
    # each launch of one call, from events the library records between them
    n0 = B.kernel_launches()
    call()
    torch.cuda.synchronize()
    per_call = B.kernel_launches() - n0
    rows = []
    for _ in range(args.steps):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(per_call + 1)]
        for e in ev:
            e.record()
        flush_w.zero_()
        flush_r.max()
        ev[0].record()
        B.set_kernel_events(ev[1:])
        call()
        B.set_kernel_events([])
        rows.append(ev)
    torch.cuda.synchronize()
    launch_us = [float(x) * 1e3 for x in np.mean([[ev[i].elapsed_time(ev[i + 1]) for i in range(per_call)]
                                                 for ev in rows], axis=0)]
    flops = 2.0 * T * (4096 * R + 128 * H + 32 * H)
    weight_bytes = 2.0 * (4096 * R + 128 * H + 32 * H)
    io_bytes = 2.0 * T * (H + R + 4096 + 128 * 2) + 4.0 * T * 32
    pk = peaks()
    tflops = flops / (us * 1e-6) / 1e12
    gbs = (weight_bytes + io_bytes) / (us * 1e-6) / 1e9
    bound = "tensor" if flops / (weight_bytes + io_bytes) > pk["bf16_tflops"] * 1e3 / pk["hbm_gbs"] else "hbm"
    roof = ({"bound": "tensor", "achieved": tflops, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
             "frac": tflops / pk["bf16_tflops"]} if bound == "tensor" else
            {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": gbs / pk["hbm_gbs"]})
    print(json.dumps({"mode": "project", "T": T, "hidden": H, "q_rank": R, "steps": args.steps,
                      "us_per_call": us, "launch_us": launch_us, "tflops": tflops,
                      "bytes_per_call": weight_bytes + io_bytes,
                      "roofline": roof, "gemm": "library tcgen05 GEMM (bf16 in, fp32 accumulate)",
                      "l2": "flushed between calls: 256 MB written, then 256 MB read"}), flush=True)


def _mla_lengths(name: str):
    if name == "decode_batch":
        return [8192, 12288, 16384, 24576, 32768, 40960, 49152, 65536]
    if name == "long_decode":
        w = wl.by_index(5)
        return list(np.diff(w.cu_k).astype(np.int64))
    raise ValueError(f"unknown --mla workload {name}")


def run_mla(args):
    """Sparse MLA attention over 2048 selected positions per query (one GPU):
    96 heads, 576-wide bf16 cache rows; synthetic seeded inputs made on the device."""
    import torch
    from sparse_attention_key_gb300 import build as lib_build
    lib_build.build()
    from sparse_attention_key_gb300 import binding as B
    dev = torch.device("cuda", 0)
    lens = _mla_lengths(args.mla)
    H, K = 96, 2048
    T, L = len(lens), int(sum(lens))
    gen = torch.Generator(device=dev).manual_seed(17)
    if args.fp8:   # E4M3 codes spread like workloads.fp8_codes, fp32 row scales 2^U(-3,0)
        cache = torch.empty((L, 576), dtype=torch.uint8, device=dev)
        for r0 in range(0, L, 1 << 18):
            r1 = min(L, r0 + (1 << 18))
            shape = (r1 - r0, 576)
            sign = torch.randint(0, 2, shape, generator=gen, device=dev, dtype=torch.int32)
            expo = (7 + 1.5 * torch.randn(shape, generator=gen, device=dev)).round().clamp(0, 15).int()
            mant = torch.randint(0, 8, shape, generator=gen, device=dev, dtype=torch.int32)
            mant = torch.where((expo == 15) & (mant == 7), torch.full_like(mant, 6), mant)
            cache[r0:r1] = ((sign << 7) | (expo << 3) | mant).to(torch.uint8)
        row_scale = torch.exp2(torch.rand((L,), generator=gen, device=dev) * -3.0).float()
    else:
        cache = torch.empty((L, 576), dtype=torch.bfloat16, device=dev)
        for r0 in range(0, L, 1 << 20):   # N(0,1) rows, in chunks
            r1 = min(L, r0 + (1 << 20))
            cache[r0:r1] = torch.randn((r1 - r0, 576), generator=gen, device=dev).to(torch.bfloat16)
    q = torch.randn((T, H, 576), generator=gen, device=dev).to(torch.bfloat16)
    idx = torch.full((T, K), -1, dtype=torch.int32, device=dev)
    for t, n in enumerate(lens):   # distinct positions, ascending, as the indexer emits them
        idx[t] = torch.randperm(int(n), generator=gen, device=dev)[:K].sort().values.to(torch.int32)
    cnt = torch.full((T,), K, dtype=torch.int32, device=dev)
    cu_k = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=dev)
    cu_q = torch.arange(T + 1, dtype=torch.int32, device=dev)
    scale = 1.0 / np.sqrt(192.0)
    out = torch.empty((T, H, 512), dtype=torch.float32, device=dev)
    lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    ws = B.workspace(B.sparse_mla_workspace_size(T, H, K), dev)
    flush_w = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.int32, device=dev)
    flush_r = torch.ones(256 * 1024 * 1024 // 4, dtype=torch.int32, device=dev)
    if args.fp8:
        call = lambda: B.sparse_mla_fp8(q, cache, row_scale, idx, cnt, cu_q, cu_k, scale, out=out, lse=lse,
                                        ws=ws)
    else:
        call = lambda: B.sparse_mla(q, cache, idx, cnt, cu_q, cu_k, scale, out=out, lse=lse, ws=ws)
    for _ in range(max(args.warmup, 3)):
        call()
    torch.cuda.synchronize()
    assert B.get_status(ws)[0] == 0
    n0 = B.kernel_launches()
    ms = []
    for _ in range(args.steps):
        flush_w.zero_()
        flush_r.max()
        a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        call()
        e.record()
        torch.cuda.synchronize()
        ms.append(a.elapsed_time(e))
    launches = (B.kernel_launches() - n0) // max(args.steps, 1)
    us = float(np.median(ms)) * 1e3
    pairs = T * K
    row_bytes = 576 + 4 if args.fp8 else 576 * 2   # a selected row (FP8: codes + its scale)
    bytes_alg = pairs * row_bytes + T * H * 576 * 2 + T * H * 512 * 4 + T * H * 4 + T * K * 4
    flops = 2.0 * pairs * H * (576 + 512)
    pk = peaks()
    gbs = bytes_alg / (us * 1e-6) / 1e9
    tflops = flops / (us * 1e-6) / 1e12
    print(json.dumps({
        "mode": "sparse_mla", "metric": "sparse MLA (query, selected position) pairs/s",
        "value": pairs / (us * 1e-6), "unit": "pairs/s", "higher_is_better": True,
        "config": {"workload": args.mla, "queries": T, "heads": H, "topk": K, "cache_rows": L,
                   "row": ("576 E4M3 codes + an fp32 scale" if args.fp8 else "576 bf16")
                   + " (512 latent + 64 key dims)", "scale": "1/sqrt(192)"},
        "steps": args.steps, "us_per_call": us, "gpu_launches_per_call": launches,
        "dtype": ("e4m3 cache, bf16 q and MMA operands" if args.fp8 else "bf16 in")
        + ", fp32 accumulate and out",
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / pk["hbm_gbs"], "bytes_per_call": bytes_alg},
        "tensor": {"achieved": tflops, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                   "frac": tflops / pk["bf16_tflops"], "flops_per_call": flops},
        "data": "synthetic, seeded on the device",
        "l2": "flushed between calls: 256 MB written, then 256 MB read"}), flush=True)


# ---------------------------------------------------------------------------
# CPU oracle (baseline / reference arm)
# ---------------------------------------------------------------------------

def _oracle_sample(w: wl.Workload, budget_pairs: int):
    """Rows of the workload, spread over its queries, totalling about budget_pairs."""
    n = w.q_pos.astype(np.int64) + 1
    order = np.argsort(np.random.default_rng(0).random(w.T))
    rows, tot = [], 0
    for t in order:
        if tot >= budget_pairs and rows:
            break
        rows.append(int(t))
        tot += int(n[t])
    return sorted(rows), tot


def _oracle_inputs(w: wl.Workload):
    import oracle
    if w.k is None:  # the chained LayerNorm, computed by the oracle itself
        k, _ = oracle.key_layernorm(w.k_raw, oracle.bf16_bits_to_f64(w.ln_w),
                                    oracle.bf16_bits_to_f64(w.ln_b), float(np.float32(w.eps)))
        return k
    return w.k


def _oracle_rate(w, k, rows, threads):
    import oracle
    t0 = time.time()
    oracle.score_topk(w.q, k, w.w, w.q_pos, w.cu_q, w.cu_k, K=w.topk, rows=rows, threads=threads)
    return time.time() - t0


def cpu_baseline(w: wl.Workload, args):
    """The fp64 oracle, as it stands, on the host: single-threaded and on all
    cores (one thread per query row), each on a bounded row sample."""
    cores = os.cpu_count() or 1
    k = _oracle_inputs(w)
    rows, tot = _oracle_sample(w, 20_000)          # calibration: a few ms of work
    rate1 = tot / max(_oracle_rate(w, k, rows, 1), 1e-6)
    # single thread: about a third of the budget
    rows1, tot1 = _oracle_sample(w, int(rate1 * args.cpu_seconds / 3))
    dt1 = _oracle_rate(w, k, rows1, 1)
    # all cores: the rest, on enough rows to keep every core busy
    rows_n, tot_n = _oracle_sample(w, max(int(rate1 * cores * args.cpu_seconds * 2 / 3), 1))
    dt_n = _oracle_rate(w, k, rows_n, cores)
    used = min(cores, len(rows_n))
    return {"value": tot_n / dt_n, "unit": UNIT, "cores": used, "kind": "oracle",
            "sample": f"{len(rows_n)} of {w.T} query rows ({tot_n} pairs) of {wl.NAMES[args.workload]}, "
                      f"fp64 C oracle, one thread per row on {used} of {cores} host cores, {dt_n:.1f} s",
            "single_thread": {"value": tot1 / dt1, "unit": UNIT, "cores": 1,
                              "sample": f"{len(rows1)} query rows ({tot1} pairs), {dt1:.1f} s"},
            "host_cores": cores}


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    w = wl.by_index(args.workload)
    k = _oracle_inputs(w)
    cores = os.cpu_count() or 1
    rows, tot = _oracle_sample(w, 20_000)
    t0 = time.time()
    oracle.score_topk(w.q, k, w.w, w.q_pos, w.cu_q, w.cu_k, K=w.topk, rows=rows, threads=cores)
    rate = tot / max(time.time() - t0, 1e-6)
    per_step = max(1.0, min(10.0, 120.0 / max(args.steps + args.warmup, 1)))
    rows, tot = _oracle_sample(w, int(rate * per_step))
    for _ in range(args.warmup):
        oracle.score_topk(w.q, k, w.w, w.q_pos, w.cu_q, w.cu_k, K=w.topk, rows=rows[:1], threads=1)
    t0 = time.time()
    for _ in range(args.steps):
        oracle.score_topk(w.q, k, w.w, w.q_pos, w.cu_q, w.cu_k, K=w.topk, rows=rows, threads=cores)
    dt = time.time() - t0
    value = tot * args.steps / dt
    used = min(cores, len(rows))
    sample = (f"{len(rows)} of {w.T} query rows ({tot} pairs) per step of "
              f"{wl.NAMES[args.workload]}; fp64 C oracle, one thread per row")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": wl.NAMES[args.workload], "B": w.B, "T": w.T, "L": w.L,
                       "pairs_per_step": w.pairs, "topk": w.topk},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": used, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", type=int, default=DEFAULT_WORKLOAD, choices=[1, 2, 3, 4, 5, 6])
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="CPU work for the cpu_baseline sample")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--no-by-workload", dest="by_workload", action="store_false",
                    help="skip timing the other full-size workloads (by_workload block)")
    ap.add_argument("--other-steps", type=int, default=20,
                    help="timed fused calls per workload in the by_workload block")
    ap.add_argument("--ln-append", type=int, metavar="ROWS", default=0,
                    help="time the key LayerNorm fused into the key-cache append of ROWS new keys "
                         "(random distinct slots of a 4*ROWS-row cache) against LayerNorm into a "
                         "staging buffer plus a scatter copy; prints its own JSON line")
    ap.add_argument("--project", type=int, metavar="T", default=0,
                    help="time the indexer projections (q, key LayerNorm into the cache, w) of T "
                         "tokens; prints its own JSON line")
    ap.add_argument("--hidden", type=int, default=7168, help="--project: attention input width")
    ap.add_argument("--q-rank", type=int, default=1536,
                    help="--project: q-LoRA rank (not given by the pages; a stand-in)")
    ap.add_argument("--mla", choices=["decode_batch", "long_decode"], default=None,
                    help="time the sparse MLA attention over 2048 selected positions per query "
                         "(96 heads) on that workload's shapes; prints its own JSON line")
    ap.add_argument("--fp8", action="store_true",
                    help="--mla: FP8 (E4M3) cache rows with an fp32 scale each")
    ap.add_argument("--fused-only", action="store_true",
                    help="time only the fused steps (for profiler captures); prints a short line")
    ap.add_argument("--record-traffic", metavar="CSV",
                    help="record per-launch DRAM bytes of --workload's kernels from an ncu CSV "
                         "(gpu__time_duration.sum, dram__bytes_read.sum, dram__bytes_write.sum of "
                         "a --fused-only run) into profiles/dram_traffic.json, then exit")
    args = ap.parse_args()
    if args.record_traffic:
        record_traffic(args.workload, args.record_traffic)
        return
    if args.ln_append:
        run_ln_append(args)
        return
    if args.project:
        run_project(args)
        return
    if args.mla:
        run_mla(args)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
