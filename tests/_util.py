"""Shared helpers of the test suite (device upload, comparisons, property checks)."""
from __future__ import annotations

import numpy as np

HEADS, DIM = 32, 128


def to_device(wl, device="cuda"):
    """Upload a workloads.Workload's arrays as torch tensors (bf16 kept as int16 bits)."""
    import torch

    def t(a, dt=None):
        x = torch.from_numpy(np.ascontiguousarray(a))
        if dt is not None:
            x = x.view(dt)
        return x.to(device)

    d = {
        "q": t(wl.q, torch.int16),
        "w": t(wl.w),
        "q_pos": t(wl.q_pos),
        "cu_q": t(wl.cu_q),
        "cu_k": t(wl.cu_k),
    }
    if wl.k is not None:
        d["k"] = t(wl.k, torch.int16)
    if wl.k_raw is not None:
        d["k_raw"] = t(wl.k_raw, torch.int16)
    if wl.ln_w is not None:
        d["ln_w"] = t(wl.ln_w, torch.int16)
        d["ln_b"] = t(wl.ln_b, torch.int16)
    return d


def bits_of(t) -> np.ndarray:
    """Device int16/bf16 tensor -> numpy uint16 bit patterns."""
    import torch
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in bf16 ulps between two arrays of bf16 bit patterns."""
    def ordered(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, 0x8000 - (x & 0x7FFF), 0x8000 + x)
    return np.abs(ordered(a) - ordered(b))


def rule_order_ok(S: np.ndarray, idx_row: np.ndarray, K: int) -> str | None:
    """Check one output row against the selection rule on the given scores.

    S: the row's n scores (any float dtype); idx_row: [K] output. Returns None if
    the row is the exact top-K of S under (score desc, position asc) emitted in
    the rule's order, else a description of the first violation.
    """
    n = S.size
    idx_row = np.asarray(idx_row)
    if n <= K:
        exp = np.concatenate([np.arange(n), -np.ones(K - n, dtype=np.int64)])
        return None if np.array_equal(idx_row, exp) else "keep-all row differs"
    sel = idx_row
    if (sel < 0).any() or (sel >= n).any():
        return "index out of range"
    if np.unique(sel).size != K:
        return "duplicate index"
    Sz = S.astype(np.float64) + 0.0          # fold -0 onto +0
    order = np.lexsort((np.arange(n), -Sz))[:K]
    if set(order.tolist()) != set(sel.tolist()):
        return "selected set is not the top-K"
    tau = Sz[order[-1]]
    above = np.sort(order[Sz[order] > tau])
    ties = np.sort(order[Sz[order] == tau])
    exp = np.concatenate([above, ties])
    return None if np.array_equal(sel, exp) else "order rule violated"


def tolerance_set_check(S_ref: np.ndarray, idx_gpu: np.ndarray, idx_ref: np.ndarray, K: int,
                        rel: float = 1e-3) -> str | None:
    """Real-valued rule: GPU and oracle index sets may differ only at positions
    whose oracle score lies within `rel` (relative) of the oracle threshold."""
    n = S_ref.size
    if n <= K:
        return None if np.array_equal(idx_gpu, idx_ref) else "keep-all row differs"
    a, b = set(idx_gpu.tolist()), set(idx_ref.tolist())
    diff = a ^ b
    if not diff:
        return None
    tau = float(np.min(S_ref[idx_ref]))
    floor = 1e-6 * float(np.max(np.abs(S_ref)))
    for p in diff:
        if p < 0 or p >= n:
            return f"position {p} out of range"
        if abs(S_ref[p] - tau) > rel * abs(tau) + floor:
            return f"position {p} (score {S_ref[p]!r}) is not near the threshold {tau!r}"
    return None


def scores_close(S_gpu: np.ndarray, S_ref: np.ndarray, rel: float = 1e-3) -> str | None:
    """Per score: |S_gpu - S_ref| <= rel*|S_ref| + 1e-6*max|S_ref|."""
    floor = 1e-6 * float(np.max(np.abs(S_ref))) if S_ref.size else 0.0
    err = np.abs(S_gpu.astype(np.float64) - S_ref)
    bad = err > rel * np.abs(S_ref) + floor
    if bad.any():
        i = int(np.flatnonzero(bad)[0])
        return f"score {i}: gpu {S_gpu[i]!r} vs oracle {S_ref[i]!r}"
    return None
