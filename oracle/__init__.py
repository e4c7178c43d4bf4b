"""CPU oracle for the Lightning Indexer — TEST INFRASTRUCTURE ONLY.

The arithmetic lives in ``indexer_oracle.c`` (plain C11, fp64); this module
only compiles it with gcc and marshals numpy arrays through ctypes. Only the
tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import it. The CUDA library never imports it, and it imports nothing from the
CUDA library.

Method source: Hugging Face discussion "Notes from an NVFP4 port of Kimi K3.1
Pro" — the indexer paragraph and item (4) of "Details that silently change the
answer". All functions here are pinned by ``tests/test_oracle.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "indexer_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

HEADS = 32
DIM = 128
MLA_DIM = 576    # MLA cache row: 512-wide latent + 64 key dims
MLA_VDIM = 512

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (gcc, no GPU)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"],
                       check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i64, i32 = ctypes.c_int64, ctypes.c_int32
            lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_double.restype = ctypes.c_double
            lib.oracle_double_to_bf16.argtypes = [ctypes.c_double]
            lib.oracle_double_to_bf16.restype = ctypes.c_uint16
            lib.oracle_key_layernorm.argtypes = [P, P, P, ctypes.c_double, i64, P, P]
            lib.oracle_key_layernorm.restype = None
            lib.oracle_scores.argtypes = [P, P, P, i64, P]
            lib.oracle_scores.restype = None
            lib.oracle_select.argtypes = [P, i64, i32, P]
            lib.oracle_select.restype = i64
            lib.oracle_score_topk.argtypes = [P, P, P, P, P, P, i32, i32, P, P, P, i64, i64, i64]
            lib.oracle_score_topk.restype = ctypes.c_int
            lib.oracle_sparse_mla.argtypes = [P, P, P, i64, i32, ctypes.c_double, P, P]
            lib.oracle_sparse_mla.restype = None
            lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_to_double.restype = ctypes.c_double
            lib.oracle_sparse_mla_fp8.argtypes = [P, P, P, P, i64, i32, ctypes.c_double, P, P]
            lib.oracle_sparse_mla_fp8.restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------

def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns, as float64 (bf16 = top half of fp32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x) -> np.ndarray:
    """Round float64 values to bf16 (nearest, ties to even), one rounding step."""
    lib = _load()
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    flat_in, flat_out = x.reshape(-1), out.reshape(-1)
    for i in range(flat_in.size):
        flat_out[i] = lib.oracle_double_to_bf16(float(flat_in[i]))
    return out


# ---------------------------------------------------------------------------
# the indexer
# ---------------------------------------------------------------------------

def key_layernorm(k_raw_bits, gamma, beta, eps: float):
    """LayerNorm of each 128-wide key row -> (bf16 bits [n,128], fp64 [n,128]).

    ``gamma``/``beta`` are given as exact float64 values of the parameters.
    """
    lib = _load()
    k_raw = _c(k_raw_bits, np.uint16).reshape(-1, DIM)
    g = _c(gamma, np.float64).reshape(DIM)
    b = _c(beta, np.float64).reshape(DIM)
    n = k_raw.shape[0]
    out = np.empty((n, DIM), dtype=np.uint16)
    y = np.empty((n, DIM), dtype=np.float64)
    lib.oracle_key_layernorm(_ptr(k_raw), _ptr(g), _ptr(b), float(eps), n, _ptr(out), _ptr(y))
    return out, y


def indexer_project(x_bits, qlora_bits, wq_bits, wk_bits, ww_bits, gamma, beta, eps: float):
    """The indexer's projections from a layer's activations, in fp64.

    Port notes, indexer paragraph: the query comes off the normalised q-LoRA
    projection, the key from the attention input through the key LayerNorm,
    and a per-head weight vector sums the heads. Per token (weights in the
    [out, in] layout of a linear layer): q = W_q qlora and k_pre = W_k x, each
    rounded once to bf16 (the 16-bit activations of the model); k = the key
    LayerNorm of k_pre; w = W_w x, kept in fp64. The products are float64
    matrix products of the exact bf16 values (a library matmul as one step).
    Returns (q bits [T,32,128], k bits [T,128], w fp64 [T,32], k_pre bits [T,128]).
    """
    x = bf16_bits_to_f64(x_bits)
    ql = bf16_bits_to_f64(qlora_bits)
    q = f64_to_bf16_bits(ql @ bf16_bits_to_f64(wq_bits).T).reshape(-1, HEADS, DIM)
    k_pre = f64_to_bf16_bits(x @ bf16_bits_to_f64(wk_bits).T)
    w = x @ bf16_bits_to_f64(ww_bits).T
    k, _ = key_layernorm(k_pre, gamma, beta, eps)
    return q, k, w, k_pre


def scores(q_t_bits, k_seq_bits, w_t, n: int) -> np.ndarray:
    """S[s] = sum_h w[h] relu(q_h . k_s) for s < n, in fp64 (one query)."""
    lib = _load()
    q = _c(q_t_bits, np.uint16).reshape(HEADS * DIM)
    k = _c(k_seq_bits, np.uint16).reshape(-1, DIM)
    w = _c(w_t, np.float32).reshape(HEADS)
    assert k.shape[0] >= n
    S = np.empty(max(n, 1), dtype=np.float64)
    lib.oracle_scores(_ptr(q), _ptr(k), _ptr(w), n, _ptr(S))
    return S[:n]


def select(S, K: int) -> np.ndarray:
    """Exact top-K of one score row under the tie/order rule -> int32 [K] (-1 padded)."""
    lib = _load()
    s = _c(S, np.float64).reshape(-1)
    out = np.empty(K, dtype=np.int32)
    r = lib.oracle_select(_ptr(s), s.size, int(K), _ptr(out))
    if r < 0:
        raise MemoryError("oracle_select")
    return out


def score_topk(q_bits, k_bits, w, q_pos, cu_q, cu_k, K: int = 2048, rows=None,
               want_scores: bool = False, threads: int = 1):
    """Indexer over a packed ragged batch.

    Returns (idx [T,K] int32, cnt [T] int32, scores [T,ld] float64 or None).
    ``rows`` restricts the work to an iterable of query rows (other rows of idx
    stay -1 and cnt 0). ``threads`` > 1 runs disjoint row subsets in parallel
    threads (each a separate call of the same C function).
    """
    lib = _load()
    q = _c(q_bits, np.uint16).reshape(-1, HEADS, DIM)
    k = _c(k_bits, np.uint16).reshape(-1, DIM)
    w_ = _c(w, np.float32).reshape(-1, HEADS)
    qp = _c(q_pos, np.int32).reshape(-1)
    cq = _c(cu_q, np.int32).reshape(-1)
    ck = _c(cu_k, np.int32).reshape(-1)
    T, B = q.shape[0], cq.size - 1
    idx = np.full((T, K), -1, dtype=np.int32)
    cnt = np.zeros(T, dtype=np.int32)
    ld = int(qp.max()) + 1 if (want_scores and T) else 0
    sc = np.full((T, ld), np.nan, dtype=np.float64) if want_scores else None
    row_list = list(range(T)) if rows is None else sorted(set(int(r) for r in rows))

    def run(r0, r1):
        rc = lib.oracle_score_topk(_ptr(q), _ptr(k), _ptr(w_), _ptr(qp), _ptr(cq), _ptr(ck),
                                   B, int(K), _ptr(idx), _ptr(cnt), _ptr(sc), ld, r0, r1)
        if rc != 0:
            raise ValueError("oracle_score_topk: query position outside its sequence")

    # contiguous runs of requested rows
    runs = []
    for r in row_list:
        if runs and runs[-1][1] == r:
            runs[-1][1] = r + 1
        else:
            runs.append([r, r + 1])
    if threads <= 1 or len(row_list) <= 1:
        for r0, r1 in runs:
            run(r0, r1)
    else:
        # split into single rows, handed to a thread pool (ctypes drops the GIL)
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(lambda r: run(r, r + 1), row_list))
    return idx, cnt, sc


# ---------------------------------------------------------------------------
# sparse MLA attention over the selected positions (the indexer's consumer)
# ---------------------------------------------------------------------------

def sparse_mla(q_t_bits, cache_bits, rows, scale: float):
    """Attention of one query token over the selected cache rows, in fp64.

    Port notes (opening paragraph, item (5)) and the TokenSpeed K3 post
    (section 2, MLA): NoPE latent attention, a 512-wide latent plus 64 key dims
    per cached token. Per head h: l_j = scale * (q_h . c_j) over the selected
    rows c_j (576 wide), p = softmax(l), o_h = sum_j p_j c_j[:512],
    lse_h = log sum_j exp(l_j). ``rows`` are absolute row numbers of
    ``cache_bits`` [L, 576]; q is [H, 576]. Returns (o [H, 512], lse [H]).
    """
    lib = _load()
    q = _c(q_t_bits, np.uint16).reshape(-1, MLA_DIM)
    c = _c(cache_bits, np.uint16).reshape(-1, MLA_DIM)
    r = _c(rows, np.int64).reshape(-1)
    assert r.size == 0 or (r.min() >= 0 and r.max() < c.shape[0])
    H = q.shape[0]
    o = np.empty((H, MLA_VDIM), dtype=np.float64)
    lse = np.empty(H, dtype=np.float64)
    lib.oracle_sparse_mla(_ptr(q), _ptr(c), _ptr(r), r.size, H, float(scale), _ptr(o), _ptr(lse))
    return o, lse


def sparse_mla_batch(q_bits, cache_bits, idx, cnt, cu_q, cu_k, scale: float, rows=None):
    """sparse_mla for each query row t of a packed ragged batch.

    The selected positions of row t are idx[t, :cnt[t]], positions inside the
    row's sequence (cache rows cu_k[b] .. cu_k[b+1]). Returns (o [T, H, 512],
    lse [T, H]); rows outside ``rows`` (when given) are left NaN.
    """
    q = _c(q_bits, np.uint16)
    T, H = q.shape[0], q.shape[1]
    cq = np.asarray(cu_q).reshape(-1)
    ck = np.asarray(cu_k).reshape(-1)
    o = np.full((T, H, MLA_VDIM), np.nan)
    lse = np.full((T, H), np.nan)
    for t in (range(T) if rows is None else rows):
        b = int(np.searchsorted(cq, t, side="right")) - 1
        pos = np.asarray(idx[t][:int(cnt[t])], dtype=np.int64)
        o[t], lse[t] = sparse_mla(q[t], cache_bits, ck[b] + pos, scale)
    return o, lse


# ---------------------------------------------------------------------------
# FP8 (E4M3) MLA cache rows
# ---------------------------------------------------------------------------

def e4m3_to_f64(codes) -> np.ndarray:
    """Exact values of E4M3 codes (uint8), as float64 (NaN for the NaN codes)."""
    lib = _load()
    table = np.array([lib.oracle_e4m3_to_double(b) for b in range(256)], dtype=np.float64)
    return table[np.asarray(codes, dtype=np.uint8)]


def sparse_mla_fp8(q_t_bits, cache8, row_scale, rows, scale: float):
    """sparse_mla over FP8 rows: row r's value is row_scale[r] x e4m3(cache8[r]).

    TokenSpeed's K3 post (section 2, MLA) stores the MLA cache in FP8; a row
    holds 576 E4M3 codes and one scale. ``cache8`` uint8 [L, 576], ``row_scale``
    [L] (any float dtype, used exactly), ``rows`` absolute row numbers, q [H, 576]
    bf16 bits. Returns (o [H, 512], lse [H]) in fp64.
    """
    lib = _load()
    q = _c(q_t_bits, np.uint16).reshape(-1, MLA_DIM)
    c = _c(cache8, np.uint8).reshape(-1, MLA_DIM)
    sc = _c(row_scale, np.float64).reshape(-1)
    r = _c(rows, np.int64).reshape(-1)
    assert r.size == 0 or (r.min() >= 0 and r.max() < c.shape[0])
    H = q.shape[0]
    o = np.empty((H, MLA_VDIM), dtype=np.float64)
    lse = np.empty(H, dtype=np.float64)
    lib.oracle_sparse_mla_fp8(_ptr(q), _ptr(c), _ptr(sc), _ptr(r), r.size, H, float(scale), _ptr(o),
                              _ptr(lse))
    return o, lse


def sparse_mla_fp8_batch(q_bits, cache8, row_scale, idx, cnt, cu_q, cu_k, scale: float, rows=None):
    """sparse_mla_fp8 for each query row t of a packed ragged batch (see
    sparse_mla_batch). Returns (o [T, H, 512], lse [T, H]); rows outside
    ``rows`` (when given) are left NaN."""
    q = _c(q_bits, np.uint16)
    T, H = q.shape[0], q.shape[1]
    cq = np.asarray(cu_q).reshape(-1)
    ck = np.asarray(cu_k).reshape(-1)
    o = np.full((T, H, MLA_VDIM), np.nan)
    lse = np.full((T, H), np.nan)
    for t in (range(T) if rows is None else rows):
        b = int(np.searchsorted(cq, t, side="right")) - 1
        pos = np.asarray(idx[t][:int(cnt[t])], dtype=np.int64)
        o[t], lse[t] = sparse_mla_fp8(q[t], cache8, row_scale, ck[b] + pos, scale)
    return o, lse
