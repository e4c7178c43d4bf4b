"""Python binding of the Lightning Indexer C ABI (``include/lightning_indexer.h``).

Argument marshalling only: every step of the indexer runs in the CUDA library
``_lib/liblightning_indexer.so``. Tensors must live on the current CUDA device,
be contiguous and have the documented dtypes; bf16 tensors may be
``torch.bfloat16`` or ``torch.uint16``/``torch.int16`` bit patterns. Work is
enqueued on the current torch stream. If the library has not been built the
first call raises ``RuntimeError`` — there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

HEADS = 32
DIM = 128
TOPK_MAX = 2048

IDX_OK = 0
STATUS_NAMES = {0: "IDX_OK", 1: "IDX_ERR_INVALID_ARG", 2: "IDX_ERR_UNSUPPORTED",
                3: "IDX_ERR_WORKSPACE", 4: "IDX_ERR_CUDA", 5: "IDX_ERR_TIMEOUT",
                6: "IDX_ERR_DEVICE_ARG"}
PARAM_BF16, PARAM_F32 = 0, 1

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib",
                         "liblightning_indexer.so")
_lib = None
_lock = threading.Lock()

EXPORTS = ("idx_key_layernorm", "idx_score", "idx_score_workspace_size", "idx_topk",
           "idx_topk_workspace_size", "idx_score_topk", "idx_score_topk_workspace_size",
           "idx_get_status", "idx_last_error", "idx_version", "idx_kernel_launches",
           "idx_score_topk_noalloc", "idx_set_wait_limit_ns", "idx_key_layernorm_append",
           "idx_indexer_project", "idx_indexer_project_workspace_size", "idx_sparse_mla",
           "idx_sparse_mla_workspace_size", "idx_sparse_mla_fp8", "idx_set_kernel_events")


class IndexerError(RuntimeError):
    def __init__(self, code: int, where: str, message: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)}: {message}")
        self.code = code


def library_path() -> str:
    return _LIB_PATH


def lib():
    """Load the CUDA library (raises RuntimeError if it is missing)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    f"Lightning Indexer CUDA library not built ({_LIB_PATH} missing); run "
                    "`python -m sparse_attention_key_gb300.build`")
            L = ctypes.CDLL(_LIB_PATH)
            P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
            L.idx_key_layernorm.argtypes = [P, P, P, ctypes.c_int, ctypes.c_float, P, i64, P]
            L.idx_score.argtypes = [P, P, P, P, P, P, i32, i32, i64, i64, P, i64, P, sz, P]
            L.idx_score_workspace_size.argtypes = [i32, i32, i64]
            L.idx_score_workspace_size.restype = sz
            L.idx_topk.argtypes = [P, i64, P, i32, i64, i32, P, P, P, sz, P]
            L.idx_topk_workspace_size.argtypes = [i32, i64, i32]
            L.idx_topk_workspace_size.restype = sz
            L.idx_score_topk.argtypes = [P, P, P, P, P, P, i32, i32, i64, i64, i32, P, P, P, sz,
                                         P]
            L.idx_score_topk_workspace_size.argtypes = [i32, i32, i64, i32]
            L.idx_score_topk_workspace_size.restype = sz
            L.idx_get_status.argtypes = [P, P, ctypes.POINTER(i32)]
            L.idx_last_error.argtypes = []
            L.idx_last_error.restype = ctypes.c_char_p
            L.idx_version.argtypes = []
            L.idx_version.restype = i32
            L.idx_kernel_launches.argtypes = []
            L.idx_kernel_launches.restype = ctypes.c_uint64
            L.idx_sparse_mla_workspace_size.argtypes = [i32, i32, i32]
            L.idx_sparse_mla_workspace_size.restype = sz
            L.idx_sparse_mla.argtypes = [P, P, i64, P, P, P, P, i32, i32, i32, i32, ctypes.c_float, P,
                                         P, P, sz, P]
            L.idx_sparse_mla_fp8.argtypes = [P, P, P, i64, P, P, P, P, i32, i32, i32, i32,
                                             ctypes.c_float, P, P, P, sz, P]
            for name in ("idx_key_layernorm", "idx_score", "idx_topk", "idx_score_topk",
                         "idx_get_status", "idx_sparse_mla", "idx_sparse_mla_fp8"):
                getattr(L, name).restype = ctypes.c_int
            _lib = L
    return _lib


def _check(code: int, where: str):
    if code != IDX_OK:
        msg = lib().idx_last_error().decode(errors="replace")
        raise IndexerError(code, where, msg)


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _dev(t: torch.Tensor, name: str, dtypes, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)} != {tuple(shape)}")
    return t


_BF16 = (torch.bfloat16, torch.int16, torch.uint16)
_I32 = (torch.int32,)
_F32 = (torch.float32,)


def workspace(nbytes: int, device=None) -> torch.Tensor:
    """A 256-byte aligned device buffer of at least ``nbytes`` (torch allocation)."""
    buf = torch.empty(max(int(nbytes), 256) + 256, dtype=torch.uint8,
                      device=device if device is not None else torch.cuda.current_device())
    off = (-buf.data_ptr()) % 256
    return buf[off:off + max(int(nbytes), 256)]


# ---------------------------------------------------------------------------
# entry points (same names as the C ABI, without the idx_ prefix)
# ---------------------------------------------------------------------------

def key_layernorm(k_raw: torch.Tensor, ln_w: torch.Tensor, ln_b: torch.Tensor, eps: float,
                  out: torch.Tensor | None = None) -> torch.Tensor:
    _dev(k_raw, "k_raw", _BF16)
    if k_raw.dim() != 2 or k_raw.shape[1] != DIM:
        raise ValueError("k_raw must be [n,128]")
    if ln_w.dtype != ln_b.dtype:
        raise TypeError("ln_w and ln_b must share a dtype")
    _dev(ln_w, "ln_w", _BF16 + _F32, (DIM,))
    _dev(ln_b, "ln_b", _BF16 + _F32, (DIM,))
    pdt = PARAM_F32 if ln_w.dtype == torch.float32 else PARAM_BF16
    if out is None:
        out = torch.empty_like(k_raw)
    _dev(out, "out", _BF16, tuple(k_raw.shape))
    _check(lib().idx_key_layernorm(_ptr(k_raw), _ptr(ln_w), _ptr(ln_b), pdt, float(eps),
                                   _ptr(out), k_raw.shape[0], _stream()), "idx_key_layernorm")
    return out


def key_layernorm_append(k_raw: torch.Tensor, ln_w: torch.Tensor, ln_b: torch.Tensor, eps: float,
                         k_cache: torch.Tensor, slot: torch.Tensor) -> torch.Tensor:
    """LayerNorm of the new raw keys written into rows `slot` of `k_cache` (in place)."""
    _dev(k_raw, "k_raw", _BF16)
    if k_raw.dim() != 2 or k_raw.shape[1] != DIM:
        raise ValueError("k_raw must be [n,128]")
    if ln_w.dtype != ln_b.dtype:
        raise TypeError("ln_w and ln_b must share a dtype")
    _dev(ln_w, "ln_w", _BF16 + _F32, (DIM,))
    _dev(ln_b, "ln_b", _BF16 + _F32, (DIM,))
    _dev(k_cache, "k_cache", _BF16)
    if k_cache.dim() != 2 or k_cache.shape[1] != DIM:
        raise ValueError("k_cache must be [rows,128]")
    _dev(slot, "slot", (torch.int64,), (k_raw.shape[0],))
    pdt = PARAM_F32 if ln_w.dtype == torch.float32 else PARAM_BF16
    fn = lib().idx_key_layernorm_append
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_float,
                   ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    _check(fn(_ptr(k_raw), _ptr(ln_w), _ptr(ln_b), pdt, float(eps), _ptr(k_cache),
              k_cache.shape[0], _ptr(slot), k_raw.shape[0], _stream()), "idx_key_layernorm_append")
    return k_cache


def indexer_project_workspace_size(T: int) -> int:
    """Bytes of workspace idx_indexer_project needs for T tokens on this device."""
    L = lib()
    L.idx_indexer_project_workspace_size.argtypes = [ctypes.c_int32]
    L.idx_indexer_project_workspace_size.restype = ctypes.c_size_t
    return int(L.idx_indexer_project_workspace_size(T))


def indexer_project(x: torch.Tensor, q_lora: torch.Tensor, w_q: torch.Tensor, w_k: torch.Tensor,
                    w_w: torch.Tensor, ln_w: torch.Tensor, ln_b: torch.Tensor, eps: float,
                    k_cache: torch.Tensor, slot: torch.Tensor, q: torch.Tensor | None = None,
                    w: torch.Tensor | None = None, ws: torch.Tensor | None = None):
    """Indexer projections -> (q [T,32,128] bf16, w [T,32] fp32); keys go to k_cache[slot]."""
    _dev(x, "x", _BF16)
    _dev(q_lora, "q_lora", _BF16)
    if x.dim() != 2 or q_lora.dim() != 2 or x.shape[0] != q_lora.shape[0]:
        raise ValueError("x [T,hidden] and q_lora [T,rank] with the same T")
    T, hidden, rank = x.shape[0], x.shape[1], q_lora.shape[1]
    _dev(w_q, "w_q", _BF16, (HEADS * DIM, rank))
    _dev(w_k, "w_k", _BF16, (DIM, hidden))
    _dev(w_w, "w_w", _BF16, (HEADS, hidden))
    if ln_w.dtype != ln_b.dtype:
        raise TypeError("ln_w and ln_b must share a dtype")
    _dev(ln_w, "ln_w", _BF16 + _F32, (DIM,))
    _dev(ln_b, "ln_b", _BF16 + _F32, (DIM,))
    _dev(k_cache, "k_cache", _BF16)
    _dev(slot, "slot", (torch.int64,), (T,))
    if q is None:
        q = torch.empty((T, HEADS, DIM), dtype=x.dtype, device=x.device)
    if w is None:
        w = torch.empty((T, HEADS), dtype=torch.float32, device=x.device)
    _dev(q, "q", _BF16, (T, HEADS, DIM))
    _dev(w, "w", _F32, (T, HEADS))
    L = lib()
    need = indexer_project_workspace_size(T)
    if ws is None:
        ws = workspace(need, x.device)
    P = ctypes.c_void_p
    fn = L.idx_indexer_project
    fn.argtypes = [P, P, P, P, P, P, P, ctypes.c_int, ctypes.c_float, ctypes.c_int32, ctypes.c_int32,
                   ctypes.c_int32, P, P, ctypes.c_int64, P, P, P, ctypes.c_size_t, P]
    fn.restype = ctypes.c_int
    pdt = PARAM_F32 if ln_w.dtype == torch.float32 else PARAM_BF16
    _check(fn(_ptr(x), _ptr(q_lora), _ptr(w_q), _ptr(w_k), _ptr(w_w), _ptr(ln_w), _ptr(ln_b), pdt,
              float(eps), T, hidden, rank, _ptr(q), _ptr(k_cache), k_cache.shape[0], _ptr(slot),
              _ptr(w), _ptr(ws), ws.numel(), _stream()), "idx_indexer_project")
    return q, w


def _batch(q, k, w, q_pos, cu_q, cu_k):
    _dev(q, "q", _BF16)
    if q.dim() != 3 or q.shape[1:] != (HEADS, DIM):
        raise ValueError("q must be [T,32,128]")
    T = q.shape[0]
    _dev(k, "k", _BF16)
    if k.dim() != 2 or k.shape[1] != DIM:
        raise ValueError("k must be [L,128]")
    _dev(w, "w", _F32, (T, HEADS))
    _dev(q_pos, "q_pos", _I32, (T,))
    _dev(cu_q, "cu_q", _I32)
    _dev(cu_k, "cu_k", _I32)
    if cu_q.dim() != 1 or cu_q.shape != cu_k.shape or cu_q.numel() < 2:
        raise ValueError("cu_q and cu_k must be [B+1] with B >= 1")
    return T, cu_q.numel() - 1


def score_workspace_size(B: int, T: int, max_len: int) -> int:
    return int(lib().idx_score_workspace_size(B, T, max_len))


def topk_workspace_size(T: int, max_len: int, topk: int) -> int:
    return int(lib().idx_topk_workspace_size(T, max_len, topk))


def score_topk_workspace_size(B: int, T: int, max_len: int, topk: int = TOPK_MAX) -> int:
    return int(lib().idx_score_topk_workspace_size(B, T, max_len, topk))


def score(q, k, w, q_pos, cu_q, cu_k, max_len: int, ld: int | None = None,
          out: torch.Tensor | None = None, ws: torch.Tensor | None = None) -> torch.Tensor:
    """fp32 scores [T, ld]; row t holds n(t) = q_pos[t]+1 valid entries."""
    T, B = _batch(q, k, w, q_pos, cu_q, cu_k)
    if ld is None:
        ld = (max_len + 3) // 4 * 4
    if out is None:
        out = torch.full((T, ld), float("nan"), dtype=torch.float32, device=q.device)
    _dev(out, "out", _F32, (T, ld))
    need = score_workspace_size(B, T, max_len)
    if ws is None:
        ws = workspace(need, q.device)
    _check(lib().idx_score(_ptr(q), _ptr(k), _ptr(w), _ptr(q_pos), _ptr(cu_q), _ptr(cu_k), B, T,
                           k.shape[0], max_len, _ptr(out), ld, _ptr(ws), ws.numel(), _stream()),
           "idx_score")
    return out


def topk(scores: torch.Tensor, n_valid: torch.Tensor, max_len: int, k: int = TOPK_MAX,
         idx: torch.Tensor | None = None, cnt: torch.Tensor | None = None,
         ws: torch.Tensor | None = None):
    """Exact top-k of each row -> (idx [T,k] int32, cnt [T] int32)."""
    _dev(scores, "scores", _F32)
    if scores.dim() != 2:
        raise ValueError("scores must be [T, ld]")
    T, ld = scores.shape
    _dev(n_valid, "n_valid", _I32, (T,))
    if idx is None:
        idx = torch.empty((T, k), dtype=torch.int32, device=scores.device)
    if cnt is None:
        cnt = torch.empty((T,), dtype=torch.int32, device=scores.device)
    _dev(idx, "idx", _I32, (T, k))
    _dev(cnt, "cnt", _I32, (T,))
    need = topk_workspace_size(T, max_len, k)
    if ws is None:
        ws = workspace(need, scores.device)
    _check(lib().idx_topk(_ptr(scores), ld, _ptr(n_valid), T, max_len, k, _ptr(idx), _ptr(cnt),
                          _ptr(ws), ws.numel(), _stream()), "idx_topk")
    return idx, cnt


def score_topk(q, k, w, q_pos, cu_q, cu_k, max_len: int, topk: int = TOPK_MAX,
               idx: torch.Tensor | None = None, cnt: torch.Tensor | None = None,
               ws: torch.Tensor | None = None):
    """The whole indexer -> (idx [T,topk] int32, cnt [T] int32)."""
    T, B = _batch(q, k, w, q_pos, cu_q, cu_k)
    if idx is None:
        idx = torch.empty((T, topk), dtype=torch.int32, device=q.device)
    if cnt is None:
        cnt = torch.empty((T,), dtype=torch.int32, device=q.device)
    _dev(idx, "idx", _I32, (T, topk))
    _dev(cnt, "cnt", _I32, (T,))
    need = score_topk_workspace_size(B, T, max_len, topk)
    if ws is None:
        ws = workspace(need, q.device)
    _check(lib().idx_score_topk(_ptr(q), _ptr(k), _ptr(w), _ptr(q_pos), _ptr(cu_q), _ptr(cu_k), B,
                                T, k.shape[0], max_len, topk, _ptr(idx), _ptr(cnt), _ptr(ws),
                                ws.numel(), _stream()), "idx_score_topk")
    return idx, cnt


def get_status(ws: torch.Tensor) -> tuple[int, int]:
    """(status code, detail) of the last call that used workspace ``ws`` (synchronises)."""
    detail = ctypes.c_int32(0)
    code = lib().idx_get_status(_ptr(ws), _stream(), ctypes.byref(detail))
    return int(code), int(detail.value)


def version() -> int:
    return int(lib().idx_version())


def kernel_launches() -> int:
    """Kernels this library has enqueued in this process."""
    return int(lib().idx_kernel_launches())


def score_topk_noalloc(q, k, w, q_pos, cu_q, cu_k, max_len: int, topk: int = TOPK_MAX,
                       idx: torch.Tensor | None = None, cnt: torch.Tensor | None = None):
    """The whole indexer with no workspace: scratch lives inside the library.

    For callers that cannot supply extra device memory (a fixed memory plan, or
    a host that hands over only inputs and outputs). The library's scratch is
    39 MiB per GPU: T * round_up(max_len, 4) * 4 bytes must fit in its 32 MiB
    of staged scores, T + B <= 40,000, and the selection scratch in 6 MiB. All calls on a
    device share it, so calls that may overlap on the GPU must be serialised;
    the first call on a device resolves the scratch address and should precede
    any stream capture. ``idx``/``cnt`` may be preallocated by the caller.
    """
    T, B = _batch(q, k, w, q_pos, cu_q, cu_k)
    if idx is None:
        idx = torch.empty((T, topk), dtype=torch.int32, device=q.device)
    if cnt is None:
        cnt = torch.empty((T,), dtype=torch.int32, device=q.device)
    _dev(idx, "idx", _I32, (T, topk))
    _dev(cnt, "cnt", _I32, (T,))
    fn = lib().idx_score_topk_noalloc
    P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    fn.argtypes = [P, P, P, P, P, P, i32, i32, i64, i64, i32, P, P, P]
    fn.restype = ctypes.c_int
    _check(fn(_ptr(q), _ptr(k), _ptr(w), _ptr(q_pos), _ptr(cu_q), _ptr(cu_k), B, T, k.shape[0],
              max_len, topk, _ptr(idx), _ptr(cnt), _stream()), "idx_score_topk_noalloc")
    return idx, cnt


def set_wait_limit_ns(limit_ns: int) -> int:
    """Test hook: bound (ns) of every wait in the tensor-core scorer; returns the old one."""
    fn = lib().idx_set_wait_limit_ns
    fn.argtypes = [ctypes.c_uint64]
    fn.restype = ctypes.c_uint64
    return int(fn(int(limit_ns)))


def set_kernel_events(events) -> int:
    """Measurement hook: record ``events`` (torch.cuda.Event with timing, each
    recorded once before so that it exists) right after each of the next
    len(events) kernels this thread enqueues through the library; [] disarms."""
    handles = [ctypes.c_void_p(int(e.cuda_event)) for e in events]
    arr = (ctypes.c_void_p * max(len(handles), 1))(*handles)
    fn = lib().idx_set_kernel_events
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int32]
    fn.restype = ctypes.c_int32
    r = int(fn(arr if handles else None, len(handles)))
    if r < 0:
        raise IndexerError(1, "idx_set_kernel_events", lib().idx_last_error().decode(errors="replace"))
    return r


MLA_DIM = 576    # MLA cache row: 512-wide latent + 64 key dims
MLA_VDIM = 512


def sparse_mla_workspace_size(T: int, heads: int, topk: int) -> int:
    return int(lib().idx_sparse_mla_workspace_size(T, heads, topk))


def sparse_mla(q, cache, idx, cnt, cu_q, cu_k, scale: float, out: torch.Tensor | None = None,
               lse: torch.Tensor | None = None, ws: torch.Tensor | None = None):
    """Sparse MLA attention over the selected positions -> (out [T,H,512] fp32, lse [T,H] fp32).

    q bf16 [T, H, 576]; cache bf16 [rows, 576]; idx int32 [T, topk] and cnt int32 [T]
    as the indexer writes them; cu_q / cu_k int32 [B+1].
    """
    _dev(q, "q", _BF16)
    _dev(cache, "cache", _BF16)
    _dev(idx, "idx", _I32)
    _dev(cnt, "cnt", _I32)
    _dev(cu_q, "cu_q", _I32)
    _dev(cu_k, "cu_k", _I32)
    if q.dim() != 3 or q.shape[2] != MLA_DIM:
        raise ValueError("q must be [T, heads, 576]")
    if cache.dim() != 2 or cache.shape[1] != MLA_DIM:
        raise ValueError("cache must be [rows, 576]")
    T, H = int(q.shape[0]), int(q.shape[1])
    if idx.dim() != 2 or idx.shape[0] != T:
        raise ValueError("idx must be [T, topk]")
    topk = int(idx.shape[1])
    _dev(cnt, "cnt", _I32, (T,))
    B = int(cu_q.numel()) - 1
    if out is None:
        out = torch.empty((T, H, MLA_VDIM), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
    _dev(out, "out", _F32, (T, H, MLA_VDIM))
    _dev(lse, "lse", _F32, (T, H))
    need = sparse_mla_workspace_size(T, H, topk)
    if ws is None:
        ws = workspace(need, q.device)
    _check(lib().idx_sparse_mla(_ptr(q), _ptr(cache), int(cache.shape[0]), _ptr(idx), _ptr(cnt),
                                _ptr(cu_q), _ptr(cu_k), B, T, H, topk, float(scale), _ptr(out),
                                _ptr(lse), _ptr(ws), ws.numel(), _stream()),
           "idx_sparse_mla")
    return out, lse


def sparse_mla_fp8(q, cache8, row_scale, idx, cnt, cu_q, cu_k, scale: float,
                   out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                   ws: torch.Tensor | None = None):
    """Sparse MLA attention over an FP8 cache -> (out [T,H,512] fp32, lse [T,H] fp32).

    cache8 uint8 (or float8_e4m3fn) [rows, 576] of E4M3 codes, row_scale fp32 [rows]:
    row s stands for row_scale[s] * e4m3(cache8[s]). Other arguments as sparse_mla.
    """
    _dev(q, "q", _BF16)
    _dev(cache8, "cache8", (torch.uint8, torch.float8_e4m3fn))
    _dev(idx, "idx", _I32)
    _dev(cnt, "cnt", _I32)
    _dev(cu_q, "cu_q", _I32)
    _dev(cu_k, "cu_k", _I32)
    if q.dim() != 3 or q.shape[2] != MLA_DIM:
        raise ValueError("q must be [T, heads, 576]")
    if cache8.dim() != 2 or cache8.shape[1] != MLA_DIM:
        raise ValueError("cache8 must be [rows, 576]")
    _dev(row_scale, "row_scale", _F32, (int(cache8.shape[0]),))
    T, H = int(q.shape[0]), int(q.shape[1])
    if idx.dim() != 2 or idx.shape[0] != T:
        raise ValueError("idx must be [T, topk]")
    topk = int(idx.shape[1])
    _dev(cnt, "cnt", _I32, (T,))
    B = int(cu_q.numel()) - 1
    if out is None:
        out = torch.empty((T, H, MLA_VDIM), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
    _dev(out, "out", _F32, (T, H, MLA_VDIM))
    _dev(lse, "lse", _F32, (T, H))
    need = sparse_mla_workspace_size(T, H, topk)
    if ws is None:
        ws = workspace(need, q.device)
    _check(lib().idx_sparse_mla_fp8(_ptr(q), _ptr(cache8), _ptr(row_scale), int(cache8.shape[0]),
                                    _ptr(idx), _ptr(cnt), _ptr(cu_q), _ptr(cu_k), B, T, H, topk,
                                    float(scale), _ptr(out), _ptr(lse), _ptr(ws), ws.numel(),
                                    _stream()),
           "idx_sparse_mla_fp8")
    return out, lse
