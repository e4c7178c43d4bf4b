"""idx_score_topk_noalloc against idx_score_topk, through the C ABI.

The no-allocation entry point serves callers that cannot give the library any
device memory of its own (a serving engine with a fixed memory plan that bans
cudaMalloc on its request path, or a plugin handed only its input and output
buffers). Its scratch is a fixed array inside the library, shared by every
call, so this test makes two different calls in a row and checks both against
the workspace entry point. It lives in its own file, collected last, so that a
run stopping at the first failure has already run every other test; it also
passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest

from sparse_attention_key_gb300 import workloads as wl
from tests._util import to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_attention_key_gb300 import build
    build.build()
    from sparse_attention_key_gb300 import binding
    lib = binding.lib()
    P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    lib.idx_score_topk_noalloc.argtypes = [P, P, P, P, P, P, i32, i32, i64, i64, i32, P, P, P]
    lib.idx_score_topk_noalloc.restype = ctypes.c_int
    return lib


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(L, d, T, B, max_len, K):
    idx = torch.full((T, K), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((T,), -7, dtype=torch.int32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = L.idx_score_topk_noalloc(_p(d["q"]), _p(d["k"]), _p(d["w"]), _p(d["q_pos"]),
                                  _p(d["cu_q"]), _p(d["cu_k"]), B, T, d["k"].shape[0], max_len,
                                  K, _p(idx), _p(cnt), stream)
    assert rc == 0, L.idx_last_error()
    return idx, cnt


def _with_workspace(d, max_len, K):
    from sparse_attention_key_gb300 import binding
    return binding.score_topk(d["q"], d["k"], d["w"], d["q_pos"], d["cu_q"], d["cu_k"], max_len, K)


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row(L):
    # call 1: integer inputs with heavy ties (bit-exact bar); call 2: a different,
    # smaller real-valued batch that reuses the shared scratch after call 1.
    w1 = wl.custom(901, q_counts=[40, 3], k_lens=[3000, 2600], kind="int2")
    # (call 2 is decode-shaped: few queries with long histories)
    w2 = wl.custom(902, q_counts=[1, 1, 1, 2], k_lens=[20000, 2049, 7, 14000], kind="normal")
    for w in (w1, w2):
        d = to_device(w)
        idx_a, cnt_a = _noalloc(L, d, w.T, w.B, w.max_len, w.topk)
        idx_b, cnt_b = _with_workspace(d, w.max_len, w.topk)
        torch.cuda.synchronize()
        # same kernels on the same inputs: identical results (within-tolerance
        # for real inputs reduces to equality here)
        assert torch.equal(idx_a, idx_b)
        assert torch.equal(cnt_a, cnt_b)


def test_noalloc_rejects_calls_beyond_its_scratch(L):
    w = wl.custom(903, q_counts=[2], k_lens=[64], kind="int2")
    d = to_device(w)
    T, too_long = 65, 131_073       # 65 * 131,076 * 4 bytes > 32 MiB
    idx = torch.empty((T, 2048), dtype=torch.int32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = L.idx_score_topk_noalloc(_p(d["q"]), _p(d["k"]), _p(d["w"]), _p(d["q_pos"]),
                                  _p(d["cu_q"]), _p(d["cu_k"]), 1, T, d["k"].shape[0], too_long,
                                  2048, _p(idx), None, stream)
    assert rc == 3
    assert b"32 MiB" in L.idx_last_error()
