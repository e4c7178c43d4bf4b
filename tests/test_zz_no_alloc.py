"""idx_score_topk_noalloc against idx_score_topk, through the C ABI.

The no-allocation entry point serves callers that cannot give the library any
device memory of its own (a serving engine with a fixed memory plan that bans
cudaMalloc on its request path, or a plugin handed only its input and output
buffers). Its scratch is a fixed array inside the library, shared by every
call, so this test makes two different calls in a row and checks both against
the workspace entry point, then checks a call that fills the 32 MiB of staged
scores against the CPU oracle itself, and a call whose scorer gives up. It
lives in its own file, collected last, so that a run stopping at the first
failure has already run every other test; it also passes on its own in a
fresh process.
"""
import ctypes
import os

import numpy as np
import pytest

import oracle
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


def test_noalloc_at_its_scratch_limit_matches_the_oracle(L):
    # 64 queries at the end of one 131,072-key history: 64 * 131,072 * 4 bytes
    # of staged scores, exactly the 32 MiB the library holds. Integer inputs
    # with heavy ties: indices and counts bit-exact against the oracle.
    n, T = 131_072, 64
    w = wl.custom(904, q_counts=[T], k_lens=[n], kind="int2")
    assert w.T * ((w.max_len + 3) // 4 * 4) * 4 == 32 << 20
    d = to_device(w)
    idx, cnt = _noalloc(L, d, w.T, w.B, w.max_len, w.topk)
    torch.cuda.synchronize()
    ridx, rcnt, _ = oracle.score_topk(w.q, w.k, w.w, w.q_pos, w.cu_q, w.cu_k, K=w.topk,
                                      threads=os.cpu_count() or 8)
    assert np.array_equal(cnt.cpu().numpy(), rcnt)
    assert np.array_equal(idx.cpu().numpy(), ridx)


def test_noalloc_scorer_timeout_leaves_every_row_skipped_then_recovers(L):
    # With the wait bound at 0 the scorer gives up; the call has no status word
    # to read, so every row must come back as skipped (cnt 0, idx -1) instead
    # of a selection from half-written scores. The next call, with the normal
    # bound, reuses the same scratch and must match the oracle again.
    from sparse_attention_key_gb300 import binding
    w = wl.custom(905, q_counts=[1, 1, 1], k_lens=[30000, 9000, 20000], kind="int2")
    d = to_device(w)
    old = binding.set_wait_limit_ns(0)
    try:
        idx, cnt = _noalloc(L, d, w.T, w.B, w.max_len, w.topk)
        torch.cuda.synchronize()
    finally:
        binding.set_wait_limit_ns(old)
    assert (cnt.cpu().numpy() == 0).all()
    assert (idx.cpu().numpy() == -1).all()
    idx, cnt = _noalloc(L, d, w.T, w.B, w.max_len, w.topk)
    torch.cuda.synchronize()
    ridx, rcnt, _ = oracle.score_topk(w.q, w.k, w.w, w.q_pos, w.cu_q, w.cu_k, K=w.topk, threads=3)
    assert np.array_equal(cnt.cpu().numpy(), rcnt)
    assert np.array_equal(idx.cpu().numpy(), ridx)
