"""Failure detection on the GPU without a fault: the scorer's bounded waits.

Every wait inside the tensor-core scorer has a time bound. This test lowers
the bound to zero through the library's test hook, so the first wait that is
not already satisfied gives up: the kernel must record IDX_ERR_TIMEOUT in the
status word, drain its copies and tensor-core work, free its tensor memory and
return. The test then restores the bound and checks that the same CUDA context
still computes correct results. No GPU is faulted, trapped or hung.
"""
import numpy as np
import pytest

import oracle
from sparse_attention_key_gb300 import workloads as wl
from tests._util import to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

IDX_ERR_TIMEOUT = 5


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_attention_key_gb300 import build
    build.build()
    from sparse_attention_key_gb300 import binding
    return binding


@pytest.mark.parametrize("shape", ["decode", "prefill", "decode_steal", "verify_steal"])
def test_zero_wait_bound_reports_timeout_and_context_survives(B, shape):
    # "_steal": a cache of more than 32 key tiles per SM, so the decode (one
    # query per sequence) and verification (four) scorers share work between
    # their CTAs, and their scheduling warp's waits are bounded too
    if shape == "decode":
        w = wl.custom(701, q_counts=[1, 1, 1], k_lens=[30000, 9000, 20000], kind="int2")
    elif shape == "prefill":
        w = wl.custom(702, q_counts=[300], k_lens=[3000], kind="int2")
    else:
        per = 1 if shape == "decode_steal" else 4
        w = wl.custom(703, q_counts=[per] * 3, k_lens=[300000, 200000, 150000], kind="int2")
        assert int(w.cu_k[-1]) // 128 >= 32 * 152
    d = to_device(w)
    ws = B.workspace(B.score_topk_workspace_size(w.B, w.T, w.max_len), "cuda")
    old = B.set_wait_limit_ns(0)
    try:
        idx, cnt = B.score_topk(d["q"], d["k"], d["w"], d["q_pos"], d["cu_q"], d["cu_k"],
                                w.max_len, ws=ws)
        code, _ = B.get_status(ws)          # synchronises: the kernel returned
    finally:
        B.set_wait_limit_ns(old)
    assert code == IDX_ERR_TIMEOUT
    # nothing is selected from the incomplete scores: every row is skipped
    assert (cnt.cpu().numpy() == 0).all() and (idx.cpu().numpy() == -1).all()
    # same context, normal bound: a correct result again
    idx, cnt = B.score_topk(d["q"], d["k"], d["w"], d["q_pos"], d["cu_q"], d["cu_k"], w.max_len,
                            ws=ws)
    assert B.get_status(ws) == (0, 0)
    ridx, rcnt, _ = oracle.score_topk(w.q, w.k, w.w, w.q_pos, w.cu_q, w.cu_k, K=2048, threads=8)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    assert np.array_equal(cnt.cpu().numpy(), rcnt)


def test_sparse_mla_zero_wait_bound_reports_timeout_and_context_survives(B):
    """The same for the sparse MLA attention: every role leaves through its
    bounded drain, the status word says IDX_ERR_TIMEOUT, and the context then
    computes the oracle's result again."""
    q, cache, idx, cnt, cu_q, cu_k = wl.mla_case(721, [9000, 3000, 20000], q_per_seq=1)
    dv = lambda a, dt=None: torch.from_numpy(np.ascontiguousarray(a if dt is None else a.view(dt))).cuda()
    args = (dv(q, np.int16), dv(cache, np.int16), dv(idx), dv(cnt), dv(cu_q), dv(cu_k), 0.072)
    ws = B.workspace(B.sparse_mla_workspace_size(q.shape[0], q.shape[1], 2048), "cuda")
    old = B.set_wait_limit_ns(0)
    try:
        B.sparse_mla(*args, ws=ws)
        code, _ = B.get_status(ws)
    finally:
        B.set_wait_limit_ns(old)
    assert code == IDX_ERR_TIMEOUT
    out, lse = B.sparse_mla(*args, ws=ws)
    assert B.get_status(ws) == (0, 0)
    o_ref, l_ref = oracle.sparse_mla_batch(q, cache, idx, cnt, cu_q, cu_k, 0.072)
    lat = oracle.bf16_bits_to_f64(cache[:, :512])
    o, l = out.cpu().numpy(), lse.cpu().numpy()
    for t in range(q.shape[0]):
        b = t
        vmax = np.abs(lat[cu_k[b] + idx[t, :cnt[t]]]).max()
        assert np.abs(o[t] - o_ref[t]).max() <= 2.0 ** -8 * vmax
        np.testing.assert_allclose(l[t], l_ref[t], atol=2e-4)


def test_projection_gemm_zero_wait_bound_reports_timeout_and_context_survives(B):
    """The projection GEMM's waits are bounded too: with a bound of 0 the call
    reports IDX_ERR_TIMEOUT in its workspace's status word, and the same context
    then computes the exact projections again."""
    rng = np.random.default_rng(731)
    T, hidden, rank = 40, 512, 256
    mk = lambda shape: wl.f32_to_bf16_bits(rng.integers(-2, 3, size=shape).astype(np.float32))
    x, ql = mk((T, hidden)), mk((T, rank))
    wq, wk, ww = mk((4096, rank)), mk((128, hidden)), mk((32, hidden))
    g = wl.f32_to_bf16_bits(np.ones(128, np.float32))
    b = wl.f32_to_bf16_bits(np.zeros(128, np.float32))
    dv = lambda a: torch.from_numpy(a.view(np.int16)).cuda()
    args = (dv(x), dv(ql), dv(wq), dv(wk), dv(ww), dv(g), dv(b), 1e-6)
    cache = torch.zeros((T, 128), dtype=torch.int16, device="cuda")
    slot = torch.arange(T, dtype=torch.int64, device="cuda")
    from sparse_attention_key_gb300 import binding
    ws = B.workspace(int(binding.lib().idx_indexer_project_workspace_size(T)), "cuda")
    old = B.set_wait_limit_ns(0)
    try:
        B.indexer_project(*args, cache, slot, ws=ws)
        code, _ = B.get_status(ws)
    finally:
        B.set_wait_limit_ns(old)
    assert code == IDX_ERR_TIMEOUT
    q, w = B.indexer_project(*args, cache, slot, ws=ws)
    assert B.get_status(ws) == (0, 0)
    rq, _, rw, _ = oracle.indexer_project(x, ql, wq, wk, ww, np.ones(128), np.zeros(128), 1e-6)
    assert np.array_equal(q.view(torch.int16).cpu().numpy().view(np.uint16), rq)
    assert np.array_equal(w.cpu().numpy(), rw.astype(np.float32))
