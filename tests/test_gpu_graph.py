"""The workspace entry points inside a CUDA graph.

Serving engines capture a decode step once and replay it. The fused call
launches only kernels (programmatic dependent launches; the plan kernel clears
the status word and the selection histograms itself), so it can be captured
after one direct call has done the per-process set-up. These tests capture it
in a torch CUDA graph, replay it, change the inputs in place and replay again,
comparing with direct calls.
"""
import numpy as np
import pytest

from sparse_attention_key_gb300 import workloads as wl
from tests._util import to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_attention_key_gb300 import build
    build.build()
    from sparse_attention_key_gb300 import binding
    return binding


@pytest.mark.parametrize("shape", ["decode", "prefill"])
def test_fused_call_replays_in_a_cuda_graph(B, shape):
    if shape == "decode":   # one query per sequence: scorer histogram + cluster selection
        w = wl.custom(801, q_counts=[1, 1, 1, 1], k_lens=[30000, 14000, 5000, 20000], kind="normal")
    else:                   # many queries per sequence: 16-query scorer + staged selection
        w = wl.custom(802, q_counts=[200, 40], k_lens=[4000, 900], kind="normal")
    d = to_device(w)
    T = w.T
    ws = B.workspace(B.score_topk_workspace_size(w.B, T, w.max_len), "cuda")
    idx = torch.empty((T, 2048), dtype=torch.int32, device="cuda")
    cnt = torch.empty((T,), dtype=torch.int32, device="cuda")
    call = lambda: B.score_topk(d["q"], d["k"], d["w"], d["q_pos"], d["cu_q"], d["cu_k"],
                                w.max_len, idx=idx, cnt=cnt, ws=ws)
    call()                                   # per-process set-up outside the capture
    torch.cuda.synchronize()
    ref_idx, ref_cnt = idx.clone(), cnt.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    idx.fill_(-7)
    cnt.fill_(-7)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(idx, ref_idx) and torch.equal(cnt, ref_cnt)
    assert B.get_status(ws) == (0, 0)
    # new weights in place: the replay follows them
    rng = np.random.default_rng(803)
    d["w"].copy_(torch.from_numpy(rng.uniform(0, 1.0 / 32, size=(T, 32)).astype(np.float32)))
    g.replay()
    torch.cuda.synchronize()
    got = idx.clone()
    call()
    torch.cuda.synchronize()
    assert torch.equal(got, idx)
    assert not torch.equal(got, ref_idx)


def test_concurrent_calls_from_several_host_threads(B):
    # the library's host-side state (device info, shared-memory opt-ins, the
    # tensor-map encoder) is shared; calls from several threads, each on its
    # own stream and workspace, must give the results of sequential calls
    import threading
    ws_list, outs, refs, errors = [], [], [], []
    batches = [wl.custom(810 + i, q_counts=[1, 2, 1], k_lens=[9000 + 1000 * i, 20000, 3000],
                         kind="int2") for i in range(4)]
    devs = [to_device(w) for w in batches]
    for w, d in zip(batches, devs):
        ws_list.append(B.workspace(B.score_topk_workspace_size(w.B, w.T, w.max_len), "cuda"))
        refs.append(B.score_topk(d["q"], d["k"], d["w"], d["q_pos"], d["cu_q"], d["cu_k"], w.max_len,
                                 ws=ws_list[-1])[0].clone())
        outs.append(None)
    torch.cuda.synchronize()

    def work(i):
        try:
            s = torch.cuda.Stream()
            w, d = batches[i], devs[i]
            with torch.cuda.stream(s):
                for _ in range(20):
                    idx, _ = B.score_topk(d["q"], d["k"], d["w"], d["q_pos"], d["cu_q"], d["cu_k"],
                                          w.max_len, ws=ws_list[i])
                s.synchronize()
            outs[i] = idx
        except Exception as e:   # reported below
            errors.append(repr(e))

    threads = [threading.Thread(target=work, args=(i,)) for i in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not errors, errors
    for i in range(4):
        assert torch.equal(outs[i], refs[i]), i
        assert B.get_status(ws_list[i]) == (0, 0)


def test_sparse_mla_replays_in_a_cuda_graph(B):
    """The attention over the selection (memset of the status word, attention,
    merge) captured once and replayed, following new query values in place."""
    q, cache, idx, cnt, cu_q, cu_k = wl.mla_case(811, [9000, 3000, 20000], q_per_seq=1)
    dv = lambda a, dt=None: torch.from_numpy(np.ascontiguousarray(a if dt is None else a.view(dt))).cuda()
    dq, dc, di, dn, dcq, dck = dv(q, np.int16), dv(cache, np.int16), dv(idx), dv(cnt), dv(cu_q), dv(cu_k)
    T, H = q.shape[0], q.shape[1]
    out = torch.empty((T, H, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((T, H), dtype=torch.float32, device="cuda")
    ws = B.workspace(B.sparse_mla_workspace_size(T, H, 2048), "cuda")
    call = lambda: B.sparse_mla(dq, dc, di, dn, dcq, dck, 0.072, out=out, lse=lse, ws=ws)
    call()
    torch.cuda.synchronize()
    ref_out, ref_lse = out.clone(), lse.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    out.fill_(7.0)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
    assert B.get_status(ws) == (0, 0)
    q2 = wl.f32_to_bf16_bits(np.random.default_rng(812).standard_normal(q.shape).astype(np.float32))
    dq.copy_(dv(q2, np.int16))
    g.replay()
    torch.cuda.synchronize()
    got = out.clone()
    call()
    torch.cuda.synchronize()
    assert torch.equal(got, out) and not torch.equal(got, ref_out)
