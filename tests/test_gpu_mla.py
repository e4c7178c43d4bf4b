"""Sparse MLA attention over the selected positions: CUDA path against the oracle.

Tolerance (derived from the arithmetic): the kernel rounds the softmax weights
to bf16 before the weighted sum of the latents (relative error <= 2^-9 per
weight, while the normaliser keeps fp32 weights), accumulates in fp32 and uses
exp2f. So |out - oracle| <= 2^-8 * max |latent| over the selected rows, and
lse (from an fp32 sum of at most 2048 terms) within 2e-4.
"""
import numpy as np
import pytest
import torch

import oracle
from sparse_attention_key_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from sparse_attention_key_gb300 import binding
    binding.lib()
    return binding


def _run(B, q, cache, idx, cnt, cu_q, cu_k, scale):
    dv = lambda a, dt=None: torch.from_numpy(np.ascontiguousarray(a if dt is None else a.view(dt))).cuda()
    out, lse = B.sparse_mla(dv(q, np.int16), dv(cache, np.int16), dv(idx), dv(cnt), dv(cu_q), dv(cu_k), scale)
    return out.cpu().numpy(), lse.cpu().numpy()


def _check(o_gpu, l_gpu, o_ref, l_ref, cache, idx, cnt, cu_q, cu_k, rows):
    lat = oracle.bf16_bits_to_f64(cache[:, :512])
    for t in rows:
        b = int(np.searchsorted(cu_q, t, side="right")) - 1
        n = int(cnt[t])
        if n == 0:
            assert np.all(o_gpu[t] == 0) and np.all(np.isneginf(l_gpu[t])), f"row {t}"
            continue
        vmax = np.abs(lat[cu_k[b] + idx[t, :n]]).max()
        err = np.abs(o_gpu[t] - o_ref[t]).max()
        assert err <= 2.0 ** -8 * vmax, f"row {t}: |d out| {err} > {2.0 ** -8 * vmax}"
        np.testing.assert_allclose(l_gpu[t], l_ref[t], rtol=0, atol=2e-4, err_msg=f"row {t}")


@pytest.mark.parametrize("heads", [32, 64, 96])
def test_mla_small_batches_against_oracle(B, heads):
    # selections of 0, 1, 17 (one partial tile), 33, 100 rows and full ones
    lens = [40, 3000, 2100, 5000]
    n_sel = [0, 1, 17, 33, 100, 2048, 2048, 1500]
    q, cache, idx, cnt, cu_q, cu_k = wl.mla_case(11 + heads, lens, q_per_seq=2, heads=heads,
                                                  n_sel=[min(s, l) for s, l in zip(n_sel, np.repeat(lens, 2))])
    scale = 1.0 / np.sqrt(192.0)
    o, l = _run(B, q, cache, idx, cnt, cu_q, cu_k, scale)
    o_ref, l_ref = oracle.sparse_mla_batch(q, cache, idx, cnt, cu_q, cu_k, scale)
    _check(o, l, o_ref, l_ref, cache, idx, cnt, cu_q, cu_k, range(q.shape[0]))


def test_mla_peaked_softmax_rescales_across_tiles(B):
    """A large scale: the running maximum grows by more than 2^8 between tiles,
    so the kernel rescales its accumulator."""
    q, cache, idx, cnt, cu_q, cu_k = wl.mla_case(21, [4096, 2500], q_per_seq=1)
    for scale in (0.5, 2.0):
        o, l = _run(B, q, cache, idx, cnt, cu_q, cu_k, scale)
        o_ref, l_ref = oracle.sparse_mla_batch(q, cache, idx, cnt, cu_q, cu_k, scale)
        _check(o, l, o_ref, l_ref, cache, idx, cnt, cu_q, cu_k, range(q.shape[0]))


@pytest.mark.parametrize("topk", [1, 33])
def test_mla_short_index_rows(B, topk):
    """idx rows of stride 1 and 33: selections shorter than one tile, and a
    second tile holding one row."""
    lens = [1, 50, 700, 33]
    q, cache, idx, cnt, cu_q, cu_k = wl.mla_case(25 + topk, lens, q_per_seq=1, heads=64, topk=topk)
    assert idx.shape == (4, topk) and list(cnt) == [1, min(topk, 50), min(topk, 700), min(topk, 33)]
    scale = 1.0 / np.sqrt(192.0)
    o, l = _run(B, q, cache, idx, cnt, cu_q, cu_k, scale)
    o_ref, l_ref = oracle.sparse_mla_batch(q, cache, idx, cnt, cu_q, cu_k, scale)
    _check(o, l, o_ref, l_ref, cache, idx, cnt, cu_q, cu_k, range(q.shape[0]))


def test_mla_many_rows_single_split(B):
    """T >= the SM count: one CTA per query row writes the result directly."""
    lens = [3000] * 40
    q, cache, idx, cnt, cu_q, cu_k = wl.mla_case(31, lens, q_per_seq=4, heads=32, topk=256)
    scale = 1.0 / np.sqrt(192.0)
    o, l = _run(B, q, cache, idx, cnt, cu_q, cu_k, scale)
    rows = list(range(0, q.shape[0], 7)) + [q.shape[0] - 1]
    o_ref, l_ref = oracle.sparse_mla_batch(q, cache, idx, cnt, cu_q, cu_k, scale, rows=rows)
    _check(o, l, o_ref, l_ref, cache, idx, cnt, cu_q, cu_k, rows)


def test_mla_positions_outside_the_sequence_are_left_out(B):
    q, cache, idx, cnt, cu_q, cu_k = wl.mla_case(41, [300, 400], q_per_seq=1, topk=64)
    idx[1, 5] = 400          # one past the sequence
    idx[1, 9] = -3
    scale = 0.1
    dv = lambda a, dt=None: torch.from_numpy(np.ascontiguousarray(a if dt is None else a.view(dt))).cuda()
    ws = B.workspace(B.sparse_mla_workspace_size(2, 96, 64), "cuda")
    out, lse = B.sparse_mla(dv(q, np.int16), dv(cache, np.int16), dv(idx), dv(cnt), dv(cu_q), dv(cu_k),
                            scale, ws=ws)
    code, detail = B.get_status(ws)
    assert code == 6 and detail == 1
    keep = [p for j, p in enumerate(idx[1, :cnt[1]]) if j not in (5, 9)]
    o_ref, l_ref = oracle.sparse_mla(q[1], cache, 300 + np.asarray(keep), scale)
    o, l = out.cpu().numpy()[1], lse.cpu().numpy()[1]
    vmax = np.abs(oracle.bf16_bits_to_f64(cache[300 + np.asarray(keep), :512])).max()
    assert np.abs(o - o_ref).max() <= 2.0 ** -8 * vmax
    np.testing.assert_allclose(l, l_ref, atol=2e-4)


def test_mla_consumes_the_indexer_selection(B):
    """idx_score_topk's output fed straight into the attention."""
    w = wl.custom(51, q_counts=[1, 1, 1], k_lens=[3000, 5000, 2100], kind="normal", positions="chunk")
    dv = lambda a, dt=None: torch.from_numpy(np.ascontiguousarray(a if dt is None else a.view(dt))).cuda()
    qi, k, wt = dv(w.q, np.int16), dv(w.k, np.int16), dv(w.w)
    qp, cq, ck = dv(w.q_pos), dv(w.cu_q), dv(w.cu_k)
    idx, cnt = B.score_topk(qi, k, wt, qp, cq, ck, w.max_len)
    rng = np.random.default_rng(52)
    cache = wl.f32_to_bf16_bits(rng.standard_normal((int(w.cu_k[-1]), 576)).astype(np.float32))
    qm = wl.f32_to_bf16_bits(rng.standard_normal((w.T, 96, 576)).astype(np.float32))
    out, lse = B.sparse_mla(dv(qm, np.int16), dv(cache, np.int16), idx, cnt, cq, ck, 0.07)
    idx_h, cnt_h = idx.cpu().numpy(), cnt.cpu().numpy()
    ref_idx, ref_cnt, _ = oracle.score_topk(w.q, w.k, w.w, w.q_pos, w.cu_q, w.cu_k)
    assert np.array_equal(cnt_h, ref_cnt)
    o_ref, l_ref = oracle.sparse_mla_batch(qm, cache, idx_h, cnt_h, w.cu_q, w.cu_k, 0.07)
    _check(out.cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, cache, idx_h, cnt_h, w.cu_q, w.cu_k,
           range(w.T))


def test_mla_decode_batch_full_size(B):
    """The decode batch's shapes: 8 sequences of 8K..64K cached rows, one query
    each, 2048 selected rows, 96 heads; every row against the oracle."""
    lens = [8192, 12288, 16384, 24576, 32768, 40960, 49152, 65536]
    q, cache, idx, cnt, cu_q, cu_k = wl.mla_case(61, lens)
    scale = 1.0 / np.sqrt(192.0)
    o, l = _run(B, q, cache, idx, cnt, cu_q, cu_k, scale)
    o_ref, l_ref = oracle.sparse_mla_batch(q, cache, idx, cnt, cu_q, cu_k, scale)
    _check(o, l, o_ref, l_ref, cache, idx, cnt, cu_q, cu_k, range(q.shape[0]))


def test_mla_bad_counts_and_empty_sequences(B):
    """A count above topk is reported (status, that row's output zero, lse
    -inf); an empty sequence and an empty selection change nothing else."""
    lens = [5000, 0, 3000, 2500]
    q, cache, idx, cnt, cu_q, cu_k = wl.mla_case(71, [5000, 1, 3000, 2500], q_per_seq=1, topk=256)
    cu_k = np.array([0, 5000, 5000, 8000, 10500], np.int32)   # sequence 1: no cached rows
    cu_q = np.array([0, 1, 1, 2, 3], np.int32)                # ... and no query rows
    q = q[[0, 2, 3]]
    idx = idx[[0, 2, 3]]
    cnt = cnt[[0, 2, 3]].copy()
    cache = cache[:10500]
    cnt[1] = 0          # an empty selection
    cnt[2] = 300        # above topk = 256
    dv = lambda a, dt=None: torch.from_numpy(np.ascontiguousarray(a if dt is None else a.view(dt))).cuda()
    ws = B.workspace(B.sparse_mla_workspace_size(3, 96, 256), "cuda")
    out, lse = B.sparse_mla(dv(q, np.int16), dv(cache, np.int16), dv(idx), dv(cnt), dv(cu_q), dv(cu_k),
                            0.07, ws=ws)
    code, detail = B.get_status(ws)
    assert code == 6 and detail == 2
    o, l = out.cpu().numpy(), lse.cpu().numpy()
    assert np.all(o[1] == 0) and np.all(np.isneginf(l[1]))
    assert np.all(o[2] == 0) and np.all(np.isneginf(l[2]))
    o_ref, l_ref = oracle.sparse_mla(q[0], cache, idx[0, :cnt[0]], 0.07)
    vmax = np.abs(oracle.bf16_bits_to_f64(cache[idx[0, :cnt[0]], :512])).max()
    assert np.abs(o[0] - o_ref).max() <= 2.0 ** -8 * vmax
    np.testing.assert_allclose(l[0], l_ref, atol=2e-4)


def test_mla_long_decode_full_size_sampled(B):
    """64 queries over histories of 64K..128K rows (a 7 GB cache made on the
    device from a seeded generator), 2048 selected rows each, 96 heads: the
    launch configuration bench.py --mla long_decode times (two splits per
    query). Three sampled queries against the oracle on their gathered rows."""
    dev = torch.device("cuda", 0)
    lens = np.random.default_rng(81).integers(65536, 131073, size=64).astype(np.int64)
    T, H, K = 64, 96, 2048
    gen = torch.Generator(device=dev).manual_seed(82)
    L = int(lens.sum())
    cache = torch.empty((L, 576), dtype=torch.bfloat16, device=dev)
    for r0 in range(0, L, 1 << 20):
        r1 = min(L, r0 + (1 << 20))
        cache[r0:r1] = torch.randn((r1 - r0, 576), generator=gen, device=dev).to(torch.bfloat16)
    q = torch.randn((T, H, 576), generator=gen, device=dev).to(torch.bfloat16)
    idx = torch.stack([torch.randperm(int(n), generator=gen, device=dev)[:K].sort().values
                       for n in lens]).to(torch.int32)
    cnt = torch.full((T,), K, dtype=torch.int32, device=dev)
    cu_k_h = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    cu_k = torch.from_numpy(cu_k_h).to(dev)
    cu_q = torch.arange(T + 1, dtype=torch.int32, device=dev)
    scale = 1.0 / np.sqrt(192.0)
    ws = B.workspace(B.sparse_mla_workspace_size(T, H, K), dev)
    out, lse = B.sparse_mla(q, cache, idx, cnt, cu_q, cu_k, scale, ws=ws)
    assert B.get_status(ws) == (0, 0)
    for t in (0, 31, 63):
        rows = int(cu_k_h[t]) + idx[t].long()
        sel = cache[rows].view(torch.int16).cpu().numpy().view(np.uint16)      # [2048, 576]
        qt = q[t].view(torch.int16).cpu().numpy().view(np.uint16)
        o_ref, l_ref = oracle.sparse_mla(qt, sel, np.arange(K), scale)
        vmax = np.abs(oracle.bf16_bits_to_f64(sel[:, :512])).max()
        err = np.abs(out[t].cpu().numpy() - o_ref).max()
        assert err <= 2.0 ** -8 * vmax, f"row {t}: |d out| {err}"
        np.testing.assert_allclose(lse[t].cpu().numpy(), l_ref, atol=2e-4, err_msg=f"row {t}")


# ---------------------------------------------------------------------------
# FP8 (E4M3) cache. Same tolerance: the codes convert to bf16 exactly, the row
# scale multiplies the logits in fp32 and the weights before their bf16
# rounding, so |out - oracle| <= 2^-8 * max |row_scale x e4m3(code)| over the
# selected rows' latents. lse: 2e-4 plus 2^-18 relative, since the logits are
# fp32 (a 576-term tensor-core sum, then two products) and the extreme row
# scales below make them reach thousands.
# ---------------------------------------------------------------------------

def _run8(B, q, cache8, row_scale, idx, cnt, cu_q, cu_k, scale, ws=None):
    dv = lambda a, dt=None: torch.from_numpy(np.ascontiguousarray(a if dt is None else a.view(dt))).cuda()
    out, lse = B.sparse_mla_fp8(dv(q, np.int16), dv(cache8), dv(row_scale), dv(idx), dv(cnt), dv(cu_q),
                                dv(cu_k), scale, ws=ws)
    return out.cpu().numpy(), lse.cpu().numpy()


def _check8(o_gpu, l_gpu, o_ref, l_ref, cache8, row_scale, idx, cnt, cu_q, cu_k, rows):
    for t in rows:
        b = int(np.searchsorted(cu_q, t, side="right")) - 1
        n = int(cnt[t])
        if n == 0:
            assert np.all(o_gpu[t] == 0) and np.all(np.isneginf(l_gpu[t])), f"row {t}"
            continue
        r = cu_k[b] + idx[t, :n]
        vmax = np.abs(row_scale[r].astype(np.float64)[:, None] * oracle.e4m3_to_f64(cache8[r, :512])).max()
        err = np.abs(o_gpu[t] - o_ref[t]).max()
        assert err <= 2.0 ** -8 * vmax, f"row {t}: |d out| {err} > {2.0 ** -8 * vmax}"
        np.testing.assert_allclose(l_gpu[t], l_ref[t], rtol=2.0 ** -18, atol=2e-4, err_msg=f"row {t}")


@pytest.mark.parametrize("heads", [32, 64, 96])
def test_mla_fp8_small_batches_against_oracle(B, heads):
    lens = [40, 3000, 2100, 5000]
    n_sel = [0, 1, 17, 33, 100, 2048, 2048, 1500]
    case = wl.mla_fp8_case(111 + heads, lens, q_per_seq=2, heads=heads,
                           n_sel=[min(s, l) for s, l in zip(n_sel, np.repeat(lens, 2))])
    q, cache8, rs, idx, cnt, cu_q, cu_k = case
    scale = 1.0 / np.sqrt(192.0)
    o, l = _run8(B, *case, scale)
    o_ref, l_ref = oracle.sparse_mla_fp8_batch(q, cache8, rs, idx, cnt, cu_q, cu_k, scale)
    _check8(o, l, o_ref, l_ref, cache8, rs, idx, cnt, cu_q, cu_k, range(q.shape[0]))


def test_mla_fp8_every_code_and_extreme_scales(B):
    """Every non-NaN code (zeros of both signs, subnormals, +-448) placed in
    every column over the selected rows, with row scales from 2^-20 to 2^6."""
    q, cache8, rs, idx, cnt, cu_q, cu_k = wl.mla_fp8_case(121, [700, 1200], q_per_seq=1, heads=64, topk=512)
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    L = cache8.shape[0]
    cache8 = codes[(np.arange(L)[:, None] * 7 + np.arange(576)[None, :] * 3) % codes.size]
    rs = np.exp2(np.random.default_rng(122).integers(-20, 7, size=L)).astype(np.float32)
    scale = 0.02
    o, l = _run8(B, q, cache8, rs, idx, cnt, cu_q, cu_k, scale)
    o_ref, l_ref = oracle.sparse_mla_fp8_batch(q, cache8, rs, idx, cnt, cu_q, cu_k, scale)
    _check8(o, l, o_ref, l_ref, cache8, rs, idx, cnt, cu_q, cu_k, range(q.shape[0]))


def test_mla_fp8_peaked_softmax_and_short_rows(B):
    """A large scale (the running maximum grows past 2^8 between tiles) and
    selections of 1 and 33 rows."""
    case = wl.mla_fp8_case(131, [4096, 2500, 1, 33], q_per_seq=1, heads=96)
    q, cache8, rs, idx, cnt, cu_q, cu_k = case
    for scale in (0.5, 2.0):
        o, l = _run8(B, *case, scale)
        o_ref, l_ref = oracle.sparse_mla_fp8_batch(q, cache8, rs, idx, cnt, cu_q, cu_k, scale)
        _check8(o, l, o_ref, l_ref, cache8, rs, idx, cnt, cu_q, cu_k, range(q.shape[0]))


def test_mla_fp8_positions_outside_the_sequence_are_left_out(B):
    q, cache8, rs, idx, cnt, cu_q, cu_k = wl.mla_fp8_case(141, [300, 400], q_per_seq=1, topk=64)
    idx[1, 5] = 400
    idx[1, 9] = -3
    ws = B.workspace(B.sparse_mla_workspace_size(2, 96, 64), "cuda")
    o, l = _run8(B, q, cache8, rs, idx, cnt, cu_q, cu_k, 0.1, ws=ws)
    assert B.get_status(ws) == (6, 1)
    keep = 300 + np.asarray([p for j, p in enumerate(idx[1, :cnt[1]]) if j not in (5, 9)])
    o_ref, l_ref = oracle.sparse_mla_fp8(q[1], cache8, rs, keep, 0.1)
    vmax = np.abs(rs[keep].astype(np.float64)[:, None] * oracle.e4m3_to_f64(cache8[keep, :512])).max()
    assert np.abs(o[1] - o_ref).max() <= 2.0 ** -8 * vmax
    np.testing.assert_allclose(l[1], l_ref, rtol=2.0 ** -18, atol=2e-4)


def test_mla_fp8_many_rows_single_split(B):
    case = wl.mla_fp8_case(151, [3000] * 40, q_per_seq=4, heads=32, topk=256)
    q, cache8, rs, idx, cnt, cu_q, cu_k = case
    scale = 1.0 / np.sqrt(192.0)
    o, l = _run8(B, *case, scale)
    rows = list(range(0, q.shape[0], 7)) + [q.shape[0] - 1]
    o_ref, l_ref = oracle.sparse_mla_fp8_batch(q, cache8, rs, idx, cnt, cu_q, cu_k, scale, rows=rows)
    _check8(o, l, o_ref, l_ref, cache8, rs, idx, cnt, cu_q, cu_k, rows)


def test_mla_fp8_decode_batch_full_size(B):
    """The decode batch's shapes over an FP8 cache; every row against the oracle."""
    lens = [8192, 12288, 16384, 24576, 32768, 40960, 49152, 65536]
    case = wl.mla_fp8_case(161, lens)
    q, cache8, rs, idx, cnt, cu_q, cu_k = case
    scale = 1.0 / np.sqrt(192.0)
    o, l = _run8(B, *case, scale)
    o_ref, l_ref = oracle.sparse_mla_fp8_batch(q, cache8, rs, idx, cnt, cu_q, cu_k, scale)
    _check8(o, l, o_ref, l_ref, cache8, rs, idx, cnt, cu_q, cu_k, range(q.shape[0]))


def test_mla_fp8_long_decode_full_size_sampled(B):
    """64 queries over 64K..128K-row histories in FP8 (a 3.5 GB cache made on
    the device from seeded random bytes), 2048 selected
    rows each, 96 heads, the launch bench.py --mla long_decode --fp8 times;
    three sampled queries against the oracle on their gathered rows."""
    dev = torch.device("cuda", 0)
    lens = np.random.default_rng(181).integers(65536, 131073, size=64).astype(np.int64)
    T, H, K = 64, 96, 2048
    gen = torch.Generator(device=dev).manual_seed(182)
    L = int(lens.sum())
    cache8 = torch.empty((L, 576), dtype=torch.uint8, device=dev)
    for r0 in range(0, L, 1 << 18):
        r1 = min(L, r0 + (1 << 18))
        blk = torch.randint(0, 1024, (r1 - r0, 576), generator=gen, device=dev, dtype=torch.int32)
        # keep magnitudes moderate: clear the top exponent bit of 3 codes in 4
        # (bits 8-9 choose), then move the NaN codes to 0
        blk = torch.where((blk & 0x300) != 0, blk & 0xBF, blk) & 0xFF
        blk = torch.where((blk & 0x7F) == 0x7F, torch.zeros_like(blk), blk)
        cache8[r0:r1] = blk.to(torch.uint8)
    rs = torch.exp2(torch.rand((L,), generator=gen, device=dev) * -3.0).float()
    q = torch.randn((T, H, 576), generator=gen, device=dev).to(torch.bfloat16)
    idx = torch.stack([torch.randperm(int(n), generator=gen, device=dev)[:K].sort().values
                       for n in lens]).to(torch.int32)
    cnt = torch.full((T,), K, dtype=torch.int32, device=dev)
    cu_k_h = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    cu_k = torch.from_numpy(cu_k_h).to(dev)
    cu_q = torch.arange(T + 1, dtype=torch.int32, device=dev)
    scale = 1.0 / np.sqrt(192.0)
    ws = B.workspace(B.sparse_mla_workspace_size(T, H, K), dev)
    out, lse = B.sparse_mla_fp8(q, cache8, rs, idx, cnt, cu_q, cu_k, scale, ws=ws)
    assert B.get_status(ws) == (0, 0)
    for t in (0, 31, 63):
        rows = int(cu_k_h[t]) + idx[t].long()
        sel8 = cache8[rows].cpu().numpy()
        sel_s = rs[rows].cpu().numpy()
        qt = q[t].view(torch.int16).cpu().numpy().view(np.uint16)
        o_ref, l_ref = oracle.sparse_mla_fp8(qt, sel8, sel_s, np.arange(K), scale)
        vmax = np.abs(sel_s.astype(np.float64)[:, None] * oracle.e4m3_to_f64(sel8[:, :512])).max()
        err = np.abs(out[t].cpu().numpy() - o_ref).max()
        assert err <= 2.0 ** -8 * vmax, f"row {t}: |d out| {err}"
        np.testing.assert_allclose(lse[t].cpu().numpy(), l_ref, rtol=2.0 ** -18, atol=2e-4,
                                   err_msg=f"row {t}")
