"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

Bars (from the indexer's statement of the problem):
  - integer-valued inputs (exact in fp32 in any summation order): indices and
    counts bit-exact, scores exactly equal;
  - real-valued inputs: every score within 1e-3 relative (+1e-6 x row max), and
    the GPU's and the oracle's index sets may differ only at positions whose
    oracle score is within 1e-3 of the oracle threshold; the GPU output must be
    the exact rule-ordered top-K of the GPU's own fp32 scores;
  - the stand-alone top-K on given fp32 rows: bit-exact (both sides decide on the
    same fp32 values);
  - LayerNorm: within 1 bf16 ulp of the fp64 oracle, or within the fp32
    evaluation bound 2^-17 * (|y - beta| + |beta|) where the output is near zero
    after cancellation (there a bf16 ulp is far below fp32's absolute error).
The stages are compared on identical inputs: a 1-ulp LayerNorm difference in one
key element moves a score by ~1e-3 relative, so the scoring of the decode batch
takes the oracle's post-LayerNorm keys on both sides, and the GPU-chained path is
checked for consistency with its own scores.
Full-size workloads are checked on every row against the oracle (run on all
host cores), plus quick variants on sampled rows.
"""
import os
import zlib

import numpy as np
import pytest

import oracle
from sparse_attention_key_gb300 import workloads as wl
from tests._util import (bf16_ulp_distance, bits_of, rule_order_ok, scores_close,
                         to_device, tolerance_set_check)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ORACLE_THREADS = max(os.cpu_count() or 1, 1)


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_attention_key_gb300 import build
    build.build()
    from sparse_attention_key_gb300 import binding
    return binding


_cache = {}


def workload(i):
    if i not in _cache:
        _cache[i] = wl.by_index(i)
    return _cache[i]


def gpu_scores(B, d, max_len):
    return B.score(d["q"], d["k"], d["w"], d["q_pos"], d["cu_q"], d["cu_k"], max_len)


def oracle_rows(w, rows, want_scores=True, K=2048, k_bits=None):
    return oracle.score_topk(w.q, w.k if k_bits is None else k_bits, w.w, w.q_pos, w.cu_q, w.cu_k,
                             K=K, rows=rows, want_scores=want_scores, threads=ORACLE_THREADS)


# ---------------------------------------------------------------------------
# LayerNorm
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("f32_params", [False, True])
def test_layernorm_cache_append(B, f32_params):
    # new keys normalised straight into their cache rows: the same values as
    # idx_key_layernorm (bit-identical) and within the oracle's tolerance;
    # padding (-1) and out-of-range slots write nothing; other rows untouched
    rng = np.random.default_rng(9 + f32_params)
    n_new, rows = 1000, 5000
    x = wl.f32_to_bf16_bits(rng.standard_normal((n_new, 128)).astype(np.float32) * 1.5 - 0.2)
    g = wl.f32_to_bf16_bits((1 + 0.1 * rng.standard_normal(128)).astype(np.float32))
    b = wl.f32_to_bf16_bits((0.1 * rng.standard_normal(128)).astype(np.float32))
    slot = rng.permutation(rows)[:n_new].astype(np.int64)
    slot[::97] = -1
    slot[5] = rows            # out of range: ignored
    slot[6] = -7
    if f32_params:
        gw = torch.from_numpy(wl.bf16_bits_to_f32(g)).cuda()
        gb = torch.from_numpy(wl.bf16_bits_to_f32(b)).cuda()
    else:
        gw, gb = torch.from_numpy(g.view(np.int16)).cuda(), torch.from_numpy(b.view(np.int16)).cuda()
    guard = np.int16(0x7FBF)  # a bf16 NaN pattern no LayerNorm output takes
    cache = torch.full((rows, 128), int(guard), dtype=torch.int16, device="cuda")
    xd = torch.from_numpy(x.view(np.int16)).cuda()
    B.key_layernorm_append(xd, gw, gb, 1e-6, cache, torch.from_numpy(slot).cuda())
    plain = bits_of(B.key_layernorm(xd, gw, gb, 1e-6))
    got = bits_of(cache)
    ok = (slot >= 0) & (slot < rows)
    assert np.array_equal(got[slot[ok]], plain[ok])
    untouched = np.ones(rows, bool)
    untouched[slot[ok]] = False
    assert (got[untouched] == np.uint16(guard)).all()
    ref = _ln_check(B, x[ok], g, b, 1e-6, f32_params=f32_params)
    assert np.array_equal(ref, plain[ok])


def _ln_check(B, k_raw_bits, ln_w_bits, ln_b_bits, eps, f32_params=False):
    dev = torch.from_numpy(k_raw_bits.view(np.int16)).cuda()
    if f32_params:
        gw = torch.from_numpy(wl.bf16_bits_to_f32(ln_w_bits)).cuda()
        gb = torch.from_numpy(wl.bf16_bits_to_f32(ln_b_bits)).cuda()
    else:
        gw = torch.from_numpy(ln_w_bits.view(np.int16)).cuda()
        gb = torch.from_numpy(ln_b_bits.view(np.int16)).cuda()
    out = bits_of(B.key_layernorm(dev, gw, gb, eps))
    beta = oracle.bf16_bits_to_f64(ln_b_bits)
    ref, y = oracle.key_layernorm(k_raw_bits, oracle.bf16_bits_to_f64(ln_w_bits), beta,
                                  float(np.float32(eps)))
    dist = bf16_ulp_distance(out, ref)
    err = np.abs(oracle.bf16_bits_to_f64(out) - y)
    fp32_bound = 2.0 ** -17 * (np.abs(y - beta[None, :]) + np.abs(beta[None, :]))
    bad = (dist > 1) & (err > fp32_bound)
    assert not bad.any(), f"{bad.sum()} outputs outside 1 ulp and the fp32 bound"
    assert (dist == 0).mean() > 0.99
    return out


def test_layernorm_tiny_exact_params(B):
    w = workload(1)
    _ln_check(B, w.k_raw, w.ln_w, w.ln_b, w.eps)


def test_layernorm_decode_batch_params(B):
    w = workload(2)
    _ln_check(B, w.k_raw, w.ln_w, w.ln_b, w.eps)


def test_layernorm_fp32_params_and_ragged_rows(B):
    rng = np.random.default_rng(7)
    x = wl.f32_to_bf16_bits(rng.standard_normal((1237, 128)).astype(np.float32) * 2 + 0.3)
    g = wl.f32_to_bf16_bits((1 + 0.1 * rng.standard_normal(128)).astype(np.float32))
    b = wl.f32_to_bf16_bits((0.1 * rng.standard_normal(128)).astype(np.float32))
    _ln_check(B, x, g, b, 1e-5, f32_params=True)


def test_layernorm_in_place(B):
    rng = np.random.default_rng(8)
    x = wl.f32_to_bf16_bits(rng.standard_normal((300, 128)).astype(np.float32))
    g = wl.f32_to_bf16_bits(np.ones(128, np.float32))
    b = wl.f32_to_bf16_bits(np.zeros(128, np.float32))
    d = torch.from_numpy(x.view(np.int16)).cuda()
    gw, gb = torch.from_numpy(g.view(np.int16)).cuda(), torch.from_numpy(b.view(np.int16)).cuda()
    expect = bits_of(B.key_layernorm(d.clone(), gw, gb, 1e-6))
    B.key_layernorm(d, gw, gb, 1e-6, out=d)
    assert np.array_equal(bits_of(d), expect)


# ---------------------------------------------------------------------------
# scores
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("kind", ["int2", "int4s3"])
def test_scores_exact_on_integer_inputs(B, kind):
    w = wl.custom(101, q_counts=[3, 130, 1, 0, 17], k_lens=[300, 700, 5000, 9, 129], kind=kind)
    d = to_device(w)
    S = gpu_scores(B, d, w.max_len).cpu().numpy()
    _, _, ref = oracle_rows(w, range(w.T))
    for t in range(w.T):
        n = int(w.q_pos[t]) + 1
        assert np.array_equal(S[t, :n].astype(np.float64), ref[t, :n]), t
        assert np.isnan(S[t, n:]).all(), "entries past the causal length must stay untouched"


def test_scores_real_inputs_within_tolerance(B):
    w = wl.custom(102, q_counts=[5, 64, 1], k_lens=[1000, 2300, 4097], kind="normal",
                  positions="random")
    d = to_device(w)
    S = gpu_scores(B, d, w.max_len).cpu().numpy()
    _, _, ref = oracle_rows(w, range(w.T))
    for t in range(w.T):
        n = int(w.q_pos[t]) + 1
        msg = scores_close(S[t, :n], ref[t, :n])
        assert msg is None, f"row {t}: {msg}"


# ---------------------------------------------------------------------------
# stand-alone top-K on given fp32 rows: bit-exact
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("kind", ["ties", "normal", "mixed", "const", "tiny"])
@pytest.mark.parametrize("K", [1, 7, 2048])
@pytest.mark.parametrize("lens", ["short", "mid", "wide", "long", "cap", "over_cap"])
def test_topk_bit_exact_on_synthetic_rows(B, kind, K, lens):
    rng = np.random.default_rng(zlib.crc32(f"{kind}/{K}/{lens}".encode()))
    if lens == "short":
        n_valid = np.concatenate([[0, 1, K - 1 if K > 1 else 0, K, K + 1, 2047, 2048, 2049, 4096],
                                  rng.integers(1, 20000, size=20), [50_000]]).astype(np.int32)
    elif lens == "mid":   # many rows of 16K..30K positions: the streamed kernel
        n_valid = rng.integers(16_000, 30_001, size=400).astype(np.int32)
        # around the candidate list's capacity (8192): const rows are all candidates
        n_valid[:10] = [30_000, 16_385, K + 1, 2047, 2048, 2051, 8191, 8192, 8195, 12_289]
        n_valid[:10] = np.maximum(n_valid[:10], K + 1)
    elif lens == "wide":  # many rows of 40K..53K positions (the agentic chunk's row lengths)
        n_valid = rng.integers(40_000, 53_001, size=200).astype(np.int32)
        n_valid[:8] = [53_000, 52_999, 12_289, K + 1, 2048, 2047, 49_999, 1]
    elif lens == "long":   # few long rows
        n_valid = np.array([70_000, 131_072, 65_537, K + 3, 100_001], np.int32)
        if kind in ("normal", "ties"):
            n_valid = np.append(n_valid, np.int32(700_001))
    elif lens == "cap":   # few rows up to exactly 2^21 positions: one cluster per row
        n_valid = np.array([2_097_152, 12_289, K + 1, 262_145, 131_071], np.int32)
    else:                 # one position beyond it: the slice-parallel kernels
        n_valid = np.array([2_097_153, 12_289, 40_000], np.int32)
    max_len = int(n_valid.max())
    ld = (max_len + 3) // 4 * 4
    S = wl.score_rows(int(rng.integers(1 << 30)), n_valid.size, n_valid, ld, kind=kind)
    dS = torch.from_numpy(S).cuda()
    idx, cnt = B.topk(dS, torch.from_numpy(n_valid).cuda(), max_len, K)
    idx, cnt = idx.cpu().numpy(), cnt.cpu().numpy()
    for t, n in enumerate(n_valid):
        ref = oracle.select(S[t, :n].astype(np.float64), K)
        assert np.array_equal(idx[t], ref), f"row {t} (n={n})"
        assert cnt[t] == min(n, K)


# ---------------------------------------------------------------------------
# projections (q-LoRA -> q, attention input -> key LayerNorm -> cache, -> w)
# ---------------------------------------------------------------------------

def _proj_inputs(seed, T, hidden, rank, integer):
    rng = np.random.default_rng(seed)
    if integer:
        mk = lambda shape, lo, hi: wl.f32_to_bf16_bits(rng.integers(lo, hi + 1, size=shape).astype(np.float32))
        x, ql = mk((T, hidden), -2, 2), mk((T, rank), -2, 2)
        wq, wk, ww = mk((4096, rank), -1, 1), mk((128, hidden), -1, 1), mk((32, hidden), -1, 1)
    else:
        mk = lambda shape, s: wl.f32_to_bf16_bits((rng.standard_normal(shape) * s).astype(np.float32))
        x, ql = mk((T, hidden), 1.0), mk((T, rank), 1.0)
        wq, wk, ww = mk((4096, rank), rank ** -0.5), mk((128, hidden), hidden ** -0.5), mk((32, hidden), 0.01)
    g = wl.f32_to_bf16_bits((1 + 0.1 * rng.standard_normal(128)).astype(np.float32))
    b = wl.f32_to_bf16_bits((0.1 * rng.standard_normal(128)).astype(np.float32))
    return x, ql, wq, wk, ww, g, b


def _proj_run(B, x, ql, wq, wk, ww, g, b, cache_rows, slot):
    dv = lambda a: torch.from_numpy(a.view(np.int16)).cuda()
    cache = torch.zeros((cache_rows, 128), dtype=torch.int16, device="cuda")
    q, w = B.indexer_project(dv(x), dv(ql), dv(wq), dv(wk), dv(ww), dv(g), dv(b), 1e-6, cache,
                             torch.from_numpy(slot).cuda())
    return bits_of(q), w.cpu().numpy(), bits_of(cache)


def test_indexer_project_integer_inputs_exact(B):
    T, hidden, rank = 37, 7168, 1536
    x, ql, wq, wk, ww, g, b = _proj_inputs(41, T, hidden, rank, integer=True)
    slot = np.random.default_rng(1).permutation(100)[:T].astype(np.int64)
    q, w, cache = _proj_run(B, x, ql, wq, wk, ww, g, b, 100, slot)
    rq, rk, rw, rk_pre = oracle.indexer_project(x, ql, wq, wk, ww, oracle.bf16_bits_to_f64(g),
                                                oracle.bf16_bits_to_f64(b), float(np.float32(1e-6)))
    assert np.array_equal(q, rq)                    # exact integers, rounded once to bf16
    assert np.array_equal(w, rw.astype(np.float32))
    # identical pre-LayerNorm keys on both sides: the key LayerNorm's tolerance
    beta = oracle.bf16_bits_to_f64(b)
    _, y = oracle.key_layernorm(rk_pre, oracle.bf16_bits_to_f64(g), beta, float(np.float32(1e-6)))
    got = cache[slot]
    dist = bf16_ulp_distance(got, rk)
    err = np.abs(oracle.bf16_bits_to_f64(got) - y)
    bound = 2.0 ** -17 * (np.abs(y - beta[None, :]) + np.abs(beta[None, :]))
    assert not ((dist > 1) & (err > bound)).any()
    untouched = np.setdiff1d(np.arange(100), slot)
    assert (cache[untouched] == 0).all()


def _proj_check_exact(B, seed, T, hidden, rank, cache_rows):
    x, ql, wq, wk, ww, g, b = _proj_inputs(seed, T, hidden, rank, integer=True)
    slot = np.random.default_rng(seed).permutation(cache_rows)[:T].astype(np.int64)
    q, w, cache = _proj_run(B, x, ql, wq, wk, ww, g, b, cache_rows, slot)
    rq, rk, rw, rk_pre = oracle.indexer_project(x, ql, wq, wk, ww, oracle.bf16_bits_to_f64(g),
                                                oracle.bf16_bits_to_f64(b), float(np.float32(1e-6)))
    assert np.array_equal(q, rq)
    assert np.array_equal(w, rw.astype(np.float32))
    beta = oracle.bf16_bits_to_f64(b)
    _, y = oracle.key_layernorm(rk_pre, oracle.bf16_bits_to_f64(g), beta, float(np.float32(1e-6)))
    got = cache[slot]
    dist = bf16_ulp_distance(got, rk)
    err = np.abs(oracle.bf16_bits_to_f64(got) - y)
    bound = 2.0 ** -17 * (np.abs(y - beta[None, :]) + np.abs(beta[None, :]))
    assert not ((dist > 1) & (err > bound)).any()


def test_indexer_project_many_tokens_exact(B):
    # 1,300 tokens: 11 row tiles (6 pairs, the last with a tile past the end)
    # x 16 column tiles of q, enough work without splitting K (bf16 written
    # straight from the accumulators); the key/weight product splits K.
    # Integer inputs: exact.
    _proj_check_exact(B, 43, 1300, 7168, 1536, 1400)


def test_indexer_project_ragged_k_and_rows_exact(B):
    # hidden and q_rank not multiples of the 64-wide K block (the last block
    # reads zeros past the matrix), and a second row tile with 2 valid rows
    _proj_check_exact(B, 44, 130, 1000, 520, 200)


def test_indexer_project_real_valued(B):
    T, hidden, rank = 64, 1024, 512
    x, ql, wq, wk, ww, g, b = _proj_inputs(42, T, hidden, rank, integer=False)
    slot = np.arange(T, dtype=np.int64)
    q, w, cache = _proj_run(B, x, ql, wq, wk, ww, g, b, T, slot)
    rq, rk, rw, _ = oracle.indexer_project(x, ql, wq, wk, ww, oracle.bf16_bits_to_f64(g),
                                           oracle.bf16_bits_to_f64(b), float(np.float32(1e-6)))
    # one bf16 rounding of an fp32-accumulated sum: 1 ulp, or the fp32
    # accumulation bound where the sum cancels (sum of |products| x 2^-20)
    dist = bf16_ulp_distance(q, rq)
    err = np.abs(oracle.bf16_bits_to_f64(q) - oracle.bf16_bits_to_f64(rq)).reshape(T, -1)
    mag = np.abs(oracle.bf16_bits_to_f64(ql)) @ np.abs(oracle.bf16_bits_to_f64(wq)).T
    assert not ((dist.reshape(T, -1) > 1) & (err > 2.0 ** -20 * mag + 2.0 ** -9 * np.abs(
        oracle.bf16_bits_to_f64(rq).reshape(T, -1)))).any()
    assert (dist <= 1).mean() > 0.999
    assert np.allclose(w, rw, rtol=1e-5, atol=1e-6)
    # a one-ulp flip of a pre-LayerNorm key can move its row's outputs by ~2 ulps
    d = np.abs(oracle.bf16_bits_to_f64(cache) - oracle.bf16_bits_to_f64(rk))
    assert (d <= 2.0 ** -6 * np.maximum(np.abs(oracle.bf16_bits_to_f64(rk)), 1.0)).all()
    assert (cache == rk).mean() > 0.95


# ---------------------------------------------------------------------------
# the whole indexer
# ---------------------------------------------------------------------------

def _check_exact(B, w, rows=None, K=2048):
    d = to_device(w)
    idx, cnt = B.score_topk(d["q"], d["k"], d["w"], d["q_pos"], d["cu_q"], d["cu_k"], w.max_len, K)
    idx, cnt = idx.cpu().numpy(), cnt.cpu().numpy()
    rows = list(range(w.T)) if rows is None else rows
    ridx, rcnt, _ = oracle_rows(w, rows, want_scores=False, K=K)
    for t in rows:
        assert np.array_equal(idx[t], ridx[t]), f"row {t}"
        assert cnt[t] == rcnt[t]
    return idx, cnt


def test_indexer_tiny_exact_all_rows(B):
    w = workload(1)
    idx, cnt = _check_exact(B, w)
    assert cnt.tolist() == [101, 2048, 2048, 2048, 2048, 2048, 2048, 2048]


def test_indexer_small_ragged_prefill_ties_all_rows(B):
    w = wl.custom(103, q_counts=[300, 45, 1], k_lens=[3000, 2049, 2050], kind="int2")
    _check_exact(B, w)


@pytest.mark.parametrize("K", [1, 16, 333])
def test_indexer_small_topk_values(B, K):
    w = wl.custom(104, q_counts=[40, 7], k_lens=[500, 390], kind="int4s3", positions="random",
                  topk=K)
    _check_exact(B, w, K=K)


def test_indexer_prefill_ties_full_size_sampled(B):
    w = workload(3)
    rows = [0, 1, 127, 128, 2046, 2047, 2048, 2049, 4095, 5000, 6143, 8190, 8191]
    _check_exact(B, w, rows=rows)


def test_indexer_prefill_ties_full_size_all_rows(B):
    # every one of the 8,192 rows bit-exact, tie order included (integer inputs)
    w = workload(3)
    d = to_device(w)
    idx, cnt = B.score_topk(d["q"], d["k"], d["w"], d["q_pos"], d["cu_q"], d["cu_k"], w.max_len)
    ridx, rcnt, _ = oracle_rows(w, None, want_scores=False)
    got_idx, got_cnt = idx.cpu().numpy(), cnt.cpu().numpy()
    bad = np.flatnonzero((got_idx != ridx).any(axis=1) | (got_cnt != rcnt))
    assert bad.size == 0, f"{bad.size} rows differ, first {bad[:8].tolist()}"


def _check_tolerance(B, w, rows, d=None, k_oracle=None):
    d = to_device(w) if d is None else d
    idx, cnt = B.score_topk(d["q"], d["k"], d["w"], d["q_pos"], d["cu_q"], d["cu_k"], w.max_len)
    S = gpu_scores(B, d, w.max_len)
    idx, cnt = idx.cpu().numpy(), cnt.cpu().numpy()
    ridx, rcnt, rS = oracle_rows(w, rows, k_bits=k_oracle)
    for t in rows:
        n = int(w.q_pos[t]) + 1
        S_gpu = S[t, :n].cpu().numpy()
        assert cnt[t] == rcnt[t] == min(n, 2048)
        msg = scores_close(S_gpu, rS[t, :n])
        assert msg is None, f"row {t}: {msg}"
        msg = tolerance_set_check(rS[t, :n], idx[t], ridx[t], 2048)
        assert msg is None, f"row {t}: {msg}"
        msg = rule_order_ok(S_gpu, idx[t], 2048)
        assert msg is None, f"row {t}: {msg}"


def test_indexer_decode_batch(B):
    w = workload(2)
    k_ref, _ = oracle.key_layernorm(w.k_raw, oracle.bf16_bits_to_f64(w.ln_w),
                                    oracle.bf16_bits_to_f64(w.ln_b), float(np.float32(w.eps)))
    d = to_device(w)
    d["k"] = torch.from_numpy(k_ref.view(np.int16)).cuda()   # identical keys on both sides
    _check_tolerance(B, w, rows=list(range(w.T)), d=d, k_oracle=k_ref)


def test_indexer_decode_batch_gpu_chained_is_self_consistent(B):
    w = workload(2)
    d = to_device(w)
    d["k"] = B.key_layernorm(d["k_raw"], d["ln_w"], d["ln_b"], w.eps)
    idx, cnt = B.score_topk(d["q"], d["k"], d["w"], d["q_pos"], d["cu_q"], d["cu_k"], w.max_len)
    S = gpu_scores(B, d, w.max_len).cpu().numpy()
    idx = idx.cpu().numpy()
    for t in range(w.T):
        n = int(w.q_pos[t]) + 1
        assert rule_order_ok(S[t, :n], idx[t], 2048) is None, t


def test_indexer_agentic_chunk_sampled(B):
    w = workload(4)
    rows = [0, 1, 399, 799, 800, 1600, 2401, 3199]
    _check_tolerance(B, w, rows)


def test_indexer_agentic_chunk_all_rows(B):
    # all 3,200 rows: scores within tolerance, sets within the threshold rule,
    # and the GPU output the rule-ordered top-K of its own scores
    w = workload(4)
    _check_tolerance(B, w, list(range(w.T)))


def test_indexer_long_decode_all_rows(B):
    w = workload(5)
    _check_tolerance(B, w, list(range(w.T)))


def test_indexer_spec_verify_all_rows(B):
    w = workload(6)
    _check_tolerance(B, w, list(range(w.T)))


def test_indexer_long_decode_sampled(B):
    w = workload(5)
    rows = [0, 7, 31, 32, 50, 63]
    _check_tolerance(B, w, rows)
    # every row: the GPU output is the rule-ordered top-K of the GPU's own scores
    d = to_device(w)
    idx, _ = B.score_topk(d["q"], d["k"], d["w"], d["q_pos"], d["cu_q"], d["cu_k"], w.max_len)
    S = gpu_scores(B, d, w.max_len).cpu().numpy()
    idx = idx.cpu().numpy()
    for t in range(w.T):
        n = int(w.q_pos[t]) + 1
        assert rule_order_ok(S[t, :n], idx[t], 2048) is None, t


def test_indexer_spec_verify_sampled(B):
    w = workload(6)
    rows = [0, 3, 4, 29, 30, 63]
    _check_tolerance(B, w, rows)
    d = to_device(w)
    idx, _ = B.score_topk(d["q"], d["k"], d["w"], d["q_pos"], d["cu_q"], d["cu_k"], w.max_len)
    S = gpu_scores(B, d, w.max_len).cpu().numpy()
    idx = idx.cpu().numpy()
    for t in range(w.T):
        n = int(w.q_pos[t]) + 1
        assert rule_order_ok(S[t, :n], idx[t], 2048) is None, t


# ---------------------------------------------------------------------------
# edge cases and errors
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("L", [1, 2, 127, 128, 129, 2047, 2048, 2049, 2050])
def test_indexer_history_lengths_around_tiles_and_budget(B, L):
    w = wl.custom(200 + L, q_counts=[min(L, 3)], k_lens=[L], kind="int2")
    _check_exact(B, w)


def test_indexer_few_chunk_queries_with_long_histories(B):
    # many queries per sequence (tensor-core prefill tiles) but few rows in all:
    # the few-rows selection path, with its own histogram pass
    w = wl.custom(401, q_counts=[60, 40], k_lens=[20000, 15000], kind="int2")
    _check_exact(B, w)


def test_indexer_spec_verify_shapes_exact(B):
    # a few queries per sequence (the speculative-verification configuration,
    # 4 queries per tensor-core group), one history long enough for the
    # cluster selection; integer inputs: bit-exact
    w = wl.custom(404, q_counts=[4, 4, 3, 4, 1], k_lens=[20000, 3000, 9000, 130, 2100], kind="int2")
    assert w.B < w.T <= 4 * w.B
    _check_exact(B, w)


def test_indexer_many_rows_long_histories_integer_ties_exact(B):
    # more than 128 rows of more than 32,768 keys: the streamed selection reads
    # the scorer's segment maxima; with integer inputs the tie groups at the
    # bound overflow its candidate list on some rows (general path) and not on
    # others. Bit-exact.
    w = wl.custom(405, q_counts=[140, 20], k_lens=[40000, 33000], kind="int2")
    _check_exact(B, w)


@pytest.mark.parametrize("kind", ["int4s3", "int2"])
def test_indexer_many_rows_mixed_lengths_exact(B, kind):
    # random query positions: rows that keep everything, rows too short for
    # the segment bound (fewer than 2,048 segments of 16) and rows that use it,
    # in one call
    w = wl.custom(406, q_counts=[100, 60], k_lens=[60000, 34000], kind=kind, positions="random")
    _check_exact(B, w)


def test_indexer_many_rows_long_histories_real_values(B):
    w = wl.custom(407, q_counts=[90, 50], k_lens=[45000, 70000], kind="normal")
    _check_tolerance(B, w, list(range(w.T)))


def _stealing_batch(seed, per_seq, kind, positions):
    # 30 sequences of 1..60K keys: more than 32 key tiles of cache per SM, so
    # the decode (1 query per sequence) and verification (4) scorers share
    # their work between CTAs
    rng = np.random.default_rng(seed)
    k_lens = rng.integers(per_seq, 60_001, size=30).tolist()
    k_lens[:3] = [60_000, per_seq, 2049]
    w = wl.custom(seed, q_counts=[per_seq] * 30, k_lens=k_lens, kind=kind, positions=positions)
    assert int(w.cu_k[-1]) // 128 >= 32 * 152
    return w


@pytest.mark.parametrize("per_seq", [1, 4])
def test_indexer_work_stealing_scorers_integer_ties_exact(B, per_seq):
    _check_exact(B, _stealing_batch(411 + per_seq, per_seq, "int2", "random"))


@pytest.mark.parametrize("per_seq", [1, 4])
def test_indexer_work_stealing_scorers_real_values_all_rows(B, per_seq):
    w = _stealing_batch(421 + per_seq, per_seq, "normal", "chunk")
    _check_tolerance(B, w, list(range(w.T)))


def test_indexer_decode_integer_ties_long_histories(B):
    # one query per sequence (the scorer histograms the first digit itself) on
    # integer inputs: tie groups far larger than the selection's candidate list
    w = wl.custom(402, q_counts=[1, 1, 1, 1], k_lens=[40000, 13000, 30000, 12289], kind="int2")
    _check_exact(B, w)


def test_indexer_many_sequences(B):
    # more sequences than the fast plan kernel takes (2048): the general plan,
    # one query per sequence, some sequences without queries
    rng = np.random.default_rng(403)
    k_lens = rng.integers(1, 600, size=2100)
    q_counts = np.where(rng.random(2100) < 0.1, 0, 1)
    w = wl.custom(403, q_counts=q_counts, k_lens=k_lens, kind="int2")
    _check_exact(B, w)


def test_indexer_batch_with_empty_sequences(B):
    w = wl.custom(301, q_counts=[0, 4, 0, 2, 0], k_lens=[0, 2500, 10, 3000, 0], kind="int2")
    _check_exact(B, w)


def test_indexer_zero_queries(B):
    w = wl.custom(302, q_counts=[0], k_lens=[100], kind="int2")
    d = to_device(w)
    idx, cnt = B.score_topk(d["q"], d["k"], d["w"], d["q_pos"], d["cu_q"], d["cu_k"], 100)
    torch.cuda.synchronize()
    assert idx.shape == (0, 2048) and cnt.shape == (0,)


def test_indexer_output_guard_bands_untouched(B):
    w = wl.custom(303, q_counts=[20], k_lens=[4000], kind="int2")
    d = to_device(w)
    guard = 4096
    buf = torch.full((w.T * 2048 + 2 * guard,), -7, dtype=torch.int32, device="cuda")
    cbuf = torch.full((w.T + 2 * 64,), -7, dtype=torch.int32, device="cuda")
    idx = buf[guard:guard + w.T * 2048].view(w.T, 2048)
    cnt = cbuf[64:64 + w.T]
    B.score_topk(d["q"], d["k"], d["w"], d["q_pos"], d["cu_q"], d["cu_k"], w.max_len, idx=idx,
                 cnt=cnt)
    b = buf.cpu().numpy()
    c = cbuf.cpu().numpy()
    assert (b[:guard] == -7).all() and (b[-guard:] == -7).all()
    assert (c[:64] == -7).all() and (c[-64:] == -7).all()
    ridx, _, _ = oracle_rows(w, range(w.T), want_scores=False)
    assert np.array_equal(idx.cpu().numpy(), ridx)


def test_device_argument_error_is_reported_and_row_skipped(B):
    w = wl.custom(304, q_counts=[3], k_lens=[3000], kind="int2")
    bad = w.q_pos.copy()
    bad[1] = 3000                                   # == len_k: outside the sequence
    d = to_device(w)
    d["q_pos"] = torch.from_numpy(bad).cuda()
    ws = B.workspace(B.score_topk_workspace_size(1, 3, 3001), "cuda")
    idx, cnt = B.score_topk(d["q"], d["k"], d["w"], d["q_pos"], d["cu_q"], d["cu_k"], 3001, ws=ws)
    code, detail = B.get_status(ws)
    assert code == 6 and detail == 1
    ridx, _, _ = oracle_rows(w, [0, 2], want_scores=False)
    got = idx.cpu().numpy()
    assert np.array_equal(got[0], ridx[0]) and np.array_equal(got[2], ridx[2])
    # a later good call on the same workspace clears the status
    d["q_pos"] = torch.from_numpy(w.q_pos).cuda()
    B.score_topk(d["q"], d["k"], d["w"], d["q_pos"], d["cu_q"], d["cu_k"], 3001, ws=ws)
    assert B.get_status(ws) == (0, 0)


def test_host_argument_errors_raise(B):
    w = wl.custom(305, q_counts=[2], k_lens=[100], kind="int2")
    d = to_device(w)
    with pytest.raises(B.IndexerError) as e:
        B.score_topk(d["q"], d["k"], d["w"], d["q_pos"], d["cu_q"], d["cu_k"], 100, topk=4096)
    assert e.value.code == 1
    ws = B.workspace(256, "cuda")
    with pytest.raises(B.IndexerError) as e:
        B.score_topk(d["q"], d["k"], d["w"], d["q_pos"], d["cu_q"], d["cu_k"], 100, ws=ws)
    assert e.value.code == 3
