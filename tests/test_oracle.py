"""Pins for the CPU oracle (no GPU).

Each test checks the oracle against something other than itself: values fixed
by the page's rule (hand-derived golden cases), brute force over all subsets,
closed forms, special cases that reduce to a library routine (numpy/torch
float64), and invariants. Method source: "Notes from an NVFP4 port of Kimi
K3.1 Pro" (indexer paragraph; item (4) of "Details that silently change the
answer"; the closing paragraph on dormant selection).
"""
import itertools
import os

import numpy as np
import pytest

import oracle
from sparse_attention_key_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tie_rule_cases.txt")


def _golden_cases():
    cases = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, s, e = (p.strip() for p in line.split("|"))
            cases.append((int(k), [float(x) for x in s.split()], [int(x) for x in e.split()]))
    return cases


# ---------------------------------------------------------------------------
# select: the tie / order rule
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("K,scores,expected", _golden_cases())
def test_select_golden_tie_rule(K, scores, expected):
    got = oracle.select(np.array(scores), K)
    assert got.tolist() == expected


def _rule_order(S, sel):
    """The page's output order for a selected set: above-threshold ascending, then the tie group."""
    tau = min(S[a] for a in sel)
    return sorted(a for a in sel if S[a] > tau) + sorted(a for a in sel if S[a] == tau)


def test_select_brute_force_all_subsets():
    rng = np.random.default_rng(11)
    checked = 0
    for n in range(2, 10):
        for K in range(1, n):
            for _ in range(6):
                S = rng.integers(0, 4, size=n).astype(np.float64)  # heavy ties
                valid = []
                for sel in itertools.combinations(range(n), K):
                    ss = set(sel)
                    ok = all(S[a] > S[b] or (S[a] == S[b] and a < b)
                             for a in ss for b in range(n) if b not in ss)
                    if ok:
                        valid.append(sel)
                assert len(valid) == 1, "the defining property must give a unique set"
                got = oracle.select(S, K)
                assert sorted(got.tolist()) == list(valid[0])
                assert got.tolist() == _rule_order(S, valid[0])
                checked += 1
    assert checked > 100


def test_select_keep_all_when_history_fits():
    rng = np.random.default_rng(12)
    for n in (1, 5, 2047, 2048):
        S = rng.standard_normal(n)
        got = oracle.select(S, 2048)
        assert got[:n].tolist() == list(range(n))
        assert (got[n:] == -1).all()


def test_select_empty_row():
    got = oracle.select(np.zeros(0), 4)
    assert got.tolist() == [-1, -1, -1, -1]


def test_select_all_equal_keeps_lowest_positions():
    for n in (2049, 5000):
        got = oracle.select(np.full(n, 0.75), 2048)
        assert got.tolist() == list(range(2048))


def test_select_distinct_scores_against_library_sort():
    rng = np.random.default_rng(13)
    for n, K in ((3000, 2048), (10000, 2048), (50, 7)):
        S = rng.permutation(n).astype(np.float64) * 0.5 - 100.0  # distinct
        order = np.argsort(-S, kind="stable")
        top = order[:K]
        # distinct scores: all but the K-th are above tau (ascending), then the K-th
        expected = sorted(top[:K - 1].tolist()) + [int(top[K - 1])]
        assert oracle.select(S, K).tolist() == expected


def test_select_signed_zero_compares_equal():
    S = np.array([0.0, -0.0, -0.0, 0.0, 1.0])
    assert oracle.select(S, 3).tolist() == [4, 0, 1]
    S2 = np.array([-0.0, 0.0, 0.0])
    assert oracle.select(S2, 2).tolist() == [0, 1]


def test_select_invariants_random_rows():
    rng = np.random.default_rng(14)
    for trial in range(20):
        n = int(rng.integers(2049, 9000))
        kind = trial % 3
        if kind == 0:
            S = rng.integers(0, 8, size=n).astype(np.float64)
        elif kind == 1:
            S = rng.standard_normal(n)
        else:
            S = np.maximum(rng.standard_normal(n), 0.0)
        got = oracle.select(S, 2048)
        assert got.size == 2048 and (got >= 0).all() and (got < n).all()
        assert len(set(got.tolist())) == 2048
        tau = S[got].min()
        above = [a for a in got.tolist() if S[a] > tau]
        ties = [a for a in got.tolist() if S[a] == tau]
        assert got.tolist() == above + ties
        assert above == sorted(above) and ties == sorted(ties)
        assert len(above) == int((S > tau).sum())       # every above-tau key kept
        tie_all = np.flatnonzero(S == tau)
        assert ties == tie_all[:len(ties)].tolist()     # lowest positions of the tie group


# ---------------------------------------------------------------------------
# scores: relu(q_h . k), head-weighted sum, causal history
# ---------------------------------------------------------------------------

def _rand_qk(rng, n):
    k = wl.f32_to_bf16_bits(rng.standard_normal((n, 128), dtype=np.float32))
    q = wl.f32_to_bf16_bits(rng.standard_normal((32, 128), dtype=np.float32))
    return q, k


def test_scores_single_head_is_relu_of_a_gemm():
    rng = np.random.default_rng(21)
    q, k = _rand_qk(rng, 300)
    qf = oracle.bf16_bits_to_f64(q)
    kf = oracle.bf16_bits_to_f64(k)
    for h in (0, 7, 31):
        w = np.zeros(32, np.float32)
        w[h] = 1.0
        got = oracle.scores(q, k, w, 300)
        ref = np.maximum(kf @ qf[h], 0.0)            # library GEMV, float64
        assert (ref == 0).sum() > 50                  # the relu is exercised
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_scores_linear_in_head_weights():
    """S(w) = sum_h w_h S(e_h), for weights of either sign (relu before the weight)."""
    rng = np.random.default_rng(22)
    q, k = _rand_qk(rng, 200)
    basis = []
    for h in range(32):
        e = np.zeros(32, np.float32)
        e[h] = 1.0
        basis.append(oracle.scores(q, k, e, 200))
    basis = np.stack(basis)
    w = rng.uniform(-1, 1, size=32).astype(np.float32)
    got = oracle.scores(q, k, w, 200)
    ref = w.astype(np.float64) @ basis
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_scores_integer_inputs_are_exact_integers():
    rng = np.random.default_rng(23)
    k = wl.f32_to_bf16_bits(rng.integers(-2, 3, (64, 128)).astype(np.float32))
    q = wl.f32_to_bf16_bits(rng.integers(-2, 3, (32, 128)).astype(np.float32))
    w = rng.integers(0, 2, 32).astype(np.float32)
    got = oracle.scores(q, k, w, 64)
    assert np.array_equal(got, np.round(got))
    qi = oracle.bf16_bits_to_f64(q).astype(np.int64)
    ki = oracle.bf16_bits_to_f64(k).astype(np.int64)
    ref = (np.maximum(ki @ qi.T, 0) * w.astype(np.int64)).sum(axis=1)   # integer GEMM
    assert np.array_equal(got, ref.astype(np.float64))


def test_causal_history_is_inclusive_and_bounded():
    """A query at position p scores keys 0..p and nothing after."""
    rng = np.random.default_rng(24)
    L = 40
    k = wl.f32_to_bf16_bits(rng.integers(-1, 2, (L, 128)).astype(np.float32) * 0.0)
    q = np.zeros((3, 32, 128), np.uint16)
    one = wl.f32_to_bf16_bits(np.ones(1, np.float32))[0]
    q[:, 0, 0] = one                                   # head 0 reads feature 0
    k = k.copy()
    for s in (9, 10, 30):                              # keys with a large feature 0
        k[s, 0] = wl.f32_to_bf16_bits(np.array([5.0], np.float32))[0]
    w = np.zeros((3, 32), np.float32)
    w[:, 0] = 1.0
    q_pos = np.array([9, 29, 39], np.int32)
    idx, cnt, sc = oracle.score_topk(q, k, w, q_pos, [0, 3], [0, L], K=1, want_scores=True)
    # query at 9 sees key 9 (inclusive) -> picks it; at 29 the earliest max is 9; at 39 too
    assert idx[:, 0].tolist() == [9, 9, 9]
    assert cnt.tolist() == [1, 1, 1]
    assert np.isfinite(sc[0, :10]).all() and np.isnan(sc[0, 10:]).all()
    assert np.isfinite(sc[1, :30]).all() and np.isnan(sc[1, 30:]).all()
    # K=2: the query at 9 cannot see key 10 or 30 (future) -> tie group of zeros fills in at 0
    idx2, _, _ = oracle.score_topk(q, k, w, q_pos, [0, 3], [0, L], K=2)
    assert idx2[0].tolist() == [9, 0]
    assert idx2[1].tolist() == [9, 10]
    assert idx2[2].tolist() == [9, 10]


def test_keep_all_boundary_2047_vs_2048():
    """Positions 2047 and 2048 straddle the 2048-key budget (keep-all vs drop-one)."""
    rng = np.random.default_rng(25)
    L = 2100
    k = wl.f32_to_bf16_bits(rng.integers(-2, 3, (L, 128)).astype(np.float32))
    q = wl.f32_to_bf16_bits(rng.integers(-2, 3, (2, 32, 128)).astype(np.float32))
    w = np.ones((2, 32), np.float32)
    idx, cnt, sc = oracle.score_topk(q, k, w, np.array([2047, 2048], np.int32), [0, 2], [0, L],
                                     want_scores=True)
    assert idx[0].tolist() == list(range(2048)) and cnt[0] == 2048
    S = sc[1, :2049]
    assert cnt[1] == 2048
    dropped = set(range(2049)) - set(idx[1].tolist())
    assert len(dropped) == 1
    d = dropped.pop()
    # the dropped key is the lowest-scoring one, and the highest position among those lowest
    assert S[d] == S.min() and d == int(np.flatnonzero(S == S.min()).max())


def test_ragged_batch_against_independent_numpy_restatement():
    """A small ragged batch against numpy float64 matmuls + a library lexsort selection.

    Not a pin on its own (it restates the definition); it checks the packed-batch
    indexing (cu_q / cu_k offsets, per-sequence local positions) end to end.
    """
    w_ = wl.custom(31, q_counts=[3, 0, 5, 2], k_lens=[40, 7, 90, 33], kind="int2",
                   positions="random", topk=16)
    idx, cnt, _ = oracle.score_topk(w_.q, w_.k, w_.w, w_.q_pos, w_.cu_q, w_.cu_k, K=16)
    kf = oracle.bf16_bits_to_f64(w_.k)
    qf = oracle.bf16_bits_to_f64(w_.q)
    for b in range(w_.B):
        for t in range(w_.cu_q[b], w_.cu_q[b + 1]):
            n = int(w_.q_pos[t]) + 1
            keys = kf[w_.cu_k[b]:w_.cu_k[b] + n]
            S = (np.maximum(keys @ qf[t].T, 0.0) * w_.w[t].astype(np.float64)).sum(axis=1)
            if n <= 16:
                exp = list(range(n)) + [-1] * (16 - n)
            else:
                order = np.lexsort((np.arange(n), -S))[:16]
                exp = _rule_order(S, set(order.tolist()))
            assert idx[t].tolist() == exp
            assert cnt[t] == min(n, 16)


def test_out_of_range_position_is_rejected():
    w_ = wl.custom(32, q_counts=[1], k_lens=[10], kind="int2")
    bad = w_.q_pos.copy()
    bad[0] = 10
    with pytest.raises(ValueError):
        oracle.score_topk(w_.q, w_.k, w_.w, bad, w_.cu_q, w_.cu_k, K=4)


# ---------------------------------------------------------------------------
# LayerNorm and bf16 rounding
# ---------------------------------------------------------------------------

def _bf16(vals):
    return wl.f32_to_bf16_bits(np.asarray(vals, np.float32))


def test_bf16_rounding_matches_fp32_bit_rule():
    rng = np.random.default_rng(41)
    x = np.concatenate([rng.standard_normal(5000).astype(np.float32) * 10,
                        rng.standard_normal(1000).astype(np.float32) * 1e-30])
    assert np.array_equal(oracle.f64_to_bf16_bits(x.astype(np.float64)), wl.f32_to_bf16_bits(x))


def test_bf16_rounding_special_cases():
    cases = [
        (1.0 + 2.0 ** -8, 0x3F80),                 # halfway, ties to even (down)
        (1.0 + 3 * 2.0 ** -8, 0x3F82),             # halfway, ties to even (up)
        (1.0 + 2.0 ** -8 + 2.0 ** -30, 0x3F81),    # just above halfway: one rounding step
        (-(1.0 + 2.0 ** -8 + 2.0 ** -30), 0xBF81),
        (2.0 ** -130, 0x0008),                     # subnormal, exact
        (3 * 2.0 ** -134, 0x0002),                 # subnormal halfway -> even
        (0.0, 0x0000),
        (-0.0, 0x8000),
        (2.5, 0x4020),
    ]
    for x, bits in cases:
        assert int(oracle.f64_to_bf16_bits([x])[0]) == bits, x


def test_layernorm_constant_row_gives_bias():
    g = oracle.bf16_bits_to_f64(_bf16(np.linspace(0.5, 1.5, 128)))
    b = oracle.bf16_bits_to_f64(_bf16(np.linspace(-1, 1, 128)))
    x = np.tile(_bf16([3.25]), (2, 128))
    out, y = oracle.key_layernorm(x, g, b, 1e-6)
    assert np.array_equal(out[0], _bf16(b.astype(np.float32)))
    assert np.array_equal(y[1], b)


@pytest.mark.parametrize("a,gamma,beta,eps", [(1.0, 1.0, 0.0, 1e-6), (1.0, 2.0, 0.5, 1e-6),
                                              (2.0 ** -10, 1.0, 0.0, 1e-6), (3.0, 0.5, -1.0, 1e-5)])
def test_layernorm_plus_minus_a_closed_form(a, gamma, beta, eps):
    """Row of +a/-a: mean 0, biased variance a^2 -> y = +-a/sqrt(a^2+eps)*gamma+beta."""
    row = np.array([a if d % 2 == 0 else -a for d in range(128)])
    x = _bf16(row)[None, :]
    out, y = oracle.key_layernorm(x, np.full(128, gamma), np.full(128, beta), eps)
    yp = a / np.sqrt(a * a + eps) * gamma + beta
    ym = -a / np.sqrt(a * a + eps) * gamma + beta
    exp = np.array([yp if d % 2 == 0 else ym for d in range(128)])
    np.testing.assert_allclose(y[0], exp, rtol=1e-14, atol=1e-15)
    assert np.array_equal(out[0], oracle.f64_to_bf16_bits(exp))
    if (a, gamma, beta) == (1.0, 1.0, 0.0):
        assert out[0, 0] == 0x3F80 and out[0, 1] == 0xBF80
    if (a, gamma, beta) == (1.0, 2.0, 0.5):
        assert out[0, 0] == 0x4020 and out[0, 1] == 0xBFC0


def test_layernorm_against_torch_float64():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(42)
    x = _bf16(rng.standard_normal((64, 128)).astype(np.float32) * 3 + 0.7)
    g = oracle.bf16_bits_to_f64(_bf16(1 + 0.1 * rng.standard_normal(128)))
    b = oracle.bf16_bits_to_f64(_bf16(0.1 * rng.standard_normal(128)))
    out, y = oracle.key_layernorm(x, g, b, 1e-6)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(oracle.bf16_bits_to_f64(x)), (128,),
                                         torch.from_numpy(g), torch.from_numpy(b), eps=1e-6)
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)
    assert np.array_equal(out, oracle.f64_to_bf16_bits(ref.numpy()))


def test_workloads_shapes_and_pairs():
    w1 = wl.tiny_exact()
    assert w1.pairs == 18913 and w1.T == 8 and w1.L == 3072 and w1.exact
    w3 = wl.prefill_ties(L=512)
    assert w3.pairs == 512 * 513 // 2
    w2 = wl.decode_batch()
    assert w2.pairs == 249856 and w2.k is None and w2.k_raw.shape == (249856, 128)
    # speculative verification: 16 users x the last 4 positions of their histories
    w6 = wl.spec_verify(B=3, lo=100, hi=200)
    lens = np.diff(w6.cu_k)
    assert w6.T == 12 and w6.B == 3 and np.array_equal(np.diff(w6.cu_q), [4, 4, 4])
    assert np.array_equal(w6.q_pos, np.concatenate([np.arange(l - 4, l) for l in lens]))
    assert w6.pairs == int(sum(4 * l - 6 for l in lens))
    assert wl.NAMES[6] == "spec_verify" and wl.by_index(6).T == 64


# ---------------------------------------------------------------------------
# projections (indexer paragraph: q from the normalised q-LoRA, k from the
# attention input through the key LayerNorm, per-head weights)
# ---------------------------------------------------------------------------

def _int_bf16_bits(rng, shape, lo, hi):
    return wl.f32_to_bf16_bits(rng.integers(lo, hi + 1, size=shape).astype(np.float32))


def test_projection_integer_inputs_match_int64_matmul():
    # small integers: every product sum is an exact integer; q and k_pre are
    # those integers rounded once to bf16, w is the integer itself
    rng = np.random.default_rng(31)
    T, hidden, rank = 5, 96, 40
    x, ql = _int_bf16_bits(rng, (T, hidden), -2, 2), _int_bf16_bits(rng, (T, rank), -2, 2)
    wq = _int_bf16_bits(rng, (32 * 128, rank), -1, 1)
    wk = _int_bf16_bits(rng, (128, hidden), -1, 1)
    ww = _int_bf16_bits(rng, (32, hidden), -1, 1)
    g, b = np.ones(128), np.zeros(128)
    q, k, w, k_pre = oracle.indexer_project(x, ql, wq, wk, ww, g, b, 1e-6)
    xi = wl.bf16_bits_to_f32(x).astype(np.int64)
    qli = wl.bf16_bits_to_f32(ql).astype(np.int64)
    q_int = qli @ wl.bf16_bits_to_f32(wq).astype(np.int64).T
    k_int = xi @ wl.bf16_bits_to_f32(wk).astype(np.int64).T
    w_int = xi @ wl.bf16_bits_to_f32(ww).astype(np.int64).T
    assert np.array_equal(w, w_int.astype(np.float64))
    assert np.array_equal(q.reshape(T, -1), wl.f32_to_bf16_bits(q_int.astype(np.float32)))
    assert np.array_equal(k_pre, wl.f32_to_bf16_bits(k_int.astype(np.float32)))
    assert np.array_equal(k, oracle.key_layernorm(k_pre, g, b, 1e-6)[0])


def test_projection_identity_weights_select_inputs():
    # W = [I | 0]: the outputs are the leading inputs themselves
    rng = np.random.default_rng(32)
    T, hidden, rank = 3, 160, 4096
    x = wl.f32_to_bf16_bits(rng.standard_normal((T, hidden)).astype(np.float32))
    ql = wl.f32_to_bf16_bits(rng.standard_normal((T, rank)).astype(np.float32))
    eye = lambda n, m: wl.f32_to_bf16_bits(np.eye(n, m, dtype=np.float32))
    q, k, w, k_pre = oracle.indexer_project(x, ql, eye(4096, rank), eye(128, hidden), eye(32, hidden),
                                            np.ones(128), np.zeros(128), 1e-6)
    assert np.array_equal(q.reshape(T, -1), ql)
    assert np.array_equal(k_pre, x[:, :128])
    assert np.array_equal(w, wl.bf16_bits_to_f32(x[:, :32]).astype(np.float64))


# ---------------------------------------------------------------------------
# sparse MLA attention over the selected positions
# ---------------------------------------------------------------------------

def _mla_inputs(seed, H=4, L=40, qscale=1.0):
    rng = np.random.default_rng(seed)
    q = wl.f32_to_bf16_bits((qscale * rng.standard_normal((H, oracle.MLA_DIM))).astype(np.float32))
    c = wl.f32_to_bf16_bits(rng.standard_normal((L, oracle.MLA_DIM)).astype(np.float32))
    return q, c


def test_mla_single_row_returns_its_latent():
    q, c = _mla_inputs(1)
    o, lse = oracle.sparse_mla(q, c, [17], 0.07)
    lat = oracle.bf16_bits_to_f64(c[17, :oracle.MLA_VDIM])
    for h in range(q.shape[0]):
        assert np.array_equal(o[h], lat)
        dot = float(oracle.bf16_bits_to_f64(q[h]) @ oracle.bf16_bits_to_f64(c[17]))
        assert lse[h] == pytest.approx(0.07 * dot, rel=1e-12, abs=1e-12)


def test_mla_identical_rows_and_zero_query():
    q, c = _mla_inputs(2)
    c[5:9] = c[5]          # four identical rows
    o, lse = oracle.sparse_mla(q, c, [5, 6, 7, 8], 0.1)
    lat = oracle.bf16_bits_to_f64(c[5, :oracle.MLA_VDIM])
    np.testing.assert_allclose(o, np.broadcast_to(lat, o.shape), rtol=1e-13, atol=1e-13)
    # a zero query: every logit is 0, so o is the mean latent and lse = log n
    rows = [0, 3, 9, 21, 30]
    oz, lz = oracle.sparse_mla(np.zeros_like(q), c, rows, 0.1)
    mean = oracle.bf16_bits_to_f64(c[rows, :oracle.MLA_VDIM]).mean(axis=0)
    np.testing.assert_allclose(oz, np.broadcast_to(mean, oz.shape), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(lz, np.log(len(rows)), rtol=1e-14)


def test_mla_large_scale_tends_to_the_top_row():
    q, c = _mla_inputs(3)
    rows = list(range(0, 40, 3))
    o, _ = oracle.sparse_mla(q, c, rows, 50.0)
    qd, cd = oracle.bf16_bits_to_f64(q), oracle.bf16_bits_to_f64(c)
    for h in range(q.shape[0]):
        logits = 50.0 * (cd[rows] @ qd[h])
        i = int(np.argmax(logits))
        top = cd[rows[i], :oracle.MLA_VDIM]
        # |o - c_top| = |sum_j p_j (c_j - c_top)| <= (1 - p_top) max_j |c_j - c_top|,
        # and 1 - p_top <= sum over the other rows of exp(l_j - l_top)
        rest = np.exp(np.delete(logits, i) - logits[i]).sum()
        spread = np.abs(cd[rows, :oracle.MLA_VDIM] - top).max()
        assert np.abs(o[h] - top).max() <= rest * spread + 1e-12


def test_mla_row_order_does_not_matter():
    q, c = _mla_inputs(4)
    rows = [2, 11, 19, 7, 33, 25]
    o1, l1 = oracle.sparse_mla(q, c, rows, 0.05)
    o2, l2 = oracle.sparse_mla(q, c, rows[::-1], 0.05)
    np.testing.assert_allclose(o1, o2, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(l1, l2, rtol=1e-14)


def test_mla_empty_selection():
    q, c = _mla_inputs(5)
    o, lse = oracle.sparse_mla(q, c, [], 0.05)
    assert np.all(o == 0.0) and np.all(np.isneginf(lse))


def test_mla_against_scipy_softmax_over_numpy_matmul():
    """The definition through library routines: a float64 matmul of the
    selected rows, scipy's softmax and logsumexp, another matmul for o."""
    special = pytest.importorskip("scipy.special")
    q, c = _mla_inputs(6, H=8, L=300, qscale=0.5)
    rows = np.random.default_rng(7).choice(300, size=120, replace=False)
    scale = 1.0 / np.sqrt(192.0)
    o, lse = oracle.sparse_mla(q, c, rows, scale)
    cd = oracle.bf16_bits_to_f64(c)[rows]
    logits = scale * (oracle.bf16_bits_to_f64(q) @ cd.T)          # [H, n]
    p = special.softmax(logits, axis=1)
    np.testing.assert_allclose(o, p @ cd[:, :oracle.MLA_VDIM], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse, special.logsumexp(logits, axis=1), rtol=1e-12)


def test_mla_batch_maps_positions_through_the_sequence_offsets():
    q, c = _mla_inputs(8, H=4, L=60)
    qb = np.stack([q, q[::-1]])                    # two query rows, one per sequence
    cu_q, cu_k = [0, 1, 2], [0, 25, 60]
    idx = np.array([[3, 0, 24, -1], [0, 34, 10, -1]], np.int32)
    cnt = np.array([3, 3], np.int32)
    o, lse = oracle.sparse_mla_batch(qb, c, idx, cnt, cu_q, cu_k, 0.05)
    o0, l0 = oracle.sparse_mla(qb[0], c, [3, 0, 24], 0.05)
    o1, l1 = oracle.sparse_mla(qb[1], c, [25, 59, 35], 0.05)
    assert np.array_equal(o[0], o0) and np.array_equal(o[1], o1)
    assert np.array_equal(lse[0], l0) and np.array_equal(lse[1], l1)


def test_mla_inputs_follow_the_indexer_output_format():
    """workloads.mla_case: each query keeps min(topk, its causal length)
    distinct positions inside its sequence, ascending and -1 padded, as
    idx_score_topk writes them; shapes of q and the 576-wide cache."""
    q, cache, idx, cnt, cu_q, cu_k = wl.mla_case(3, [10, 5000, 2049], q_per_seq=2, heads=32, topk=2048)
    assert q.shape == (6, 32, 576) and cache.shape == (int(cu_k[-1]), 576)
    assert list(cu_q) == [0, 2, 4, 6] and list(cu_k) == [0, 10, 5010, 7059]
    lens = [10, 5000, 2049]
    for t in range(6):
        n = lens[t // 2] - (1 - t % 2)                 # the query's causal length
        assert cnt[t] == min(2048, n)
        sel = idx[t, :cnt[t]]
        assert np.all(np.diff(sel) > 0) and sel.min() >= 0 and sel.max() < n
        assert np.all(idx[t, cnt[t]:] == -1)


# ---------------------------------------------------------------------------
# FP8 (E4M3) MLA cache rows
# ---------------------------------------------------------------------------

def test_e4m3_hand_derived_codes():
    # sign | exponent (4 bits, bias 7) | mantissa (3 bits); exponent 0: m/8 x 2^-6
    cases = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6,
             0x38: 1.0, 0x39: 1.125, 0x40: 2.0, 0x7E: 448.0, 0xB8: -1.0, 0xFE: -448.0}
    got = oracle.e4m3_to_f64(list(cases))
    assert np.array_equal(got, np.array(list(cases.values())))
    assert np.signbit(oracle.e4m3_to_f64([0x80]))[0]
    assert np.isnan(oracle.e4m3_to_f64([0x7F, 0xFF])).all()


def test_e4m3_every_code_against_torch():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_to_f64(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def _bf16_exact_fp8_rows(rng, n, pow2_scales=True):
    # codes with |value| <= 8 and power-of-two row scales: every dequantised
    # value is an exact bf16 value (<= 4 significant bits)
    codes = rng.integers(0, 256, size=(n, 576)).astype(np.uint8)
    codes[(codes & 0x7F) >= 0x58] &= 0x47          # keep exponents small (|v| < 2^4), no NaN
    scale = 2.0 ** rng.integers(-3, 2, size=n).astype(np.float64)
    return codes, scale


def test_mla_fp8_equals_bf16_attention_on_exact_rows():
    rng = np.random.default_rng(31)
    codes, scale = _bf16_exact_fp8_rows(rng, 40)
    vals = scale[:, None] * oracle.e4m3_to_f64(codes)
    bits = oracle.f64_to_bf16_bits(vals)
    assert np.array_equal(oracle.bf16_bits_to_f64(bits), vals)   # exact in bf16
    q = wl.f32_to_bf16_bits(rng.standard_normal((6, 576)).astype(np.float32) * 0.1)
    rows = np.array([3, 17, 0, 39, 22, 5])
    o8, l8 = oracle.sparse_mla_fp8(q, codes, scale, rows, 0.07)
    ob, lb = oracle.sparse_mla(q, bits, rows, 0.07)
    assert np.array_equal(o8, ob) and np.array_equal(l8, lb)


def test_mla_fp8_single_row_returns_its_dequantised_latent():
    rng = np.random.default_rng(32)
    codes, scale = _bf16_exact_fp8_rows(rng, 5)
    scale[2] = 0.3                                   # any real scale
    q = wl.f32_to_bf16_bits(rng.standard_normal((4, 576)).astype(np.float32))
    o, lse = oracle.sparse_mla_fp8(q, codes, scale, np.array([2]), 0.05)
    c = 0.3 * oracle.e4m3_to_f64(codes[2])
    assert np.allclose(o, np.broadcast_to(c[:512], o.shape), rtol=0, atol=1e-15)
    assert np.allclose(lse, 0.05 * (oracle.bf16_bits_to_f64(q) @ c), rtol=1e-14, atol=1e-14)
