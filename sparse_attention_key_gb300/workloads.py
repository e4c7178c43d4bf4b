"""Seeded synthetic workloads for the Lightning Indexer.

This module only draws inputs: shapes, value distributions, ragged lengths and
query positions. It holds none of the indexer's arithmetic, and it is the one
module that both the CUDA path's callers and the CPU oracle's callers share.

All randomness comes from ``numpy.random.default_rng(seed)``; real values are
drawn in fp32 and rounded to bf16 (nearest-even) as input data. Arrays are
host numpy arrays; bf16 tensors are carried as uint16 bit patterns.

Named workloads (sizes from the indexer's use in Kimi K3.1 Pro's MLA layers:
32 heads x 128 dims, top-2048, causal histories up to 128K keys):

1. ``tiny_exact``     1 sequence of 3072 keys, 8 queries at positions
                      {100, 2047, 2048, 2500, 3000, 3069, 3070, 3071}; q, k are
                      integers in [-4, 4] x 2^-3, w integers in [0, 3] x 2^-2;
                      LayerNorm weight 1, bias 0, eps 1e-6 (checked on k).
2. ``decode_batch``   8 sequences, one query each at the end of 8K/12K/16K/24K/
                      32K/40K/48K/64K-key histories; raw keys and q ~ N(0,1),
                      w ~ U(0, 1/32), LayerNorm weight ~ N(1, 0.1), bias ~
                      N(0, 0.1); the keys are LayerNormed before scoring.
3. ``prefill_ties``   1 sequence, T = L = 8192, every position a query; q, k
                      integers in [-2, 2], w integers in [0, 1] (heavy ties).
4. ``agentic_chunk``  4 sequences, each a 50,000-key cached prefix plus an
                      800-query causal chunk (L = 50,800, positions 50,000..
                      50,799); q, k ~ N(0,1), w ~ U(0, 1/32). Stands in for a
                      multi-turn agentic session (~50K prompt, ~800 new tokens
                      per turn); no dataset is used.
5. ``long_decode``    64 sequences, one query each, histories uniform in
                      [65,536, 131,072] keys; post-LN keys ~ N(0,1), q ~ N(0,1),
                      w ~ U(0, 1/32).
6. ``spec_verify``    speculative-decoding verification: 16 sequences, each
                      with 4 queries at the last 4 positions of a history
                      uniform in [50,000, 100,000] keys (64 rows); post-LN keys
                      ~ N(0,1), q ~ N(0,1), w ~ U(0, 1/32).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

HEADS = 32
DIM = 128
TOPK = 2048

NAMES = {1: "tiny_exact", 2: "decode_batch", 3: "prefill_ties", 4: "agentic_chunk",
         5: "long_decode", 6: "spec_verify"}


def f32_to_bf16_bits(x) -> np.ndarray:
    """Round fp32 values to bf16 bit patterns (nearest, ties to even). Finite input."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + r) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits) -> np.ndarray:
    """bf16 bit patterns -> exact fp32 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


@dataclass
class Workload:
    name: str
    q: np.ndarray            # uint16 [T,32,128] bf16 bits
    w: np.ndarray            # float32 [T,32]
    q_pos: np.ndarray        # int32 [T], position of each query inside its sequence
    cu_q: np.ndarray         # int32 [B+1], query rows of sequence b: cu_q[b]..cu_q[b+1]
    cu_k: np.ndarray         # int32 [B+1], key rows of sequence b: cu_k[b]..cu_k[b+1]
    k: np.ndarray | None     # uint16 [L,128] scoring keys (post-LayerNorm cache), or None
    k_raw: np.ndarray | None = None   # uint16 [L,128] raw keys when LayerNorm runs first
    ln_w: np.ndarray | None = None    # uint16 [128] bf16 bits
    ln_b: np.ndarray | None = None    # uint16 [128] bf16 bits
    eps: float = 1e-6
    topk: int = TOPK
    exact: bool = False      # integer-valued inputs: indices must match bit-exactly
    meta: dict = field(default_factory=dict)

    @property
    def T(self) -> int:
        return int(self.q.shape[0])

    @property
    def B(self) -> int:
        return int(self.cu_q.size - 1)

    @property
    def L(self) -> int:
        return int(self.cu_k[-1])

    @property
    def pairs(self) -> int:
        """Query-key pairs scored: sum over queries of the causal length q_pos + 1."""
        return int(np.sum(self.q_pos.astype(np.int64) + 1))

    @property
    def max_len(self) -> int:
        return int(self.q_pos.max()) + 1 if self.T else 0


def _normal_bf16(rng, shape, chunk=1 << 24) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for i in range(0, n, chunk):
        m = min(chunk, n - i)
        out[i:i + m] = f32_to_bf16_bits(rng.standard_normal(m, dtype=np.float32))
    return out.reshape(shape)


def _int_bf16(rng, shape, lo, hi, scale) -> np.ndarray:
    v = rng.integers(lo, hi + 1, size=shape, dtype=np.int32).astype(np.float32) * np.float32(scale)
    return f32_to_bf16_bits(v)


def _ragged(q_counts, k_lens):
    cu_q = np.zeros(len(q_counts) + 1, dtype=np.int32)
    cu_k = np.zeros(len(k_lens) + 1, dtype=np.int32)
    cu_q[1:] = np.cumsum(q_counts)
    cu_k[1:] = np.cumsum(k_lens)
    return cu_q, cu_k


def tiny_exact(seed: int = 1) -> Workload:
    rng = np.random.default_rng(seed)
    L = 3072
    pos = np.array([100, 2047, 2048, 2500, 3000, 3069, 3070, 3071], dtype=np.int32)
    k = _int_bf16(rng, (L, DIM), -4, 4, 2.0 ** -3)
    q = _int_bf16(rng, (pos.size, HEADS, DIM), -4, 4, 2.0 ** -3)
    w = (rng.integers(0, 4, size=(pos.size, HEADS)).astype(np.float32) * np.float32(0.25))
    cu_q, cu_k = _ragged([pos.size], [L])
    ones = f32_to_bf16_bits(np.ones(DIM, np.float32))
    zeros = f32_to_bf16_bits(np.zeros(DIM, np.float32))
    return Workload("tiny_exact", q, w, pos, cu_q, cu_k, k, k_raw=k, ln_w=ones, ln_b=zeros,
                    eps=1e-6, exact=True)


def decode_batch(seed: int = 2) -> Workload:
    rng = np.random.default_rng(seed)
    lens = [l * 1024 for l in (8, 12, 16, 24, 32, 40, 48, 64)]
    cu_q, cu_k = _ragged([1] * len(lens), lens)
    k_raw = _normal_bf16(rng, (int(cu_k[-1]), DIM))
    q = _normal_bf16(rng, (len(lens), HEADS, DIM))
    w = rng.uniform(0.0, 1.0 / 32, size=(len(lens), HEADS)).astype(np.float32)
    ln_w = f32_to_bf16_bits((1.0 + 0.1 * rng.standard_normal(DIM)).astype(np.float32))
    ln_b = f32_to_bf16_bits((0.1 * rng.standard_normal(DIM)).astype(np.float32))
    pos = np.array([l - 1 for l in lens], dtype=np.int32)
    return Workload("decode_batch", q, w, pos, cu_q, cu_k, None, k_raw=k_raw, ln_w=ln_w,
                    ln_b=ln_b, eps=1e-6, exact=False)


def prefill_ties(seed: int = 3, L: int = 8192) -> Workload:
    rng = np.random.default_rng(seed)
    k = _int_bf16(rng, (L, DIM), -2, 2, 1.0)
    q = _int_bf16(rng, (L, HEADS, DIM), -2, 2, 1.0)
    w = rng.integers(0, 2, size=(L, HEADS)).astype(np.float32)
    cu_q, cu_k = _ragged([L], [L])
    pos = np.arange(L, dtype=np.int32)
    return Workload("prefill_ties", q, w, pos, cu_q, cu_k, k, exact=True)


def agentic_chunk(seed: int = 4, B: int = 4, prefix: int = 50_000, chunk: int = 800) -> Workload:
    rng = np.random.default_rng(seed)
    L = prefix + chunk
    cu_q, cu_k = _ragged([chunk] * B, [L] * B)
    k = _normal_bf16(rng, (B * L, DIM))
    q = _normal_bf16(rng, (B * chunk, HEADS, DIM))
    w = rng.uniform(0.0, 1.0 / 32, size=(B * chunk, HEADS)).astype(np.float32)
    pos = np.tile(np.arange(prefix, L, dtype=np.int32), B)
    return Workload("agentic_chunk", q, w, pos, cu_q, cu_k, k, exact=False)


def long_decode(seed: int = 5, B: int = 64, lo: int = 65_536, hi: int = 131_072) -> Workload:
    rng = np.random.default_rng(seed)
    lens = rng.integers(lo, hi + 1, size=B).astype(np.int64)
    cu_q, cu_k = _ragged([1] * B, lens)
    k = _normal_bf16(rng, (int(cu_k[-1]), DIM))
    q = _normal_bf16(rng, (B, HEADS, DIM))
    w = rng.uniform(0.0, 1.0 / 32, size=(B, HEADS)).astype(np.float32)
    pos = (lens - 1).astype(np.int32)
    return Workload("long_decode", q, w, pos, cu_q, cu_k, k, exact=False)


def spec_verify(seed: int = 6, B: int = 16, m: int = 4, lo: int = 50_000,
                hi: int = 100_000) -> Workload:
    rng = np.random.default_rng(seed)
    lens = rng.integers(lo, hi + 1, size=B).astype(np.int64)
    cu_q, cu_k = _ragged([m] * B, lens)
    k = _normal_bf16(rng, (int(cu_k[-1]), DIM))
    q = _normal_bf16(rng, (B * m, HEADS, DIM))
    w = rng.uniform(0.0, 1.0 / 32, size=(B * m, HEADS)).astype(np.float32)
    pos = np.concatenate([np.arange(l - m, l, dtype=np.int32) for l in lens])
    return Workload("spec_verify", q, w, pos, cu_q, cu_k, k, exact=False)


def by_index(i: int, seed: int | None = None) -> Workload:
    """Workload i in 1..6 (see the module docstring); the default seed is i."""
    fn = {1: tiny_exact, 2: decode_batch, 3: prefill_ties, 4: agentic_chunk, 5: long_decode,
          6: spec_verify}[i]
    return fn(i if seed is None else seed)


def custom(seed: int, q_counts, k_lens, kind: str = "normal", positions: str = "chunk",
           topk: int = TOPK) -> Workload:
    """A ragged batch for tests.

    ``q_counts[b]`` queries and ``k_lens[b]`` keys for sequence b. ``positions``:
    "chunk" puts the queries at the end of the history (a causal chunk: query i
    of n_q at k_len - n_q + i); "random" draws distinct positions in [0, k_len).
    ``kind``: "normal" (q, k ~ N(0,1), w ~ U(0,1/32)), "int2" (integers in
    [-2, 2], w in {0,1}: exact with heavy ties), "int4s3" (integers in [-4,4] x
    2^-3, w in {0,..,3} x 2^-2: exact).
    """
    rng = np.random.default_rng(seed)
    q_counts = [int(c) for c in q_counts]
    k_lens = [int(l) for l in k_lens]
    cu_q, cu_k = _ragged(q_counts, k_lens)
    L, T = int(cu_k[-1]), int(cu_q[-1])
    if kind == "normal":
        k = _normal_bf16(rng, (L, DIM))
        q = _normal_bf16(rng, (T, HEADS, DIM))
        w = rng.uniform(0.0, 1.0 / 32, size=(T, HEADS)).astype(np.float32)
        exact = False
    elif kind == "int2":
        k = _int_bf16(rng, (L, DIM), -2, 2, 1.0)
        q = _int_bf16(rng, (T, HEADS, DIM), -2, 2, 1.0)
        w = rng.integers(0, 2, size=(T, HEADS)).astype(np.float32)
        exact = True
    elif kind == "int4s3":
        k = _int_bf16(rng, (L, DIM), -4, 4, 2.0 ** -3)
        q = _int_bf16(rng, (T, HEADS, DIM), -4, 4, 2.0 ** -3)
        w = rng.integers(0, 4, size=(T, HEADS)).astype(np.float32) * np.float32(0.25)
        exact = True
    else:
        raise ValueError(kind)
    pos = np.empty(T, dtype=np.int32)
    for b in range(len(q_counts)):
        nq, lk = q_counts[b], k_lens[b]
        if nq == 0:
            continue
        if positions == "chunk":
            if nq > lk:
                raise ValueError("more queries than keys in a causal chunk")
            pos[cu_q[b]:cu_q[b + 1]] = np.arange(lk - nq, lk, dtype=np.int32)
        elif positions == "random":
            pos[cu_q[b]:cu_q[b + 1]] = rng.choice(lk, size=nq, replace=nq > lk).astype(np.int32)
        else:
            raise ValueError(positions)
    return Workload(f"custom_{kind}", q, w, pos, cu_q, cu_k, k, exact=exact, topk=topk)


def score_rows(seed: int, T: int, n_valid, ld: int, kind: str = "ties") -> np.ndarray:
    """Synthetic fp32 score rows [T, ld] for exercising a stand-alone top-K.

    kind: "ties" (small integers: large tie groups at the boundary), "normal"
    (continuous, mostly distinct), "mixed" (relu-like: ~half exact zeros, the
    rest continuous, some -0.0), "const" (all equal), "tiny" (+-0, +-denormals
    and the smallest normals, with repeats).
    """
    rng = np.random.default_rng(seed)
    n_valid = np.asarray(n_valid, dtype=np.int64)
    S = np.full((T, ld), np.nan, dtype=np.float32)
    for t in range(T):
        n = int(n_valid[t])
        if kind == "ties":
            v = rng.integers(0, 16, size=n).astype(np.float32)
        elif kind == "normal":
            v = rng.standard_normal(n, dtype=np.float32)
        elif kind == "mixed":
            v = rng.standard_normal(n, dtype=np.float32)
            v[v < 0] = 0.0
            neg0 = rng.random(n) < 0.1
            v[neg0 & (v == 0)] = -0.0
        elif kind == "const":
            v = np.full(n, 1.5, dtype=np.float32)
        elif kind == "tiny":
            # values around zero: +-0, +-denormals, the smallest normals and a
            # few ordinary values; many exact repeats
            pool = np.array([0.0, -0.0, 1e-45, -1e-45, 3e-42, -3e-42, 1.1754942e-38,
                             -1.1754942e-38, 1.1754944e-38, 2.5e-39, 1.0, -1.0, 5e-40],
                            dtype=np.float32)
            v = pool[rng.integers(0, pool.size, size=n)]
            m = rng.random(n) < 0.3
            v[m] = (rng.standard_normal(int(m.sum())) * 1e-38).astype(np.float32)
        else:
            raise ValueError(kind)
        S[t, :n] = v
    return S


# ---------------------------------------------------------------------------
# Sparse MLA attention inputs (the consumer of the indexer's selection)
# ---------------------------------------------------------------------------
MLA_DIM = 576     # cache row: 512-wide latent + 64 key dims
MLA_HEADS = 96


def mla_case(seed: int, k_lens, q_per_seq: int = 1, heads: int = MLA_HEADS, topk: int = 2048,
             n_sel=None, qscale: float = 1.0):
    """Seeded inputs of one sparse MLA call over a packed ragged batch.

    Sequence b holds k_lens[b] cached rows (bf16 ~ N(0,1), 576 wide) and
    q_per_seq query rows at its last positions (absorbed queries, bf16 ~
    N(0, qscale^2)). Each query keeps min(topk, its causal length) distinct
    positions (or n_sel[t] when given), drawn uniformly and sorted ascending,
    as the indexer emits them; idx is -1 padded to topk. Returns
    (q [T,H,576] bits, cache [L,576] bits, idx [T,topk] int32, cnt [T] int32,
    cu_q, cu_k).
    """
    rng = np.random.default_rng(seed)
    k_lens = np.asarray(k_lens, dtype=np.int64)
    cache = _normal_bf16(rng, (int(k_lens.sum()), MLA_DIM))
    return _mla_queries(rng, cache, k_lens, q_per_seq, heads, topk, n_sel, qscale)


def fp8_codes(rng, shape) -> np.ndarray:
    """E4M3 code bytes with a bell-shaped spread of magnitudes: random sign,
    exponent field 7 + round(N(0, 1.5)) clipped to 0..15 (so mostly values of
    2^-2 .. 2^3, with some subnormals and some near the top of the range),
    uniform mantissa; the two NaN codes are never drawn (mantissa 7 of the top
    exponent becomes 6)."""
    sign = rng.integers(0, 2, size=shape, dtype=np.uint8)
    expo = np.clip(np.rint(7 + 1.5 * rng.standard_normal(shape)), 0, 15).astype(np.uint8)
    mant = rng.integers(0, 8, size=shape, dtype=np.uint8)
    mant = np.where((expo == 15) & (mant == 7), np.uint8(6), mant)
    return ((sign << 7) | (expo << 3) | mant).astype(np.uint8)


def mla_fp8_case(seed: int, k_lens, q_per_seq: int = 1, heads: int = MLA_HEADS, topk: int = 2048,
                 n_sel=None, qscale: float = 1.0):
    """mla_case over an FP8 cache: rows of 576 E4M3 codes (fp8_codes) with
    one fp32 scale each, 2^U(-3, 0). Returns (q bits, cache8 [L,576] uint8,
    row_scale [L] fp32, idx, cnt, cu_q, cu_k)."""
    rng = np.random.default_rng(seed)
    k_lens = np.asarray(k_lens, dtype=np.int64)
    L = int(k_lens.sum())
    cache8 = fp8_codes(rng, (L, MLA_DIM))
    row_scale = np.exp2(rng.uniform(-3.0, 0.0, size=L)).astype(np.float32)
    q, _, idx, cnt, cu_q, cu_k = _mla_queries(rng, cache8, k_lens, q_per_seq, heads, topk, n_sel, qscale)
    return q, cache8, row_scale, idx, cnt, cu_q, cu_k


def _mla_queries(rng, cache, k_lens, q_per_seq, heads, topk, n_sel, qscale):
    B = k_lens.size
    cu_k = np.concatenate([[0], np.cumsum(k_lens)]).astype(np.int32)
    cu_q = (np.arange(B + 1) * q_per_seq).astype(np.int32)
    T = B * q_per_seq
    q = f32_to_bf16_bits((qscale * rng.standard_normal((T, heads, MLA_DIM))).astype(np.float32))
    idx = np.full((T, topk), -1, dtype=np.int32)
    cnt = np.zeros(T, dtype=np.int32)
    for t in range(T):
        b = t // q_per_seq
        n = int(k_lens[b]) - (q_per_seq - 1 - t % q_per_seq)   # causal length of this query
        m = min(topk, max(n, 0)) if n_sel is None else int(n_sel[t])
        if m > 0:
            idx[t, :m] = np.sort(rng.choice(n, size=m, replace=False)).astype(np.int32)
        cnt[t] = m
    return q, cache, idx, cnt, cu_q, cu_k
