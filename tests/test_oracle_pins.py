"""Pins of the CPU oracle against what the SparCML pages and mathematics fix.

No GPU. Each test checks the oracle against something other than itself:
brute force on tiny inputs, closed forms, invariants, published known-answer
values. A plausible slip in the oracle (a dropped term, a wrong sign or index,
a flipped tie-break, a transposed operand) breaks at least one of these.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from top_gradient_compression_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
GOLDEN_RATIO_INC = 0x9E3779B97F4A7C15
M64 = (1 << 64) - 1


def keys(x):
    return np.asarray(x, np.float32).view(np.uint32) & np.uint32(0x7FFFFFFF)


# --------------------------------------------------------------------------
# SplitMix64: published known-answer vector (Rosetta Code, seed 1234567).
# --------------------------------------------------------------------------
def test_splitmix64_known_answer_vector():
    with open(os.path.join(GOLDEN, "splitmix64_seed1234567.txt")) as f:
        expect = [int(l) for l in f if l.strip() and not l.startswith("#")]
    assert len(expect) == 5
    state = 1234567
    for e in expect:
        # one generator step: output = finaliser(state + increment)
        assert oracle.splitmix64(state) == e
        state = (state + GOLDEN_RATIO_INC) & M64


# --------------------------------------------------------------------------
# Top-k with error feedback (§2.2, §4).
# --------------------------------------------------------------------------
def brute_topk(acc_seg, k):
    """O(n^2) definition: i is kept iff fewer than k entries beat it, where j
    beats i when |acc_j| > |acc_i|, or they are equal and j < i."""
    kk = keys(acc_seg).astype(np.int64)
    n = len(kk)
    keep = []
    for i in range(n):
        beaten_by = sum(1 for j in range(n) if kk[j] > kk[i] or (kk[j] == kk[i] and j < i))
        if beaten_by < k:
            keep.append(i)
    return keep


def tie_heavy(rng, shape):
    pool = np.array([0.0, -0.0, 1.0, -1.0, 2.0, -2.0, 0.5, -0.5, 3.0], np.float32)
    return pool[rng.integers(0, len(pool), size=shape)]


@pytest.mark.parametrize("seed", range(6))
def test_topk_brute_force_all_k_tiny(seed):
    rng = np.random.default_rng(seed)
    P = int(rng.integers(1, 6))
    N = int(rng.integers(1, 41))
    grad = tie_heavy(rng, (P, N)) if seed % 2 else rng.standard_normal((P, N)).astype(np.float32)
    res0 = tie_heavy(rng, (P, N)) * np.float32(0.25)
    for k in range(0, N + 1):
        res = res0.copy()
        idx, val, nnz = oracle.topk_ef(grad, res, seg_len=N, k_num=k, k_den=N, cap=N + 1)
        acc = res0 + grad
        for p in range(P):
            want = brute_topk(acc[p], k)
            assert nnz[p] == k
            assert list(idx[p, :k]) == want
            assert np.array_equal(val[p, :k].view(np.uint32), acc[p, want].view(np.uint32))


CANON_NAN = np.uint32(0x7FFFFFFF)


def test_topk_orders_non_finite_magnitudes_by_bit_pattern():
    """Non-finite inputs are not rejected; the magnitude key is the bit
    pattern of |x|, so a NaN ranks above +-inf, which ranks above every
    finite value. Every NaN that the error-feedback add produces is the
    canonical NaN 0x7fffffff (IEEE 754 leaves a NaN result's payload open),
    so NaNs of any payload tie and the lower index wins; +inf and -inf have
    one key, so the lower index wins between them too."""
    f = np.float32
    qnan, big_nan = np.uint32(0x7FC00000).view(f), np.uint32(0xFFC00001).view(f)
    grad = np.array([[1.0, -np.inf, 3.0e38, qnan, -2.0, np.inf, big_nan, 0.0]], f)
    acc_bits = grad.view(np.uint32).copy()
    acc_bits[0, [3, 6]] = CANON_NAN
    for k, want in [(1, [3]), (2, [3, 6]), (3, [1, 3, 6]), (4, [1, 3, 5, 6]), (5, [1, 2, 3, 5, 6])]:
        res = np.zeros_like(grad)
        idx, val, nnz = oracle.topk_ef(grad, res, seg_len=8, k_num=k, k_den=8, cap=8)
        assert nnz[0] == k and list(idx[0, :k]) == want
        assert np.array_equal(val[0, :k].view(np.uint32), acc_bits[0, want])
        kept = np.zeros(8, bool)
        kept[want] = True
        assert np.array_equal(res[0, ~kept].view(np.uint32), acc_bits[0, ~kept])
        assert (res[0, kept].view(np.uint32) == 0).all()


def test_fp32_additions_give_the_canonical_nan():
    """Every NaN an addition produces is 0x7fffffff whatever the input
    payloads (the EF add, the sum reduce and SSAR's pairwise sums), while
    finite sums and the signs of infinities are untouched."""
    f = np.float32
    pay = [np.uint32(x).view(f) for x in (0x7FC00000, 0xFFC00001, 0x7F800001, 0x7FFFFFFF)]
    for a in pay:
        g = np.array([[a, np.inf, 1.5]], f)
        r = np.array([[0.0, -np.inf, 2.25]], f)
        oracle.topk_ef(g, r, 3, 0, 1)  # k = 0: residual = acc everywhere
        assert list(r.view(np.uint32)[0]) == [CANON_NAN, CANON_NAN, np.float32(3.75).view(np.uint32)]
    idx = np.array([[0, 1, 2], [0, 1, 3]], np.uint32)
    val = np.array([[pay[1], np.inf, 1.0], [1.0, -np.inf, np.inf]], f)
    out = oracle.sparse_reduce(idx, val, np.array([3, 3], np.uint32), 16)
    assert list(out["idx"]) == [0, 1, 2, 3]
    assert list(out["val"].view(np.uint32)) == [CANON_NAN, CANON_NAN,
                                                 np.float32(1.0).view(np.uint32),
                                                 np.float32(np.inf).view(np.uint32)]
    ri, rv, _ = oracle.ssar(idx, val, np.array([3, 3], np.uint32), 16)
    assert np.array_equal(rv.view(np.uint32), out["val"].view(np.uint32))


def brute_table(grad_row, seg_begin, seg_k):
    want = []
    for s in range(len(seg_k)):
        b, e = seg_begin[s], seg_begin[s + 1]
        want += [b + i for i in brute_topk(grad_row[b:e], seg_k[s])]
    return want


@pytest.mark.parametrize("seed", range(4))
def test_topk_ragged_segment_table_brute_force(seed):
    """Layer-wise sparsification (§8.4) over an arbitrary segment table:
    segments of 1, 2, 7 and more entries, each with its own k_s from 0 to n_s,
    against the O(n^2) definition segment by segment; the EF invariant holds
    bitwise and nnz is the sum of the k_s."""
    rng = np.random.default_rng(100 + seed)
    lens = [1, 7, 2, 40, 1, 13, 64, 3] if seed % 2 else [5, 1, 1, 29, 7, 70]
    seg_begin = [0] + list(np.cumsum(lens))
    N = seg_begin[-1]
    seg_k = [int(rng.integers(0, n + 1)) for n in lens]
    seg_k[0], seg_k[-1] = 0, lens[-1]  # both ends of the k range
    P = 3
    grad = tie_heavy(rng, (P, N)) if seed < 2 else rng.standard_normal((P, N)).astype(np.float32)
    res0 = tie_heavy(rng, (P, N)) * np.float32(0.5)
    res = res0.copy()
    idx, val, nnz = oracle.topk_ef_segments(grad, res, seg_begin, seg_k)
    acc = res0 + grad
    K = sum(seg_k)
    for p in range(P):
        want = brute_table(acc[p], seg_begin, seg_k)
        assert int(nnz[p]) == K == len(want)
        assert list(idx[p, :K]) == want
        assert np.array_equal(val[p, :K].view(np.uint32), acc[p, want].view(np.uint32))
        rebuilt = res[p].copy()
        rebuilt[want] = val[p, :K]
        assert np.array_equal(rebuilt.view(np.uint32), acc[p].view(np.uint32))
        assert (res[p, want].view(np.uint32) == 0).all()


def test_topk_uniform_form_is_the_equal_segment_table():
    rng = np.random.default_rng(9)
    P, N, L = 2, 1000, 300
    g = rng.standard_normal((P, N)).astype(np.float32)
    r1, r2 = np.zeros_like(g), np.zeros_like(g)
    a = oracle.topk_ef(g, r1, L, 3, 100)
    b, k = oracle.uniform_segments(N, L, 3, 100)
    assert b == [0, 300, 600, 900, 1000] and k == [9, 9, 9, 3]
    c = oracle.topk_ef_segments(g, r2, b, k)
    for x, y in zip(a, c):
        assert np.array_equal(x, y)
    assert np.array_equal(r1, r2)


def test_topk_segment_table_is_checked():
    g = np.zeros((1, 10), np.float32)
    for b, k in [([0, 5, 5, 10], [1, 0, 1]),  # empty segment
                 ([0, 5, 9], [1, 1]),         # does not end at N
                 ([1, 5, 10], [1, 1]),        # does not start at 0
                 ([0, 5, 10], [6, 1])]:       # k_s > n_s
        with pytest.raises(oracle.OracleError):
            oracle.topk_ef_segments(g, np.zeros_like(g), b, k)


def test_threaded_drivers_give_the_sequential_results():
    """The all-core timing drivers (pairs (node, segment) on threads; the
    reduce cut into index ranges) reproduce the sequential oracle bit for bit,
    for sparse and dense results and for bad streams."""
    rng = np.random.default_rng(4)
    P, N = 5, 20_011
    g = rng.standard_normal((P, N)).astype(np.float32)
    lens = [1, 999, 7, 5000, 14_004]
    b = [0] + list(np.cumsum(lens))
    k = [1, 20, 0, 50, 1300]
    r1, r2 = np.zeros_like(g), np.zeros_like(g)
    a = oracle.topk_ef_segments(g, r1, b, k)
    c = oracle.topk_ef_segments(g, r2, b, k, threads=7)
    for x, y in zip(a, c):
        assert np.array_equal(x, y)
    assert np.array_equal(r1.view(np.uint32), r2.view(np.uint32))
    for kk, dense in [(400, False), (6000, True)]:
        idx, val, nnz = W.uniform_streams(P, N, kk, 77 + kk)
        s1 = oracle.sparse_reduce(idx, val, nnz, N)
        s2 = oracle.sparse_reduce(idx, val, nnz, N, threads=6)
        assert s1["nnz"] == s2["nnz"] and s1["is_dense"] == s2["is_dense"] == dense
        for key in ("idx", "val", "dense"):
            if s1[key] is not None:
                assert np.array_equal(np.asarray(s1[key]).view(np.uint32),
                                      np.asarray(s2[key]).view(np.uint32))
    idx, val, nnz = W.uniform_streams(2, 100, 10, 5)
    idx[1, 4] = idx[1, 3]  # not strictly ascending
    with pytest.raises(oracle.OracleError) as e:
        oracle.sparse_reduce(idx, val, nnz, 100, threads=3)
    assert e.value.code == oracle.BAD_STREAM


@pytest.mark.parametrize("N,seg_len,k_num,k_den", [(50, 16, 3, 8), (37, 5, 2, 5), (64, 64, 1, 100),
                                                    (33, 1, 1, 1), (40, 7, 0, 3)])
def test_topk_segments_brute_force(N, seg_len, k_num, k_den):
    rng = np.random.default_rng(N * 7 + seg_len)
    P = 3
    grad = tie_heavy(rng, (P, N))
    res = np.zeros((P, N), np.float32)
    idx, val, nnz = oracle.topk_ef(grad, res, seg_len, k_num, k_den, cap=N)
    for p in range(P):
        want = []
        for b in range(0, N, seg_len):
            n_s = min(seg_len, N - b)
            k_s = n_s * k_num // k_den  # App. A style: last segment takes the remainder
            want += [b + i for i in brute_topk(grad[p, b:b + n_s], k_s)]
        assert int(nnz[p]) == len(want)
        assert list(idx[p, :len(want)]) == want


def test_topk_k_equals_n_keeps_everything_and_zero_keeps_nothing():
    rng = np.random.default_rng(3)
    g = rng.standard_normal((2, 17)).astype(np.float32)
    r = np.zeros_like(g)
    idx, val, nnz = oracle.topk_ef(g, r, 17, 1, 1)
    assert list(nnz) == [17, 17] and (idx[:, :17] == np.arange(17)).all()
    assert not r.any()
    r = np.zeros_like(g)
    idx, val, nnz = oracle.topk_ef(g, r, 17, 0, 1)
    assert list(nnz) == [0, 0] and np.array_equal(r, g)


def test_topk_floor_rounding_of_k_matches_tiny_workload():
    # 1% of 65,536 per node is 655 entries: k_s is floor(d * n_s).
    assert oracle.segment_ks(65_536, 65_536, 1, 100) == [655]
    ks = oracle.segment_ks(25_557_032, 100_000, 1, 1000)
    assert len(ks) == 256 and ks[:-1] == [100] * 255 and ks[-1] == 57


@pytest.mark.parametrize("steps", [1, 4])
def test_error_feedback_invariant_transmitted_plus_residual_is_accumulated(steps):
    """§2.2/§4: what is not sent stays in the residual, bit for bit."""
    P, N = 3, 3000
    res = np.zeros((P, N), np.float32)
    for t in range(steps):
        g = W.normal_grad(P, N, 1.0, 100 + t).numpy()
        acc = res + g  # fp32 round-to-nearest add
        idx, val, nnz = oracle.topk_ef(g, res, 500, 1, 50)
        for p in range(P):
            sel = idx[p, :nnz[p]]
            assert np.all(np.diff(sel.astype(np.int64)) > 0)
            sent = np.zeros(N, np.float32)
            sent[sel] = val[p, :nnz[p]]
            assert np.array_equal((sent + res[p]).view(np.uint32), acc[p].view(np.uint32))
            assert not res[p, sel].view(np.uint32).any()  # +0.0 exactly
            # every kept magnitude >= every dropped one inside each segment
            for b in range(0, N, 500):
                m = np.zeros(N, bool)
                m[sel] = True
                seg = slice(b, b + 500)
                kept = keys(acc[p, seg][m[seg]])
                drop = keys(acc[p, seg][~m[seg]])
                assert kept.min() >= drop.max()


# --------------------------------------------------------------------------
# Sparse sum-reduction (§5.2) and dense switch (§5.1, §5.3.3).
# --------------------------------------------------------------------------
def brute_dense_sum(idx, val, nnz, N):
    out = np.zeros(N, np.float32)  # neutral element +0.0
    for p in range(idx.shape[0]):
        d = np.zeros(N, np.float32)
        d[idx[p, :nnz[p]]] = val[p, :nnz[p]]
        out = out + d
    return out


def random_streams(rng, P, N, maxk, tie_vals=False):
    cap = maxk
    idx = np.zeros((P, cap), np.uint32)
    val = np.zeros((P, cap), np.float32)
    nnz = np.zeros(P, np.uint32)
    for p in range(P):
        k = int(rng.integers(0, maxk + 1))
        sel = np.sort(rng.choice(N, size=k, replace=False))
        idx[p, :k] = sel
        val[p, :k] = tie_heavy(rng, k) if tie_vals else rng.standard_normal(k).astype(np.float32)
        nnz[p] = k
    return idx, val, nnz


@pytest.mark.parametrize("seed", range(8))
def test_reduce_equals_brute_force_dense_sum(seed):
    rng = np.random.default_rng(1000 + seed)
    P = int(rng.integers(1, 9))
    N = int(rng.integers(1, 200))
    idx, val, nnz = random_streams(rng, P, N, min(N, 60), tie_vals=seed % 2 == 1)
    r = oracle.sparse_reduce(idx, val, nnz, N)
    want = brute_dense_sum(idx, val, nnz, N)
    union = set()
    for p in range(P):
        union |= set(idx[p, :nnz[p]].tolist())
    assert r["nnz"] == len(union)
    assert r["is_dense"] == (4 * len(union) > N)
    if r["is_dense"]:
        assert np.array_equal(r["dense"].view(np.uint32), want.view(np.uint32))
    else:
        assert list(r["idx"]) == sorted(union)
        assert np.array_equal(r["val"].view(np.uint32), want[sorted(union)].view(np.uint32))


def test_reduce_size_bounds_disjoint_and_identical():
    N, P, k = 4096, 8, 100
    rng = np.random.default_rng(5)
    perm = rng.permutation(N)[: P * k].reshape(P, k)
    idx = np.sort(perm, axis=1).astype(np.uint32)
    val = rng.standard_normal((P, k)).astype(np.float32)
    nnz = np.full(P, k, np.uint32)
    r = oracle.sparse_reduce(idx, val, nnz, N)
    assert r["nnz"] == P * k  # App. B: union bound tight for disjoint sets (allgather)
    same = np.tile(idx[:1], (P, 1))
    r2 = oracle.sparse_reduce(same, val, nnz, N)
    assert r2["nnz"] == k  # §5.3.1: full overlap keeps k items
    for P2 in (1, 3, 16):
        i2, v2, n2 = uniform_small = W.uniform_streams(P2, N, 300, 77)
        assert oracle.sparse_reduce(i2, v2, n2, N)["nnz"] <= min(N, P2 * 300)


def test_dense_switch_exactly_at_quarter():
    N = 64
    for U, dense in ((16, False), (17, True)):
        idx = np.arange(U, dtype=np.uint32)[None, :]
        val = np.ones((1, U), np.float32)
        r = oracle.sparse_reduce(idx, val, np.array([U], np.uint32), N)
        assert r["nnz"] == U and r["is_dense"] == dense
        if dense:
            assert r["dense"][:U].tolist() == [1.0] * U and not r["dense"][U:].any()


def test_reduce_signed_zero_and_cancellation_keep_structural_support():
    idx = np.array([[3, 5], [3, 5]], np.uint32)
    val = np.array([[-0.0, 2.5], [-0.0, -2.5]], np.float32)
    r = oracle.sparse_reduce(idx, val, np.array([2, 2], np.uint32), 1000)
    assert r["nnz"] == 2 and list(r["idx"]) == [3, 5]
    assert r["val"].view(np.uint32).tolist() == [0, 0]  # +0.0 both (sum from +0.0)


def test_reduce_rejects_bad_streams():
    with pytest.raises(oracle.OracleError):
        oracle.sparse_reduce(np.array([[4, 2]], np.uint32), np.ones((1, 2), np.float32),
                             np.array([2], np.uint32), 10)
    with pytest.raises(oracle.OracleError):
        oracle.sparse_reduce(np.array([[4, 10]], np.uint32), np.ones((1, 2), np.float32),
                             np.array([2], np.uint32), 10)


@pytest.mark.parametrize("P,dnum,dden", [(2, 1, 100), (8, 1, 100), (8, 10, 100), (32, 5, 100)])
def test_density_law_uniform_indices(P, dnum, dden):
    """App. B.1 / uniform model: E[U]/N = 1 - (1 - d)^P for k = dN distinct indices."""
    N = 1 << 18
    k = N * dnum // dden
    idx, val, nnz = W.uniform_streams(P, N, k, 900 + P)
    r = oracle.sparse_reduce(idx, val, nnz, N)
    d = k / N
    q = 1 - (1 - d) ** P
    assert abs(r["nnz"] / N - q) <= 6 * math.sqrt(q * (1 - q) / N)
    assert r["is_dense"] == (4 * r["nnz"] > N)


def test_density_law_small_n_mean_over_seeds():
    """Figure 7's setting (N = 512): mean union size over seeds follows the closed form."""
    N, P, k, M = 512, 8, 32, 300
    us = []
    for s in range(M):
        idx, val, nnz = W.uniform_streams(P, N, k, 5000 + s)
        us.append(oracle.sparse_reduce(idx, val, nnz, N)["nnz"])
    q = 1 - (1 - k / N) ** P
    sd = math.sqrt(N * q * (1 - q))
    assert abs(np.mean(us) - N * q) <= 6 * sd / math.sqrt(M)
    assert max(us) <= min(N, P * k)


# --------------------------------------------------------------------------
# 4-bit stochastic quantisation (§2.2, §6).
# --------------------------------------------------------------------------
def unpack(codes, n):
    lo = codes & 0x0F
    hi = codes >> 4
    out = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out[..., :n]


def test_quantizer_bounds_levels_signs_and_max_entry():
    rng = np.random.default_rng(11)
    P, cap, bucket = 3, 1300, 512
    val = (rng.laplace(size=(P, cap)) * 1e-3).astype(np.float32)
    idx = np.tile(np.arange(cap, dtype=np.uint32) * 3, (P, 1))
    nnz = np.array([1300, 1025, 7], np.uint32)
    codes, scales = oracle.quantize4(idx, val, nnz, bucket, seed=42)
    deq = oracle.dequantize4(codes, scales, nnz, cap, bucket)
    cl = unpack(codes, cap)
    for p in range(P):
        n = int(nnz[p])
        for b0 in range(0, n, bucket):
            b1 = min(b0 + bucket, n)
            v = val[p, b0:b1]
            s = scales[p, b0 // bucket]
            assert s == np.abs(v).max()
            lv = cl[p, b0:b1] & 7
            sg = cl[p, b0:b1] >> 3
            assert np.array_equal(sg, (v < 0).astype(np.uint8))
            for j in range(len(v)):
                r = Fraction(float(abs(v[j]))) / Fraction(float(s)) * 7
                assert math.floor(r - Fraction(1, 10**5)) <= lv[j] <= math.ceil(r + Fraction(1, 10**5))
            assert np.all(np.abs(deq[p, b0:b1].astype(np.float64) - v) <= s / 7 * (1 + 1e-6))
            m = int(np.argmax(np.abs(v)))
            assert deq[p, b0 + m] == v[m]  # the bucket maximum is exact (level 7)


def test_quantizer_zero_bucket_gives_positive_zeros():
    idx = np.arange(10, dtype=np.uint32)[None]
    val = np.array([[0.0, -0.0] * 5], np.float32)
    codes, scales = oracle.quantize4(idx, val, np.array([10], np.uint32), 4, seed=1)
    assert not scales.any() and not codes.any()
    deq = oracle.dequantize4(codes, scales, np.array([10], np.uint32), 10, 4)
    assert not deq.view(np.uint32).any()


def test_quantizer_rounds_up_with_probability_frac():
    """r = 2.25 for every entry: about a quarter round up to level 3."""
    n = 40000
    val = np.full((1, n), 2.25, np.float32)
    val[0, 0] = 7.0  # bucket scale 7 => r = |v| exactly
    idx = np.arange(n, dtype=np.uint32)[None]
    codes, _ = oracle.quantize4(idx, val, np.array([n], np.uint32), n, seed=9)
    lv = unpack(codes, n)[0, 1:] & 7
    assert set(np.unique(lv).tolist()) <= {2, 3}
    frac_up = np.mean(lv == 3)
    assert abs(frac_up - 0.25) <= 6 * math.sqrt(0.25 * 0.75 / (n - 1))


def test_quantizer_is_unbiased_over_seeds():
    """§2.2: zero-mean quantisation noise, E[Q(v)] = v."""
    rng = np.random.default_rng(2)
    n, M = 64, 3000
    val = rng.standard_normal((1, n)).astype(np.float32)
    idx = np.arange(n, dtype=np.uint32)[None] * 11
    nnz = np.array([n], np.uint32)
    acc = np.zeros(n)
    for s in range(M):
        c, sc = oracle.quantize4(idx, val, nnz, n, seed=s * 7919 + 1)
        acc += oracle.dequantize4(c, sc, nnz, n, n)[0]
    scale = np.abs(val).max()
    sd = scale / 14  # level spacing scale/7, Bernoulli sd <= 1/2 of it
    assert np.all(np.abs(acc / M - val[0]) <= 6 * sd / math.sqrt(M) + 1e-7)


def test_quantizer_draw_depends_only_on_seed_node_index():
    rng = np.random.default_rng(4)
    n = 512
    val = rng.standard_normal((2, n)).astype(np.float32)
    val[:, 0] = 10.0  # same scale in both nodes
    idx = np.tile(np.arange(n, dtype=np.uint32), (2, 1))
    nnz = np.array([n, n], np.uint32)
    c1, _ = oracle.quantize4(idx, val, nnz, n, seed=5)
    val2 = val.copy()
    val2[:, 1:] = val[:, 1:][:, ::-1]  # move other entries around
    c2, _ = oracle.quantize4(idx, val2, nnz, n, seed=5)
    l1, l2 = unpack(c1, n), unpack(c2, n)
    # entry j of val2 equals entry (n - j) of val: different index, so its draw may differ,
    # but the unchanged entry 0 and its code are fixed
    assert l1[0, 0] == l2[0, 0] == 7
    # same values, same (node, index) => same code whatever the other entries are
    val3 = val.copy()
    val3[0, 2:] *= 0.5
    c3, _ = oracle.quantize4(idx, val3, nnz, n, seed=5)
    assert unpack(c3, n)[0, 1] == l1[0, 1]
    # a different node key changes some draws
    c4, _ = oracle.quantize4(idx[::-1].copy(), val[::-1].copy(), nnz, n, seed=5)
    assert not np.array_equal(unpack(c4, n)[1], l1[0])


def sm64_py(x):
    """SplitMix64 output for state x in Python integers, written from the
    published algorithm (Steele, Lea and Flood 2014, with Vigna's 64-bit
    finaliser): add the golden gamma, then two xor-shift-multiply rounds and a
    last xor-shift."""
    z = (x + GOLDEN_RATIO_INC) & M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
    return z ^ (z >> 31)


def test_python_splitmix64_matches_the_published_vector():
    with open(os.path.join(GOLDEN, "splitmix64_seed1234567.txt")) as f:
        expect = [int(l) for l in f if l.strip() and not l.startswith("#")]
    state = 1234567
    for e in expect:
        assert sm64_py(state) == e
        state = (state + GOLDEN_RATIO_INC) & M64


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("seed", [5, 0x0123456789ABCDEF])
def test_quantizer_draw_key_known_answers(bits, seed):
    """Known answers for the rounding draw u = (h >> 40) 2^-24 with
    h = sm(sm(sm(seed) ^ node) ^ index): each case puts frac(r) a hair above
    or below the u of its (seed, node, index), computed here with the
    independent Python SplitMix64, so the level (floor(r) or floor(r) + 1)
    pins the whole key. A slip in the key (a dropped sm(seed), node and index
    folded into one state, a swapped pair) draws another u and flips about
    half of the 24 decisions."""
    s = (1 << (bits - 1)) - 1
    base = {2: 0, 4: 3, 8: 60}[bits]
    rng = np.random.default_rng(seed & 0xFFFF)
    P, per_row = 4, 6
    f32 = np.float32
    cap = 2 * per_row
    idx = np.zeros((P, cap), np.uint32)
    val = np.zeros((P, cap), f32)
    expect = np.zeros((P, per_row), np.int64)
    for p in range(P):
        ix = np.sort(rng.choice(1 << 32, size=cap, replace=False)).astype(np.uint64)
        for c in range(per_row):
            i0, i = int(ix[2 * c]), int(ix[2 * c + 1])
            h = sm64_py(sm64_py(sm64_py(seed) ^ p) ^ i)
            u = f32(h >> 40) * f32(1.0 / 16777216.0)
            up = (c + p) % 2 == 0  # half the cases just above u, half just below
            target = float(base) + float(u) + (3e-6 if up else -3e-6)
            if not (0.0 < target - base < 1.0):
                target = float(base) + 0.5
            v = f32(target / s)
            r = f32(f32(v / f32(1.0)) * f32(s))
            frac = r - np.floor(r)
            assert abs(float(frac) - float(u)) < 1e-5 or target == base + 0.5
            expect[p, c] = int(np.floor(r)) + (1 if u < frac else 0)
            idx[p, 2 * c], idx[p, 2 * c + 1] = i0, i
            val[p, 2 * c], val[p, 2 * c + 1] = 1.0, v
    nnz = np.full(P, cap, np.uint32)
    codes, scales = oracle.quantize(val, 4, bits, seed, idx=idx, nnz=nnz)  # scale 1 per bucket
    lv = unpack_bits(codes, cap, bits) & s
    assert (scales == 1.0).all()
    assert (lv[:, 0::2] == s).all()  # the bucket maximum: r = s exactly
    assert np.array_equal(lv[:, 1::2], expect)
    if bits == 4:
        c4, _ = oracle.quantize4(idx, val, nnz, 4, seed)
        assert np.array_equal(c4, codes)


def unpack_bits(codes, n, bits):
    """codes [P][ceil(n / (8/b))] -> [P][n], the earliest entry in the lowest bits."""
    per = 8 // bits
    out = np.empty(codes.shape[:-1] + (codes.shape[-1] * per,), np.uint8)
    for k in range(per):
        out[..., k::per] = (codes >> (k * bits)) & ((1 << bits) - 1)
    return out[..., :n]


def test_general_quantizer_at_4_bits_is_the_4bit_form():
    rng = np.random.default_rng(21)
    P, cap = 3, 1300
    val = (rng.laplace(size=(P, cap)) * 1e-3).astype(np.float32)
    idx = np.tile(np.arange(cap, dtype=np.uint32) * 5, (P, 1))
    nnz = np.array([1300, 1025, 7], np.uint32)
    c4, s4 = oracle.quantize4(idx, val, nnz, 512, seed=3)
    c, sc = oracle.quantize(val, 512, 4, 3, idx=idx, nnz=nnz)
    assert np.array_equal(c, c4) and np.array_equal(sc.view(np.uint32), s4.view(np.uint32))
    d4 = oracle.dequantize4(c4, s4, nnz, cap, 512)
    d = oracle.dequantize(c, sc, cap, 512, 4, nnz=nnz)
    assert np.array_equal(d.view(np.uint32), d4.view(np.uint32))


@pytest.mark.parametrize("bits", [2, 8])
def test_b_bit_quantizer_bounds_levels_signs_and_max_entry(bits):
    """§6, 2- and 8-bit outputs: s = 2^(b-1) - 1 levels of the bucket max."""
    rng = np.random.default_rng(bits)
    s_lv = (1 << (bits - 1)) - 1
    P, cap, bucket = 2, 1000, 256
    val = rng.standard_normal((P, cap)).astype(np.float32)
    idx = np.tile(np.arange(cap, dtype=np.uint32) * 2, (P, 1))
    nnz = np.array([1000, 513], np.uint32)
    codes, scales = oracle.quantize(val, bucket, bits, 77, idx=idx, nnz=nnz)
    deq = oracle.dequantize(codes, scales, cap, bucket, bits, nnz=nnz)
    cl = unpack_bits(codes, cap, bits)
    for p in range(P):
        n = int(nnz[p])
        for b0 in range(0, n, bucket):
            b1 = min(b0 + bucket, n)
            v = val[p, b0:b1]
            s = scales[p, b0 // bucket]
            assert s == np.abs(v).max()
            lv = cl[p, b0:b1] & s_lv
            assert np.array_equal(cl[p, b0:b1] >> (bits - 1), (v < 0).astype(np.uint8))
            for j in range(len(v)):
                r = Fraction(float(abs(v[j]))) / Fraction(float(s)) * s_lv
                assert math.floor(r - Fraction(1, 10**5)) <= lv[j] <= math.ceil(r + Fraction(1, 10**5))
            assert np.all(np.abs(deq[p, b0:b1].astype(np.float64) - v) <= s / s_lv * (1 + 1e-6))
            m = int(np.argmax(np.abs(v)))
            assert deq[p, b0 + m] == v[m]  # level s: the bucket maximum is exact


@pytest.mark.parametrize("bits,r", [(2, 0.3), (8, 40.75)])
def test_b_bit_quantizer_rounds_up_with_probability_frac(bits, r):
    s_lv = (1 << (bits - 1)) - 1
    n = 40000
    val = np.full((1, n), r, np.float32)
    val[0, 0] = float(s_lv)  # scale s => r = |v| exactly
    codes, _ = oracle.quantize(val, n, bits, 13)  # dense row: the position is the key
    lv = unpack_bits(codes, n, bits)[0, 1:] & s_lv
    f = r - math.floor(r)
    assert set(np.unique(lv).tolist()) <= {math.floor(r), math.floor(r) + 1}
    assert abs(np.mean(lv == math.floor(r) + 1) - f) <= 6 * math.sqrt(f * (1 - f) / (n - 1))


@pytest.mark.parametrize("bits", [2, 8])
def test_b_bit_quantizer_is_unbiased_over_seeds(bits):
    """§2.2: zero-mean quantisation noise at every width."""
    rng = np.random.default_rng(5)
    s_lv = (1 << (bits - 1)) - 1
    n, M = 64, 2000
    val = rng.standard_normal((1, n)).astype(np.float32)
    acc = np.zeros(n)
    for k in range(M):
        c, sc = oracle.quantize(val, n, bits, k * 104729 + 3)
        acc += oracle.dequantize(c, sc, n, n, bits)[0]
    sd = np.abs(val).max() / s_lv / 2
    assert np.all(np.abs(acc / M - val[0]) <= 6 * sd / math.sqrt(M) + 1e-7)


def test_dense_rows_quantise_like_a_stream_of_every_position():
    """A dense row is the stream idx = 0..n-1 of all its entries."""
    rng = np.random.default_rng(8)
    P, n = 3, 3000
    val = rng.standard_normal((P, n)).astype(np.float32)
    for bits in (2, 4, 8):
        cd, sd = oracle.quantize(val, 1024, bits, 99)
        cs, ss = oracle.quantize(val, 1024, bits, 99,
                                 idx=np.tile(np.arange(n, dtype=np.uint32), (P, 1)),
                                 nnz=np.full(P, n, np.uint32))
        assert np.array_equal(cd, cs) and np.array_equal(sd, ss)


def test_quantisation_error_output_completes_the_value():
    """Error feedback option: dequantised value + error gives the value back
    up to the one rounding of v - q, and the error is bounded by one level."""
    rng = np.random.default_rng(9)
    val = rng.standard_normal((2, 700)).astype(np.float32)
    for bits in (2, 4, 8):
        s_lv = (1 << (bits - 1)) - 1
        c, sc, err = oracle.quantize(val, 128, bits, 4, with_error=True)
        deq = oracle.dequantize(c, sc, 700, 128, bits)
        back = deq.astype(np.float64) + err.astype(np.float64)
        ulp = np.spacing(np.maximum(np.abs(val), np.abs(deq))).astype(np.float64)
        assert np.all(np.abs(back - val) <= ulp / 2)  # one rounding of v - q
        bmax = np.repeat(sc, 128, axis=1)[:, :700]
        assert np.all(np.abs(err) <= bmax / s_lv * (1 + 1e-6))


def test_quantizer_rejects_bucket_not_whole_bytes():
    val = np.ones((1, 8), np.float32)
    with pytest.raises(RuntimeError):
        oracle.quantize(val, 6, 2, 1)  # 2-bit codes pack 4 per byte


# --------------------------------------------------------------------------
# Other associative reductions with a neutral element (§5.2).
# --------------------------------------------------------------------------
NEUTRAL = {"sum": 0.0, "max": -np.inf, "min": np.inf, "or": 0.0}


def dense_fold(dense_rows, op):
    """Fold [P][N] rows over nodes in order with numpy's own elementwise ops."""
    if op == "or":
        r = np.bitwise_or.reduce(dense_rows.view(np.uint32), axis=0)
        return r.view(np.float32)
    if op == "sum":
        acc = np.zeros(dense_rows.shape[1], np.float32)
        for row in dense_rows:
            acc = acc + row
        return acc
    f = np.maximum if op == "max" else np.minimum
    return f.reduce(dense_rows, axis=0)


@pytest.mark.parametrize("op", ["max", "min", "or"])
@pytest.mark.parametrize("seed", range(3))
def test_reduce_op_equals_brute_force_dense_fold(op, seed):
    """Each stream is the vector with the neutral element at unlisted indices;
    the reduced vector is the elementwise fold, and U the union's size."""
    rng = np.random.default_rng(100 + seed)
    P, N = 5, 300
    k = int(rng.integers(10, 120))
    idx = np.zeros((P, k), np.uint32)
    val = rng.standard_normal((P, k)).astype(np.float32)
    nnz = rng.integers(0, k + 1, size=P).astype(np.uint32)
    dense = np.full((P, N), NEUTRAL[op], np.float32)
    union = set()
    for p in range(P):
        sel = np.sort(rng.choice(N, size=int(nnz[p]), replace=False)).astype(np.uint32)
        idx[p, :nnz[p]] = sel
        dense[p, sel] = val[p, :nnz[p]]
        union |= set(sel.tolist())
    want = dense_fold(dense, op)
    r = oracle.sparse_reduce_op(idx, val, nnz, N, op, 1, 1000)  # forced dense
    assert r["is_dense"] and r["nnz"] == len(union)
    assert np.array_equal(r["dense"].view(np.uint32), want.view(np.uint32))
    r = oracle.sparse_reduce_op(idx, val, nnz, N, op, 1, 1)  # never dense
    assert np.array_equal(r["idx"], np.array(sorted(union), np.uint32))
    assert np.array_equal(r["val"].view(np.uint32), want[r["idx"]].view(np.uint32))


def test_reduce_op_sum_is_the_sum_reduce_and_idempotent_ops_keep_a_stream():
    rng = np.random.default_rng(7)
    P, N, k = 4, 5000, 900
    idx, val, nnz = (np.zeros((P, k), np.uint32), rng.standard_normal((P, k)).astype(np.float32),
                     np.full(P, k, np.uint32))
    for p in range(P):
        idx[p] = np.sort(rng.choice(N, k, replace=False))
    a = oracle.sparse_reduce(idx, val, nnz, N, 1, 1)  # sparse output either way
    b = oracle.sparse_reduce_op(idx, val, nnz, N, "sum", 1, 1)
    assert a["nnz"] == b["nnz"] and np.array_equal(a["idx"], b["idx"])
    assert np.array_equal(a["val"].view(np.uint32), b["val"].view(np.uint32))
    same_i = np.tile(idx[:1], (3, 1))
    same_v = np.tile(val[:1], (3, 1))
    for op in ("max", "min", "or"):  # x op x = x: three copies reduce to the stream
        r = oracle.sparse_reduce_op(same_i, same_v, np.full(3, k, np.uint32), N, op)
        assert np.array_equal(r["idx"], idx[0])
        assert np.array_equal(r["val"].view(np.uint32), val[0].view(np.uint32))


def test_reduce_op_ties_keep_the_lower_node_and_dense_absent_is_neutral():
    idx = np.array([[3], [3]], np.uint32)
    nnz = np.array([1, 1], np.uint32)
    pz_nz = np.array([[0.0], [-0.0]], np.float32)
    r = oracle.sparse_reduce_op(idx, pz_nz, nnz, 4, "max", 1, 8)
    assert r["dense"][3].view(np.uint32) == np.float32(0.0).view(np.uint32)  # +0 kept
    r = oracle.sparse_reduce_op(idx, pz_nz[::-1].copy(), nnz, 4, "min", 1, 8)
    assert r["dense"][3].view(np.uint32) == np.float32(-0.0).view(np.uint32)  # -0 kept
    for op in ("max", "min", "or"):
        r = oracle.sparse_reduce_op(idx, pz_nz, nnz, 4, op, 1, 8)
        assert r["is_dense"] and r["nnz"] == 1
        rest = np.delete(r["dense"], 3)
        assert np.array_equal(rest.view(np.uint32),
                              np.full(3, NEUTRAL[op], np.float32).view(np.uint32))


# --------------------------------------------------------------------------
# Static sparse allreduce by recursive doubling (§5.3.1).
# --------------------------------------------------------------------------
def disjoint_or_same(P, k, N, same, rng):
    if same:
        base = np.sort(rng.choice(N, k, replace=False)).astype(np.uint32)
        idx = np.tile(base, (P, 1))
    else:
        perm = rng.permutation(N)[:P * k].reshape(P, k)
        idx = np.sort(perm, axis=1).astype(np.uint32)
    return idx, rng.standard_normal((P, k)).astype(np.float32), np.full(P, k, np.uint32)


@pytest.mark.parametrize("P", [2, 4, 8, 16])
def test_ssar_fill_in_identical_and_disjoint_sets(P):
    """§5.3.1: fully overlapping indices keep every intermediate result at k
    items; disjoint indices double them at each stage (App. B: union of
    disjoint sets = sum of sizes)."""
    rng = np.random.default_rng(P)
    k, N = 300, 100_000
    stages = P.bit_length() - 1
    idx, val, nnz = disjoint_or_same(P, k, N, True, rng)
    _, _, fill = oracle.ssar(idx, val, nnz, N)
    assert fill.tolist() == [(P >> (s + 1)) * k for s in range(stages)]
    idx, val, nnz = disjoint_or_same(P, k, N, False, rng)
    oi, _, fill = oracle.ssar(idx, val, nnz, N)
    assert fill.tolist() == [P * k] * stages
    assert np.array_equal(oi, np.sort(idx.reshape(-1)))


@pytest.mark.parametrize("P", [2, 8, 32])
def test_ssar_equals_the_sequential_reduce_when_sums_are_exact(P):
    """With small integer values every sum is exact, so the recursive-doubling
    order gives the sequential reduce's result bit for bit; with P = 2 it is
    that reduce for any values."""
    rng = np.random.default_rng(40 + P)
    N, k = 5000, 700
    idx = np.zeros((P, k), np.uint32)
    for p in range(P):
        idx[p] = np.sort(rng.choice(N, k, replace=False))
    val = rng.integers(-1000, 1000, size=(P, k)).astype(np.float32)
    nnz = rng.integers(0, k + 1, size=P).astype(np.uint32)
    oi, ov, _ = oracle.ssar(idx, val, nnz, N)
    ref = oracle.sparse_reduce(idx, val, nnz, N, 1, 1)
    assert np.array_equal(oi, ref["idx"]) and np.array_equal(ov.view(np.uint32), ref["val"].view(np.uint32))
    if P == 2:
        val2 = rng.standard_normal((2, k)).astype(np.float32)
        oi, ov, _ = oracle.ssar(idx, val2, nnz, N)
        ref = oracle.sparse_reduce(idx, val2, nnz, N, 1, 1)
        assert np.array_equal(ov.view(np.uint32), ref["val"].view(np.uint32))


@pytest.mark.parametrize("P", [4, 8, 16])
def test_ssar_equals_a_dense_pairwise_tree_brute_force(P):
    """Recursive doubling (§5.3.1) written out densely with numpy: at stage s
    group g adds (+0 + lower half) + upper half element-wise, absent entries
    being +0.0, and the support is the union of the halves' supports. With
    N(0, 1) values the sums round, so this pins the tree order bit for bit,
    and the stage sizes are the unions' sizes (App. B)."""
    rng = np.random.default_rng(70 + P)
    N, k = 3000, 400
    idx = np.zeros((P, k), np.uint32)
    for p in range(P):
        idx[p] = np.sort(rng.choice(N, k, replace=False))
    val = rng.standard_normal((P, k)).astype(np.float32)
    val[:, ::11] = -0.0
    nnz = rng.integers(0, k + 1, size=P).astype(np.uint32)
    dense = np.zeros((P, N), np.float32)
    here = np.zeros((P, N), bool)
    for p in range(P):
        dense[p, idx[p, :nnz[p]]] = val[p, :nnz[p]]
        here[p, idx[p, :nnz[p]]] = True
    fill = []
    while dense.shape[0] > 1:
        dense = (np.float32(0.0) + dense[0::2]) + dense[1::2]
        here = here[0::2] | here[1::2]
        fill.append(int(here.sum()))
    oi, ov, of = oracle.ssar(idx, val, nnz, N)
    assert of.tolist() == fill
    assert np.array_equal(oi, np.flatnonzero(here[0]).astype(np.uint32))
    assert np.array_equal(ov.view(np.uint32), dense[0, oi].view(np.uint32))


def test_ssar_needs_a_power_of_two():
    with pytest.raises(RuntimeError):
        oracle.ssar(np.zeros((3, 1), np.uint32), np.zeros((3, 1), np.float32),
                    np.zeros(3, np.uint32), 10)


# --------------------------------------------------------------------------
# Pack and densify (§5.1).
# --------------------------------------------------------------------------
def test_pack_and_densify_round_trip():
    rng = np.random.default_rng(8)
    P, N = 4, 999
    x = rng.standard_normal((P, N)).astype(np.float32)
    x[rng.random((P, N)) < 0.7] = 0.0
    x[0, 5] = -0.0
    idx, val, nnz, st = oracle.pack(x, 0.0, N)
    assert st == oracle.OK
    d = oracle.densify(idx, val, nnz, N)
    assert np.array_equal(d, x)
    for p in range(P):
        assert int(nnz[p]) == sum(1 for i in range(N) if abs(float(x[p, i])) > 0.0)
    idx2, val2, nnz2, st2 = oracle.pack(x, 0.5, N)
    for p in range(P):
        sel = idx2[p, :nnz2[p]]
        assert np.all(np.abs(x[p, sel]) > 0.5)
        rest = np.setdiff1d(np.arange(N), sel)
        assert np.all(np.abs(x[p, rest]) <= 0.5)
    _, _, nnz3, st3 = oracle.pack(x, 0.0, 5)
    assert st3 == oracle.CAPACITY and list(nnz3) == [5] * P


def test_reduce_single_node_is_densify():
    rng = np.random.default_rng(9)
    N = 100
    idx = np.sort(rng.choice(N, size=90, replace=False)).astype(np.uint32)[None]
    val = rng.standard_normal((1, 90)).astype(np.float32)
    nnz = np.array([90], np.uint32)
    r = oracle.sparse_reduce(idx, val, nnz, N)
    d = oracle.densify(idx, val, nnz, N)[0]
    assert r["is_dense"]
    assert np.array_equal((d + np.float32(0)).view(np.uint32), r["dense"].view(np.uint32))
