"""GPU parity of Top-k with error feedback (SparCML §2.2, §4, §8.4) against the
oracle: indices, nnz, values and the residual must match bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from top_gradient_compression_gb300 import api, workloads as W

from gpu_helpers import DEV, bits, check_topk_steps, check_topk_table_steps, u32

pytestmark = pytest.mark.gpu


def make(dist, P, N, seed):
    rng = np.random.default_rng(seed)
    if dist == "normal":
        return rng.standard_normal((P, N)).astype(np.float32)
    if dist == "laplace":
        return (rng.laplace(size=(P, N)) * 1e-3).astype(np.float32)
    if dist == "ties":  # a handful of magnitudes: large equal-key groups at the boundary
        pool = np.array([0.0, -0.0, 1.0, -1.0, 2.0, -2.0, 0.5, -0.5, 3.0], np.float32)
        return pool[rng.integers(0, len(pool), size=(P, N))]
    if dist == "const":  # one magnitude everywhere: every entry ties
        return np.where(rng.random((P, N)) < 0.5, 1.5, -1.5).astype(np.float32)
    raise ValueError(dist)


def test_tiny_workload_three_steps():
    c = W.TINY
    grads = [W.tiny_grads(t).numpy() for t in range(c["steps"])]
    check_topk_steps(grads, c["seg_len"], c["k_num"], c["k_den"], fallback=False)


@pytest.mark.parametrize("P,N,seg_len,k_num,k_den,dist,fallback", [
    (3, 1001, 100, 3, 100, "normal", False),         # node bases not 16-byte aligned
    (2, 50_000, 7_000, 1, 50, "ties", False),         # ragged segments, heavy ties
    (1, 3 * 8192 + 5, 8192, 1, 10, "normal", False),  # chunk-sized segments + ragged tail
    (2, 40, 1, 1, 1, "normal", False),                # segment length 1, k = n
    (2, 1000, 1000, 0, 1, "normal", False),           # k = 0
    (2, 777, 777, 1, 1, "ties", False),               # k = n with ties
    (1, 1 << 21, 1 << 21, 1, 100, "normal", False),   # one long segment
    (2, 4_194_304, 4_194_304, 1, 100, "laplace", False),  # long segments
    (2, 300_000, 100_000, 1, 1000, "normal", False),  # layer-sized segments, k = 100
    (4, 65_536, 65_536, 30, 100, "ties", False),      # 30 %: range-parallel select, ties
    (2, 20_000, 20_000, 1, 100, "const", True),       # all keys equal: sub-slots overflow
])
def test_topk_shapes(P, N, seg_len, k_num, k_den, dist, fallback):
    grads = [make(dist, P, N, s) for s in range(2)]
    check_topk_steps(grads, seg_len, k_num, k_den, fallback=fallback)


def table(lens, ks):
    return [0] + list(np.cumsum(lens).astype(int)), list(ks)


def test_topk_segment_table_mixed_sizes():
    """Layer-wise sparsification over a ragged table in one call (§8.4):
    segments of 1, 7, 100,000 and more than 2^18 entries, every kind of
    segment (k = 0, k = n, sampled whole, layer-sized, long), offsets that are
    not multiples of 4, k_s from 0 to n_s."""
    lens = [1, 7, 100_000, 300_001, 1, 7, 13, 8_192, 8_193, 262_144, 262_147, 1_100_000, 5]
    ks = [0, 7, 100, 3_000, 1, 0, 13, 81, 1_000, 2_621, 26_214, 11_000, 2]
    P = 3
    b, k = table(lens, ks)
    grads = [make("normal", P, b[-1], 40 + t) for t in range(3)]
    check_topk_table_steps(grads, b, k, fallback=False)


@pytest.mark.parametrize("seed", range(3))
def test_topk_segment_table_random(seed):
    rng = np.random.default_rng(500 + seed)
    lens = list(rng.choice([1, 3, 64, 1_000, 9_000, 70_000, 300_000], size=24))
    ks = [int(rng.integers(0, n + 1)) if rng.random() < 0.3 else max(0, n // 100) for n in lens]
    b, k = table(lens, ks)
    P = 2
    grads = [make("laplace" if seed % 2 else "normal", P, b[-1], 60 + 3 * seed + t)
             for t in range(2)]
    check_topk_table_steps(grads, b, k)


def test_topk_long_segments_keep_all_none_and_dense():
    """Long segments (> 2^18) that keep nothing, everything (written straight
    from the stream pass), 90 % (candidates almost everywhere) and 0.01 %."""
    lens = [300_000, 400_003, 600_000, 350_000]
    ks = [0, 400_003, 540_000, 35]
    b, k = table(lens, ks)
    grads = [make("normal", 2, b[-1], 70 + t) for t in range(2)]
    check_topk_table_steps(grads, b, k, fallback=False)


@pytest.mark.parametrize("dist", ["ties", "const"])
def test_topk_long_segment_falls_back_to_the_raw_select(dist):
    """A long segment whose candidates cannot decide the select (a boundary
    bin far above its buffer, or sub-slots that overflow): the raw select
    re-reads the segment's acc and gives the same bits."""
    P, N = 2, 1 << 21
    grads = [make(dist, P, N, 80 + t) for t in range(2)]
    # the first EF step sees the raw tie groups; later steps add the residual,
    # which splits them, so only the first step is sure to fall back
    check_topk_steps(grads[:1], N, 1, 100, fallback=True)
    check_topk_steps(grads, N, 1, 100)
    b, k = table([N // 2 + 3, N // 2 - 3], [10_000, 5])
    check_topk_table_steps(grads[:1], b, k, fallback=True)
    check_topk_table_steps(grads, b, k)


def test_topk_const_keeps_lowest_indices():
    P, N = 2, 100_000  # sampled segment, every key equal: candidate slots overflow
    g = make("const", P, N, 7)
    res = torch.zeros((P, N), device=DEV)
    idx, val, nnz = api.topk_ef(torch.from_numpy(g).to(DEV), res, N, 1, 100)
    k = N // 100
    assert (u32(idx)[:, :k] == np.arange(k)).all()
    check_topk_steps([g], N, 1, 100)


def test_topk_sample_overestimates_then_falls_back():
    """Large values only where the guess pass samples: too few candidates, so the
    select pass re-reads the segment. The result is still exact."""
    P, N = 1, 1 << 20
    n_runs, run = 32, 256  # the guess pass reads 32 runs of 256 entries of a long segment
    g = (np.random.default_rng(3).standard_normal((P, N)) * 0.01).astype(np.float32)
    for i in range(n_runs):
        st = (i * (N - run) // (n_runs - 1)) & ~(run - 1)
        g[0, st:st + run] = 10.0 + i
    check_topk_steps([g], N, 1, 100, fallback=True)  # k = 10,485 > 8,192 sampled entries


def test_topk_nonzero_initial_residual():
    rng = np.random.default_rng(5)
    P, N = 3, 70_000
    res0 = rng.standard_normal((P, N)).astype(np.float32)
    grads = [rng.standard_normal((P, N)).astype(np.float32) for _ in range(3)]
    check_topk_steps(grads, 30_000, 1, 100, res0=res0)


def test_topk_deterministic_and_capacity_checked():
    P, N = 2, 100_000
    g = torch.from_numpy(make("normal", P, N, 1)).to(DEV)
    r1 = torch.zeros_like(g)
    r2 = torch.zeros_like(g)
    a = api.topk_ef(g, r1, N, 1, 100)
    b = api.topk_ef(g, r2, N, 1, 100)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1]) and torch.equal(r1, r2)
    with pytest.raises(api.SparcmlError):
        small = (torch.empty((P, 10), dtype=torch.int32, device=DEV),
                 torch.empty((P, 10), device=DEV), torch.empty(P, dtype=torch.int32, device=DEV))
        api.topk_ef(g, r1, N, 1, 100, out=small)


@pytest.mark.slow
def test_resnet50_workload_sampled_segments_ten_steps():
    """Full ResNet-50-sized workload (P=8, N=25,557,032, 256 layer blocks, k=0.1%)
    through the same calls the benchmark times; the oracle checks a sample of
    (node, segment) pairs over all 10 EF steps (segments are independent)."""
    c = W.RESNET50
    P, N, L = c["P"], c["N"], c["seg_len"]
    # one segment on every node, node 7's ragged last segment, and a few more
    picks = [(0, 0), (1, 37), (2, 74), (3, 111), (4, 148), (5, 185), (6, 222), (7, 255),
             (0, 137), (5, 1), (3, 200)]
    res_g = torch.zeros((P, N), device=DEV)
    ws = api.workspace(api.topk_ef_workspace_size(P, N, L, c["k_num"], c["k_den"]), DEV)
    res_o = {pk: np.zeros((1, min(L, N - pk[1] * L)), np.float32) for pk in picks}
    for t in range(c["steps"]):
        g = W.resnet50_grads(t, device=DEV)
        idx, val, nnz = api.topk_ef(g, res_g, L, c["k_num"], c["k_den"], ws=ws)
        assert api.get_status(ws) == 0
        gi, gv, gr = u32(idx), bits(val.cpu().numpy()), None
        for (p, s) in picks:
            lo, n = s * L, res_o[(p, s)].shape[1]
            gs = g[p, lo:lo + n].cpu().numpy()[None]
            oi, ov, on = oracle.topk_ef(gs, res_o[(p, s)], n, c["k_num"], c["k_den"])
            k = int(on[0])
            off = s * (L * c["k_num"] // c["k_den"])
            assert np.array_equal(gi[p, off:off + k], oi[0, :k] + lo)
            assert np.array_equal(gv[p, off:off + k], bits(ov[0, :k]))
            assert np.array_equal(bits(res_g[p, lo:lo + n].cpu().numpy()), bits(res_o[(p, s)][0]))
        assert (u32(nnz) == api.segment_k_total(N, L, c["k_num"], c["k_den"])).all()
    # every node's stream is strictly ascending and inside [0, N)
    for p in range(P):
        s = gi[p, :int(u32(nnz)[p])].astype(np.int64)
        assert (np.diff(s) > 0).all() and s[-1] < N


@pytest.mark.slow
def test_asr_workload_nodes_0_8_15_three_steps_then_quantised_reduce():
    """Full LSTM/ASR-like workload (P=16, N=67,108,864, one segment per node,
    k=1%, Laplace(0, 1e-3)): nodes 0, 8 and 15 (whose rows start at byte 0,
    2^31 and 4.03e9 of the batch) are checked against the oracle on all 3 EF
    steps, streams and residual; then every node's stream is 4-bit quantised
    (buckets of 512) and reduced with the fused dequantising reduce, checked
    against the oracle quantiser, dequantiser and map-based sum."""
    c = W.ASR
    P, N, L = c["P"], c["N"], c["seg_len"]
    nodes = [0, 8, 15]
    res_g = torch.zeros((P, N), device=DEV)
    res_o = np.zeros((len(nodes), N), np.float32)
    ws = api.workspace(api.topk_ef_workspace_size(P, N, L, c["k_num"], c["k_den"]), DEV)
    seg_b, seg_k = oracle.uniform_segments(N, L, c["k_num"], c["k_den"])
    for t in range(c["steps"]):
        g = W.asr_grads(t, device=DEV)
        idx, val, nnz = api.topk_ef(g, res_g, L, c["k_num"], c["k_den"], ws=ws)
        assert api.get_status(ws) == 0
        gh = np.stack([g[p].cpu().numpy() for p in nodes])
        del g
        oi, ov, on = oracle.topk_ef_segments(gh, res_o, seg_b, seg_k, threads=len(nodes))
        k = int(on[0])
        assert k == N // 100 and (u32(nnz) == k).all()
        for q, p in enumerate(nodes):
            assert np.array_equal(u32(idx[p]), oi[q, :k]), f"node {p} step {t}: indices"
            assert np.array_equal(bits(val[p].cpu().numpy()), bits(ov[q, :k])), f"node {p}: values"
            assert np.array_equal(bits(res_g[p].cpu().numpy()), bits(res_o[q])), f"node {p}: residual"
    del res_o
    bucket, seed = c["bucket"], W.quant_seed(c["steps"] - 1)
    codes, scales = api.quantize4(idx, val, nnz, bucket, seed)
    hi, hv, hn = u32(idx), val.cpu().numpy(), u32(nnz)
    oc, osc = oracle.quantize4(hi, hv, hn, bucket, seed)
    assert np.array_equal(codes.cpu().numpy(), oc)  # k is even: every nibble is valid
    assert np.array_equal(bits(scales.cpu().numpy()), bits(osc))
    deq = oracle.dequantize4(oc, osc, hn, hi.shape[1], bucket)
    ref = oracle.sparse_reduce(hi, deq, hn, N, threads=8)
    out = api.sparse_reduce_q4(idx, codes, scales, nnz, bucket, N)
    U = int(out.nnz.item())
    assert U == ref["nnz"] and not ref["is_dense"] and not bool(out.is_dense.item())
    assert np.array_equal(u32(out.idx[:U]), ref["idx"])
    assert np.array_equal(bits(out.val[:U].cpu().numpy()), bits(ref["val"]))


def test_ef_state_checkpoint_and_resume_is_bitwise():
    """The error-feedback residual is the only state carried between steps:
    ten steps in one go equal five steps, a torch.save / torch.load round
    trip of the residual through host memory, and five more, bit for bit
    (every step's streams and the final residual)."""
    import io
    P, N, L = 4, 300_000, 100_000
    grads = [torch.from_numpy(make("normal", P, N, 100 + s)).to(DEV) for s in range(10)]

    def run(res, steps):
        outs = []
        for g in steps:
            idx, val, nnz = api.topk_ef(g, res, L, 1, 100)
            outs.append((idx.clone(), val.clone(), nnz.clone()))
        return outs

    res_a = torch.zeros((P, N), device=DEV)
    a = run(res_a, grads)
    res_b = torch.zeros((P, N), device=DEV)
    b = run(res_b, grads[:5])
    buf = io.BytesIO()
    torch.save(res_b.cpu(), buf)
    buf.seek(0)
    res_c = torch.load(buf).to(DEV)
    b += run(res_c, grads[5:])
    for (ia, va, na), (ib, vb, nb) in zip(a, b):
        assert torch.equal(na, nb) and torch.equal(ia, ib)
        assert torch.equal(va.view(torch.int32), vb.view(torch.int32))
    assert torch.equal(res_a.view(torch.int32), res_c.view(torch.int32))
