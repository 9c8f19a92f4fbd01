"""GPU parity of the sparse sum-reduce with the dense switch (SparCML §5.1-§5.3,
App. B), of pack, densify and the 4-bit quantiser (§2.2, §6), against the oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
from top_gradient_compression_gb300 import api, workloads as W

from gpu_helpers import DEV, bits, check_reduce, streams_to_dev, u32

pytestmark = pytest.mark.gpu


def rand_streams(rng, P, N, maxk, cap=None):
    cap = max(maxk, 1) if cap is None else cap
    idx = np.zeros((P, cap), np.uint32)
    val = np.zeros((P, cap), np.float32)
    nnz = np.zeros(P, np.uint32)
    for p in range(P):
        k = int(rng.integers(0, maxk + 1))
        idx[p, :k] = np.sort(rng.choice(N, size=k, replace=False))
        val[p, :k] = rng.standard_normal(k).astype(np.float32)
        nnz[p] = k
    return idx, val, nnz


@pytest.mark.parametrize("seed", range(10))
def test_reduce_random(seed):
    rng = np.random.default_rng(seed)
    P = int(rng.integers(1, 12))
    N = int(rng.choice([1, 7, 1000, 8192, 8193, 3 * 8192 + 7, 100_003]))
    maxk = int(min(N, rng.choice([1, 50, 3000, 30_000])))
    idx, val, nnz = rand_streams(rng, P, N, maxk)
    check_reduce(idx, val, nnz, N, repeat=2)


def test_reduce_all_empty_and_single_entry():
    N = 100_000
    idx = np.zeros((3, 4), np.uint32)
    check_reduce(idx, np.zeros((3, 4), np.float32), np.zeros(3, np.uint32), N)
    idx[1, 0] = N - 1
    r = check_reduce(idx, np.ones((3, 4), np.float32), np.array([0, 1, 0], np.uint32), N)
    assert r["nnz"] == 1


@pytest.mark.parametrize("N", [64, 8192 * 4, 8192 * 4 + 4])
def test_reduce_switch_exactly_at_quarter(N):
    for extra, dense in ((0, False), (1, True)):
        U = N // 4 + extra
        rng = np.random.default_rng(N + extra)
        sel = np.sort(rng.choice(N, size=U, replace=False)).astype(np.uint32)
        # spread the union over 3 nodes so no single node decides it
        parts = np.array_split(sel, 3)
        cap = max(len(x) for x in parts)
        idx = np.zeros((3, cap), np.uint32)
        val = np.zeros((3, cap), np.float32)
        nnz = np.zeros(3, np.uint32)
        for p, part in enumerate(parts):
            idx[p, :len(part)] = part
            val[p, :len(part)] = rng.standard_normal(len(part))
            nnz[p] = len(part)
        r = check_reduce(idx, val, nnz, N)
        assert r["nnz"] == U and r["is_dense"] == dense


def test_reduce_dense_paths():
    rng = np.random.default_rng(11)
    N = 200_000
    # (a) one node alone is above the threshold: dense from the first tile
    idx, val, nnz = W.uniform_streams(3, N, 60_000, 21)
    check_reduce(idx, val, nnz, N, repeat=2)
    # (b) every node small, the union crosses 25% part-way: leading tiles are fixed up
    idx, val, nnz = W.uniform_streams(16, N, 4_000, 22)
    r = check_reduce(idx, val, nnz, N, repeat=2)
    assert r["is_dense"]


@pytest.mark.parametrize("P,dnum,dden", [(2, 1, 1000), (4, 10, 100), (8, 5, 100), (32, 1, 100)])
def test_reduce_density_sweep_cells_exact(P, dnum, dden):
    idx, val, nnz = W.sweep_streams(P, dnum, dden)
    check_reduce(idx, val, nnz, W.SWEEP_N)


def test_reduce_density_sweep_all_cells_follow_the_closed_form():
    """All 24 (P, d) cells at N = 4,194,304: U/N tracks 1 - (1 - d)^P (App. B.1) and
    the result is dense exactly when 4U > N."""
    N = W.SWEEP_N
    for P in W.SWEEP_P:
        for dnum, dden in W.SWEEP_D:
            idx, val, nnz = W.sweep_streams(P, dnum, dden)
            di, dv, dn = streams_to_dev(idx, val, nnz)
            out = api.sparse_reduce(di, dv, dn, N)
            U = int(out.nnz.item())
            d = (N * dnum // dden) / N
            q = 1 - (1 - d) ** P
            assert abs(U / N - q) <= 6 * math.sqrt(q * (1 - q) / N) + 1e-12, (P, dnum, dden)
            assert bool(out.is_dense.item()) == (4 * U > N)
            assert U <= min(N, P * (N * dnum // dden))


def test_reduce_logreg_workload_exact():
    idx, val, nnz = W.logreg_streams()
    r = check_reduce(idx, val, nnz, W.LOGREG["N"], repeat=2)
    assert not r["is_dense"]


def test_reduce_detects_bad_streams():
    N = 50_000
    cases = [np.array([[5, 3, 9, 0]], np.uint32),        # not ascending
             np.array([[5, 5, 9, 0]], np.uint32),        # duplicate
             np.array([[5, 9, N, 0]], np.uint32),        # index out of range
             np.array([[9000, 20, 30000, 40000]], np.uint32)]  # out of order across tiles
    nn = [3, 3, 3, 4]
    for idx, n in zip(cases, nn):
        di, dv, dn = streams_to_dev(idx, np.ones((1, 4), np.float32), np.array([n], np.uint32))
        ws = api.workspace(api.reduce_workspace_size(1, N), DEV)
        api.sparse_reduce(di, dv, dn, N, ws=ws)
        assert api.get_status(ws) == api.STATUS_CODE["SPARCML_ERR_BAD_STREAM"]
        assert api.get_status(ws) == 0  # reading clears it


def test_pack_parity_and_capacity():
    rng = np.random.default_rng(2)
    P, N = 3, 100_003
    x = rng.standard_normal((P, N)).astype(np.float32)
    x[rng.random((P, N)) < 0.9] = 0.0
    x[0, 1] = -0.0
    xd = torch.from_numpy(x).to(DEV)
    for thr, cap in ((0.0, N), (1.5, N), (0.0, 5000)):
        oi, ov, on, ost = oracle.pack(x, thr, cap)
        idx, val, nnz, ws = api.pack(xd, thr, cap)
        st = api.get_status(ws)
        assert st == (api.STATUS_CODE["SPARCML_ERR_CAPACITY"] if ost else 0)
        assert np.array_equal(u32(nnz), on)
        for p in range(P):
            n = int(on[p])
            assert np.array_equal(u32(idx)[p, :n], oi[p, :n])
            assert np.array_equal(bits(val.cpu().numpy()[p, :n]), bits(ov[p, :n]))


def test_densify_parity():
    rng = np.random.default_rng(4)
    P, N = 4, 9999
    idx, val, nnz = rand_streams(rng, P, N, 3000)
    di, dv, dn = streams_to_dev(idx, val, nnz)
    got = api.densify(di, dv, dn, N)
    assert np.array_equal(bits(got.cpu().numpy()), bits(oracle.densify(idx, val, nnz, N)))


def test_quantize_dequantize_parity():
    rng = np.random.default_rng(6)
    P, cap, bucket = 3, 2000, 512
    val = (rng.laplace(size=(P, cap)) * 1e-3).astype(np.float32)
    val[1, 600:700] = 0.0  # a partly zero bucket
    val[2, :] = 0.0        # an all-zero node
    idx = np.sort(rng.choice(1 << 24, size=(P, cap), replace=False), axis=1).astype(np.uint32)
    nnz = np.array([2000, 1025, 7], np.uint32)
    for seed in (0, 123456789, 2**63 + 5):
        oc, osc = oracle.quantize4(idx, val, nnz, bucket, seed)
        di, dv, dn = streams_to_dev(idx, val, nnz)
        codes, scales = api.quantize4(di, dv, dn, bucket, seed)
        gc, gs = codes.cpu().numpy(), scales.cpu().numpy()
        for p in range(P):
            n = int(nnz[p])
            lo_o, hi_o = oc[p] & 15, oc[p] >> 4
            lo_g, hi_g = gc[p] & 15, gc[p] >> 4
            assert np.array_equal(lo_g[: (n + 1) // 2], lo_o[: (n + 1) // 2])
            assert np.array_equal(hi_g[: n // 2], hi_o[: n // 2])
            nb = (n + bucket - 1) // bucket
            assert np.array_equal(bits(gs[p, :nb]), bits(osc[p, :nb]))
        od = oracle.dequantize4(oc, osc, nnz, cap, bucket)
        gd = api.dequantize4(codes, scales, dn, cap, bucket).cpu().numpy()
        for p in range(P):
            n = int(nnz[p])
            assert np.array_equal(bits(gd[p, :n]), bits(od[p, :n]))


@pytest.mark.parametrize("k,dense,bucket", [(1_000, False, 512), (5_000, False, 96),
                                             (20_000, True, 512), (30_000, True, 6)])
def test_reduce_q4_equals_dequantize_then_reduce(k, dense, bucket):
    P, N = 6, 300_000
    idx, val, nnz = W.uniform_streams(P, N, k, 31, std=1e-3)
    nnz[2] = k // 2 + 345
    seed = W.quant_seed(0)
    oc, osc = oracle.quantize4(idx, val, nnz, bucket, seed)
    deq = oracle.dequantize4(oc, osc, nnz, k, bucket)
    ref = oracle.sparse_reduce(idx, deq, nnz, N)
    assert ref["is_dense"] == dense
    di, dv, dn = streams_to_dev(idx, val, nnz)
    codes, scales = api.quantize4(di, dv, dn, bucket, seed)
    out = api.sparse_reduce_q4(di, codes, scales, dn, bucket, N)
    U = int(out.nnz.item())
    assert U == ref["nnz"] and bool(out.is_dense.item()) == ref["is_dense"]
    if dense:
        assert np.array_equal(bits(out.dense.cpu().numpy()), bits(ref["dense"]))
    else:
        assert np.array_equal(u32(out.idx[:U]), ref["idx"])
        assert np.array_equal(bits(out.val[:U].cpu().numpy()), bits(ref["val"]))


def test_reduce_sparse_regime_skewed_tile():
    """Sparse inputs take wide tiles with a compact accumulator; a tile that
    still receives many thousand entries (skew) is accumulated in several slot
    windows from re-read entries. Checked bit for bit against the oracle."""
    rng = np.random.default_rng(12)
    P, N, cap = 3, 4_194_304, 20_000
    idx = np.zeros((P, cap), np.uint32)
    val = rng.standard_normal((P, cap)).astype(np.float32)
    nnz = np.full(P, cap, np.uint32)
    idx[0] = np.arange(cap, dtype=np.uint32) * 3            # 20,000 entries in the first wide tile
    idx[1] = np.sort(rng.choice(60_000, cap, replace=False))  # overlapping the same tile
    idx[2] = np.sort(rng.choice(N, cap, replace=False))       # spread out
    r = check_reduce(idx, val, nnz, N, repeat=2)
    assert not r["is_dense"] and r["nnz"] > 8192


def test_reduce_dense_regime_sparse_result_is_compacted():
    """Inputs that cover the index space (P * cap >= N) take the dense-first
    tiles; when the streams overlap so much that the union stays under 25%, the
    sparse result is rebuilt from the dense slices. Bit for bit vs the oracle."""
    rng = np.random.default_rng(21)
    P, N, k = 24, 200_000, 10_000  # P * k = 1.2 N
    base = np.sort(rng.choice(N, 12_000, replace=False)).astype(np.uint32)
    idx = np.zeros((P, k), np.uint32)
    for p in range(P):
        idx[p] = np.sort(rng.choice(base, k, replace=False))
    val = rng.standard_normal((P, k)).astype(np.float32)
    r = check_reduce(idx, val, np.full(P, k, np.uint32), N, repeat=2)
    assert not r["is_dense"] and r["nnz"] <= 12_000


@pytest.mark.parametrize("P,N,maxk,note", [
    (64, 100_003, 3_000, "warp-per-1,024-index tiles, 64 nodes, ragged last tile, dense result"),
    (33, 50_001, 400, "warp-per-1,024-index tiles, nodes 32.., result near the switch"),
    (5, 700, 200, "one ragged warp tile shorter than 1,024 indices"),
    (40, 30_000, 1_500, "rounds spanning several nodes, some nodes empty"),
    (4, 10_000, 1_001, "rows not 16-byte aligned (cap = 1,001): quad split pass with a lead"),
    (7, 20_001, 1_001, "P * cap not a multiple of 4: scalar split pass"),
    (80, 100_000, 2_000, "more than 64 nodes covering the index space: staged CTA tiles"),
    (100, 200_000, 1_000, "more than 64 nodes, union crosses 25% part-way: look-back + fix-up"),
    (8, 200_000, 4_000, "P * cap between N/16 and N/2: sparse-first warp tiles, look-back"),
    (16, 100_000, 2_800, "sparse-first warp tiles, union crosses 25% part-way: fix-up"),
    (200, 1_000_000, 500, "more than 64 nodes, P * cap below N/4: compact-accumulator tiles"),
    (1100, 100_000, 60, "more than 1,024 nodes: staged CTA tiles with look-back"),
])
def test_reduce_each_regime_exact(P, N, maxk, note):
    """Every tiling regime of the reduce, bit for bit against the oracle; node
    sizes vary from 0 to maxk so tiles see empty and short per-node runs."""
    rng = np.random.default_rng(P * 1000 + maxk)
    idx, val, nnz = rand_streams(rng, P, N, maxk)
    nnz[P // 2] = 0  # an empty node in the middle of the order
    check_reduce(idx, val, nnz, N, repeat=2)


@pytest.mark.parametrize("N,k", [
    (4_096, 1_100), (4_096, 1_101),     # dense-first warp tiles: quad / scalar split pass
    (65_536, 3_000), (65_536, 3_001),   # sparse-first warp tiles: quad / scalar split pass
])
def test_reduce_detects_bad_streams_in_warp_tiles(N, k):
    """Streams that cover a large share of the index space take the
    warp-per-tile path; a step down, a repeat, an index past N or two entries
    swapped across tiles is flagged there too, by either form of the split
    pass and with either output order."""
    rng = np.random.default_rng(4)
    good = np.sort(rng.choice(N - 1, size=k, replace=False)).astype(np.uint32)
    bad = [good.copy() for _ in range(4)]
    bad[0][500], bad[0][501] = bad[0][501], bad[0][500]  # step down inside a tile
    bad[1][700] = bad[1][699]                              # repeated index
    bad[2][-1] = N                                         # index past the end
    bad[3][100], bad[3][900] = bad[3][900], bad[3][100]    # out of order across tiles
    for b in bad:
        idx = np.stack([good, b])
        di, dv, dn = streams_to_dev(idx, np.ones((2, k), np.float32), np.full(2, k, np.uint32))
        ws = api.workspace(api.reduce_workspace_size(2, N), DEV)
        api.sparse_reduce(di, dv, dn, N, ws=ws)
        assert api.get_status(ws) == api.STATUS_CODE["SPARCML_ERR_BAD_STREAM"]


@pytest.mark.parametrize("P,N,k,note", [
    (64, 65_536, 6_553, "64 nodes at 10 %, the largest sweep cell's per-tile load"),
    (64, 70_001, 7_000, "ragged last tile"),
    (8, 50_000, 5_001, "rows not 16-byte aligned (cap = 5,001)"),
    (3, 100_000, 8_000, "sparse-first with look-back"),
])
def test_reduce_warp_tiles_heavy_nodes_exact(P, N, k, note):
    """About a hundred entries per node and 1,024-index tile: a round of 32
    quads holds one node's tail and the next node's head, so nearly every
    round is added one node at a time. Bit for bit against the oracle."""
    idx, val, nnz = W.uniform_streams(P, N, k, 70 + P)
    nnz[P // 2] = 2 * k // 3  # a shorter node among full ones
    check_reduce(idx, val, nnz, N, repeat=2)


def test_reduce_largest_sweep_cell_sampled():
    """P = 64, d = 10 % at N = 4,194,304, launched as the benchmark does: the
    union size against a count of the distinct indices, and the values at
    two whole tiles plus 2,048 random indices against the oracle run on the
    streams restricted to those indices (each index sums independently)."""
    P, N = 64, W.SWEEP_N
    idx, val, nnz = W.sweep_streams(P, 10, 100)
    di, dv, dn = streams_to_dev(idx, val, nnz)
    ws = api.workspace(api.reduce_workspace_size(P, N), DEV)
    out = api.sparse_reduce(di, dv, dn, N, ws=ws)
    assert api.get_status(ws) == 0
    U = int(out.nnz.item())
    assert U == np.unique(idx.reshape(-1)).size
    assert bool(out.is_dense.item()) == (4 * U > N) and 4 * U > N
    rng = np.random.default_rng(12)
    sample = np.union1d(np.arange(7 * 1024, 9 * 1024), rng.choice(N, 2_048, replace=False))
    keep = np.isin(idx, sample)
    cnt = keep.sum(axis=1)
    sub_i = np.zeros((P, int(cnt.max())), np.uint32)
    sub_v = np.zeros((P, int(cnt.max())), np.float32)
    for p in range(P):
        sub_i[p, :cnt[p]] = idx[p][keep[p]]
        sub_v[p, :cnt[p]] = val[p][keep[p]]
    ref = oracle.sparse_reduce(sub_i, sub_v, cnt.astype(np.uint32), N)
    assert not ref["is_dense"]
    want = np.zeros(N, np.float32)
    want[ref["idx"]] = ref["val"]
    got = out.dense.cpu().numpy()
    assert np.array_equal(bits(got[sample]), bits(want[sample]))


@pytest.mark.parametrize("P,N,k", [(6, 30_000, 2_000), (64, 65_536, 3_001)])
def test_reduce_warp_tiles_with_unaligned_buffers(P, N, k):
    """Warp tiles read 16-byte quads only from 16-byte aligned buffers; stream
    buffers that start 4 bytes off a 16-byte boundary take the entry-by-entry
    loads. Same bits as the oracle either way."""
    idx, val, nnz = W.uniform_streams(P, N, k, 40 + P)
    ref = oracle.sparse_reduce(idx, val, nnz, N)
    flat_i = torch.zeros(P * k + 1, dtype=torch.int32, device=DEV)
    flat_v = torch.zeros(P * k + 1, dtype=torch.float32, device=DEV)
    flat_i[1:] = torch.from_numpy(idx.view(np.int32).reshape(-1)).to(DEV)
    flat_v[1:] = torch.from_numpy(val.reshape(-1)).to(DEV)
    di, dv = flat_i[1:].view(P, k), flat_v[1:].view(P, k)
    assert di.data_ptr() % 16 == 4 and dv.data_ptr() % 16 == 4
    dn = torch.from_numpy(nnz.view(np.int32)).to(DEV)
    ws = api.workspace(api.reduce_workspace_size(P, N), DEV)
    out = api.sparse_reduce(di, dv, dn, N, ws=ws)
    assert api.get_status(ws) == 0
    U = int(out.nnz.item())
    assert U == ref["nnz"] and bool(out.is_dense.item()) == ref["is_dense"]
    if ref["is_dense"]:
        assert np.array_equal(bits(out.dense.cpu().numpy()), bits(ref["dense"]))
    else:
        assert np.array_equal(u32(out.idx[:U]), ref["idx"])
        assert np.array_equal(bits(out.val[:U].cpu().numpy()), bits(ref["val"]))


def hot_head_streams(P, N, head, k, seed):
    """Every node holds all of [0, head) plus k - head random others: the
    first tiles hold P * 1,024 entries each (a skewed, Zipf-like head)."""
    rng = np.random.default_rng(seed)
    idx = np.zeros((P, k), np.uint32)
    for p in range(P):
        rest = rng.choice(np.arange(head, N), size=k - head, replace=False)
        idx[p] = np.sort(np.concatenate([np.arange(head), rest])).astype(np.uint32)
    val = rng.standard_normal((P, k)).astype(np.float32)
    return idx, val, np.full(P, k, np.uint32)


@pytest.mark.parametrize("P,k", [(16, 6_000), (17, 6_001)])  # quad / entry-by-entry warp tiles
def test_reduce_hot_head_tiles(P, k):
    """A skewed head: the first tiles hold P * 1,024 entries each (every node
    has every index there). Bit for bit against the oracle (sum, and max)."""
    N = 100_000
    idx, val, nnz = hot_head_streams(P, N, 3_100, k, P)
    r = check_reduce(idx, val, nnz, N, repeat=2)
    assert r["nnz"] >= 3_100
    ref = oracle.sparse_reduce_op(idx, val, nnz, N, "max")
    di, dv, dn = streams_to_dev(idx, val, nnz)
    out = api.sparse_reduce_op(di, dv, dn, N, "max")
    assert int(out.nnz.item()) == ref["nnz"] and bool(out.is_dense.item()) == ref["is_dense"]
    got = out.dense if ref["is_dense"] else out.val[:ref["nnz"]]
    want = ref["dense"] if ref["is_dense"] else ref["val"]
    assert np.array_equal(bits(got.cpu().numpy()), bits(want))


def test_reduce_hot_head_tiles_with_4bit_values():
    P, N, k, bucket = 16, 100_000, 6_000, 512
    idx, val, nnz = hot_head_streams(P, N, 3_100, k, 5)
    val *= 1e-2
    seed = W.quant_seed(2)
    oc, osc = oracle.quantize4(idx, val, nnz, bucket, seed)
    deq = oracle.dequantize4(oc, osc, nnz, k, bucket)
    ref = oracle.sparse_reduce(idx, deq, nnz, N)
    di, dv, dn = streams_to_dev(idx, val, nnz)
    codes, scales = api.quantize4(di, dv, dn, bucket, seed)
    out = api.sparse_reduce_q4(di, codes, scales, dn, bucket, N)
    U = int(out.nnz.item())
    assert U == ref["nnz"] and bool(out.is_dense.item()) == ref["is_dense"]
    if ref["is_dense"]:
        assert np.array_equal(bits(out.dense.cpu().numpy()), bits(ref["dense"]))
    else:
        assert np.array_equal(u32(out.idx[:U]), ref["idx"])
        assert np.array_equal(bits(out.val[:U].cpu().numpy()), bits(ref["val"]))


def test_reduce_sparse_first_head_tiles_past_staging():
    """Sparse-first warp tiles (P * cap < N / 4) whose first tiles hold every
    index: 1,024 union entries, more than the 512 a tile stages for its
    coalesced output, and 16,384 entries, several load batches. Those tiles
    take the per-lane output; 4-bit values and unaligned fp32 rows (the
    scalar warp tiles), bit for bit."""
    P, N, k, bucket = 16, 1 << 22, 50_000, 512
    idx, val, nnz = hot_head_streams(P, N, 3_100, k, 11)
    assert 4 * P * k < N  # the sparse-first form
    val *= 1e-2
    seed = W.quant_seed(3)
    oc, osc = oracle.quantize4(idx, val, nnz, bucket, seed)
    ref = oracle.sparse_reduce(idx, oracle.dequantize4(oc, osc, nnz, k, bucket), nnz, N)
    assert not ref["is_dense"]
    di, dv, dn = streams_to_dev(idx, val, nnz)
    codes, scales = api.quantize4(di, dv, dn, bucket, seed)
    out = api.sparse_reduce_q4(di, codes, scales, dn, bucket, N)
    U = int(out.nnz.item())
    assert U == ref["nnz"] and not bool(out.is_dense.item())
    assert np.array_equal(u32(out.idx[:U]), ref["idx"])
    assert np.array_equal(bits(out.val[:U].cpu().numpy()), bits(ref["val"]))
    wide = k + 1  # rows no longer 16-byte aligned: the scalar warp tiles
    i2 = np.zeros((P, wide), np.uint32)
    v2 = np.zeros((P, wide), np.float32)
    i2[:, :k], v2[:, :k] = idx, val
    r = check_reduce(i2, v2, nnz, N, repeat=2)
    assert not r["is_dense"]


def test_reduce_skewed_head_every_warp_tile_path():
    """A Zipf head puts about a thousand entries per node into each of the first
    1,024-index tiles: those tiles are spread over a CTA (dense-first warp-tile
    mode) in every variant, fp32 quads, unaligned fp32, the fused 4-bit decode
    and max, and the result stays bit-exact."""
    from test_gpu_reduce_ops import check_op
    P, N, k = 16, 1 << 20, 30_000
    idx, val, nnz = W.zipf_streams(P, N, k, 1.1, 1.0, 99)
    check_reduce(idx, val, nnz, N, repeat=2)  # 16-byte quads
    wide = k + 1  # rows no longer 16-byte aligned: the scalar warp tiles
    i2 = np.zeros((P, wide), np.uint32)
    v2 = np.zeros((P, wide), np.float32)
    i2[:, :k], v2[:, :k] = idx, val
    check_reduce(i2, v2, nnz, N, repeat=2)
    check_op(idx, val, nnz, N, "max")
    bucket, seed = 512, 1234
    di, dv, dn = streams_to_dev(idx, val, nnz)
    codes, scales = api.quantize4(di, dv, dn, bucket, seed)
    oc, osc = oracle.quantize4(idx, val, nnz, bucket, seed)
    assert np.array_equal(codes.cpu().numpy(), oc)
    ref = oracle.sparse_reduce(idx, oracle.dequantize4(oc, osc, nnz, k, bucket), nnz, N)
    out = api.sparse_reduce_q4(di, codes, scales, dn, bucket, N)
    U = int(out.nnz.item())
    assert U == ref["nnz"] and bool(out.is_dense.item()) == ref["is_dense"]
    if ref["is_dense"]:
        assert np.array_equal(bits(out.dense.cpu().numpy()), bits(ref["dense"]))
    else:
        assert np.array_equal(u32(out.idx[:U]), ref["idx"])
        assert np.array_equal(bits(out.val[:U].cpu().numpy()), bits(ref["val"]))
