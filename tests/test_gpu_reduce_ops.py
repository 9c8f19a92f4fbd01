"""GPU parity of the reduce with max, min and bitwise or (SparCML §5.2: any
coordinate-wise associative operation with a neutral element) against the
oracle, bit for bit, in every tiling regime."""
import numpy as np
import pytest
import torch

import oracle
from top_gradient_compression_gb300 import api, workloads as W

from gpu_helpers import DEV, bits, streams_to_dev, u32

pytestmark = pytest.mark.gpu


def check_op(idx, val, nnz, N, op, repeat=2):
    ref = oracle.sparse_reduce_op(idx, val, nnz, N, op)
    di, dv, dn = streams_to_dev(idx, val, nnz)
    ws = api.workspace(api.reduce_workspace_size(idx.shape[0], N), DEV)
    for _ in range(repeat):
        out = api.sparse_reduce_op(di, dv, dn, N, op, ws=ws)
        assert api.get_status(ws) == 0
        U = int(out.nnz.item())
        assert U == ref["nnz"] and bool(out.is_dense.item()) == ref["is_dense"]
        if ref["is_dense"]:
            assert np.array_equal(bits(out.dense.cpu().numpy()), bits(ref["dense"]))
        else:
            assert np.array_equal(u32(out.idx[:U]), ref["idx"])
            assert np.array_equal(bits(out.val[:U].cpu().numpy()), bits(ref["val"]))
    return ref


@pytest.mark.parametrize("op", ["max", "min", "or"])
@pytest.mark.parametrize("P,N,k", [
    (3, 4_194_304, 2_000),     # compact-accumulator CTA tiles
    (8, 200_000, 4_000),       # sparse-first warp tiles (or: CTA tiles)
    (16, 200_000, 12_000),     # dense-first warp tiles, dense result
    (4, 100_000, 8_000),       # ~80 entries per node and tile: dense-first warp tiles
    (3, 100_000, 8_000),       # the same load, sparse-first warp tiles with look-back
    (80, 100_000, 2_000),      # more than 64 nodes: staged CTA tiles, dense-first
    (100, 200_000, 1_000),     # staged CTA tiles, look-back, dense by fix-up
])
def test_reduce_op_each_regime(op, P, N, k):
    idx, val, nnz = W.uniform_streams(P, N, k, 50 + P, std=1.0)
    nnz[P // 2] = k // 3
    check_op(idx, val, nnz, N, op)


@pytest.mark.parametrize("op", ["max", "min", "or"])
def test_reduce_op_density_sweep_cell_and_signed_zero_ties(op):
    idx, val, nnz = W.sweep_streams(32, 5, 100)
    val[:, ::7] = 0.0
    val[1::2, ::7] = -0.0  # equal magnitudes of both signs at shared indices
    r = check_op(idx, val, nnz, W.SWEEP_N, op)
    assert r["is_dense"]


def test_reduce_op_sum_matches_the_sum_reduce():
    idx, val, nnz = W.sweep_streams(16, 1, 100)
    di, dv, dn = streams_to_dev(idx, val, nnz)
    a = api.sparse_reduce(di, dv, dn, W.SWEEP_N)
    b = api.sparse_reduce_op(di, dv, dn, W.SWEEP_N, "sum")
    U = int(a.nnz.item())
    assert U == int(b.nnz.item())
    assert torch.equal(a.idx[:U], b.idx[:U]) and torch.equal(a.val[:U], b.val[:U])
