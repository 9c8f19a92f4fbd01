"""GPU parity of the emulated SSAR recursive-doubling allreduce (SparCML
§5.3.1) against the oracle's stage-by-stage schedule: final indices, values
(bit for bit) and the fill-in of every stage."""
import numpy as np
import pytest
import torch

import oracle
from top_gradient_compression_gb300 import api, workloads as W

from gpu_helpers import DEV, bits, streams_to_dev, u32

pytestmark = pytest.mark.gpu


def check_ssar(idx, val, nnz, N):
    oi, ov, ofill = oracle.ssar(idx, val, nnz, N)
    di, dv, dn = streams_to_dev(idx, val, nnz)
    P, cap = idx.shape
    ws = api.workspace(api.ssar_workspace_size(P, cap, N), DEV)
    gi, gv, gn, gfill = api.ssar_allreduce(di, dv, dn, N, ws=ws)
    assert api.get_status(ws) == 0
    U = int(gn.item())
    assert U == len(oi)
    assert np.array_equal(u32(gi[:U]), oi)
    assert np.array_equal(bits(gv[:U].cpu().numpy()), bits(ov))
    assert np.array_equal(gfill.cpu().numpy().astype(np.uint64), ofill)
    return ofill


@pytest.mark.parametrize("P,N,k", [
    (2, 100_000, 3_000),
    (4, 1_000, 999),           # nearly full: long runs of equal indices across streams
    (8, 200_003, 5_000),
    (16, 4_194_304, 4_194),    # density-sweep-like, 0.1 %
    (64, 4_194_304, 41_943),   # density-sweep cell P=64, d=1 %
])
def test_ssar_uniform_streams(P, N, k):
    idx, val, nnz = W.uniform_streams(P, N, k, 70 + P)
    nnz[P // 2] = k // 3
    nnz[-1] = 0  # an empty node
    check_ssar(idx, val, nnz, N)


@pytest.mark.parametrize("same", [True, False])
def test_ssar_identical_and_disjoint_sets(same):
    """§5.3.1's extremes: identical index sets stay at k per partial result,
    disjoint ones double at every stage."""
    P, N, k = 16, 1_000_000, 20_000
    rng = np.random.default_rng(9)
    if same:
        idx = np.tile(np.sort(rng.choice(N, k, replace=False)).astype(np.uint32), (P, 1))
    else:
        idx = np.sort(rng.permutation(N)[:P * k].reshape(P, k), axis=1).astype(np.uint32)
    val = rng.standard_normal((P, k)).astype(np.float32)
    fill = check_ssar(idx, val, np.full(P, k, np.uint32), N)
    if same:
        assert fill.tolist() == [(P >> (s + 1)) * k for s in range(4)]
    else:
        assert fill.tolist() == [P * k] * 4


def test_ssar_flags_bad_streams():
    N = 10_000
    idx = np.array([[5, 3, 9, 0], [1, 2, 3, 4]], np.uint32)
    di, dv, dn = streams_to_dev(idx, np.ones((2, 4), np.float32), np.array([3, 4], np.uint32))
    ws = api.workspace(api.ssar_workspace_size(2, 4, N), DEV)
    api.ssar_allreduce(di, dv, dn, N, ws=ws)
    assert api.get_status(ws) == api.STATUS_CODE["SPARCML_ERR_BAD_STREAM"]
