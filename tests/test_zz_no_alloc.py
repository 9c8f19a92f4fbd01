"""The allocation-free sparse reduce: same results as the oracle and as the
workspace reduce.

sparcml_sparse_reduce_noalloc serves callers that cannot allocate device
memory at the point where they reduce (for example a plug-in whose host
framework owns all device memory through its own pool), so they cannot hand
the library a workspace. Its scratch is a fixed array inside the library that
every call shares. These tests call it through the C ABI: twice in a row on a
dense and then a sparse case (the second call reuses the scratch the first
one left behind), compared bit for bit with the oracle and with
sparcml_sparse_reduce; then more than 64 nodes, a Zipf-skewed head, the exact
25 % switch, bad streams and an overfull node, each checked against the
oracle or the status word. The file is collected last.
"""
import numpy as np
import pytest
import torch

import oracle
from top_gradient_compression_gb300 import _lib, api, workloads as W

from gpu_helpers import DEV, bits, streams_to_dev, u32

pytestmark = pytest.mark.gpu


def _reduce_noalloc(di, dv, dn, N, out, status, cap=None):
    P = di.shape[0]
    cap = di.shape[1] if cap is None else cap
    return _lib.load().sparcml_sparse_reduce_noalloc(
        di.data_ptr(), dv.data_ptr(), dn.data_ptr(), P, cap, N, 1, 4, out.idx.data_ptr(),
        out.val.data_ptr(), out.idx.numel(), out.dense.data_ptr(), out.nnz.data_ptr(),
        out.is_dense.data_ptr(), status.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _check_against_oracle(idx, val, nnz, N, status):
    di, dv, dn = streams_to_dev(idx, val, nnz)
    out = api.reduce_out(N, DEV)
    assert _reduce_noalloc(di, dv, dn, N, out, status) == 0
    assert api.get_status(status) == 0
    ref = oracle.sparse_reduce(idx, val, nnz, N)
    U = int(out.nnz.item())
    assert U == ref["nnz"] and bool(out.is_dense.item()) == ref["is_dense"]
    if ref["is_dense"]:
        assert np.array_equal(bits(out.dense.cpu().numpy()), bits(ref["dense"]))
    else:
        assert np.array_equal(u32(out.idx[:U]), ref["idx"])
        assert np.array_equal(bits(out.val[:U].cpu().numpy()), bits(ref["val"]))
    return ref, out


def test_noalloc_reduce_matches_oracle_and_workspace_reduce_on_two_calls_in_a_row():
    cases = [(W.uniform_streams(16, 200_000, 4_000, 22), 200_000, True),      # dense + fix-up
             (W.uniform_streams(8, 1_000_003, 20_000, 23), 1_000_003, False)]  # sparse
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    for (idx, val, nnz), N, dense in cases:
        ref, out = _check_against_oracle(idx, val, nnz, N, status)
        assert ref["is_dense"] == dense
        di, dv, dn = streams_to_dev(idx, val, nnz)
        ws_out = api.sparse_reduce(di, dv, dn, N)
        U = int(out.nnz.item())
        assert U == int(ws_out.nnz.item())
        if dense:
            assert torch.equal(out.dense.view(torch.int32), ws_out.dense.view(torch.int32))
        else:
            assert torch.equal(out.idx[:U], ws_out.idx[:U])
            assert torch.equal(out.val[:U].view(torch.int32), ws_out.val[:U].view(torch.int32))


@pytest.mark.parametrize("case", ["many_nodes", "zipf_head", "quarter", "quarter_plus_one",
                                  "ragged"])
def test_noalloc_reduce_against_oracle(case):
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    if case == "many_nodes":  # more than 64 nodes
        idx, val, nnz = W.uniform_streams(100, 300_000, 700, 41)
        nnz[::7] = 0
        N = 300_000
    elif case == "zipf_head":  # the logistic-regression streams: hot low indices
        idx, val, nnz = W.logreg_streams()
        N = W.LOGREG["N"]
    elif case == "ragged":  # N not a multiple of the tile, empty and full nodes
        N = 3 * 8192 + 5
        idx, val, nnz = W.uniform_streams(5, N, 2_000, 43)
        nnz[1] = 0
        idx[4, :] = np.arange(N - 2_000, N, dtype=np.uint32)
    else:  # the union is exactly N/4 (sparse) or N/4 + 1 (dense), over 3 nodes
        N = 8192 * 4 + 4
        U = N // 4 + (case == "quarter_plus_one")
        rng = np.random.default_rng(U)
        sel = np.sort(rng.choice(N, size=U, replace=False)).astype(np.uint32)
        parts = np.array_split(sel, 3)
        cap = max(len(x) for x in parts)
        idx = np.zeros((3, cap), np.uint32)
        val = np.zeros((3, cap), np.float32)
        nnz = np.zeros(3, np.uint32)
        for p, part in enumerate(parts):
            idx[p, :len(part)] = part
            val[p, :len(part)] = rng.standard_normal(len(part))
            nnz[p] = len(part)
    ref, _ = _check_against_oracle(idx, val, nnz, N, status)
    if case.startswith("quarter"):
        assert ref["is_dense"] == (case == "quarter_plus_one")


def test_noalloc_reduce_reports_bad_streams_and_capacity():
    N = 50_000
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    bad = api.STATUS_CODE["SPARCML_ERR_BAD_STREAM"]
    for row, n in [([5, 3, 9, 0], 3),              # not ascending
                   ([5, 5, 9, 0], 3),              # duplicate
                   ([5, 9, N, 0], 3),              # index out of range
                   ([9000, 20, 30000, 40000], 4)]:  # out of order across tiles
        di, dv, dn = streams_to_dev(np.array([row], np.uint32), np.ones((1, 4), np.float32),
                                    np.array([n], np.uint32))
        out = api.reduce_out(N, DEV)
        assert _reduce_noalloc(di, dv, dn, N, out, status) == 0
        assert api.get_status(status) == bad, row
    # nnz above the capacity: the node is read up to cap and the status says so
    idx, val, nnz = W.uniform_streams(2, N, 100, 44)
    nnz[1] = 101
    di, dv, dn = streams_to_dev(idx, val, nnz)
    out = api.reduce_out(N, DEV)
    assert _reduce_noalloc(di, dv, dn, N, out, status) == 0
    assert api.get_status(status) == api.STATUS_CODE["SPARCML_ERR_CAPACITY"]
    # and the next clean call is clean
    _check_against_oracle(*W.uniform_streams(2, N, 100, 45), N, status)


def test_noalloc_reduce_rejects_sizes_beyond_its_scratch():
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    di, dv, dn = streams_to_dev(np.zeros((1, 1), np.uint32), np.zeros((1, 1), np.float32),
                                np.zeros(1, np.uint32))
    out = api.reduce_out(16, DEV)
    big = (1 << 27) + 1
    rc = _reduce_noalloc(di, dv, dn, big, out, status)
    assert rc == api.STATUS_CODE["SPARCML_ERR_WORKSPACE"]
