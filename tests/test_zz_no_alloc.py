"""The allocation-free sparse reduce gives the same results as the workspace one.

sparcml_sparse_reduce_noalloc serves callers that cannot allocate device
memory at the point where they reduce (for example a plug-in whose host
framework owns all device memory through its own pool), so they cannot hand
the library a workspace. Its scratch is a fixed array inside the library that
every call shares. This test calls it through the C ABI twice in a row, on a
dense and then a sparse case (the second call reuses the scratch the first one
left behind), and compares each result bit for bit with sparcml_sparse_reduce.
It lives in its own file, collected last.
"""
import numpy as np
import pytest
import torch

from top_gradient_compression_gb300 import _lib, api, workloads as W

from gpu_helpers import DEV, bits, streams_to_dev, u32

pytestmark = pytest.mark.gpu


def _reduce_noalloc(di, dv, dn, N, out, status):
    P, cap = di.shape
    return _lib.load().sparcml_sparse_reduce_noalloc(
        di.data_ptr(), dv.data_ptr(), dn.data_ptr(), P, cap, N, 1, 4, out.idx.data_ptr(),
        out.val.data_ptr(), out.idx.numel(), out.dense.data_ptr(), out.nnz.data_ptr(),
        out.is_dense.data_ptr(), status.data_ptr(), torch.cuda.current_stream().cuda_stream)


def test_noalloc_reduce_matches_workspace_reduce_on_two_calls_in_a_row():
    cases = [(W.uniform_streams(16, 200_000, 4_000, 22), 200_000, True),      # dense + fix-up
             (W.uniform_streams(8, 1_000_003, 20_000, 23), 1_000_003, False)]  # sparse
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    for (idx, val, nnz), N, dense in cases:
        di, dv, dn = streams_to_dev(idx, val, nnz)
        ref = api.sparse_reduce(di, dv, dn, N)
        out = api.reduce_out(N, DEV)
        assert _reduce_noalloc(di, dv, dn, N, out, status) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        U = int(out.nnz.item())
        assert U == int(ref.nnz.item())
        assert bool(out.is_dense.item()) == bool(ref.is_dense.item()) == dense
        if dense:
            assert np.array_equal(bits(out.dense.cpu().numpy()), bits(ref.dense.cpu().numpy()))
        else:
            assert np.array_equal(u32(out.idx[:U]), u32(ref.idx[:U]))
            assert np.array_equal(bits(out.val[:U].cpu().numpy()),
                                  bits(ref.val[:U].cpu().numpy()))


def test_noalloc_reduce_rejects_sizes_beyond_its_scratch():
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    di, dv, dn = streams_to_dev(np.zeros((1, 1), np.uint32), np.zeros((1, 1), np.float32),
                                np.zeros(1, np.uint32))
    out = api.reduce_out(16, DEV)
    big = (1 << 27) + 1
    rc = _reduce_noalloc(di, dv, dn, big, out, status)
    assert rc == api.STATUS_CODE["SPARCML_ERR_WORKSPACE"]
