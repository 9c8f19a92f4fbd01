"""Failure detection without a GPU fault: a host-set fault-injection word
makes the first publisher of every decoupled look-back chain withhold its
prefix, so the bounded waits behind it run out. The call still completes,
the status word reports SPARCML_ERR_TIMEOUT, every access stays in bounds,
and the next call with the injection cleared is clean and bit-exact against
the oracle. Nothing here traps, faults or waits without a bound."""
import time

import numpy as np
import pytest
import torch

import oracle
from top_gradient_compression_gb300 import api, workloads as W

from gpu_helpers import DEV, bits, streams_to_dev, u32

pytestmark = pytest.mark.gpu

TIMEOUT = api.STATUS_CODE["SPARCML_ERR_TIMEOUT"]


def _reduce_matches_oracle(out, idx, val, nnz, N):
    ref = oracle.sparse_reduce(idx, val, nnz, N)
    U = int(out.nnz.item())
    assert U == ref["nnz"] and bool(out.is_dense.item()) == ref["is_dense"]
    if ref["is_dense"]:
        assert np.array_equal(bits(out.dense.cpu().numpy()), bits(ref["dense"]))
    else:
        assert np.array_equal(u32(out.idx[:U]), ref["idx"])
        assert np.array_equal(bits(out.val[:U].cpu().numpy()), bits(ref["val"]))


@pytest.mark.parametrize("P,N,k", [
    (8, 200_000, 4_000),     # warp tiles, sparse-first: warp-wide look-back per CTA group
    (3, 4_194_304, 2_000),   # compact-accumulator CTA tiles: CTA look-back
    (100, 200_000, 1_000),   # staged CTA tiles with look-back
])
def test_reduce_lookback_wait_runs_out_then_recovers(P, N, k):
    idx, val, nnz = W.uniform_streams(P, N, k, 300 + P)
    di, dv, dn = streams_to_dev(idx, val, nnz)
    ws = api.workspace(api.reduce_workspace_size(P, N), DEV)
    out = api.reduce_out(N, DEV)
    api.set_fault_injection(ws, api.INJECT_WITHHOLD_FIRST)
    t0 = time.perf_counter()
    api.sparse_reduce(di, dv, dn, N, out=out, ws=ws)
    assert api.get_status(ws) == TIMEOUT
    assert time.perf_counter() - t0 < 30.0  # the shortened waits end within milliseconds each
    api.sparse_reduce(di, dv, dn, N, out=out, ws=ws)  # still armed: times out again
    assert api.get_status(ws) == TIMEOUT
    api.set_fault_injection(ws, 0)
    api.sparse_reduce(di, dv, dn, N, out=out, ws=ws)
    assert api.get_status(ws) == 0
    _reduce_matches_oracle(out, idx, val, nnz, N)


def test_ssar_chunk_wait_runs_out_then_recovers():
    P, N, k = 8, 200_003, 5_000  # several chunks per pair: chunk 1 waits on chunk 0
    idx, val, nnz = W.uniform_streams(P, N, k, 77)
    di, dv, dn = streams_to_dev(idx, val, nnz)
    ws = api.workspace(api.ssar_workspace_size(P, k, N), DEV)
    api.set_fault_injection(ws, api.INJECT_WITHHOLD_FIRST)
    api.ssar_allreduce(di, dv, dn, N, ws=ws)
    assert api.get_status(ws) == TIMEOUT
    api.set_fault_injection(ws, 0)
    gi, gv, gn, _ = api.ssar_allreduce(di, dv, dn, N, ws=ws)
    assert api.get_status(ws) == 0
    oi, ov, _ = oracle.ssar(idx, val, nnz, N)
    U = int(gn.item())
    assert np.array_equal(u32(gi[:U]), oi) and np.array_equal(bits(gv[:U].cpu().numpy()), bits(ov))


def test_a_fresh_workspace_has_no_fault_armed():
    """A workspace whose header was zeroed at creation is never armed, and
    arming one workspace leaves another untouched."""
    P, N, k = 8, 200_000, 4_000
    idx, val, nnz = W.uniform_streams(P, N, k, 301)
    di, dv, dn = streams_to_dev(idx, val, nnz)
    armed = api.workspace(api.reduce_workspace_size(P, N), DEV)
    clean = api.workspace(api.reduce_workspace_size(P, N), DEV)
    api.set_fault_injection(armed, api.INJECT_WITHHOLD_FIRST)
    out = api.sparse_reduce(di, dv, dn, N, ws=clean)
    assert api.get_status(clean) == 0
    _reduce_matches_oracle(out, idx, val, nnz, N)
    assert int(armed[32:36].cpu().view(torch.int32).item()) != 0


def test_checked_mode_flags_non_finite_inputs():
    """sparcml_check_finite records SPARCML_ERR_NONFINITE for a NaN or an inf
    anywhere in the array (head, 16-byte quads, tail; aligned and unaligned
    starts) and nothing for finite data, however large or small."""
    NONFINITE = api.STATUS_CODE["SPARCML_ERR_NONFINITE"]
    status = api.status_word(DEV)
    g = torch.Generator(device=DEV).manual_seed(11)
    x = torch.randn(1_000_003, device=DEV, generator=g)
    x[7] = 3.0e38
    x[8] = 1.0e-40  # subnormal
    api.check_finite(x, status)
    assert api.get_status(status) == 0
    for pos, v in [(0, float("nan")), (1, float("inf")), (500_000, float("-inf")),
                   (999_999, float("nan")), (1_000_002, float("inf"))]:
        y = x.clone()
        y[pos] = v
        api.check_finite(y, status)
        assert api.get_status(status) == NONFINITE, pos
    for start in (1, 2, 3):  # views starting 4, 8 and 12 bytes past a 16-byte boundary
        y = x.clone()
        y[start] = float("nan")
        api.check_finite(y[start:], status)
        assert api.get_status(status) == NONFINITE, start
        api.check_finite(y[start + 1:], status)
        assert api.get_status(status) == 0, start
    api.check_finite(x[:0], status)
    assert api.get_status(status) == 0
    # the workspace of a reduce is a status word too: the next clean call is clean
    ws = api.workspace(api.reduce_workspace_size(2, 1000), DEV)
    y = x.clone()
    y[123] = float("nan")
    api.check_finite(y, ws)
    assert api.get_status(ws) == NONFINITE
    assert api.get_status(ws) == 0
