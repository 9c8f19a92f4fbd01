"""Shared helpers of the GPU parity tests: move seeded inputs to the device,
run the CUDA path through the C ABI and compare with the oracle bit for bit."""
import numpy as np
import torch

import oracle
from top_gradient_compression_gb300 import api

DEV = "cuda:0"


def u32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().view(np.uint32)


def bits(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, np.float32)).view(np.uint32)


def streams_to_dev(idx, val, nnz):
    return (torch.from_numpy(np.ascontiguousarray(idx).view(np.int32)).to(DEV),
            torch.from_numpy(np.ascontiguousarray(val, np.float32)).to(DEV),
            torch.from_numpy(np.ascontiguousarray(nnz).view(np.int32)).to(DEV))


def check_fallbacks(ws, fallback):
    """fallback False: no (node, segment) was decided by the raw select; True:
    at least one was; None: either."""
    n = api.topk_fallbacks(ws)
    if fallback is not None:
        assert (n > 0) == fallback, f"raw-select fallbacks: {n}"


def check_topk_steps(grads, seg_len, k_num, k_den, res0=None, fallback=None):
    """Run the EF steps on GPU and oracle side by side; everything must match bitwise."""
    P, N = grads[0].shape
    res_o = np.zeros((P, N), np.float32) if res0 is None else res0.copy()
    res_g = torch.from_numpy(res_o.copy()).to(DEV)
    ws = api.workspace(api.topk_ef_workspace_size(P, N, seg_len, k_num, k_den), DEV)
    for g in grads:
        gg = torch.from_numpy(np.ascontiguousarray(g)).to(DEV)
        idx, val, nnz = api.topk_ef(gg, res_g, seg_len, k_num, k_den, ws=ws)
        st = api.get_status(ws)
        assert st == 0, api.STATUS[st]
        check_fallbacks(ws, fallback)
        oi, ov, on = oracle.topk_ef(g, res_o, seg_len, k_num, k_den, cap=idx.shape[1])
        gn = u32(nnz)
        assert np.array_equal(gn, on)
        gi, gv = u32(idx), bits(val.cpu().numpy())
        for p in range(P):
            n = int(on[p])
            assert np.array_equal(gi[p, :n], oi[p, :n]), f"node {p}: indices differ"
            assert np.array_equal(gv[p, :n], bits(ov[p, :n])), f"node {p}: values differ"
        assert np.array_equal(bits(res_g.cpu().numpy()), bits(res_o)), "residual differs"
    return res_o


def check_topk_table_steps(grads, seg_begin, seg_k, res0=None, fallback=None):
    """The segment-table form over several EF steps against the oracle, bitwise:
    streams, nnz and the residual after every step."""
    P, N = grads[0].shape
    res_o = np.zeros((P, N), np.float32) if res0 is None else res0.copy()
    res_g = torch.from_numpy(res_o.copy()).to(DEV)
    ws = api.workspace(api.topk_ef_segments_workspace_size(P, N, seg_begin, seg_k), DEV)
    for g in grads:
        gg = torch.from_numpy(np.ascontiguousarray(g)).to(DEV)
        idx, val, nnz = api.topk_ef_segments(gg, res_g, seg_begin, seg_k, ws=ws)
        st = api.get_status(ws)
        assert st == 0, api.STATUS[st]
        check_fallbacks(ws, fallback)
        oi, ov, on = oracle.topk_ef_segments(g, res_o, seg_begin, seg_k, cap=idx.shape[1],
                                             threads=4)
        assert np.array_equal(u32(nnz), on)
        gi, gv = u32(idx), bits(val.cpu().numpy())
        for p in range(P):
            n = int(on[p])
            assert np.array_equal(gi[p, :n], oi[p, :n]), f"node {p}: indices differ"
            assert np.array_equal(gv[p, :n], bits(ov[p, :n])), f"node {p}: values differ"
        assert np.array_equal(bits(res_g.cpu().numpy()), bits(res_o)), "residual differs"
    return res_o


def check_reduce(idx, val, nnz, N, dens_num=1, dens_den=4, repeat=1):
    P = idx.shape[0]
    di, dv, dn = streams_to_dev(idx, val, nnz)
    ws = api.workspace(api.reduce_workspace_size(P, N), DEV)
    ref = oracle.sparse_reduce(idx, val, nnz, N, dens_num, dens_den)
    first = None
    for _ in range(repeat):
        out = api.sparse_reduce(di, dv, dn, N, dens_num, dens_den, ws=ws)
        st = api.get_status(ws)
        assert st == 0, api.STATUS[st]
        U = int(out.nnz.item())
        dense = bool(out.is_dense.item())
        assert U == ref["nnz"] and dense == ref["is_dense"]
        if dense:
            got = bits(out.dense.cpu().numpy())
            assert np.array_equal(got, bits(ref["dense"]))
        else:
            got = (u32(out.idx[:U]).copy(), bits(out.val[:U].cpu().numpy()).copy())
            assert np.array_equal(got[0], ref["idx"])
            assert np.array_equal(got[1], bits(ref["val"]))
        if first is None:
            first = got
        else:  # bitwise identical on a second run: no races in the fixed-order path
            if dense:
                assert np.array_equal(first, got)
            else:
                assert np.array_equal(first[0], got[0]) and np.array_equal(first[1], got[1])
    return ref
