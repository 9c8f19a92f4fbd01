"""Python binding of the C ABI (include/sparcml.h): argument marshalling only.

Every function takes torch CUDA tensors, checks dtype/shape/contiguity,
passes raw device pointers and the current CUDA stream to libsparcml.so and
returns without synchronising. All computation happens in the library's
kernels; there is no fallback path.

Stream layout (SparCML §5.1 sparse streams): ``idx`` int32 [P, cap] (read as
uint32 by the library), ``val`` float32 [P, cap], ``nnz`` int32 [P].
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass

import numpy as _np
import torch

from . import _lib

OK = 0
STATUS = {0: "SPARCML_OK", 1: "SPARCML_ERR_INVALID_ARG", 2: "SPARCML_ERR_WORKSPACE",
          3: "SPARCML_ERR_CAPACITY", 4: "SPARCML_ERR_BAD_STREAM", 5: "SPARCML_ERR_NONFINITE",
          6: "SPARCML_ERR_TIMEOUT", 7: "SPARCML_ERR_CUDA"}
STATUS_CODE = {v: k for k, v in STATUS.items()}


class SparcmlError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn}: {_lib.load().sparcml_status_string(code).decode()} ({code})")
        self.code = code


def _check(fn: str, code: int):
    if code != OK:
        raise SparcmlError(fn, code)


def _cuda(t: torch.Tensor, dtype, name: str, ndim: int | None = None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")
    return t.data_ptr()


def _opt_ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def workspace(nbytes: int, device) -> torch.Tensor:
    """Caller-owned scratch for one library call (256-byte aligned by torch's allocator)."""
    ws = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)
    assert ws.data_ptr() % 256 == 0
    ws[:64].zero_()  # header: status word, fault-injection word
    return ws


def status_word(device) -> torch.Tensor:
    return torch.zeros(64, dtype=torch.int32, device=device)


def make_events(n: int, stream=None) -> list:
    """CUDA events usable by the *_traced entry points (each recorded once so the
    underlying cudaEvent_t exists)."""
    s = torch.cuda.current_stream() if stream is None else stream
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in evs:
        e.record(s)
    return evs


def _event_array(events):
    if events is None:
        return None
    arr = (C.c_void_p * len(events))(*[e.cuda_event for e in events])
    return arr


INJECT_WITHHOLD_FIRST = 1


def set_fault_injection(ws: torch.Tensor, mode: int, stream=None):
    """Arm (mode INJECT_WITHHOLD_FIRST) or clear (0) the workspace's fault
    injection: later reduce / SSAR calls with ws see their look-back waits run
    out and record SPARCML_ERR_TIMEOUT (include/sparcml.h)."""
    _check("sparcml_set_fault_injection",
           _lib.load().sparcml_set_fault_injection(ws.data_ptr(), int(mode), _stream(stream)))


def launch_count() -> int:
    return int(_lib.load().sparcml_launch_count())


def get_status(word: torch.Tensor, stream=None) -> int:
    """Synchronise the stream, return and clear the first device-side error."""
    return int(_lib.load().sparcml_get_status(word.data_ptr(), _stream(stream)))


# ---------------------------------------------------------------------------
# Top-k with error feedback (§2.2, §4) fused with packing (§5.1), over a
# segment table (layer-wise sparsification, §8.4).
# ---------------------------------------------------------------------------
def _table(seg_begin, seg_k):
    """Host arrays of a segment table: (seg_begin uint64 [nseg+1], seg_k uint32 [nseg])."""
    b = _np.ascontiguousarray(_np.asarray(seg_begin, dtype=_np.uint64))
    k = _np.ascontiguousarray(_np.asarray(seg_k, dtype=_np.uint32))
    if b.ndim != 1 or k.ndim != 1 or b.size != k.size + 1:
        raise ValueError("seg_begin needs nseg + 1 entries and seg_k nseg")
    return b, k


def uniform_segments(N: int, seg_len: int, k_num: int, k_den: int):
    """The library's equal-segment table: (seg_begin uint64 [nseg+1], seg_k uint32 [nseg])."""
    lib = _lib.load()
    n = int(lib.sparcml_topk_uniform_segments(N, seg_len, k_num, k_den, None, None))
    if n == 0:
        raise ValueError("invalid equal-segment table parameters")
    b = _np.zeros(n + 1, _np.uint64)
    k = _np.zeros(n, _np.uint32)
    lib.sparcml_topk_uniform_segments(N, seg_len, k_num, k_den, b.ctypes.data, k.ctypes.data)
    return b, k


def total_k(seg_k) -> int:
    """Entries a node's stream holds for a table (the capacity it needs)."""
    k = _np.ascontiguousarray(_np.asarray(seg_k, dtype=_np.uint32))
    return int(_lib.load().sparcml_topk_total_k(k.ctypes.data, k.size))


def segment_k_total(N: int, seg_len: int, k_num: int, k_den: int) -> int:
    return total_k(uniform_segments(N, seg_len, k_num, k_den)[1])


def topk_fallbacks(ws: torch.Tensor, stream=None) -> int:
    """(node, segment) pairs the last Top-k call with ws decided by re-reading
    the segment (same results, slower); synchronises the stream."""
    n = int(_lib.load().sparcml_topk_ef_fallbacks(ws.data_ptr(), _stream(stream)))
    if n < 0:
        raise SparcmlError("sparcml_topk_ef_fallbacks", 7)
    return n


def topk_ef_workspace_size(P: int, N: int, seg_len: int, k_num: int, k_den: int) -> int:
    return int(_lib.load().sparcml_topk_ef_uniform_workspace_size(P, N, seg_len, k_num, k_den))


def topk_ef_segments_workspace_size(P: int, N: int, seg_begin, seg_k) -> int:
    b, k = _table(seg_begin, seg_k)
    return int(_lib.load().sparcml_topk_ef_workspace_size(P, N, b.ctypes.data, k.ctypes.data,
                                                          k.size))


def _topk_out(out, P, cap, device):
    if out is None:
        out = (torch.empty((P, max(cap, 1)), dtype=torch.int32, device=device),
               torch.empty((P, max(cap, 1)), dtype=torch.float32, device=device),
               torch.empty((P,), dtype=torch.int32, device=device))
    idx, val, nnz = out
    return out, (_cuda(idx, torch.int32, "out_idx", 2), _cuda(val, torch.float32, "out_val", 2),
                 _cuda(nnz, torch.int32, "out_nnz", 1), idx.shape[1])


def _grad_res(grad, residual):
    gp = _cuda(grad, torch.float32, "grad", 2)
    rp = _cuda(residual, torch.float32, "residual", 2)
    if residual.shape != grad.shape:
        raise ValueError("grad and residual shapes differ")
    return gp, rp


def topk_ef(grad: torch.Tensor, residual: torch.Tensor, seg_len: int, k_num: int, k_den: int,
            out=None, ws: torch.Tensor | None = None, stream=None, events=None):
    """Equal segments of seg_len, density k_num/k_den. Returns (idx int32 [P, cap],
    val float32 [P, cap], nnz int32 [P]); residual is updated. ``events``: optional
    4 CUDA events (see make_events) recorded around the phases."""
    gp, rp = _grad_res(grad, residual)
    P, N = grad.shape
    out, (ip, vp, np_, cap) = _topk_out(out, P, segment_k_total(N, seg_len, k_num, k_den)
                                        if out is None else 0, grad.device)
    if ws is None:
        ws = workspace(topk_ef_workspace_size(P, N, seg_len, k_num, k_den), grad.device)
    lib = _lib.load()
    if events is None:
        _check("sparcml_topk_ef_uniform", lib.sparcml_topk_ef_uniform(
            gp, rp, P, N, seg_len, k_num, k_den, ip, vp, np_, cap, ws.data_ptr(), ws.numel(),
            _stream(stream)))
    else:
        assert len(events) == 4
        _check("sparcml_topk_ef_uniform_traced", lib.sparcml_topk_ef_uniform_traced(
            gp, rp, P, N, seg_len, k_num, k_den, ip, vp, np_, cap, ws.data_ptr(), ws.numel(),
            _stream(stream), _event_array(events)))
    return out


def topk_ef_segments(grad: torch.Tensor, residual: torch.Tensor, seg_begin, seg_k, out=None,
                     ws: torch.Tensor | None = None, stream=None, events=None):
    """Segment s = [seg_begin[s], seg_begin[s+1]) keeps seg_k[s] entries (host
    arrays). Returns (idx, val, nnz) as topk_ef; residual is updated."""
    gp, rp = _grad_res(grad, residual)
    P, N = grad.shape
    b, k = _table(seg_begin, seg_k)
    out, (ip, vp, np_, cap) = _topk_out(out, P, total_k(k) if out is None else 0, grad.device)
    if ws is None:
        ws = workspace(topk_ef_segments_workspace_size(P, N, b, k), grad.device)
    lib = _lib.load()
    if events is None:
        _check("sparcml_topk_ef", lib.sparcml_topk_ef(
            gp, rp, P, N, b.ctypes.data, k.ctypes.data, k.size, ip, vp, np_, cap, ws.data_ptr(),
            ws.numel(), _stream(stream)))
    else:
        assert len(events) == 4
        _check("sparcml_topk_ef_traced", lib.sparcml_topk_ef_traced(
            gp, rp, P, N, b.ctypes.data, k.ctypes.data, k.size, ip, vp, np_, cap, ws.data_ptr(),
            ws.numel(), _stream(stream), _event_array(events)))
    return out


# ---------------------------------------------------------------------------
# Pack (§5.1).
# ---------------------------------------------------------------------------
def pack_workspace_size(P: int, N: int) -> int:
    return int(_lib.load().sparcml_pack_workspace_size(P, N))


def pack(x: torch.Tensor, thr: float, cap: int, out=None, ws=None, stream=None):
    xp = _cuda(x, torch.float32, "x", 2)
    P, N = x.shape
    if out is None:
        out = (torch.empty((P, cap), dtype=torch.int32, device=x.device),
               torch.empty((P, cap), dtype=torch.float32, device=x.device),
               torch.empty((P,), dtype=torch.int32, device=x.device))
    idx, val, nnz = out
    if ws is None:
        ws = workspace(pack_workspace_size(P, N), x.device)
    _check("sparcml_pack", _lib.load().sparcml_pack(
        xp, P, N, float(thr), _cuda(idx, torch.int32, "out_idx", 2),
        _cuda(val, torch.float32, "out_val", 2), _cuda(nnz, torch.int32, "out_nnz", 1),
        idx.shape[1], ws.data_ptr(), ws.numel(), _stream(stream)))
    return idx, val, nnz, ws


# ---------------------------------------------------------------------------
# 4-bit stochastic quantisation (§2.2, §6).
# ---------------------------------------------------------------------------
def quantize4(idx, val, nnz, bucket: int, seed: int, codes=None, scales=None, status=None,
              stream=None):
    P, cap = val.shape
    if codes is None:
        codes = torch.zeros((P, (cap + 1) // 2), dtype=torch.uint8, device=val.device)
    if scales is None:
        scales = torch.zeros((P, (cap + bucket - 1) // bucket), dtype=torch.float32,
                             device=val.device)
    _check("sparcml_quantize4", _lib.load().sparcml_quantize4(
        _cuda(idx, torch.int32, "idx", 2), _cuda(val, torch.float32, "val", 2),
        _cuda(nnz, torch.int32, "nnz", 1), P, cap, bucket, seed & (2**64 - 1),
        _cuda(codes, torch.uint8, "codes", 2), _cuda(scales, torch.float32, "scales", 2),
        _opt_ptr(status), _stream(stream)))
    return codes, scales


def dequantize4(codes, scales, nnz, cap: int, bucket: int, out=None, status=None, stream=None):
    P = codes.shape[0]
    if out is None:
        out = torch.zeros((P, cap), dtype=torch.float32, device=codes.device)
    _check("sparcml_dequantize4", _lib.load().sparcml_dequantize4(
        _cuda(codes, torch.uint8, "codes", 2), _cuda(scales, torch.float32, "scales", 2),
        _cuda(nnz, torch.int32, "nnz", 1), P, cap, bucket,
        _cuda(out, torch.float32, "val_out", 2), _opt_ptr(status), _stream(stream)))
    return out


def quantize(val, bucket: int, bits: int, seed: int, idx=None, nnz=None, codes=None,
             scales=None, err=None, status=None, stream=None):
    """b-bit stochastic quantisation (b in {2, 4, 8}) of stream values (idx,
    nnz given) or of dense rows (idx None: positions are the rounding keys;
    nnz None: full rows). val may be 1-D (one row). err, if given, receives
    v - dequantised(v). Returns (codes, scales)."""
    if val.dim() == 1:
        val = val.view(1, -1)
    P, cap = val.shape
    per = 8 // bits
    if codes is None:
        codes = torch.zeros((P, (cap + per - 1) // per), dtype=torch.uint8, device=val.device)
    if scales is None:
        scales = torch.zeros((P, (cap + bucket - 1) // bucket), dtype=torch.float32,
                             device=val.device)
    _check("sparcml_quantize", _lib.load().sparcml_quantize(
        None if idx is None else _cuda(idx, torch.int32, "idx", 2),
        _cuda(val, torch.float32, "val", 2),
        None if nnz is None else _cuda(nnz, torch.int32, "nnz", 1), P, cap, bucket, bits,
        seed & (2**64 - 1), _cuda(codes, torch.uint8, "codes", 2),
        _cuda(scales, torch.float32, "scales", 2),
        None if err is None else _cuda(err.view(P, cap), torch.float32, "err", 2),
        _opt_ptr(status), _stream(stream)))
    return codes, scales


def dequantize(codes, scales, cap: int, bucket: int, bits: int, nnz=None, out=None, status=None,
               stream=None):
    P = codes.shape[0]
    if out is None:
        out = torch.zeros((P, cap), dtype=torch.float32, device=codes.device)
    _check("sparcml_dequantize", _lib.load().sparcml_dequantize(
        _cuda(codes, torch.uint8, "codes", 2), _cuda(scales, torch.float32, "scales", 2),
        None if nnz is None else _cuda(nnz, torch.int32, "nnz", 1), P, cap, bucket, bits,
        _cuda(out, torch.float32, "val_out", 2), _opt_ptr(status), _stream(stream)))
    return out


# ---------------------------------------------------------------------------
# Sparse sum-reduce with the dense switch (§5.1-§5.3).
# ---------------------------------------------------------------------------
@dataclass
class ReduceOut:
    idx: torch.Tensor        # int32 [out_cap]; first nnz entries valid when sparse
    val: torch.Tensor        # float32 [out_cap]
    dense: torch.Tensor      # float32 [N]; valid when is_dense
    nnz: torch.Tensor        # int32 [1] device scalar: U
    is_dense: torch.Tensor   # int32 [1] device scalar


def reduce_workspace_size(P: int, N: int) -> int:
    return int(_lib.load().sparcml_sparse_reduce_workspace_size(P, N))


def reduce_out(N: int, device, dens_num: int = 1, dens_den: int = 4) -> ReduceOut:
    cap = max(N * dens_num // dens_den, 1)
    return ReduceOut(torch.empty(cap, dtype=torch.int32, device=device),
                     torch.empty(cap, dtype=torch.float32, device=device),
                     torch.empty(N, dtype=torch.float32, device=device),
                     torch.zeros(1, dtype=torch.int32, device=device),
                     torch.zeros(1, dtype=torch.int32, device=device))


def _reduce_out_ptrs(o: ReduceOut):
    return (_cuda(o.idx, torch.int32, "out_idx", 1), _cuda(o.val, torch.float32, "out_val", 1),
            o.idx.numel(), _cuda(o.dense, torch.float32, "out_dense", 1),
            _cuda(o.nnz, torch.int32, "out_nnz"), _cuda(o.is_dense, torch.int32, "out_is_dense"))


def sparse_reduce(idx, val, nnz, N: int, dens_num: int = 1, dens_den: int = 4,
                  out: ReduceOut | None = None, ws=None, stream=None, events=None) -> ReduceOut:
    """``events``: optional 3 CUDA events recorded around the two kernels."""
    P, cap = idx.shape
    if out is None:
        out = reduce_out(N, idx.device, dens_num, dens_den)
    if ws is None:
        ws = workspace(reduce_workspace_size(P, N), idx.device)
    oi, ov, ocap, od, on, odn = _reduce_out_ptrs(out)
    args = (_cuda(idx, torch.int32, "idx", 2), _cuda(val, torch.float32, "val", 2),
            _cuda(nnz, torch.int32, "nnz", 1), P, cap, N, dens_num, dens_den, oi, ov, ocap, od,
            on, odn, ws.data_ptr(), ws.numel(), _stream(stream))
    lib = _lib.load()
    if events is None:
        _check("sparcml_sparse_reduce", lib.sparcml_sparse_reduce(*args))
    else:
        assert len(events) == 3
        _check("sparcml_sparse_reduce_traced",
               lib.sparcml_sparse_reduce_traced(*args, _event_array(events)))
    return out


def sparse_reduce_q4(idx, codes, scales, nnz, bucket: int, N: int, dens_num: int = 1,
                     dens_den: int = 4, out: ReduceOut | None = None, ws=None,
                     stream=None) -> ReduceOut:
    P, cap = idx.shape
    if out is None:
        out = reduce_out(N, idx.device, dens_num, dens_den)
    if ws is None:
        ws = workspace(reduce_workspace_size(P, N), idx.device)
    oi, ov, ocap, od, on, odn = _reduce_out_ptrs(out)
    _check("sparcml_sparse_reduce_q4", _lib.load().sparcml_sparse_reduce_q4(
        _cuda(idx, torch.int32, "idx", 2), _cuda(codes, torch.uint8, "codes", 2),
        _cuda(scales, torch.float32, "scales", 2), _cuda(nnz, torch.int32, "nnz", 1), P, cap,
        bucket, N, dens_num, dens_den, oi, ov, ocap, od, on, odn, ws.data_ptr(), ws.numel(),
        _stream(stream)))
    return out


OPS = {"sum": 0, "max": 1, "min": 2, "or": 3}


def sparse_reduce_op(idx, val, nnz, N: int, op: str, dens_num: int = 1, dens_den: int = 4,
                     out: ReduceOut | None = None, ws=None, stream=None) -> ReduceOut:
    """Reduction with sum, max, min or bitwise or (§5.2), neutral element at
    unlisted indices; same outputs as sparse_reduce."""
    P, cap = idx.shape
    if out is None:
        out = reduce_out(N, idx.device, dens_num, dens_den)
    if ws is None:
        ws = workspace(reduce_workspace_size(P, N), idx.device)
    oi, ov, ocap, od, on, odn = _reduce_out_ptrs(out)
    _check("sparcml_sparse_reduce_op", _lib.load().sparcml_sparse_reduce_op(
        _cuda(idx, torch.int32, "idx", 2), _cuda(val, torch.float32, "val", 2),
        _cuda(nnz, torch.int32, "nnz", 1), P, cap, N, OPS[op], dens_num, dens_den, oi, ov, ocap,
        od, on, odn, ws.data_ptr(), ws.numel(), _stream(stream)))
    return out


def sparse_reduce_qb(idx, codes, scales, nnz, bucket: int, bits: int, N: int, dens_num: int = 1,
                     dens_den: int = 4, out: ReduceOut | None = None, ws=None,
                     stream=None) -> ReduceOut:
    P, cap = idx.shape
    if out is None:
        out = reduce_out(N, idx.device, dens_num, dens_den)
    if ws is None:
        ws = workspace(reduce_workspace_size(P, N), idx.device)
    oi, ov, ocap, od, on, odn = _reduce_out_ptrs(out)
    _check("sparcml_sparse_reduce_qb", _lib.load().sparcml_sparse_reduce_qb(
        _cuda(idx, torch.int32, "idx", 2), _cuda(codes, torch.uint8, "codes", 2),
        _cuda(scales, torch.float32, "scales", 2), _cuda(nnz, torch.int32, "nnz", 1), P, cap,
        bucket, bits, N, dens_num, dens_den, oi, ov, ocap, od, on, odn, ws.data_ptr(),
        ws.numel(), _stream(stream)))
    return out


def ssar_workspace_size(P: int, cap: int, N: int) -> int:
    return int(_lib.load().sparcml_ssar_workspace_size(P, cap, N))


def ssar_allreduce(idx, val, nnz, N: int, ws=None, stream=None, events=None):
    """Static sparse allreduce by recursive doubling (§5.3.1), emulated: returns
    (out_idx int32 [min(N, P*cap)], out_val, out_nnz int32 [1], stage_nnz
    int64 [log2 P]); the first out_nnz entries are the result. `events`
    (log2 P + 1 CUDA events) are recorded around the stages."""
    P, cap = idx.shape
    dev = idx.device
    out_cap = min(N, P * cap)
    out_idx = torch.empty(out_cap, dtype=torch.int32, device=dev)
    out_val = torch.empty(out_cap, dtype=torch.float32, device=dev)
    out_nnz = torch.zeros(1, dtype=torch.int32, device=dev)
    stages = P.bit_length() - 1
    stage_nnz = torch.zeros(max(stages, 1), dtype=torch.int64, device=dev)
    if ws is None:
        ws = workspace(ssar_workspace_size(P, cap, N), dev)
    lib = _lib.load()
    args = (_cuda(idx, torch.int32, "idx", 2), _cuda(val, torch.float32, "val", 2),
            _cuda(nnz, torch.int32, "nnz", 1), P, cap, N, out_idx.data_ptr(), out_val.data_ptr(),
            out_cap, out_nnz.data_ptr(), stage_nnz.data_ptr(), ws.data_ptr(), ws.numel(),
            _stream(stream))
    if events is None:
        _check("sparcml_ssar_allreduce", lib.sparcml_ssar_allreduce(*args))
    else:
        arr = (C.c_void_p * len(events))(*[e.cuda_event for e in events])
        _check("sparcml_ssar_allreduce_traced", lib.sparcml_ssar_allreduce_traced(*args, arr))
    return out_idx, out_val, out_nnz, stage_nnz[:stages]


def densify(idx, val, nnz, N: int, out=None, status=None, stream=None):
    P, cap = idx.shape
    if out is None:
        out = torch.empty((P, N), dtype=torch.float32, device=idx.device)
    _check("sparcml_densify", _lib.load().sparcml_densify(
        _cuda(idx, torch.int32, "idx", 2), _cuda(val, torch.float32, "val", 2),
        _cuda(nnz, torch.int32, "nnz", 1), P, cap, N, _cuda(out, torch.float32, "dense", 2),
        _opt_ptr(status), _stream(stream)))
    return out


def check_finite(x: torch.Tensor, status: torch.Tensor, stream=None) -> None:
    """Checked mode for an input: records SPARCML_ERR_NONFINITE in `status`
    (a status word or workspace) if x holds a NaN or an inf. Non-blocking;
    read it with get_status."""
    if not x.is_cuda or x.dtype != torch.float32 or not x.is_contiguous():
        raise ValueError("check_finite: x must be a contiguous float32 CUDA tensor")
    _check("sparcml_check_finite", _lib.load().sparcml_check_finite(
        x.data_ptr() if x.numel() else None, x.numel(), status.data_ptr(), _stream(stream)))
