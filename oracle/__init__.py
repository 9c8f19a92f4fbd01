"""CPU oracle for the SparCML sparse-reduction hot path (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg use this package. The product path never imports it. The arithmetic lives
in ``oracle.cpp`` (plain C++17: sort-based Top-k, std::map sum, SplitMix64
rounding draws); this module compiles it with g++ and marshals numpy arrays.

Every function here cites the section of "SparCML: High-Performance Sparse
Communication for Machine Learning" that it follows in ``oracle.cpp``.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK, INVALID, CAPACITY, BAD_STREAM = 0, 1, 3, 4


def build(force: bool = False) -> str:
    """Compile oracle.cpp into liboracle.so next to it (no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread",
                               "-ffp-contract=off", "-fno-fast-math", "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = C.CDLL(build())
            u32p, f32p, u8p = (np.ctypeslib.ndpointer(dtype=t, flags="C_CONTIGUOUS")
                               for t in (np.uint32, np.float32, np.uint8))
            lib.oracle_splitmix64.argtypes = [C.c_uint64]
            lib.oracle_splitmix64.restype = C.c_uint64
            lib.oracle_topk_ef.argtypes = [f32p, f32p, C.c_int32, C.c_uint64, C.c_uint64,
                                           C.c_uint64, C.c_uint64, u32p, f32p, u32p, C.c_uint64]
            u64p_ = np.ctypeslib.ndpointer(dtype=np.uint64, flags="C_CONTIGUOUS")
            lib.oracle_topk_ef_segments.argtypes = [f32p, f32p, C.c_int32, C.c_uint64, u64p_,
                                                    u64p_, C.c_uint64, u32p, f32p, u32p,
                                                    C.c_uint64]
            lib.oracle_topk_ef_segments_mt.argtypes = [f32p, f32p, C.c_int32, C.c_uint64, u64p_,
                                                       u64p_, C.c_uint64, u32p, f32p, u32p,
                                                       C.c_uint64, C.c_int32]
            lib.oracle_sparse_reduce_mt.argtypes = [u32p, f32p, u32p, C.c_int32, C.c_uint64,
                                                    C.c_uint64, C.c_uint32, C.c_uint32, u32p,
                                                    f32p, C.c_uint64, f32p,
                                                    C.POINTER(C.c_uint64), C.POINTER(C.c_int32),
                                                    C.c_int32]
            lib.oracle_pack.argtypes = [f32p, C.c_int32, C.c_uint64, C.c_float, u32p, f32p,
                                        u32p, C.c_uint64]
            lib.oracle_quantize4.argtypes = [u32p, f32p, u32p, C.c_int32, C.c_uint64,
                                             C.c_uint32, C.c_uint64, u8p, f32p]
            lib.oracle_dequantize4.argtypes = [u8p, f32p, u32p, C.c_int32, C.c_uint64,
                                               C.c_uint32, f32p]
            lib.oracle_quantize.argtypes = [C.c_void_p, f32p, C.c_void_p, C.c_int32, C.c_uint64,
                                            C.c_uint32, C.c_uint32, C.c_uint64, u8p, f32p,
                                            C.c_void_p]
            lib.oracle_dequantize.argtypes = [u8p, f32p, C.c_void_p, C.c_int32, C.c_uint64,
                                              C.c_uint32, C.c_uint32, f32p]
            lib.oracle_sparse_reduce.argtypes = [u32p, f32p, u32p, C.c_int32, C.c_uint64,
                                                 C.c_uint64, C.c_uint32, C.c_uint32, u32p, f32p,
                                                 C.c_uint64, f32p, C.POINTER(C.c_uint64),
                                                 C.POINTER(C.c_int32)]
            lib.oracle_sparse_reduce_op.argtypes = [u32p, f32p, u32p, C.c_int32, C.c_uint64,
                                                    C.c_uint64, C.c_int32, C.c_uint32,
                                                    C.c_uint32, u32p, f32p, C.c_uint64, f32p,
                                                    C.POINTER(C.c_uint64), C.POINTER(C.c_int32)]
            u64p = np.ctypeslib.ndpointer(dtype=np.uint64, flags="C_CONTIGUOUS")
            lib.oracle_ssar.argtypes = [u32p, f32p, u32p, C.c_int32, C.c_uint64, C.c_uint64,
                                        u32p, f32p, C.c_uint64, C.POINTER(C.c_uint64), u64p]
            lib.oracle_densify.argtypes = [u32p, f32p, u32p, C.c_int32, C.c_uint64, C.c_uint64,
                                           f32p]
            for f in ("oracle_topk_ef", "oracle_topk_ef_segments", "oracle_topk_ef_segments_mt",
                      "oracle_pack", "oracle_quantize4", "oracle_dequantize4",
                      "oracle_quantize", "oracle_dequantize", "oracle_sparse_reduce",
                      "oracle_sparse_reduce_op", "oracle_sparse_reduce_mt", "oracle_ssar",
                      "oracle_densify"):
                getattr(lib, f).restype = C.c_int
            _lib = lib
    return _lib


class OracleError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} returned status {code}")
        self.code = code


def _check(fn, code):
    if code != OK:
        raise OracleError(fn, code)


def _u32(a):
    return np.ascontiguousarray(np.asarray(a).view(np.uint32) if np.asarray(a).dtype == np.int32
                                else np.asarray(a, dtype=np.uint32))


def _f32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def splitmix64(x: int) -> int:
    """SplitMix64 output for state ``x`` (increment, then mix)."""
    return int(_load().oracle_splitmix64(C.c_uint64(x & 0xFFFFFFFFFFFFFFFF)))


def segment_ks(N: int, seg_len: int, k_num: int, k_den: int) -> list[int]:
    """k_s = floor(n_s * k_num / k_den) for the segments [s*seg_len, ...) of one node."""
    return [min(seg_len, N - b) * k_num // k_den for b in range(0, N, seg_len)]


def topk_ef(grad, residual, seg_len, k_num, k_den, cap=None):
    """Top-k with error feedback (SparCML §2.2 and §4).

    grad: [P, N] float32; residual: [P, N] float32, updated IN PLACE (must be a
    contiguous float32 numpy array). Returns (idx [P, cap] uint32, val [P, cap]
    float32, nnz [P] uint32)."""
    g = _f32(grad)
    assert isinstance(residual, np.ndarray) and residual.dtype == np.float32 \
        and residual.flags.c_contiguous and residual.shape == g.shape
    P, N = g.shape
    total = sum(segment_ks(N, seg_len, k_num, k_den))
    cap = max(total, 1) if cap is None else cap
    idx = np.zeros((P, cap), np.uint32)
    val = np.zeros((P, cap), np.float32)
    nnz = np.zeros((P,), np.uint32)
    _check("oracle_topk_ef", _load().oracle_topk_ef(g, residual, P, N, seg_len, k_num, k_den,
                                                    idx, val, nnz, cap))
    return idx, val, nnz


def uniform_segments(N: int, seg_len: int, k_num: int, k_den: int):
    """The equal-segment table: begins [0, L, 2L, ..., N] and k_s = floor(n_s * k_num / k_den)
    (the last segment takes the remainder, App. A)."""
    begin = list(range(0, N, seg_len)) + [N]
    return begin, segment_ks(N, seg_len, k_num, k_den)


def _seg_arrays(seg_begin, seg_k):
    b = np.ascontiguousarray(np.asarray(seg_begin, dtype=np.uint64))
    k = np.ascontiguousarray(np.asarray(seg_k, dtype=np.uint64))
    if b.ndim != 1 or k.ndim != 1 or b.size != k.size + 1:
        raise ValueError("seg_begin needs nseg + 1 entries and seg_k nseg")
    return b, k


def topk_ef_segments(grad, residual, seg_begin, seg_k, cap=None, threads: int = 1):
    """Top-k with error feedback over an arbitrary segment table (SparCML §2.2,
    §4; layer-wise sparsification, §8.4): segment s = [seg_begin[s],
    seg_begin[s+1]) keeps seg_k[s] entries. residual is updated IN PLACE.
    threads > 1 spreads the (node, segment) pairs over host threads (same
    results). Returns (idx [P, cap] uint32, val [P, cap] float32, nnz [P] uint32)."""
    g = _f32(grad)
    assert isinstance(residual, np.ndarray) and residual.dtype == np.float32 \
        and residual.flags.c_contiguous and residual.shape == g.shape
    P, N = g.shape
    b, k = _seg_arrays(seg_begin, seg_k)
    total = int(k.sum())
    cap = max(total, 1) if cap is None else cap
    idx = np.zeros((P, cap), np.uint32)
    val = np.zeros((P, cap), np.float32)
    nnz = np.zeros((P,), np.uint32)
    if threads > 1:
        _check("oracle_topk_ef_segments_mt", _load().oracle_topk_ef_segments_mt(
            g, residual, P, N, b, k, k.size, idx, val, nnz, cap, threads))
    else:
        _check("oracle_topk_ef_segments", _load().oracle_topk_ef_segments(
            g, residual, P, N, b, k, k.size, idx, val, nnz, cap))
    return idx, val, nnz


def pack(x, thr, cap):
    """Threshold selection |x| > thr into ascending streams (SparCML §5.1).
    Returns (idx, val, nnz, status) where status is CAPACITY on truncation."""
    x = _f32(x)
    P, N = x.shape
    idx = np.zeros((P, cap), np.uint32)
    val = np.zeros((P, cap), np.float32)
    nnz = np.zeros((P,), np.uint32)
    st = _load().oracle_pack(x, P, N, float(thr), idx, val, nnz, cap)
    if st not in (OK, CAPACITY):
        raise OracleError("oracle_pack", st)
    return idx, val, nnz, st


def quantize4(idx, val, nnz, bucket, seed):
    """4-bit stochastic quantisation (SparCML §2.2, §6). Returns (codes, scales)."""
    idx, val, nnz = _u32(idx), _f32(val), _u32(nnz)
    P, cap = val.shape
    codes = np.zeros((P, (cap + 1) // 2), np.uint8)
    scales = np.zeros((P, (cap + bucket - 1) // bucket), np.float32)
    _check("oracle_quantize4", _load().oracle_quantize4(idx, val, nnz, P, cap, bucket,
                                                        C.c_uint64(seed & (2**64 - 1)),
                                                        codes, scales))
    return codes, scales


def dequantize4(codes, scales, nnz, cap, bucket):
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales, nnz = _f32(scales), _u32(nnz)
    P = codes.shape[0]
    out = np.zeros((P, cap), np.float32)
    _check("oracle_dequantize4", _load().oracle_dequantize4(codes, scales, nnz, P, cap, bucket,
                                                            out))
    return out


def _ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def quantize(val, bucket, bits, seed, idx=None, nnz=None, with_error=False):
    """b-bit stochastic quantisation, b in {2, 4, 8} (SparCML §2.2, §6), of
    stream values (idx, nnz given) or dense rows (idx None: the position is
    the rounding key; nnz None: full rows). Returns (codes, scales) or, with
    with_error, (codes, scales, v - dequantised v)."""
    val = _f32(val)
    if val.ndim == 1:
        val = val[None]
    P, cap = val.shape
    idx = None if idx is None else _u32(idx)
    nnz = None if nnz is None else _u32(nnz)
    per_byte = 8 // bits
    codes = np.zeros((P, (cap + per_byte - 1) // per_byte), np.uint8)
    scales = np.zeros((P, (cap + bucket - 1) // bucket), np.float32)
    err = np.zeros((P, cap), np.float32) if with_error else None
    _check("oracle_quantize", _load().oracle_quantize(
        _ptr(idx), val, _ptr(nnz), P, cap, bucket, bits, C.c_uint64(seed & (2**64 - 1)),
        codes, scales, _ptr(err)))
    return (codes, scales, err) if with_error else (codes, scales)


def dequantize(codes, scales, cap, bucket, bits, nnz=None):
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = _f32(scales)
    nnz = None if nnz is None else _u32(nnz)
    P = codes.shape[0]
    out = np.zeros((P, cap), np.float32)
    _check("oracle_dequantize", _load().oracle_dequantize(codes, scales, _ptr(nnz), P, cap,
                                                          bucket, bits, out))
    return out


OPS = {"sum": 0, "max": 1, "min": 2, "or": 3}


def sparse_reduce_op(idx, val, nnz, N, op, dens_num=1, dens_den=4):
    """Reduction of P sparse streams with sum, max, min or bitwise or, each
    with its neutral element for unlisted coordinates (SparCML §5.2). Same
    result dict as sparse_reduce."""
    idx, val, nnz = _u32(idx), _f32(val), _u32(nnz)
    P, cap = idx.shape
    out_cap = max(N * dens_num // dens_den, 1)
    oi = np.zeros(out_cap, np.uint32)
    ov = np.zeros(out_cap, np.float32)
    od = np.zeros(N, np.float32)
    u = C.c_uint64(0)
    d = C.c_int32(0)
    _check("oracle_sparse_reduce_op", _load().oracle_sparse_reduce_op(
        idx, val, nnz, P, cap, N, OPS[op], dens_num, dens_den, oi, ov, out_cap, od,
        C.byref(u), C.byref(d)))
    U = int(u.value)
    if d.value:
        return dict(nnz=U, is_dense=True, idx=None, val=None, dense=od)
    return dict(nnz=U, is_dense=False, idx=oi[:U].copy(), val=ov[:U].copy(), dense=None)


def ssar(idx, val, nnz, N):
    """Static sparse allreduce by recursive doubling (SparCML §5.3.1): log2(P)
    stages of pairwise two-stream sum reduces. Returns (idx, val, stage_nnz)."""
    idx, val, nnz = _u32(idx), _f32(val), _u32(nnz)
    P, cap = idx.shape
    out_cap = int(min(N, P * cap))
    oi = np.zeros(max(out_cap, 1), np.uint32)
    ov = np.zeros(max(out_cap, 1), np.float32)
    stages = np.zeros(max(P.bit_length() - 1, 1), np.uint64)
    u = C.c_uint64(0)
    _check("oracle_ssar", _load().oracle_ssar(idx, val, nnz, P, cap, N, oi, ov, out_cap,
                                              C.byref(u), stages))
    U = int(u.value)
    return oi[:U].copy(), ov[:U].copy(), stages[:P.bit_length() - 1].copy()


def sparse_reduce(idx, val, nnz, N, dens_num=1, dens_den=4, threads: int = 1):
    """Sum-reduction of P sparse streams with the dense switch (SparCML §5.1-§5.3).
    threads > 1 cuts the index space into that many ranges reduced on host
    threads (same results).

    Returns dict(nnz=U, is_dense=bool, idx=uint32[U] | None, val=float32[U] | None,
    dense=float32[N] | None)."""
    idx, val, nnz = _u32(idx), _f32(val), _u32(nnz)
    P, cap = idx.shape
    out_cap = max(N * dens_num // dens_den, 1)
    oi = np.zeros(out_cap, np.uint32)
    ov = np.zeros(out_cap, np.float32)
    od = np.zeros(N, np.float32)
    u = C.c_uint64(0)
    d = C.c_int32(0)
    if threads > 1:
        _check("oracle_sparse_reduce_mt", _load().oracle_sparse_reduce_mt(
            idx, val, nnz, P, cap, N, dens_num, dens_den, oi, ov, out_cap, od,
            C.byref(u), C.byref(d), threads))
    else:
        _check("oracle_sparse_reduce", _load().oracle_sparse_reduce(
            idx, val, nnz, P, cap, N, dens_num, dens_den, oi, ov, out_cap, od,
            C.byref(u), C.byref(d)))
    U = int(u.value)
    if d.value:
        return dict(nnz=U, is_dense=True, idx=None, val=None, dense=od)
    return dict(nnz=U, is_dense=False, idx=oi[:U].copy(), val=ov[:U].copy(), dense=None)


def densify(idx, val, nnz, N):
    idx, val, nnz = _u32(idx), _f32(val), _u32(nnz)
    P, cap = idx.shape
    out = np.zeros((P, N), np.float32)
    _check("oracle_densify", _load().oracle_densify(idx, val, nnz, P, cap, N, out))
    return out
