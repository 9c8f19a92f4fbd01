"""The C ABI library loads, exports what include/sparcml.h declares, and
rejects bad arguments on the host before enqueuing any GPU work. No GPU:
every call here returns from host-side validation."""
import ctypes as C
import os
import re

import pytest

from top_gradient_compression_gb300 import _lib, api

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sparcml.h")
FAKE = 1 << 20  # a non-null, 256-byte aligned address that is never dereferenced


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sparcml_\w+)\s*\(", text)))


def test_header_declares_the_path_entry_points():
    names = declared_functions()
    for want in ("sparcml_topk_ef", "sparcml_pack", "sparcml_sparse_reduce", "sparcml_densify",
                 "sparcml_quantize4", "sparcml_dequantize4", "sparcml_sparse_reduce_q4",
                 "sparcml_get_status"):
        assert want in names


def test_library_exports_every_declared_symbol():
    lib = _lib.load()
    names = declared_functions()
    assert set(names) == set(_lib.SIGNATURES), "binding table and header disagree"
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_launch_counter():
    lib = _lib.load()
    for code, name in api.STATUS.items():
        assert lib.sparcml_status_string(code).decode() == name
    assert lib.sparcml_status_string(99) == b"SPARCML_ERR_UNKNOWN"
    assert lib.sparcml_launch_count() == 0  # nothing launched without a GPU


def test_workspace_sizes():
    lib = _lib.load()
    ws = lib.sparcml_topk_ef_uniform_workspace_size
    assert ws(0, 10, 10, 1, 100) == 0
    assert ws(1, 10, 10, 2, 1) == 0  # k_num > k_den
    assert ws(1, 1 << 32, 10, 1, 100) == 0  # N too large
    small = ws(4, 65536, 65536, 1, 100)
    big = ws(8, 25_557_032, 100_000, 1, 1000)
    assert 0 < small < big
    assert small % 256 == 0 and big % 256 == 0
    # candidate slots are bounded by the input size: at most 8 bytes per entry + overhead
    assert big < 8 * 8 * 25_557_032
    b, k = api.uniform_segments(25_557_032, 100_000, 1, 1000)
    assert api.topk_ef_segments_workspace_size(8, 25_557_032, b, k) == big
    assert lib.sparcml_sparse_reduce_workspace_size(64, 4_194_304) > 0
    assert lib.sparcml_sparse_reduce_workspace_size(5000, 100) == 0  # P above the limit
    assert lib.sparcml_pack_workspace_size(2, 100) >= 256


def test_topk_host_validation_returns_before_launch():
    import numpy as np
    lib = _lib.load()
    good_b = np.array([0, 1, 8, 500, 1000], np.uint64)
    good_k = np.array([0, 7, 5, 100], np.uint32)
    ws = api.topk_ef_segments_workspace_size(2, 1000, good_b, good_k)
    assert ws > 0

    def call(b=good_b, k=good_k, nseg=None, P=2, N=1000, cap=112, w=FAKE, wsb=ws, grad=FAKE):
        b = np.ascontiguousarray(b, np.uint64)
        k = np.ascontiguousarray(k, np.uint32)
        return lib.sparcml_topk_ef(grad, FAKE, P, N, b.ctypes.data, k.ctypes.data,
                                   k.size if nseg is None else nseg, FAKE, FAKE, FAKE, cap, w, wsb,
                                   None)
    bad = api.STATUS_CODE["SPARCML_ERR_INVALID_ARG"]
    assert call(grad=None) == bad and call(P=0) == bad and call(N=0) == bad
    assert call(nseg=0) == bad
    assert call(b=[1, 8, 500, 1000, 1000]) == bad      # does not start at 0
    assert call(b=[0, 1, 8, 500, 999]) == bad          # does not end at N
    assert call(b=[0, 8, 8, 500, 1000]) == bad         # an empty segment
    assert call(k=[2, 7, 5, 100]) == bad               # k_s > n_s
    assert call(w=FAKE + 8) == bad                     # workspace must be 256-byte aligned
    assert call(wsb=ws - 1) == api.STATUS_CODE["SPARCML_ERR_WORKSPACE"]
    assert call(cap=111) == api.STATUS_CODE["SPARCML_ERR_CAPACITY"]  # 112 entries per node
    uw = lib.sparcml_topk_ef_uniform_workspace_size(2, 1000, 100, 1, 10)
    u = lib.sparcml_topk_ef_uniform
    assert u(FAKE, FAKE, 2, 1000, 0, 1, 10, FAKE, FAKE, FAKE, 100, FAKE, uw, None) == bad
    assert u(FAKE, FAKE, 2, 1000, 100, 11, 10, FAKE, FAKE, FAKE, 100, FAKE, uw, None) == bad
    assert u(FAKE, FAKE, 2, 1000, 100, 1, 10, FAKE, FAKE, FAKE, 99, FAKE, uw, None) == 3


def test_reduce_and_other_host_validation():
    lib = _lib.load()
    ws = lib.sparcml_sparse_reduce_workspace_size(4, 1000)
    r = lib.sparcml_sparse_reduce
    assert r(FAKE, FAKE, FAKE, 4, 10, 1000, 1, 4, FAKE, FAKE, 249, FAKE, FAKE, FAKE, FAKE, ws,
             None) == 3  # out_cap < floor(N/4)
    assert r(FAKE, FAKE, FAKE, 4, 10, 1000, 1, 4, FAKE, FAKE, 250, None, FAKE, FAKE, FAKE, ws,
             None) == 1
    assert r(FAKE, FAKE, FAKE, 4, 10, 1000, 5, 4, FAKE, FAKE, 250, FAKE, FAKE, FAKE, FAKE, ws,
             None) == 1
    assert r(FAKE, FAKE, FAKE, 4, 10, 1000, 1, 4, FAKE, FAKE, 250, FAKE, FAKE, FAKE, FAKE, ws - 1,
             None) == 2
    assert lib.sparcml_sparse_reduce_workspace_size(4097, 1000) == 0  # P above 4,096
    assert r(FAKE, FAKE, FAKE, 4097, 10, 1000, 1, 4, FAKE, FAKE, 250, FAKE, FAKE, FAKE, FAKE,
             1 << 30, None) == 1
    assert r(FAKE, FAKE, FAKE, 4, 1 << 32, 1000, 1, 4, FAKE, FAKE, 250, FAKE, FAKE, FAKE, FAKE,
             ws, None) == 1  # cap of 2^32 entries
    assert lib.sparcml_quantize4(FAKE, FAKE, FAKE, 2, 100, 3, 0, FAKE, FAKE, None, None) == 1
    assert lib.sparcml_dequantize4(FAKE, FAKE, FAKE, 2, 0, 512, FAKE, None, None) == 1
    assert lib.sparcml_densify(FAKE, FAKE, FAKE, 2, 10, 0, FAKE, None, None) == 1
    assert lib.sparcml_pack(FAKE, 2, 100, C.c_float(-1.0), FAKE, FAKE, FAKE, 10, FAKE, 4096,
                            None) == 1
    assert lib.sparcml_pack(FAKE, 2, 100, C.c_float(float("nan")), FAKE, FAKE, FAKE, 10, FAKE,
                            4096, None) == 1
    assert lib.sparcml_get_status(None, None) == 1
    q = lib.sparcml_quantize
    assert q(None, FAKE, None, 1, 16, 8, 3, 0, FAKE, FAKE, None, None, None) == 1  # bits
    assert q(None, FAKE, None, 1, 16, 6, 2, 0, FAKE, FAKE, None, None, None) == 1  # bucket
    assert q(None, None, None, 1, 16, 8, 4, 0, FAKE, FAKE, None, None, None) == 1  # val
    assert lib.sparcml_dequantize(FAKE, FAKE, None, 1, 16, 8, 5, FAKE, None, None) == 1
    ws = lib.sparcml_sparse_reduce_workspace_size(2, 1000)
    assert lib.sparcml_sparse_reduce_qb(FAKE, FAKE, FAKE, FAKE, 2, 10, 6, 2, 1000, 1, 4, FAKE,
                                        FAKE, 250, FAKE, FAKE, FAKE, FAKE, ws, None) == 1
    assert lib.sparcml_sparse_reduce_op(FAKE, FAKE, FAKE, 2, 10, 1000, 4, 1, 4, FAKE, FAKE, 250,
                                        FAKE, FAKE, FAKE, FAKE, ws, None) == 1  # unknown op
    sw = lib.sparcml_ssar_workspace_size(4, 100, 1000)
    assert sw > 0 and lib.sparcml_ssar_workspace_size(3, 100, 1000) == 0  # P not a power of 2
    ss = lib.sparcml_ssar_allreduce
    assert ss(FAKE, FAKE, FAKE, 6, 100, 1000, FAKE, FAKE, 600, FAKE, None, FAKE, sw, None) == 1
    assert ss(FAKE, FAKE, FAKE, 4, 100, 1000, FAKE, FAKE, 399, FAKE, None, FAKE, sw, None) == 3
    assert ss(FAKE, FAKE, FAKE, 4, 100, 1000, FAKE, FAKE, 400, FAKE, None, FAKE, sw - 1,
              None) == 2


def test_equal_segment_table_matches_the_oracle_rule():
    """The library's equal-segment table and its k rounding (floor, the last
    segment takes the remainder) agree with the oracle's."""
    import oracle
    for N, L, kn, kd in [(65_536, 65_536, 1, 100), (25_557_032, 100_000, 1, 1000), (1001, 7, 3, 8),
                         (10, 100, 1, 1), (33, 1, 1, 2)]:
        b, k = api.uniform_segments(N, L, kn, kd)
        ob, ok = oracle.uniform_segments(N, L, kn, kd)
        assert list(b) == ob and list(k) == ok
        assert api.segment_k_total(N, L, kn, kd) == sum(oracle.segment_ks(N, L, kn, kd))
    lib = _lib.load()
    assert lib.sparcml_topk_uniform_segments(0, 10, 1, 2, None, None) == 0
    assert lib.sparcml_topk_uniform_segments(10, 0, 1, 2, None, None) == 0
    assert lib.sparcml_topk_uniform_segments(10, 3, 3, 2, None, None) == 0
    assert lib.sparcml_topk_total_k(None, 5) == 0


def test_binding_arity_matches_the_header():
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    decls = re.findall(r"\b(sparcml_\w+)\s*\(([^)]*)\)\s*;", text)
    assert decls
    for name, params in decls:
        params = params.strip()
        n = 0 if params in ("", "void") else len(params.split(","))
        assert len(_lib.SIGNATURES[name][1]) == n, name
