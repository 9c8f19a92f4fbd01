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
    assert lib.sparcml_topk_ef_workspace_size(0, 10, 10, 1, 100) == 0
    assert lib.sparcml_topk_ef_workspace_size(1, 10, 10, 2, 1) == 0  # k_num > k_den
    assert lib.sparcml_topk_ef_workspace_size(1, 1 << 32, 10, 1, 100) == 0  # N too large
    small = lib.sparcml_topk_ef_workspace_size(4, 65536, 65536, 1, 100)
    big = lib.sparcml_topk_ef_workspace_size(8, 25_557_032, 100_000, 1, 1000)
    assert 0 < small < big
    assert small % 256 == 0 and big % 256 == 0
    # candidate slots are bounded by the input size: at most 8 bytes per entry + overhead
    assert big < 8 * 8 * 25_557_032
    assert lib.sparcml_sparse_reduce_workspace_size(64, 4_194_304) > 0
    assert lib.sparcml_sparse_reduce_workspace_size(5000, 100) == 0  # P above the limit
    assert lib.sparcml_pack_workspace_size(2, 100) >= 256


def test_topk_host_validation_returns_before_launch():
    lib = _lib.load()
    ws = lib.sparcml_topk_ef_workspace_size(2, 1000, 100, 1, 10)
    args = dict(grad=FAKE, res=FAKE, P=2, N=1000, L=100, kn=1, kd=10, oi=FAKE, ov=FAKE, on=FAKE,
                cap=100, ws=FAKE, wsb=ws, s=None)

    def call(**kw):
        a = dict(args, **kw)
        return lib.sparcml_topk_ef(a["grad"], a["res"], a["P"], a["N"], a["L"], a["kn"], a["kd"],
                                   a["oi"], a["ov"], a["on"], a["cap"], a["ws"], a["wsb"], a["s"])
    assert call(grad=None) == api.STATUS_CODE["SPARCML_ERR_INVALID_ARG"]
    assert call(P=0) == 1 and call(N=0) == 1 and call(L=0) == 1 and call(kd=0) == 1
    assert call(kn=11) == 1
    assert call(ws=FAKE + 8) == 1  # workspace must be 256-byte aligned
    assert call(wsb=ws - 1) == 2
    assert call(cap=99) == 3  # 10 segments x 10 entries do not fit


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


def test_segment_k_total_matches_the_oracle_rule():
    import oracle
    for N, L, kn, kd in [(65_536, 65_536, 1, 100), (25_557_032, 100_000, 1, 1000), (1001, 7, 3, 8),
                         (10, 100, 1, 1), (33, 1, 1, 2)]:
        assert api.segment_k_total(N, L, kn, kd) == sum(oracle.segment_ks(N, L, kn, kd))


def test_binding_arity_matches_the_header():
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    decls = re.findall(r"\b(sparcml_\w+)\s*\(([^)]*)\)\s*;", text)
    assert decls
    for name, params in decls:
        params = params.strip()
        n = 0 if params in ("", "void") else len(params.split(","))
        assert len(_lib.SIGNATURES[name][1]) == n, name
