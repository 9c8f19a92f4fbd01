"""GPU parity of the b-bit stochastic quantiser (SparCML §2.2, §6; 2-, 4- and
8-bit outputs) on streams and on dense rows, of its inverse, of the
quantisation-error output, and of the reduce with fused b-bit decode, against
the oracle, bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from top_gradient_compression_gb300 import api, workloads as W

from gpu_helpers import DEV, bits, streams_to_dev, u32

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("b", [2, 4, 8])
@pytest.mark.parametrize("bucket,cap", [(512, 3_001), (96, 3_004), (512, 3_004), (1024, 3_004)])
def test_stream_quantise_dequantise_and_error(b, bucket, cap):
    """cap % 4 == 0 with buckets of 512 / 1,024 takes the register-resident
    vector kernel (rows ending inside a float4 included); the rest the
    entry-by-entry one."""
    P, N, k = 5, 400_000, 3_001
    idx, val, nnz = W.uniform_streams(P, N, k, 61, std=1e-3, cap=cap)
    k = cap
    nnz[1] = 1_237
    nnz[3] = 0
    seed = W.quant_seed(4)
    oc, osc, oe = oracle.quantize(val, bucket, b, seed, idx=idx, nnz=nnz, with_error=True)
    od = oracle.dequantize(oc, osc, k, bucket, b, nnz=nnz)
    di, dv, dn = streams_to_dev(idx, val, nnz)
    err = torch.zeros((P, k), device=DEV)
    codes, scales = api.quantize(dv, bucket, b, seed, idx=di, nnz=dn, err=err)
    deq = api.dequantize(codes, scales, k, bucket, b, nnz=dn)
    torch.cuda.synchronize()
    per = 8 // b
    gc = codes.cpu().numpy()
    for p in range(P):
        n = int(nnz[p])
        nb = (n + per - 1) // per
        assert np.array_equal(gc[p, :nb], oc[p, :nb]), f"node {p} codes"
        ns = (n + bucket - 1) // bucket
        assert np.array_equal(bits(scales[p, :ns].cpu().numpy()), bits(osc[p, :ns]))
        assert np.array_equal(bits(deq[p, :n].cpu().numpy()), bits(od[p, :n]))
        assert np.array_equal(bits(err[p, :n].cpu().numpy()), bits(oe[p, :n]))


@pytest.mark.parametrize("b", [2, 4, 8])
@pytest.mark.parametrize("N", [1_000_003, 1_049_088])
def test_dense_rows_quantise_like_the_oracle(b, N):
    """QSGD on a dense vector (the reduced result of a dense reduce), buckets of
    1,024, positions as rounding keys; a ragged last bucket (the second size
    takes the vector kernel)."""
    rng = np.random.default_rng(b)
    x = rng.standard_normal((1, N)).astype(np.float32)
    x[0, 5000:6024] = 0.0  # an all-zero bucket
    oc, osc = oracle.quantize(x, 1024, b, 12345)
    od = oracle.dequantize(oc, osc, N, 1024, b)
    dx = torch.from_numpy(x).to(DEV)
    codes, scales = api.quantize(dx, 1024, b, 12345)
    deq = api.dequantize(codes, scales, N, 1024, b)
    assert np.array_equal(codes.cpu().numpy(), oc)
    assert np.array_equal(bits(scales.cpu().numpy()), bits(osc))
    assert np.array_equal(bits(deq.cpu().numpy()), bits(od))


def test_dense_quantisation_of_a_dense_reduce_result():
    """Reduce a density-sweep cell whose result is dense, then quantise the dense
    result (4-bit, buckets of 1,024): the codes match the oracle's on the
    oracle's own reduced vector."""
    idx, val, nnz = W.sweep_streams(8, 10, 100)
    N = W.SWEEP_N
    ref = oracle.sparse_reduce(idx, val, nnz, N)
    assert ref["is_dense"]
    oc, osc = oracle.quantize(ref["dense"], 1024, 4, 777)
    di, dv, dn = streams_to_dev(idx, val, nnz)
    out = api.sparse_reduce(di, dv, dn, N)
    assert bool(out.is_dense.item())
    codes, scales = api.quantize(out.dense, 1024, 4, 777)
    assert np.array_equal(codes.cpu().numpy(), oc)
    assert np.array_equal(bits(scales.cpu().numpy()), bits(osc))


@pytest.mark.parametrize("b,k,dense", [(2, 4_000, False), (8, 4_000, False), (2, 40_000, True),
                                       (8, 40_000, True)])
def test_reduce_with_fused_b_bit_decode(b, k, dense):
    P, N, bucket = 6, 300_000, 256
    idx, val, nnz = W.uniform_streams(P, N, k, 33, std=1e-2)
    nnz[2] = k // 3
    seed = W.quant_seed(1)
    oc, osc = oracle.quantize(val, bucket, b, seed, idx=idx, nnz=nnz)
    deq = oracle.dequantize(oc, osc, k, bucket, b, nnz=nnz)
    ref = oracle.sparse_reduce(idx, deq, nnz, N)
    assert ref["is_dense"] == dense
    di, dv, dn = streams_to_dev(idx, val, nnz)
    codes, scales = api.quantize(dv, bucket, b, seed, idx=di, nnz=dn)
    out = api.sparse_reduce_qb(di, codes, scales, dn, bucket, b, N)
    U = int(out.nnz.item())
    assert U == ref["nnz"] and bool(out.is_dense.item()) == dense
    if dense:
        assert np.array_equal(bits(out.dense.cpu().numpy()), bits(ref["dense"]))
    else:
        assert np.array_equal(u32(out.idx[:U]), ref["idx"])
        assert np.array_equal(bits(out.val[:U].cpu().numpy()), bits(ref["val"]))


def test_quantiser_rejects_bad_widths_on_the_host():
    x = torch.zeros((1, 16), device=DEV)
    codes = torch.zeros((1, 16), dtype=torch.uint8, device=DEV)
    scales = torch.zeros((1, 16), device=DEV)
    for b, bucket in ((3, 8), (2, 6), (8, 0)):
        with pytest.raises(api.SparcmlError):
            api.quantize(x, bucket, b, 1, codes=codes, scales=scales)


@pytest.mark.parametrize("b", [2, 4, 8])
@pytest.mark.parametrize("cap", [3_001, 4_096])
def test_code_bytes_past_each_row_are_untouched(b, cap):
    """The encode pass stores a 32-bit word of codes only when all four bytes
    hold entries: bytes past ceil(nnz / (8/b)) keep what the caller put there,
    on 4-byte aligned rows (cap = 4,096) and unaligned ones (cap = 3,001), for
    rows ending at every offset within a word."""
    P, N = 9, 400_000
    idx, val, nnz = W.uniform_streams(P, N, cap, 62, std=1e-3, cap=cap)
    per = 8 // b
    nnz[:] = [cap, 0, 1, per, per + 1, 2 * per + 1, 3 * per + 2, cap - per, cap - 1]
    seed = W.quant_seed(5)
    oc, osc = oracle.quantize(val, 512, b, seed, idx=idx, nnz=nnz)
    di, dv, dn = streams_to_dev(idx, val, nnz)
    stride = (cap + per - 1) // per
    codes = torch.full((P, stride), 0xA5, dtype=torch.uint8, device=DEV)
    codes, scales = api.quantize(dv, 512, b, seed, idx=di, nnz=dn, codes=codes)
    gc = codes.cpu().numpy()
    for p in range(P):
        n = int(nnz[p])
        nb = (n + per - 1) // per
        if n % per:  # the last byte's unused codes are zero
            assert np.array_equal(gc[p, :nb - 1], oc[p, :nb - 1])
            mask = (1 << (b * (n % per))) - 1
            assert gc[p, nb - 1] == (oc[p, nb - 1] & mask)
        else:
            assert np.array_equal(gc[p, :nb], oc[p, :nb])
        assert (gc[p, nb:] == 0xA5).all(), p
