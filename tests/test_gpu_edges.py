"""GPU parity at the edges of the inputs, against the oracle bit for bit:
non-finite gradients in Top-k with error feedback (SparCML §2.2, §4: the
magnitude order of the bit patterns), non-finite stream values in the sum,
max, min and bitwise-or reductions (§5.2: each with its neutral element), and
densify (§5.1) over many thread blocks."""
import numpy as np
import pytest
import torch

import oracle
from top_gradient_compression_gb300 import api, workloads as W

from gpu_helpers import DEV, bits, check_topk_steps, streams_to_dev
from test_gpu_reduce_ops import check_op

pytestmark = pytest.mark.gpu

F32 = np.float32
NAN_A = np.uint32(0x7FC00000).view(F32)   # the default quiet NaN
NAN_B = np.uint32(0xFFC00001).view(F32)   # negative, another payload
NAN_S = np.uint32(0x7F800001).view(F32)   # a signalling pattern
SPECIALS = np.array([NAN_A, NAN_B, NAN_S, np.inf, -np.inf, 0.0, -0.0, 3.0e38, -3.0e38,
                     1.0e-45, -1.0e-45], F32)


def sprinkle(g, rng, frac):
    """Overwrite a fraction of the entries with NaNs, infinities, signed zeros,
    huge finite values and the smallest subnormals."""
    m = rng.random(g.shape) < frac
    g[m] = SPECIALS[rng.integers(0, len(SPECIALS), size=int(m.sum()))]
    return g


@pytest.mark.parametrize("P,N,seg_len,k_num,k_den,frac", [
    (3, 5_000, 5_000, 1, 100, 0.02),       # exact segment: more specials than k
    (2, 300_000, 100_000, 1, 1000, 0.0005),  # layer-sized segments (warp guess + short select)
    (2, 300_000, 100_000, 1, 1000, 0.003),   # specials outnumber k: the boundary key is NaN / inf
    (1, 1 << 21, 1 << 21, 1, 100, 0.001),  # one long segment: 4-CTA cluster select
    (2, 4_194_304, 4_194_304, 1, 100, 0.0002),  # long segment: grid-wide select passes
    (4, 65_536, 8_192, 30, 100, 0.05),     # dense selection, chunk-sized segments
])
def test_topk_non_finite_gradients(P, N, seg_len, k_num, k_den, frac):
    rng = np.random.default_rng(N + P)
    grads = []
    for _ in range(3):  # NaNs stay in the residual and meet the next step's gradient
        g = rng.standard_normal((P, N)).astype(F32)
        grads.append(sprinkle(g, rng, frac))
    check_topk_steps(grads, seg_len, k_num, k_den)


def test_topk_boundary_inside_an_infinity_group():
    """k falls inside a group of +-inf entries of one key: the lowest indices of
    the group are kept, NaNs (above inf) all kept, finite values dropped."""
    P, N = 2, 40_000
    rng = np.random.default_rng(3)
    g = rng.standard_normal((P, N)).astype(F32)
    inf_at = rng.choice(N, size=700, replace=False)
    nan_at = rng.choice(np.setdiff1d(np.arange(N), inf_at), size=150, replace=False)
    g[:, inf_at] = np.where(rng.random(700) < 0.5, np.inf, -np.inf).astype(F32)
    g[:, nan_at] = NAN_B
    res = torch.zeros((P, N), device=DEV)
    idx, val, nnz = api.topk_ef(torch.from_numpy(g).to(DEV), res, N, 1, 100)  # k = 400
    kept = np.sort(idx.cpu().numpy().view(np.uint32)[0, :400])
    want = np.sort(np.concatenate([nan_at, np.sort(inf_at)[:250]]))
    assert np.array_equal(kept, want)
    check_topk_steps([g], N, 1, 100)


def specials_streams(P, N, k, seed, frac=0.05):
    idx, val, nnz = W.uniform_streams(P, N, k, seed)
    rng = np.random.default_rng(seed)
    sprinkle(val, rng, frac)
    return idx, val, nnz


@pytest.mark.parametrize("op", ["sum", "max", "min", "or"])
@pytest.mark.parametrize("P,N,k", [
    (3, 4_194_304, 2_000),   # compact-accumulator CTA tiles
    (8, 200_000, 4_000),     # sparse-first warp tiles
    (16, 200_000, 12_000),   # dense-first warp tiles
    (80, 100_000, 2_000),    # staged CTA tiles, dense-first
    (100, 200_000, 1_000),   # staged CTA tiles, look-back + fix-up
])
def test_reduce_non_finite_values_each_regime(op, P, N, k):
    """NaNs of several payloads, +-inf (which meet the +-inf neutral elements of
    max and min), signed zeros and subnormals in the streams: a NaN produced by
    a sum is the canonical NaN; max and min never take a NaN; or works on the
    bit patterns."""
    idx, val, nnz = specials_streams(P, N, k, 900 + P)
    check_op(idx, val, nnz, N, op)


@pytest.mark.parametrize("op", ["sum", "max", "min"])
def test_reduce_all_entries_infinite(op):
    """Every value is +-inf: sums of opposite infinities give NaN, max / min of a
    lone -inf / +inf equal the neutral element yet the index is present."""
    P, N, k = 6, 50_000, 3_000
    idx, val, nnz = W.uniform_streams(P, N, k, 5)
    rng = np.random.default_rng(6)
    val[:] = np.where(rng.random(val.shape) < 0.5, np.inf, -np.inf).astype(F32)
    check_op(idx, val, nnz, N, op)


def test_densify_many_blocks():
    P, N, k = 8, 1_000_003, 150_001
    idx, val, nnz = W.uniform_streams(P, N, k, 31)
    nnz[3] = 0
    nnz[5] = 17
    di, dv, dn = streams_to_dev(idx, val, nnz)
    status = api.status_word(DEV)
    got = api.densify(di, dv, dn, N, status=status)
    assert api.get_status(status) == 0
    want = oracle.densify(idx, val, nnz, N)
    assert np.array_equal(bits(got.cpu().numpy()), bits(want))
