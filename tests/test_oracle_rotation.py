"""Pins of the oracle's rotation (R1) and sign generator against facts that do
not come from the oracle itself: published splitmix64 outputs, the integer
Hadamard identity H H^T = d I, a dense fp64 matrix product, orthogonality."""
import json
import os

import numpy as np
import pytest

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_splitmix64_published_values():
    g = json.load(open(os.path.join(GOLD, "splitmix64.json")))
    got = [oracle.splitmix64(g["seed"], i) for i in range(len(g["outputs_signed"]))]
    want = [v & 0xFFFFFFFFFFFFFFFF for v in g["outputs_signed"]]
    assert got == want


def test_signs_are_bit63_of_the_stream():
    s = oracle.signs(0, 4)
    g = json.load(open(os.path.join(GOLD, "splitmix64.json")))
    # negative signed outputs have bit 63 set -> sign -1
    assert s.tolist() == [-1 if v < 0 else 1 for v in g["outputs_signed"]]


def test_signs_balanced():
    s = oracle.signs(42, 4096)
    assert abs(int(s.sum())) < 4 * np.sqrt(4096)


@pytest.mark.parametrize("d", [32, 64, 128, 256])
def test_normalisation_constant(d):
    want = {32: 0x3E3504F3, 64: 0x3E000000, 128: 0x3DB504F3, 256: 0x3D800000}[d]
    assert int(oracle.inv_sqrt_d(d).view(np.uint32)) == want


def _hadamard(d):
    i = np.arange(d)
    pc = np.vectorize(lambda v: bin(v).count("1"))(i[:, None] & i[None, :])
    return np.where(pc % 2 == 0, 1, -1).astype(np.int64)


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("seed", [0, 42])
def test_rotation_matrix_is_signed_hadamard(d, seed):
    """R(e_j) * sqrt(d) must be exactly column j of H diag(s) (integers), and
    the integer matrix must satisfy M M^T = d I."""
    c = float(oracle.inv_sqrt_d(d))
    cols = oracle.rotate_fp32(np.eye(d, dtype=np.float32), seed)  # row j = R(e_j)
    M = cols.T.astype(np.float64) / c
    assert np.all(np.abs(M) == 1.0)
    Mi = M.astype(np.int64)
    assert np.array_equal(Mi @ Mi.T, d * np.eye(d, dtype=np.int64))
    s = oracle.signs(seed, d).astype(np.int64)
    assert np.array_equal(Mi, _hadamard(d) * s[None, :])


@pytest.mark.parametrize("d", [64, 128, 256])
def test_fp32_fwht_matches_dense_fp64(d):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((64, d)).astype(np.float32)
    x[:, 5] *= 20
    y = oracle.rotate_fp32(x, 42).astype(np.float64)
    s = oracle.signs(42, d).astype(np.float64)
    ref = (x.astype(np.float64) * s) @ _hadamard(d).T.astype(np.float64) / np.sqrt(d)
    err = np.linalg.norm(y - ref, axis=1) / np.linalg.norm(ref, axis=1)
    assert err.max() < 1e-6


def test_inner_products_preserved():
    """<R q, R k> = <q, k> (orthogonal transform), up to fp32 rounding."""
    rng = np.random.default_rng(4)
    q = rng.standard_normal((100, 128)).astype(np.float32)
    k = rng.standard_normal((100, 128)).astype(np.float32)
    k[:, [3, 77]] *= 20
    rq, rk = oracle.rotate_fp32(q), oracle.rotate_fp32(k)
    lhs = np.sum(rq.astype(np.float64) * rk, axis=1)
    rhs = np.sum(q.astype(np.float64) * k, axis=1)
    scale = np.linalg.norm(q, axis=1) * np.linalg.norm(k, axis=1)
    assert np.max(np.abs(lhs - rhs) / scale) < 1e-6


def test_inverse_rotation_round_trip():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((20, 128)).astype(np.float32)
    back = oracle.inverse_rotate_f64(oracle.rotate_fp32(x).astype(np.float64))
    assert np.max(np.abs(back - x)) < 1e-5 * np.max(np.abs(x))


def test_rotation_spreads_outliers():
    """After rotation a vector with two x20 channels has no coordinate much
    larger than the typical one (the reason the rotation exists)."""
    rng = np.random.default_rng(6)
    x = rng.standard_normal((200, 128)).astype(np.float32)
    x[:, [3, 77]] *= 20
    y = oracle.rotate_fp32(x)
    ratio_before = np.abs(x).max(1) / np.sqrt((x ** 2).mean(1))
    ratio_after = np.abs(y).max(1) / np.sqrt((y ** 2).mean(1))
    assert np.median(ratio_before) > 7 and np.median(ratio_after) < 4


# ---------------------------------------------------------------- fp32 inverse rotation (decode output stage)
@pytest.mark.parametrize("d", [64, 128, 256])
def test_fp32_inverse_rotation_matches_dense_fp64(d):
    # out = s .* (H o) / sqrt(d), the transpose of R (H is symmetric), by a dense product
    rng = np.random.default_rng(7)
    o = rng.standard_normal((64, d)).astype(np.float32)
    o[:, 9] *= 30
    got = oracle.inverse_rotate_fp32(o, 42).astype(np.float64)
    s = oracle.signs(42, d).astype(np.float64)
    ref = (o.astype(np.float64) @ _hadamard(d).T.astype(np.float64)) * s / np.sqrt(d)
    err = np.linalg.norm(got - ref, axis=1) / np.linalg.norm(ref, axis=1)
    assert err.max() < 1e-6


@pytest.mark.parametrize("d", [64, 128])
def test_fp32_inverse_rotation_of_basis_vectors_is_exact(d):
    # R^T e_k = s .* (column k of H) / sqrt(d): every butterfly adds zeros, so the
    # fp32 result is exactly +-fl32(1/sqrt d) with the sign s_i H[i][k]
    c = oracle.inv_sqrt_d(d)
    s = oracle.signs(42, d).astype(np.int64)
    H = _hadamard(d)
    got = oracle.inverse_rotate_fp32(np.eye(d, dtype=np.float32), 42)   # row k = R^T e_k
    want = (H.T * s[None, :]).astype(np.float32) * c                    # row k: s_i H[i][k] c
    assert np.array_equal(got.view(np.uint32), want.astype(np.float32).view(np.uint32))


def test_fp32_inverse_undoes_forward_rotation():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((50, 128)).astype(np.float32)
    x[:, [3, 77]] *= 20
    back = oracle.inverse_rotate_fp32(oracle.rotate_fp32(x))
    assert np.max(np.abs(back - x) / np.max(np.abs(x), axis=1, keepdims=True)) < 1e-6
