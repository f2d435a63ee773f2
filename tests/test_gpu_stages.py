"""Bit-exact checks of single stages of the CUDA path against the oracle:
rotation and its inverse (the decode output stage), quantiser (scale byte + E2M1 codes), the decode prologue (rotated
E4M3 query) and the E4M3 conversion."""
import numpy as np
import pytest
import torch

import oracle
import ue8m0_kv_cache_gb300 as uq

pytestmark = pytest.mark.gpu


def _rows(n, d, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(n, d, generator=g)
    x[:, 3] *= 20
    x[:, d - 5] *= 20
    x[: n // 4] *= 1e-20
    x[n // 4: n // 2] *= 1e20
    return x.float()


@pytest.mark.parametrize("d", [64, 128, 256])
def test_rotation_bit_exact(d):
    x = _rows(4096, d, 1)
    for seed in (0, 42):
        y = uq.uq_test_rotate(x.cuda(), seed).cpu().numpy()
        ref = oracle.rotate_fp32(x.numpy(), seed)
        assert np.array_equal(y.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("d", [64, 128, 256])
def test_inverse_rotation_bit_exact(d):
    # the merge kernels' output stage (D7) against the oracle's fp32 inverse rotation
    x = _rows(4096, d, 3)
    for seed in (0, 42):
        y = uq.uq_test_rotate(x.cuda(), seed, inverse=True).cpu().numpy()
        ref = oracle.inverse_rotate_fp32(x.numpy(), seed)
        assert np.array_equal(y.view(np.uint32), ref.view(np.uint32))


def _check_quant(y):
    d = y.shape[-1]
    codes, scales = uq.uq_test_quantize_rotated(torch.from_numpy(y).cuda())
    rc, rs = oracle.quantize_rotated(y)
    sc = scales.cpu().numpy()
    assert np.array_equal(sc, rs), np.argwhere(sc != rs)[:5]
    cc = codes.cpu().numpy()
    bad = np.argwhere(cc != rc)
    assert bad.size == 0, (bad[:5], cc[tuple(bad[0])], rc[tuple(bad[0])], y.reshape(-1, d)[bad[0][0]])


@pytest.mark.parametrize("d", [64, 128, 256])
def test_quantizer_random_rows(d):
    x = _rows(8192, d, 2).numpy()
    _check_quant(oracle.rotate_fp32(x, 42))


def test_quantizer_dense_code_sweep():
    """Groups whose first element is 6 (so E = 0) carry every fp32 value in a
    dense sweep around each E2M1 decision boundary, both signs."""
    vals = []
    for p in [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]:
        b = int(np.float32(p).view(np.uint32))
        vals.append(np.arange(b - 2000, b + 2001, dtype=np.int64).astype(np.uint32).view(np.float32))
    rng = np.random.default_rng(3)
    vals.append(rng.uniform(-6, 6, 200000).astype(np.float32))
    vals.append(np.array([0.0, -0.0, 1e-30, -1e-30, 1e-45, -1e-45], np.float32))
    v = np.concatenate(vals)
    v = np.concatenate([v, -v])
    v = v[np.abs(v) <= 6.0]
    n = (v.size + 30) // 31
    v = np.concatenate([v, np.zeros(n * 31 - v.size, np.float32)]).reshape(n, 31)
    y = np.concatenate([np.full((n, 1), 6.0, np.float32), v], axis=1)
    pad = (-n) % 4
    y = np.concatenate([y, np.tile(y[:1], (pad, 1))]).reshape(-1, 128)
    _check_quant(y)


def test_quantizer_scale_byte_sweep():
    """Group maxima on both sides of every sqrt(2) crossing of 0.156*m,
    including subnormal and near-overflow magnitudes."""
    ms = []
    for k in range(-150, 128):
        m0 = np.float32(2.0 ** (k + 0.5) / 0.156)
        if not np.isfinite(m0) or m0 == 0:
            continue
        b = int(m0.view(np.uint32))
        ms.append(np.arange(max(b - 3, 1), b + 4, dtype=np.int64).astype(np.uint32).view(np.float32))
    rng = np.random.default_rng(4)
    ms.append(np.exp(rng.uniform(-100, 88, 20000)).astype(np.float32))
    ms.append(np.array([0.0, 1e-45, 3.4e38], np.float32))
    m = np.concatenate(ms)
    m = m[np.isfinite(m)]
    pad = (-m.size) % 4
    m = np.concatenate([m, np.ones(pad, np.float32)])
    y = np.zeros((m.size, 32), np.float32)
    y[:, 0] = m
    y[:, 1] = -m * np.float32(0.3)
    y[:, 2] = m * np.float32(0.77)
    _check_quant(y.reshape(-1, 128))


def test_quantizer_nonfinite_groups():
    y = np.ones((4, 128), np.float32)
    y[0, 5] = np.nan
    y[1, 40] = np.inf
    y[2, 70] = -np.inf
    y[3, :] = 0.0
    _check_quant(y)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_query_prologue_bit_exact(d):
    g = torch.Generator().manual_seed(5)
    q = torch.randn(1000, d, generator=g)
    q[:, 7] *= 30
    q = q.to(torch.bfloat16)
    got = uq.uq_test_query_fp8(q.cuda()).cpu().numpy()
    ref = oracle.query_fp8(q.contiguous().view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(got, ref)


def test_query_prologue_all_bf16_values():
    bitsv = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    x = bitsv.view(torch.bfloat16)
    x = x[torch.isfinite(x.float())]
    n = (x.numel() // 128) * 128
    q = x[:n].reshape(-1, 128).contiguous()
    got = uq.uq_test_query_fp8(q.cuda()).cpu().numpy()
    ref = oracle.query_fp8(q.view(torch.int16).numpy().view(np.uint16))
    finite = np.isfinite(oracle.rotate_fp32(q.float().numpy()))
    assert np.array_equal(got[finite], ref[finite])


def test_e4m3_conversion_exhaustive_bf16_and_random_fp32():
    x = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).float()
    rng = np.random.default_rng(6)
    x = torch.cat([x, torch.from_numpy(rng.standard_normal(1 << 20).astype(np.float32) * 50)])
    got = uq.uq_test_cvt_e4m3(x.cuda()).cpu().numpy()
    xs = x.numpy()
    ref = oracle.e4m3_codes(xs)
    nan = np.isnan(xs)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.all((got[nan] & 0x7F) == 0x7F)
