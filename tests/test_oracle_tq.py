"""Pins of the oracle's TurboQuant Q_mse codebook variant (TQ4): the
Lloyd-Max codebook against closed forms, independent quadrature, the Gaussian
limit and the distortion figures the TurboQuant page prints; the quantiser
against brute-force nearest-centroid search; the stored norm against the
vector norm; the decode against exact attention within the codebook's error."""
import json
import math
import os

import numpy as np
import pytest
from scipy import integrate, stats

import oracle
from oracle import tq

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "tq_facts.json")))


@pytest.mark.parametrize("d", [64, 128, 256])
def test_one_bit_centroid_is_mean_absolute_coordinate(d):
    # 1 bit: boundary 0, centroids +-E|X| = +-Gamma(d/2) / (sqrt(pi) Gamma((d+1)/2))
    want = math.exp(math.lgamma(d / 2) - math.lgamma((d + 1) / 2)) / math.sqrt(math.pi)
    c = tq.lloyd_max(d, 1)
    assert c[1] == pytest.approx(want, rel=1e-12) and c[0] == -c[1]


def test_pdf_is_the_printed_density():
    # the pdf integrates to 1 and matches the Beta(1/2, (d-1)/2) law of X^2
    for d in (64, 128):
        total, _ = integrate.quad(lambda x: float(tq.pdf(x, d)), -1, 1, limit=200)
        assert total == pytest.approx(1.0, abs=1e-10)
        for a in (0.05, 0.1, 0.2):
            p, _ = integrate.quad(lambda x: float(tq.pdf(x, d)), -a, a, limit=200)
            assert p == pytest.approx(stats.beta(0.5, (d - 1) / 2).cdf(a * a), rel=1e-9)


@pytest.mark.parametrize("d,bits", [(128, 2), (128, 4), (256, 3), (64, 4)])
def test_centroids_are_cell_conditional_means_by_quadrature(d, bits):
    c = tq.lloyd_max(d, bits)
    edges = np.concatenate(([-1.0], 0.5 * (c[:-1] + c[1:]), [1.0]))
    for i in range(len(c)):
        m0, _ = integrate.quad(lambda x: float(tq.pdf(x, d)), edges[i], edges[i + 1], limit=200, epsabs=0, epsrel=1e-13)
        m1, _ = integrate.quad(lambda x: x * float(tq.pdf(x, d)), edges[i], edges[i + 1], limit=200, epsabs=0, epsrel=1e-13)
        assert c[i] == pytest.approx(m1 / m0, rel=1e-9, abs=1e-15)
    assert np.all(np.diff(c) > 0) and np.array_equal(c, -c[::-1])


def _gaussian_lloyd_max(bits):
    """Lloyd-Max centroids of N(0, 1) (Max 1960), by its own iteration on the
    normal law."""
    L = 1 << bits
    c = np.linspace(-2.5, 2.5, L)
    n = stats.norm
    for _ in range(20000):
        e = np.concatenate(([-np.inf], 0.5 * (c[:-1] + c[1:]), [np.inf]))
        new = (n.pdf(e[:-1]) - n.pdf(e[1:])) / (n.cdf(e[1:]) - n.cdf(e[:-1]))
        if np.max(np.abs(new - c)) < 1e-13:
            c = new
            break
        c = new
    return c


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_large_dimension_reduces_to_gaussian_lloyd_max(bits):
    # f tends to N(0, 1/d) as d grows (the page's measure concentration remark)
    d = 4096
    got = tq.lloyd_max(d, bits) * math.sqrt(d)
    want = _gaussian_lloyd_max(bits)
    np.testing.assert_allclose(got, want, rtol=2e-3, atol=2e-4)


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_distortion_matches_printed_table_and_bounds(bits):
    d_large = 4096
    D = tq.distortion(tq.lloyd_max(d_large, bits), d_large)
    printed = GOLD["mse_distortion_by_bits"]["value"][str(bits)]
    half_digit = GOLD["mse_distortion_by_bits"]["printed_digits"][str(bits)]
    assert abs(D - printed) <= half_digit
    for d in (64, 128, 256):
        D = tq.distortion(tq.lloyd_max(d, bits), d)
        assert 1.0 / 4 ** bits <= D <= math.sqrt(3) * math.pi / 2 / 4 ** bits


def test_codebook_tables():
    for d in (64, 128, 256):
        mags, tau = oracle.tq_codebook(d)
        c = tq.lloyd_max(d, 4)
        assert np.all(np.diff(mags) > 0) and mags[0] > 0
        assert np.array_equal(mags, np.float16(c[8:]).astype(np.float64))
        assert tau.dtype == np.float32 and tau[7] == 0.0 and np.array_equal(tau, -tau[::-1])
        assert np.all(tau[8:] > mags[:-1]) and np.all(tau[8:] < mags[1:])


def _rows(n, d, seed):
    g = np.random.default_rng(seed)
    x = g.standard_normal((n, d)).astype(np.float32)
    x[:, [3, 77 % d]] *= 20.0
    return x


@pytest.mark.parametrize("d", [64, 128])
def test_codes_are_nearest_centroid(d):
    # brute force over all 16 signed centroids (a different formulation from the
    # oracle's sign + magnitude rank): index of the nearest one, mapped to the
    # sign-magnitude nibble; the norm by numpy's own fp64 routine
    x = _rows(400, d, 11)
    codes, norms = oracle.tq_quantize_rows(x)
    c = tq.lloyd_max(d, 4)                                               # ascending, 16 levels
    y = oracle.rotate_fp32(x).astype(np.float64)
    n = np.linalg.norm(y, axis=1)
    np.testing.assert_allclose(norms, n.astype(np.float32), rtol=1e-7, atol=0)
    u = y / n[:, None]
    nearest = np.argmin(np.abs(u[..., None] - c), axis=-1)               # index 0..15
    want = np.where(nearest >= 8, nearest - 8, 8 | (7 - nearest))
    got = np.stack([codes & 15, codes >> 4], -1).reshape(codes.shape[0], d)
    assert np.array_equal(got, want)


def test_norm_is_the_vector_norm():
    # the rotation is orthogonal: the stored norm of R x is |x| up to fp32 rotation error
    x = _rows(200, 128, 12)
    _, norms = oracle.tq_quantize_rows(x)
    np.testing.assert_allclose(norms, np.linalg.norm(x.astype(np.float64), axis=1), rtol=2e-6)


def test_code_rule_by_hand():
    cpos = np.array([0.1, 0.2, 0.3, 0.4, 0.5, 0.6, 0.7, 0.8], np.float64)
    assert oracle.tq_code(0.0, cpos) == 0 and oracle.tq_code(-0.0, cpos) == 0
    assert oracle.tq_code(0.14, cpos) == 0 and oracle.tq_code(0.16, cpos) == 1
    assert oracle.tq_code(-0.16, cpos) == 8 | 1 and oracle.tq_code(-0.04, cpos) == 8
    assert oracle.tq_code(0.95, cpos) == 7 and oracle.tq_code(-1.0, cpos) == 15
    assert oracle.tq_code(0.349, cpos) == 2 and oracle.tq_code(0.351, cpos) == 3
    mags = np.arange(1, 9, dtype=np.float64)
    assert [oracle.tq_value(k, mags) for k in (0, 7, 8, 15)] == [1.0, 8.0, -1.0, -8.0]


def test_zero_row_stores_zero_norm_and_zero_codes():
    x = np.zeros((1, 128), np.float32)
    codes, norms = oracle.tq_quantize_rows(x)
    assert norms[0] == 0.0 and not codes.any()


def test_non_finite_row_gets_nan_norm_and_zero_codes():
    x = _rows(2, 128, 13)
    x[1, 5] = np.inf
    codes, norms = oracle.tq_quantize_rows(x)
    assert np.isnan(norms[1]) and not codes[1].any() and np.isfinite(norms[0])


def test_dequantised_mse_matches_codebook_distortion():
    x = np.random.default_rng(14).standard_normal((3000, 128)).astype(np.float32)
    codes, norms = oracle.tq_quantize_rows(x)
    mags = oracle.tq_centroids(128)
    sign = np.where(np.stack([codes & 8, (codes >> 4) & 8], -1).reshape(3000, 128) > 0, -1.0, 1.0)
    mag = mags[np.stack([codes & 7, (codes >> 4) & 7], -1).reshape(3000, 128)]
    y = oracle.rotate_fp32(x).astype(np.float64)
    err = np.sum((sign * mag * norms[:, None] - y) ** 2, 1) / np.sum(y * y, 1)
    assert np.mean(err) == pytest.approx(tq.distortion(tq.lloyd_max(128, 4), 128), rel=0.05)


def test_f16_rounding():
    for v in (1.0, 0.5, 65504.0, 2.0 ** -14, 2.0 ** -24, 3.0 ** -5):
        assert oracle.f16_round(v) == float(np.float16(v))
    assert oracle.f16_round(65520.0) == math.inf and oracle.f16_round(-1e-9) == 0.0
    g = np.random.default_rng(15).standard_normal(20000).astype(np.float32) * np.float32(30)
    assert all(oracle.f16_round(v) == float(np.float16(v)) for v in g[:2000])


def _bf16(x):
    b = np.ascontiguousarray(x, np.float32).view(np.uint32)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def test_decode_is_attention_on_dequantised_values():
    d, ps, Hkv, G, L = 128, 16, 2, 4, 70
    g = np.random.default_rng(16)
    k = _bf16(g.standard_normal((L, Hkv, d)))
    v = _bf16(g.standard_normal((L, Hkv, d)))
    q = _bf16(g.standard_normal((1, Hkv * G, d)))
    pages = (L + ps - 1) // ps
    bt = np.arange(pages, dtype=np.int32)[None, :][:, ::-1].copy()  # reversed page order
    slots = np.array([bt[0, j // ps] * ps + j % ps for j in range(L)], np.int64)
    cache = oracle.Cache(oracle.KIND_TQ4, pages, Hkv, ps, d)
    cache.append(k, v, slots)
    got = cache.decode(q, bt, np.array([L], np.int32))
    # exact attention on the unquantised rows, in the original basis
    f = lambda a: (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    K, V, Q = f(k), f(v), f(q)
    for h in range(Hkv * G):
        kv = h // G
        lg = K[:, kv] @ Q[0, h] / math.sqrt(d)
        p = np.exp(lg - lg.max())
        ref = p @ V[:, kv] / p.sum()
        # 4-bit codebook: relative error of a few percent of the value scale
        assert np.max(np.abs(got[0, h] - ref)) < 0.15
    # and the same dequantised values through a second, numpy-only route
    mags = cache.mags
    rows = lambda kv: [(bt[0, j // ps] * Hkv + kv) * ps + j % ps for j in range(L)]
    def deq(codes, norms, kv, is_k):
        out = np.empty((L, d))
        for j, row in enumerate(rows(kv)):
            for i in range(d):
                pos = oracle.kbyte_pos(i // 2, d) if is_k else i // 2
                code = (codes[row, pos] >> (4 * (i & 1))) & 15
                out[j, i] = oracle.tq_value(code, mags) * float(norms[row])
        return out
    qf = oracle.query_f16(q)
    for kv in range(Hkv):
        Kd, Vd = deq(cache.kc, cache.ks, kv, True), deq(cache.vc, cache.vs, kv, False)
        for h in range(kv * G, kv * G + G):
            lg = Kd @ qf[0, h] / math.sqrt(d)
            p = np.exp(lg - lg.max())
            o = oracle.inverse_rotate_f64((p @ Vd / p.sum())[None])[0]
            np.testing.assert_allclose(got[0, h], o, rtol=1e-12, atol=1e-12)
