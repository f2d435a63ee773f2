"""Pins of the oracle's FP4 append with a constant c of its own (the pages keep
one global c = 0.156 and name per-layer constants as an open option; the c
sweep objective picks one).  The new path must reduce to the pinned pieces:
the default constant, the quantiser stage on rotated rows (pinned in
test_oracle_quant.py, including its c sweep), and the exact power-of-two
behaviour of the scale byte under a doubled c."""
import numpy as np
import pytest

import oracle


def _rows(n=64, hkv=2, d=128, seed=3):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, hkv, d)).astype(np.float32)
    x[:, :, 5] *= 20.0  # an outlier channel, as in the workloads
    return x


def _append(x, c):
    n, hkv, d = x.shape
    oc = oracle.Cache(oracle.KIND_FP4, n, hkv, 1, d, c=c)
    oc.append(x, x * 0.5, np.arange(n))
    return oc


def test_explicit_default_constant_is_the_default():
    x = _rows()
    a, b = _append(x, None), _append(x, 0.156)
    for u, v in ((a.kc, b.kc), (a.ks, b.ks), (a.vc, b.vc), (a.vs, b.vs)):
        assert np.array_equal(u, v)


@pytest.mark.parametrize("c", [0.1, 0.195, 0.3, 1.0])
def test_own_constant_equals_quantiser_of_rotated_rows(c):
    x = _rows()
    n, hkv, d = x.shape
    oc = _append(x, c)
    codes, scales = oracle.quantize_rotated(oracle.rotate_fp32((x * 0.5).reshape(-1, d)), c=c)
    assert np.array_equal(oc.vc, codes) and np.array_equal(oc.vs, scales)
    kcodes, kscales = oracle.quantize_rotated(oracle.rotate_fp32(x.reshape(-1, d)), c=c)
    assert np.array_equal(oc.ks, kscales)
    perm = np.array([oracle.kbyte_pos(j, d) for j in range(d // 2)])
    assert np.array_equal(oc.kc[:, perm], kcodes)


def test_doubling_c_raises_every_unclamped_byte_by_one():
    x = _rows(n=256)
    a, b = _append(x, 0.156), _append(x, 0.312)
    live = (a.vs >= 1) & (a.vs <= 253)
    assert live.mean() > 0.99
    assert np.array_equal(b.vs[live].astype(int), a.vs[live].astype(int) + 1)
    live_k = (a.ks >= 1) & (a.ks <= 253)
    assert np.array_equal(b.ks[live_k].astype(int), a.ks[live_k].astype(int) + 1)
