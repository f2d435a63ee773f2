"""c calibration and caches with their own constant c.

* uq_calibrate_c: the squared error of the FP4 round trip of rotated rows for
  a list of constants equals the oracle's objective (group_mse, pinned to the
  pages' 0.156 / 0.195 optima), in both scale modes, and its minimiser on
  rotated unit vectors lands where the pages put it.
* A cache with fp4_c != 0: append bit-exact against the oracle with the same
  c, decode within the tolerance, and the fused append equal to the separate
  one."""
import numpy as np
import pytest
import torch

import oracle
import ue8m0_kv_cache_gb300 as uq
import workloads
from gpu_helpers import assert_close, bits, fill_cache, new_cache, oracle_for

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")
CS = [0.08, 0.13, 0.156, 0.18, 0.195, 0.25, 0.5, 1.0]


def _keys(n=4096, d=128, seed=5, dtype=torch.bfloat16):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    x = torch.randn((n, d), generator=g, device=DEV)
    x[:, 3] *= 20.0
    x[:, d - 51] *= 20.0
    return x.to(dtype)


@pytest.mark.parametrize("mode", [0, -1])
@pytest.mark.parametrize("d,dtype", [(128, torch.bfloat16), (64, torch.float32)])
def test_calibration_matches_oracle_objective(mode, d, dtype):
    x = _keys(d=d, dtype=dtype)
    got = uq.uq_calibrate_c(x, CS, mode=mode)
    y = oracle.rotate_fp32(x.float().cpu().numpy())
    ref = np.array([oracle.group_mse(y, c, mode if mode == 0 else oracle.ROUND_CONTINUOUS) for c in CS])
    assert np.allclose(got, ref, rtol=1e-5, atol=0), np.max(np.abs(got / ref - 1))


def test_calibration_minimiser_on_rotated_unit_vectors():
    g = torch.Generator(device=DEV)
    g.manual_seed(9)
    x = torch.randn((40000, 128), generator=g, device=DEV, dtype=torch.float64)
    x = (x / x.norm(dim=1, keepdim=True)).float()
    cs = np.arange(0.13, 0.23, 0.002)
    c_cont = cs[int(np.argmin(uq.uq_calibrate_c(x, cs[:50], mode=-1)))]
    c_pow2 = cs[int(np.argmin(uq.uq_calibrate_c(x, cs[:50], mode=0)))]
    assert 0.150 <= c_cont <= 0.172, c_cont
    assert abs(c_pow2 - 0.195) <= 0.004, c_pow2


def test_calibration_edge_cases():
    z = torch.zeros((8, 128), device=DEV)
    assert np.all(uq.uq_calibrate_c(z, [0.156]) == 0)
    x = _keys(n=33)
    x[7, 100] = float("nan")
    assert np.isnan(uq.uq_calibrate_c(x, [0.156])[0])
    with pytest.raises(uq.UqError):
        uq.uq_calibrate_c(_keys(n=4), [0.0])


@pytest.mark.parametrize("c", [0.1, 0.195, 0.3])
def test_append_with_own_constant_bit_exact(c):
    w = workloads.make("gqa8k", B=2, Hkv=2, Hq=16, seq_lens=[300, 77], seed=12, n_outlier=3, outlier_channels=None)
    cache = new_cache(w, fp4_c=c)
    fill_cache(w, [cache])
    assert uq.uq_check_device_status() == 0
    for b in range(2):
        L = w.seq_lens[b]
        k, v = w.kv(b, 0, L, device=DEV)
        oc = oracle.Cache(oracle.KIND_FP4, L, w.Hkv, 1, w.D, c=c)
        oc.append(bits(k), bits(v), np.arange(L))
        slots = w.slots(b, 0, L)
        pages, offs = slots // w.ps, slots % w.ps
        for g, r in ((cache.k_codes, oc.kc), (cache.k_scales, oc.ks), (cache.v_codes, oc.vc),
                     (cache.v_scales, oc.vs)):
            assert np.array_equal(g.cpu().numpy()[pages, :, offs].reshape(r.shape), r)


def test_decode_and_fused_append_with_own_constant():
    c = 0.195
    w = workloads.make("gqa8k", B=3, Hkv=2, Hq=16, seq_lens=[500, 33, 1200], seed=13, n_outlier=3,
                       outlier_channels=None)
    cache = new_cache(w, fp4_c=c)
    fill_cache(w, [cache], upto=None)
    bt = torch.from_numpy(w.block_table).to(DEV)
    sl = torch.tensor(w.seq_lens, dtype=torch.int32, device=DEV)
    q = w.q()
    got = uq.uq_decode_attention(q.to(DEV), cache, bt, sl).cpu().numpy()
    assert uq.uq_check_device_status() == 0
    oc, obt, ol = oracle_for(w, [0, 1, 2], c=c)
    assert_close(got, oc.decode(bits(q), obt, ol), "own c")
    # fused append of each sequence's last token == separate append, same output
    a, b = new_cache(w, fp4_c=c, fill=0), new_cache(w, fp4_c=c, fill=0)
    fill_cache(w, [a, b], upto=None)
    k_new = torch.stack([w.kv(i, w.seq_lens[i] - 1, 1, device=DEV)[0][0] for i in range(3)])
    v_new = torch.stack([w.kv(i, w.seq_lens[i] - 1, 1, device=DEV)[1][0] for i in range(3)])
    slots = torch.from_numpy(np.array([w.slots(i, w.seq_lens[i] - 1, 1)[0] for i in range(3)])).to(DEV)
    o1 = uq.uq_decode_attention_append(q.to(DEV), k_new, v_new, slots, a, bt, sl).cpu().numpy()
    uq.uq_quantize_append(k_new, v_new, slots, b)
    o2 = uq.uq_decode_attention(q.to(DEV), b, bt, sl).cpu().numpy()
    assert uq.uq_check_device_status() == 0
    assert np.array_equal(o1, o2)
    for x, y in ((a.k_codes, b.k_codes), (a.k_scales, b.k_scales), (a.v_codes, b.v_codes), (a.v_scales, b.v_scales)):
        assert torch.equal(x, y)
