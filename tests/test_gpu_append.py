"""Quantize-append parity: the packed cache written by the CUDA path must equal
the oracle's byte for byte (codes and scale bytes), on the workloads' inputs
(full size for the two smaller ones, sampled tokens for the larger ones) and
on edge cases."""
import numpy as np
import pytest
import torch

import oracle
import ue8m0_kv_cache_gb300 as uq
import workloads
from gpu_helpers import bits, fill_cache, new_cache

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _rows_of(cache_t, w, b, toks, h=None):
    """Rows of a device cache tensor [P][Hkv][ps][X] for tokens `toks` of seq b."""
    slots = w.slots(b, 0, max(toks) + 1)[toks]
    pages, offs = slots // w.ps, slots % w.ps
    t = cache_t.cpu()
    t = t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()
    return t[pages, :, offs] if h is None else t[pages, h, offs]


def _oracle_rows(w, b, toks, dtype=uq.FP4_UE8M0, k_scale=1.0, v_scale=1.0):
    """Oracle cache rows for the given tokens of seq b (one row per token and head)."""
    k, v = w.kv(b, 0, max(toks) + 1, device=DEV)
    k, v = k[toks], v[toks]
    oc = oracle.Cache({0: 0, 1: 1, 2: 2}[dtype], len(toks), w.Hkv, 1, w.D, k_scale=k_scale, v_scale=v_scale)
    oc.append(bits(k), bits(v), np.arange(len(toks)))
    sh = (len(toks), w.Hkv, -1)
    return [None if a is None else a.reshape(sh) for a in (oc.kc, oc.ks, oc.vc, oc.vs)]


def _compare(w, cache, b, toks, dtype=uq.FP4_UE8M0):
    ref = _oracle_rows(w, b, toks, dtype, cache.struct.k_scale, cache.struct.v_scale)
    got = [cache.k_codes, cache.k_scales, cache.v_codes, cache.v_scales]
    for name, g, r in zip(["k_codes", "k_scales", "v_codes", "v_scales"], got, ref):
        if g is None:
            continue
        gr = _rows_of(g, w, b, toks)
        if gr.dtype != r.dtype:
            gr = gr.view(r.dtype)
        bad = np.argwhere(gr.reshape(r.shape) != r)
        assert bad.size == 0, "%s seq %d: %d mismatches, first %s" % (name, b, len(bad), bad[:3])


@pytest.mark.parametrize("name", ["tiny", "gqa8k"])
def test_full_workload_bit_exact(name):
    w = workloads.make(name)
    cache = new_cache(w)
    fill_cache(w, [cache])
    assert uq.uq_check_device_status() == 0
    for b in range(w.B):
        _compare(w, cache, b, np.arange(w.seq_lens[b]))


@pytest.mark.parametrize("name", ["mixed", "prefix128k", "append64k"])
def test_large_workload_sampled_bit_exact(name):
    w = workloads.make(name)
    cache = new_cache(w)
    fill_cache(w, [cache])
    assert uq.uq_check_device_status() == 0
    rng = np.random.default_rng(7)
    for b in rng.choice(w.B, size=2, replace=False):
        toks = np.unique(np.concatenate([rng.choice(w.seq_lens[b], 3000, replace=False),
                                         [0, w.seq_lens[b] - 1]]))
        _compare(w, cache, int(b), toks)


@pytest.mark.parametrize("d,ps,T", [(128, 16, 1), (128, 16, 77), (64, 32, 333), (128, 256, 1000),
                                    (64, 16, 5), (256, 16, 77), (256, 64, 333)])
def test_edge_shapes(d, ps, T):
    w = workloads.make("gqa8k", B=1, Hkv=3, Hq=3, D=d, ps=ps, seq_lens=[T], seed=9, n_outlier=2,
                       outlier_channels=None)
    cache = new_cache(w)
    fill_cache(w, [cache])
    _compare(w, cache, 0, np.arange(T))


def test_skipped_and_out_of_range_slots():
    w = workloads.make("gqa8k", B=1, Hkv=2, Hq=2, seq_lens=[64], seed=10, n_outlier=2, outlier_channels=None)
    cache = new_cache(w, fill=0xAB)
    k, v = w.kv(0, 0, 64, device=DEV)
    slots = torch.from_numpy(w.slots(0, 0, 64)).to(DEV)
    slots[5] = -1
    slots[9] = w.num_pages * w.ps + 3  # beyond the cache: skipped, recorded
    uq.uq_quantize_append(k, v, slots, cache)
    assert uq.uq_check_device_status() == 7  # UQ_ERR_DEVICE_BOUNDS
    assert uq.uq_check_device_status() == 0  # cleared
    keep = np.array([t for t in range(64) if t not in (5, 9)])
    _compare(w, cache, 0, keep)
    for t in (5, 9):
        assert np.all(_rows_of(cache.k_codes, w, 0, np.array([t])) == 0xAB)


def test_nonfinite_input_row():
    w = workloads.make("gqa8k", B=1, Hkv=1, Hq=1, seq_lens=[16], seed=11, n_outlier=1, outlier_channels=None)
    cache = new_cache(w)
    k, v = w.kv(0, 0, 16, device=DEV)
    k = k.clone()
    k[3, 0, 17] = float("nan")
    uq.uq_quantize_append(k, v, torch.from_numpy(w.slots(0, 0, 16)).to(DEV), cache)
    ks = _rows_of(cache.k_scales, w, 0, np.array([3]), h=0)
    kc = _rows_of(cache.k_codes, w, 0, np.array([3]), h=0)
    assert np.all(ks == 0xFF) and np.all(kc == 0)  # a NaN spreads to every rotated coordinate


@pytest.mark.parametrize("dtype", [uq.FP8_E4M3, uq.BF16])
@pytest.mark.parametrize("fp32_in", [False, True])
def test_anchor_append_bit_exact(dtype, fp32_in):
    w = workloads.make("gqa8k", B=2, Hkv=4, Hq=8, seq_lens=[300, 129], seed=12, kv_fp32=fp32_in)
    cache = new_cache(w, dtype, k_scale=0.5, v_scale=2.0) if dtype == uq.FP8_E4M3 else new_cache(w, dtype)
    fill_cache(w, [cache])
    for b in range(w.B):
        _compare(w, cache, b, np.arange(w.seq_lens[b]), dtype)


@pytest.mark.parametrize("fp32_in", [False, True])
def test_head_dim_256_bit_exact(fp32_in):
    """D = 256 runs a warp-per-row append (a row is too long for one thread's registers)."""
    w = workloads.make("gqa8k", B=2, Hkv=2, Hq=2, D=256, ps=16, seq_lens=[300, 17], seed=12, n_outlier=4,
                       outlier_channels=None, kv_fp32=fp32_in)
    cache = new_cache(w)
    fill_cache(w, [cache])
    assert uq.uq_check_device_status() == 0
    for b in range(2):
        _compare(w, cache, b, np.arange(w.seq_lens[b]))
