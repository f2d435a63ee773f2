"""TQ4 (the TurboQuant Q_mse codebook variant): the library's codebook equals
the oracle's; the cache bytes the CUDA append writes (codes and fp32 norms)
equal the oracle's byte for byte; the decode matches the oracle's fp64
attention on the same codes within the decode tolerance."""
import numpy as np
import pytest
import torch

import oracle
import ue8m0_kv_cache_gb300 as uq
import workloads
from gpu_helpers import assert_close, bits, errors, fill_cache, new_cache, oracle_for, unquantised_attention

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("nbits", [1, 2, 3, 4])
def test_codebook_matches_oracle(d, nbits):
    mags, thr = uq.uq_tq_codebook(d, nbits)
    from oracle import tq
    c = tq.lloyd_max(d, nbits)
    h = 1 << (nbits - 1)
    assert np.array_equal(mags, np.float16(c[h:]).astype(np.float32))
    want = np.array([np.float32(0.5 * (c[j] + c[j + 1])) for j in range(2 * h - 1)], np.float32)
    assert np.array_equal(thr, want)


def _oracle_rows(w, b, toks):
    k, v = w.kv(b, 0, max(toks) + 1, device=DEV)
    k, v = k[toks], v[toks]
    oc = oracle.Cache(oracle.KIND_TQ4, len(toks), w.Hkv, 1, w.D)
    oc.append(bits(k), bits(v), np.arange(len(toks)))
    sh = (len(toks), w.Hkv, -1)
    return oc.kc.reshape(sh), oc.ks.view(np.uint8).reshape(sh), oc.vc.reshape(sh), oc.vs.view(np.uint8).reshape(sh)


def _compare(w, cache, b, toks):
    slots = w.slots(b, 0, max(toks) + 1)[toks]
    pages, offs = slots // w.ps, slots % w.ps
    ref = _oracle_rows(w, b, toks)
    for name, g, r in zip(["k_codes", "k_norms", "v_codes", "v_norms"],
                          [cache.k_codes, cache.k_scales, cache.v_codes, cache.v_scales], ref):
        gr = g.cpu().numpy()[pages, :, offs]
        bad = np.argwhere(gr.reshape(r.shape) != r)
        assert bad.size == 0, "%s seq %d: %d mismatches, first %s" % (name, b, len(bad), bad[:3])


@pytest.mark.parametrize("name", ["tiny", "gqa8k"])
def test_append_bit_exact(name):
    w = workloads.make(name)
    cache = new_cache(w, uq.TQ4)
    fill_cache(w, [cache])
    assert uq.uq_check_device_status() == 0
    for b in range(min(w.B, 4)):
        _compare(w, cache, b, np.arange(w.seq_lens[b]))


@pytest.mark.parametrize("d,ps,T", [(128, 16, 1), (128, 16, 77), (64, 32, 333), (128, 256, 1000), (64, 16, 5)])
def test_append_edge_shapes(d, ps, T):
    w = workloads.make("gqa8k", B=1, Hkv=3, Hq=3, D=d, ps=ps, seq_lens=[T], seed=9, n_outlier=2,
                       outlier_channels=None)
    cache = new_cache(w, uq.TQ4)
    fill_cache(w, [cache])
    _compare(w, cache, 0, np.arange(T))


def test_append_small_path_and_non_finite_row():
    """A decode-step sized append (the direct-load kernel) with a NaN row and a
    skipped slot: the NaN row stores a NaN norm and zero codes."""
    w = workloads.make("gqa8k", B=1, Hkv=2, Hq=2, seq_lens=[40], seed=10)
    cache = new_cache(w, uq.TQ4, fill=0)
    k, v = w.kv(0, 0, 40, device=DEV)
    k[3, 1, 7] = float("nan")
    slots = torch.from_numpy(w.slots(0, 0, 40)).to(DEV)
    slots[5] = -1
    uq.uq_quantize_append(k, v, slots, cache)
    assert uq.uq_check_device_status() == 0
    oc = oracle.Cache(oracle.KIND_TQ4, w.num_pages, w.Hkv, w.ps, w.D)
    oc.append(bits(k), bits(v), slots.cpu().numpy())
    for g, r in ((cache.k_codes, oc.kc), (cache.k_scales, oc.ks.view(np.uint8)), (cache.v_codes, oc.vc),
                 (cache.v_scales, oc.vs.view(np.uint8))):
        assert np.array_equal(g.cpu().numpy().reshape(r.shape[0], -1), r.reshape(r.shape[0], -1))
    s3 = int(w.slots(0, 3, 1)[0])
    row = (s3 // w.ps * w.Hkv + 1) * w.ps + s3 % w.ps
    assert np.isnan(oc.ks[row]) and not oc.kc[row].any()


def _run(w, cache, q, lens=None):
    bt = torch.from_numpy(w.block_table).to(DEV)
    sl = torch.tensor(w.seq_lens if lens is None else lens, dtype=torch.int32, device=DEV)
    out = uq.uq_decode_attention_tq4(q.to(DEV), cache, bt, sl)
    assert uq.uq_check_device_status() == 0
    return out.cpu().numpy()


def _ref(w, seqs, q):
    oc, bt, ol = oracle_for(w, seqs, uq.TQ4)
    return oc.decode(bits(q[seqs]), bt, ol)


@pytest.mark.parametrize("name", ["tiny", "gqa8k"])
def test_decode_full_workload(name):
    w = workloads.make(name)
    cache = new_cache(w, uq.TQ4)
    fill_cache(w, [cache])
    q = w.q()
    got = _run(w, cache, q)
    seqs = list(range(min(w.B, 4)))
    ma, rl = assert_close(got[seqs], _ref(w, seqs, q), name)
    ua, ur = errors(got[0], unquantised_attention(w, 0, q))
    print("\nTQ4 %s: vs oracle max_abs %.2e rel_l2 %.2e | vs unquantised (not gated) max_abs %.3f rel_l2 %.3f"
          % (name, ma, rl, ua, ur))


@pytest.mark.parametrize("G,d,ps", [(1, 128, 16), (4, 64, 32), (8, 128, 128), (16, 64, 16)])
def test_decode_shapes(G, d, ps):
    w = workloads.make("gqa8k", B=3, Hkv=2, Hq=2 * G, D=d, ps=ps, seq_lens=[200, 33, 517], seed=40 + G,
                       n_outlier=3, outlier_channels=None)
    cache = new_cache(w, uq.TQ4)
    fill_cache(w, [cache])
    q = w.q()
    assert_close(_run(w, cache, q), _ref(w, [0, 1, 2], q), "G=%d d=%d ps=%d" % (G, d, ps))


def test_decode_empty_short_and_garbage_slots():
    w = workloads.make("gqa8k", B=4, Hkv=2, Hq=16, seq_lens=[0, 1, 17, 250], seed=41, n_outlier=3,
                       outlier_channels=None)
    cache = new_cache(w, uq.TQ4, fill=0xFF)  # unwritten slots: NaN norms
    fill_cache(w, [cache])
    q = w.q()
    got = _run(w, cache, q)
    assert np.all(got[0] == 0)
    assert_close(got[1:], _ref(w, [1, 2, 3], q), "short")


def test_decode_large_sampled():
    w = workloads.make("mixed")
    cache = new_cache(w, uq.TQ4)
    fill_cache(w, [cache])
    q = w.q()
    got = _run(w, cache, q)
    seqs = [0, 17]
    assert_close(got[seqs], _ref(w, seqs, q), "mixed sampled")


def test_nan_row_poisons_its_heads_only():
    w = workloads.make("gqa8k", B=2, Hkv=2, Hq=4, seq_lens=[64, 64], seed=42)
    cache = new_cache(w, uq.TQ4, fill=0)
    for b in range(2):
        k, v = w.kv(b, 0, 64, device=DEV)
        if b == 0:
            v[10, 1, 3] = float("inf")
        uq.uq_quantize_append(k, v, torch.from_numpy(w.slots(b, 0, 64)).to(DEV), cache)
    got = _run(w, cache, w.q())
    assert np.all(np.isnan(got[0, 2:])) and np.all(np.isfinite(got[0, :2])) and np.all(np.isfinite(got[1]))
