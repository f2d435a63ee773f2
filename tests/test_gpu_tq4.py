"""TQ4 (the TurboQuant Q_mse codebook variant): the library's codebook table
equals the f16 / fp32 roundings of the oracle's Lloyd-Max centroids; the
CUDA append's codes and norms are a valid Q_mse quantisation of each row
(checked against the oracle's fp64 nearest-centroid codes and fp64 norm, see
check_tq4_rows); the decode matches the oracle's fp64 attention on the same
cache bytes within the decode tolerance."""
import numpy as np
import pytest
import torch

import oracle
import ue8m0_kv_cache_gb300 as uq
import workloads
from gpu_helpers import assert_close, bits, errors, fill_cache, new_cache, oracle_from_device, unquantised_attention

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


# The library decides a code by comparing y with fl32(n32 * tau32_k): n32 its fp32
# norm (relative error <= NORM_REL against the exact norm), tau32_k the fp32
# rounding of the fp64 midpoint tau_k.  That threshold is n tau_k (1 + e) with
# |e| <= NORM_REL + 2^-23, so the code equals the oracle's nearest fp64 centroid
# wherever |y/n - tau_k| > TAU_REL |tau_k| for every k; inside that band either
# of the two codes next to tau_k is a valid nearest-centroid code.
NORM_REL = 1e-6
TAU_REL = 2e-6


def _signed_index(codes):
    """Sign-magnitude nibble -> index 0..15 of the ascending 16-level codebook."""
    mag, neg = codes & 7, (codes & 8) != 0
    return np.where(neg, 7 - mag, 8 + mag)


def _nibbles(rows, d, is_k):
    """Natural-order codes [n][d] of cache rows [n][d/2] (K rows are group-interleaved)."""
    if is_k:
        rows = rows[:, [oracle.kbyte_pos(j, d) for j in range(d // 2)]]
    return np.stack([rows & 15, rows >> 4], -1).reshape(rows.shape[0], d)


def check_tq4_rows(x, gpu_codes, gpu_norms, is_k):
    """x: [n][d] fp32 input rows; gpu_codes [n][d/2] cache order; gpu_norms [n]."""
    d = x.shape[1]
    want_codes, want_norms = oracle.tq_quantize_rows(x)
    nonfin = ~np.isfinite(want_norms)
    assert np.array_equal(np.isnan(gpu_norms), nonfin), "non-finite rows differ"
    pos = ~nonfin & (want_norms > 0)
    rel = np.abs(gpu_norms[pos].astype(np.float64) - want_norms[pos]) / want_norms[pos]
    assert rel.size == 0 or rel.max() <= NORM_REL, "norm rel err %.3g" % rel.max()
    assert not gpu_codes[nonfin].any(), "non-finite rows must store zero codes"
    g = _signed_index(_nibbles(gpu_codes[pos], d, is_k))
    wnt = _signed_index(np.stack([want_codes[pos] & 15, want_codes[pos] >> 4], -1).reshape(-1, d))
    y = oracle.rotate_fp32(x[pos]).astype(np.float64)
    u = y / np.linalg.norm(y, axis=1, keepdims=True)
    c = oracle.tq_centroids(d)
    cent = np.concatenate((-c[::-1], c))
    tau = 0.5 * (cent[:-1] + cent[1:])                                   # 15 fp64 midpoints
    k = np.argmin(np.abs(u[..., None] - tau), axis=-1)                   # nearest threshold
    near = np.abs(u - tau[k]) <= TAU_REL * np.abs(tau[k])
    assert np.array_equal(g[~near], wnt[~near]), "%d codes differ away from a threshold" % \
        int(np.sum(g[~near] != wnt[~near]))
    ok = (g[near] == k[near]) | (g[near] == k[near] + 1)
    assert np.all(ok), "a code next to a threshold is neither neighbour"
    return int(np.sum(g != wnt)), int(near.sum())


def _compare(w, cache, b, toks):
    slots = w.slots(b, 0, max(toks) + 1)[toks]
    pages, offs = slots // w.ps, slots % w.ps
    k, v = w.kv(b, 0, max(toks) + 1, device=DEV)
    f32 = lambda t: t[toks].float().cpu().numpy().reshape(-1, w.D)
    for name, x, gc, gn, is_k in (("K", f32(k), cache.k_codes, cache.k_scales, True),
                                  ("V", f32(v), cache.v_codes, cache.v_scales, False)):
        codes = gc.cpu().numpy()[pages, :, offs].reshape(-1, w.D // 2)
        norms = gn.cpu().numpy().view(np.float32)[pages, :, offs].reshape(-1)
        check_tq4_rows(x, codes, norms, is_k)


@pytest.mark.parametrize("name", ["tiny", "gqa8k"])
def test_append_valid_quantisation(name):
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
    skipped slot: the NaN row stores a NaN norm and zero codes, the skipped
    slot keeps its fill bytes, every other row is a valid quantisation."""
    w = workloads.make("gqa8k", B=1, Hkv=2, Hq=2, seq_lens=[40], seed=10)
    cache = new_cache(w, uq.TQ4, fill=0)
    k, v = w.kv(0, 0, 40, device=DEV)
    k[3, 1, 7] = float("nan")
    slots = torch.from_numpy(w.slots(0, 0, 40)).to(DEV)
    slots[5] = -1
    uq.uq_quantize_append(k, v, slots, cache)
    assert uq.uq_check_device_status() == 0
    sl = slots.cpu().numpy()
    live = np.flatnonzero(sl >= 0)
    pages, offs = sl[live] // w.ps, sl[live] % w.ps
    for x, gc, gn, is_k in ((k, cache.k_codes, cache.k_scales, True), (v, cache.v_codes, cache.v_scales, False)):
        codes = gc.cpu().numpy()[pages, :, offs].reshape(-1, w.D // 2)
        norms = gn.cpu().numpy().view(np.float32)[pages, :, offs].reshape(-1)
        check_tq4_rows(x[live].float().cpu().numpy().reshape(-1, w.D), codes, norms, is_k)
    s3 = int(sl[3])
    assert np.isnan(cache.k_scales.cpu().numpy().view(np.float32)[s3 // w.ps, 1, s3 % w.ps])
    s5 = int(w.slots(0, 5, 1)[0])
    assert not cache.k_codes.cpu().numpy()[s5 // w.ps, :, s5 % w.ps].any()


def _run(w, cache, q, lens=None):
    bt = torch.from_numpy(w.block_table).to(DEV)
    sl = torch.tensor(w.seq_lens if lens is None else lens, dtype=torch.int32, device=DEV)
    out = uq.uq_decode_attention_tq4(q.to(DEV), cache, bt, sl)
    assert uq.uq_check_device_status() == 0
    return out.cpu().numpy()


def _ref(w, cache, seqs, q, table="library"):
    """The oracle's fp64 decode of sequences `seqs` on the device cache's own
    bytes (the attention parity is on the same dequantised values), with the
    library's f16 table (its stored codebook, checked against the oracle's
    centroids in test_codebook_matches_oracle) or the oracle's fp64 centroids."""
    oc = oracle_from_device(cache)
    tab = uq.uq_tq_codebook(w.D, 4)[0].astype(np.float64) if table == "library" else None
    sl = np.array([w.seq_lens[b] for b in seqs], np.int32)
    return oc.decode(bits(q[seqs]), w.block_table[seqs], sl, tq_table=tab)


@pytest.mark.parametrize("name", ["tiny", "gqa8k"])
def test_decode_full_workload(name):
    w = workloads.make(name)
    cache = new_cache(w, uq.TQ4)
    fill_cache(w, [cache])
    q = w.q()
    got = _run(w, cache, q)
    seqs = list(range(min(w.B, 4)))
    ma, rl = assert_close(got[seqs], _ref(w, cache, seqs, q), name)
    fa, fr = errors(got[seqs], _ref(w, cache, seqs, q, table="fp64"))
    ua, ur = errors(got[0], unquantised_attention(w, 0, q))
    print("\nTQ4 %s: vs oracle max_abs %.2e rel_l2 %.2e | vs fp64-centroid table (not gated) max_abs %.2e "
          "rel_l2 %.2e | vs unquantised (not gated) max_abs %.3f rel_l2 %.3f" % (name, ma, rl, fa, fr, ua, ur))


@pytest.mark.parametrize("G,d,ps", [(1, 128, 16), (4, 64, 32), (8, 128, 128), (16, 64, 16)])
def test_decode_shapes(G, d, ps):
    w = workloads.make("gqa8k", B=3, Hkv=2, Hq=2 * G, D=d, ps=ps, seq_lens=[200, 33, 517], seed=40 + G,
                       n_outlier=3, outlier_channels=None)
    cache = new_cache(w, uq.TQ4)
    fill_cache(w, [cache])
    q = w.q()
    assert_close(_run(w, cache, q), _ref(w, cache, [0, 1, 2], q), "G=%d d=%d ps=%d" % (G, d, ps))


def test_decode_empty_short_and_garbage_slots():
    w = workloads.make("gqa8k", B=4, Hkv=2, Hq=16, seq_lens=[0, 1, 17, 250], seed=41, n_outlier=3,
                       outlier_channels=None)
    cache = new_cache(w, uq.TQ4, fill=0xFF)  # unwritten slots: NaN norms
    fill_cache(w, [cache])
    q = w.q()
    got = _run(w, cache, q)
    assert np.all(got[0] == 0)
    assert_close(got[1:], _ref(w, cache, [1, 2, 3], q), "short")


def test_decode_large_sampled():
    w = workloads.make("mixed")
    cache = new_cache(w, uq.TQ4)
    fill_cache(w, [cache])
    q = w.q()
    got = _run(w, cache, q)
    seqs = [0, 17]
    assert_close(got[seqs], _ref(w, cache, seqs, q), "mixed sampled")


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
