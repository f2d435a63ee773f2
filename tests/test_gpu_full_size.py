"""Whole-tensor parity at the full sizes of the three large workloads, in the
launch configurations the benchmark uses.

  * decode: every output row of the mixed-length batch (64 sequences up to
    64K), of the shared-prefix batch (4 x 131072, 98304 shared) and of the 64K
    batch after the benchmark's fused append + decode step, against the
    oracle's fp64 attention on the same cache bytes;
  * append: every cache byte of the 64K batch (8 x 65537 tokens: the setup
    appends, the one-call prefill-append of 32768 tokens per sequence and the
    fused step's new token) and of eight whole sequences of the mixed batch,
    against the oracle's own quantisation.

The oracle runs on the host cores, threaded over sequences and token ranges."""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
import ue8m0_kv_cache_gb300 as uq
import workloads
from gpu_helpers import assert_close, bits, fill_cache, new_cache, oracle_from_device

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")
THREADS = max(1, os.cpu_count() or 1)


def _oracle_decode(oc, q_bits, bt, lens):
    """fp64 decode of every sequence, one sequence per task."""
    out = np.empty(q_bits.shape, np.float64)

    def one(b):
        out[b:b + 1] = oc.decode(q_bits[b:b + 1], bt[b:b + 1], lens[b:b + 1])

    with ThreadPoolExecutor(THREADS) as ex:
        list(ex.map(one, range(len(lens))))
    return out


def _oracle_append(oc, jobs):
    """jobs: (k, v, slots) host arrays; appended concurrently (disjoint slots)."""
    with ThreadPoolExecutor(THREADS) as ex:
        list(ex.map(lambda j: oc.append(*j), jobs))


def _kv_jobs(w, seqs, block=4096):
    for b in seqs:
        start = w.shared_prefix if (b > 0 and w.shared_prefix) else 0
        for t0 in range(start, w.seq_lens[b], block):
            n = min(block, w.seq_lens[b] - t0)
            k, v = w.kv(b, t0, n, device=DEV)
            yield bits(k), bits(v), w.slots(b, t0, n)


def _fresh_oracle(w, fill=0xFF):
    oc = oracle.Cache(oracle.KIND_FP4, w.num_pages, w.Hkv, w.ps, w.D)
    for a in (oc.kc, oc.ks, oc.vc, oc.vs):
        a[...] = fill
    return oc


def _cache_equal(cache, oc, rows=None):
    for name, g, r in (("k_codes", cache.k_codes, oc.kc), ("k_scales", cache.k_scales, oc.ks),
                       ("v_codes", cache.v_codes, oc.vc), ("v_scales", cache.v_scales, oc.vs)):
        gh = g.cpu().numpy().reshape(r.shape)
        if rows is not None:
            gh, r = gh[rows], r[rows]
        bad = np.argwhere(gh != r)
        assert bad.size == 0, "%s: %d differing bytes, first at %s" % (name, len(bad), bad[:3].tolist())


def _rows_of_seqs(w, seqs):
    rows = []
    for b in seqs:
        sl = w.slots(b, 0, w.seq_lens[b])
        rows.append(((sl // w.ps)[:, None] * w.Hkv + np.arange(w.Hkv)[None]) * w.ps + (sl % w.ps)[:, None])
    return np.concatenate([r.reshape(-1) for r in rows])


def _decode_every_row(w, cache, q):
    bt = torch.from_numpy(w.block_table).to(DEV)
    sl = torch.tensor(w.seq_lens, dtype=torch.int32, device=DEV)
    wsp = uq.workspace(w.B, w.Hq, w.Hkv, w.D, DEV)  # the benchmark's workspace (full split-K grid)
    got = uq.uq_decode_attention(q.to(DEV), cache, bt, sl, workspace=wsp).cpu().numpy()
    assert uq.uq_check_device_status() == 0
    ref = _oracle_decode(oracle_from_device(cache), bits(q), w.block_table, np.array(w.seq_lens, np.int32))
    return got, ref


def test_mixed_every_row_and_eight_whole_sequences_appended():
    w = workloads.make("mixed")
    cache = new_cache(w)
    fill_cache(w, [cache])
    q = w.q()
    got, ref = _decode_every_row(w, cache, q)
    ma, rl = assert_close(got, ref, "mixed, all %d rows" % (w.B * w.Hq))
    print("\nmixed decode, every row: max_abs %.2e rel_l2 %.2e" % (ma, rl))
    seqs = sorted(np.random.default_rng(3).choice(w.B, 8, replace=False).tolist())
    oc = _fresh_oracle(w)
    _oracle_append(oc, list(_kv_jobs(w, seqs)))
    _cache_equal(cache, oc, _rows_of_seqs(w, seqs))


def test_prefix128k_every_row_and_every_byte():
    w = workloads.make("prefix128k")
    cache = new_cache(w)
    fill_cache(w, [cache])
    q = w.q()
    got, ref = _decode_every_row(w, cache, q)
    ma, rl = assert_close(got, ref, "prefix128k, all rows")
    print("\nprefix128k decode, every row: max_abs %.2e rel_l2 %.2e" % (ma, rl))
    oc = _fresh_oracle(w)
    _oracle_append(oc, list(_kv_jobs(w, range(w.B))))
    _cache_equal(cache, oc)


def test_append64k_benchmark_step_every_row_and_every_byte():
    """The benchmark's workload and calls: 32768 tokens per sequence appended in
    8192-token calls, then 32768 more per sequence in one call for all eight
    sequences, then one fused append + decode step at context 65537 with the
    benchmark's workspace."""
    B, CTX0, APPEND = 8, 32768, 32768
    L0 = CTX0 + APPEND
    w = workloads.make("append64k", seq_lens=[L0] * B, extra_tokens=16, seed=1005)
    cache = new_cache(w)
    for b in range(B):
        for t0 in range(0, CTX0, 8192):
            k, v = w.kv(b, t0, 8192, device=DEV)
            uq.uq_quantize_append(k, v, torch.from_numpy(w.slots(b, t0, 8192)).to(DEV), cache)
    kv = [w.kv(b, CTX0, APPEND, device=DEV) for b in range(B)]
    kA = torch.cat([a for a, _ in kv])
    vA = torch.cat([b_ for _, b_ in kv])
    sA = torch.from_numpy(np.concatenate([w.slots(b, CTX0, APPEND) for b in range(B)])).to(DEV)
    uq.uq_quantize_append(kA, vA, sA, cache)
    del kv, kA, vA
    new = [w.kv(b, L0, 1, device=DEV) for b in range(B)]
    k_new = torch.stack([a[0] for a, _ in new]).contiguous()        # [B][Hkv][D]
    v_new = torch.stack([b_[0] for _, b_ in new]).contiguous()
    s_new = torch.tensor([int(w.slots(b, L0, 1)[0]) for b in range(B)], dtype=torch.int64, device=DEV)
    lens = torch.full((B,), L0 + 1, dtype=torch.int32, device=DEV)
    q = w.q(1)
    bt = torch.from_numpy(w.block_table).to(DEV)
    wsp = uq.workspace(B, w.Hq, w.Hkv, w.D, DEV)
    got = uq.uq_decode_attention_append(q.to(DEV), k_new, v_new, s_new, cache, bt, lens, workspace=wsp)
    got = got.cpu().numpy()
    assert uq.uq_check_device_status() == 0
    w1 = workloads.make("append64k", seq_lens=[L0 + 1] * B, extra_tokens=15, seed=1005)
    assert np.array_equal(w1.block_table, w.block_table)
    oc = _fresh_oracle(w1)
    _oracle_append(oc, list(_kv_jobs(w1, range(B))))
    _cache_equal(cache, oc)
    ref = _oracle_decode(oc, bits(q), w1.block_table, np.array(w1.seq_lens, np.int32))
    ma, rl = assert_close(got, ref, "append64k step, all rows")
    print("\nappend64k fused step, every row: max_abs %.2e rel_l2 %.2e" % (ma, rl))
