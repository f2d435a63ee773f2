"""Chunked-prefill attention parity: each query token of a chunk, attending
causally to its sequence's cache, must match the oracle's fp64 decode of that
token over the keys up to its own position (the same dequantised K/V and E4M3
query), within the decode tolerance."""
import numpy as np
import pytest
import torch

import ue8m0_kv_cache_gb300 as uq
import workloads
from gpu_helpers import assert_close, bits, fill_cache, new_cache, oracle_for

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _queries(w, chunks, seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    T = sum(chunks)
    return torch.randn((T, w.Hq, w.D), generator=g, device=DEV).to(torch.bfloat16)


def _run(w, cache, q, chunks, lens=None):
    cu = torch.tensor(np.concatenate(([0], np.cumsum(chunks))), dtype=torch.int32, device=DEV)
    bt = torch.from_numpy(w.block_table).to(DEV)
    sl = torch.tensor(w.seq_lens if lens is None else lens, dtype=torch.int32, device=DEV)
    out = uq.uq_prefill_attention(q, cu, cache, bt, sl)
    assert uq.uq_check_device_status() == 0
    return out.cpu().numpy()


def _ref(w, q, chunks, seqs=None):
    """Oracle: every query token as a one-token decode over keys 0..its position."""
    qb = bits(q)
    starts = np.concatenate(([0], np.cumsum(chunks)))
    out = {}
    for b in (range(w.B) if seqs is None else seqs):
        n = chunks[b]
        if n == 0:
            continue
        oc, bt, lens = oracle_for(w, [b])
        ctx = int(lens[0]) - n
        for i in range(n):
            t = starts[b] + i
            out[t] = oc.decode(qb[t:t + 1], bt, np.array([ctx + i + 1], np.int32))[0]
    return out


def _check(got, ref, what):
    ts = sorted(ref)
    assert_close(got[ts], np.stack([ref[t] for t in ts]), what)


@pytest.mark.parametrize("G,d,ps", [(8, 128, 16), (4, 64, 32), (1, 128, 64), (16, 128, 256)])
def test_prefill_matches_oracle(G, d, ps):
    lens = [300, 80, 1000]
    chunks = [37, 80, 5]  # the second sequence's chunk is the whole sequence
    w = workloads.make("gqa8k", B=3, Hkv=2, Hq=2 * G, D=d, ps=ps, seq_lens=lens, seed=50 + G, n_outlier=3,
                       outlier_channels=None)
    cache = new_cache(w)
    fill_cache(w, [cache])
    q = _queries(w, chunks, 51)
    _check(_run(w, cache, q, chunks), _ref(w, q, chunks), "G=%d d=%d ps=%d" % (G, d, ps))


def test_long_context_few_rows_uses_key_splits():
    lens, chunks = [20000], [6]
    w = workloads.make("gqa8k", B=1, Hkv=2, Hq=16, seq_lens=lens, seed=52)
    cache = new_cache(w)
    fill_cache(w, [cache])
    q = _queries(w, chunks, 53)
    _check(_run(w, cache, q, chunks), _ref(w, q, chunks), "long")


def test_table_larger_than_sequences_and_mixed_lengths():
    """Key splits come from the longest key range present, not from the block table's
    capacity: a table with room for 20000 more tokens per sequence, one long sequence and
    short ones whose later splits are empty, and few row tiles (so many splits)."""
    lens, chunks = [9000, 70, 640, 5], [3, 2, 64, 5]
    w = workloads.make("gqa8k", B=4, Hkv=2, Hq=16, seq_lens=lens, seed=63, extra_tokens=20000, n_outlier=3,
                       outlier_channels=None)
    assert w.block_table.shape[1] * w.ps >= 29000
    cache = new_cache(w)
    fill_cache(w, [cache])
    q = _queries(w, chunks, 64)
    _check(_run(w, cache, q, chunks), _ref(w, q, chunks), "capacity")


def test_empty_chunk_and_single_token():
    lens, chunks = [50, 1, 200], [0, 1, 130]
    w = workloads.make("gqa8k", B=3, Hkv=2, Hq=16, seq_lens=lens, seed=54, n_outlier=3, outlier_channels=None)
    cache = new_cache(w, fill=0xFF)  # unwritten slots of partial pages: NaN scales, masked
    fill_cache(w, [cache])
    q = _queries(w, chunks, 55)
    _check(_run(w, cache, q, chunks), _ref(w, q, chunks), "edge")


def test_one_token_chunks_equal_decode():
    """A chunk of one token per sequence is a decode step."""
    w = workloads.make("gqa8k", B=4, Hkv=2, Hq=16, seq_lens=[777, 16, 1500, 3], seed=56)
    cache = new_cache(w)
    fill_cache(w, [cache])
    q = w.q().to(DEV)
    got = _run(w, cache, q, [1] * 4)
    bt = torch.from_numpy(w.block_table).to(DEV)
    dec = uq.uq_decode_attention(q, cache, bt, torch.tensor(w.seq_lens, dtype=torch.int32, device=DEV)).cpu().numpy()
    assert np.max(np.abs(got - dec)) < 1e-4


def test_non_finite_key_poisons_later_queries_only():
    lens, chunks = [96], [40]
    w = workloads.make("gqa8k", B=1, Hkv=1, Hq=8, seq_lens=lens, seed=57)
    cache = new_cache(w, fill=0)
    k, v = w.kv(0, 0, 96, device=DEV)
    k[70, 0, 3] = float("nan")  # token 70 of the sequence; the chunk covers positions 56..95
    uq.uq_quantize_append(k, v, torch.from_numpy(w.slots(0, 0, 96)).to(DEV), cache)
    got = _run(w, cache, _queries(w, chunks, 58), chunks)
    assert np.all(np.isfinite(got[:14])) and np.all(np.isnan(got[14:]))


def test_chunk_longer_than_sequence_is_reported():
    w = workloads.make("gqa8k", B=1, Hkv=1, Hq=8, seq_lens=[32], seed=59)
    cache = new_cache(w)
    fill_cache(w, [cache])
    q = _queries(w, [40], 60)
    cu = torch.tensor([0, 40], dtype=torch.int32, device=DEV)
    bt = torch.from_numpy(w.block_table).to(DEV)
    uq.uq_prefill_attention(q, cu, cache, bt, torch.tensor([32], dtype=torch.int32, device=DEV))
    assert uq.uq_check_device_status() == 7  # UQ_ERR_DEVICE_BOUNDS


def test_anchor_cache_is_unsupported():
    w = workloads.make("gqa8k", B=1, Hkv=1, Hq=8, seq_lens=[16], seed=61)
    c = new_cache(w, uq.FP8_E4M3)
    with pytest.raises(uq.UqError):
        _run(w, c, _queries(w, [4], 62), [4])


def test_full_size_sampled():
    """The bench's prefill: 8 sequences of 64K context, the last 128 tokens of each as the
    chunk; sampled query tokens of two sequences against the oracle."""
    B, L, n = 8, 65536, 128
    w = workloads.make("gqa8k", B=B, seq_lens=[L] * B, seed=70)
    cache = new_cache(w)
    fill_cache(w, [cache])
    q = _queries(w, [n] * B, 71)
    got = _run(w, cache, q, [n] * B)
    qb = bits(q)
    for b in (2, 7):
        oc, bt, lens = oracle_for(w, [b])
        for i in (0, 77, 127):
            t = b * n + i
            ref = oc.decode(qb[t:t + 1], bt, np.array([L - n + i + 1], np.int32))[0]
            assert_close(got[t][None], ref[None], "seq %d token %d" % (b, i))
