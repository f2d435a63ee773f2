"""Decode-attention parity: the CUDA path vs the oracle's fp64 attention on the
same dequantised K/V and the same E4M3 query, within max-abs 2e-3 and
relative L2 1e-3 -- on every output row of the two smaller workloads, on
sampled sequences of the larger ones (at full size, in the launch
configuration the benchmark uses), and on edge cases.  The error against
unquantised attention is printed, not gated."""
import numpy as np
import pytest
import torch

import ue8m0_kv_cache_gb300 as uq
import workloads
from gpu_helpers import (assert_close, bits, errors, fill_cache, new_cache, oracle_for,
                         unquantised_attention)

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")

_DECODE = {uq.FP4_UE8M0: uq.uq_decode_attention, uq.FP8_E4M3: uq.uq_decode_attention_fp8,
           uq.BF16: uq.uq_decode_attention_bf16}


def _run(w, cache, q, seq_lens=None, ws=None):
    bt = torch.from_numpy(w.block_table).to(DEV)
    sl = torch.tensor(w.seq_lens if seq_lens is None else seq_lens, dtype=torch.int32, device=DEV)
    out = _DECODE[cache.dtype](q.to(DEV), cache, bt, sl, workspace=ws)
    assert uq.uq_check_device_status() == 0
    return out.cpu().numpy()


def _ref(w, seqs, q, dtype=uq.FP4_UE8M0, k_scale=1.0, v_scale=1.0, lens=None):
    oc, bt, ol = oracle_for(w, seqs, dtype, k_scale, v_scale)
    if lens is not None:
        ol = np.array(lens, np.int32)
    return oc.decode(bits(q[seqs]), bt, ol)


@pytest.mark.parametrize("name", ["tiny", "gqa8k"])
def test_full_workload(name):
    w = workloads.make(name)
    cache = new_cache(w)
    fill_cache(w, [cache])
    q = w.q()
    got = _run(w, cache, q)
    ref = _ref(w, list(range(w.B)), q)
    ma, rl = assert_close(got, ref, name)
    ua, ur = errors(got[0], unquantised_attention(w, 0, q))
    print("\n%s: vs oracle max_abs %.2e rel_l2 %.2e | vs unquantised (not gated) max_abs %.3f rel_l2 %.3f"
          % (name, ma, rl, ua, ur))


@pytest.mark.parametrize("name", ["mixed", "prefix128k", "append64k"])
def test_large_workload_sampled(name):
    w = workloads.make(name)
    cache = new_cache(w)
    fill_cache(w, [cache])
    if name == "append64k":  # the prefill-append of 32768 more tokens per sequence
        w2 = workloads.make(name, seq_lens=[65536] * w.B, extra_tokens=16)
        assert np.array_equal(w2.block_table, w.block_table) and w2.num_pages == w.num_pages
        dev = DEV
        for b in range(w.B):
            for t0 in range(32768, 65536, 8192):
                k, v = w2.kv(b, t0, 8192, device=dev)
                uq.uq_quantize_append(k, v, torch.from_numpy(w2.slots(b, t0, 8192)).to(dev), cache)
        w = w2
    q = w.q()
    got = _run(w, cache, q)
    assert np.all(np.isfinite(got))
    rng = np.random.default_rng(13)
    seqs = sorted(rng.choice(w.B, size=2 if w.B > 2 else 1, replace=False).tolist())
    ref = _ref(w, seqs, q)
    ma, rl = assert_close(got[seqs], ref, name)
    print("\n%s seqs %s: max_abs %.2e rel_l2 %.2e" % (name, seqs, ma, rl))


@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
def test_group_sizes(G):
    w = workloads.make("gqa8k", B=3, Hkv=2, Hq=2 * G, seq_lens=[200, 33, 517], seed=20 + G, n_outlier=3,
                       outlier_channels=None)
    cache = new_cache(w)
    fill_cache(w, [cache])
    q = w.q()
    assert_close(_run(w, cache, q), _ref(w, [0, 1, 2], q), "G=%d" % G)


@pytest.mark.parametrize("d,ps", [(64, 16), (128, 32), (64, 256), (128, 128), (256, 16), (256, 64)])
def test_head_dims_and_page_sizes(d, ps):
    w = workloads.make("gqa8k", B=2, Hkv=2, Hq=16, D=d, ps=ps, seq_lens=[700, 1], seed=30, n_outlier=3,
                       outlier_channels=None)
    cache = new_cache(w)
    fill_cache(w, [cache])
    q = w.q()
    assert_close(_run(w, cache, q), _ref(w, [0, 1], q), "d=%d ps=%d" % (d, ps))


def test_empty_and_short_sequences_with_garbage_slots():
    """seq_len 0 gives zeros; ragged tails read pages whose unused slots hold
    0xFF bytes (NaN scales) without contaminating the result."""
    w = workloads.make("gqa8k", B=4, Hkv=2, Hq=16, seq_lens=[0, 1, 17, 250], seed=31, n_outlier=3,
                       outlier_channels=None)
    cache = new_cache(w, fill=0xFF)
    fill_cache(w, [cache])
    q = w.q()
    got = _run(w, cache, q)
    assert np.all(got[0] == 0)
    assert_close(got[1:], _ref(w, [1, 2, 3], q), "short")


def test_split_count_invariance():
    """A workspace that only fits a few blocks gives a different split of the
    keys; the merged result must agree within the tolerance."""
    w = workloads.make("gqa8k", B=2, Hkv=8, Hq=64, seq_lens=[3000, 5000], seed=32)
    cache = new_cache(w)
    fill_cache(w, [cache])
    q = w.q()
    full = _run(w, cache, q)
    pairs = w.B * w.Hkv
    per_slot = 8 * (w.D + 2) * 4
    small = torch.empty(((pairs * 8 + 255) // 256) * 256 + (pairs + 3) * per_slot, dtype=torch.uint8, device=DEV)
    few = _run(w, cache, q, ws=small)
    ma, rl = errors(few, full)
    assert ma < 1e-4 and rl < 1e-5
    assert_close(few, _ref(w, [0, 1], q), "3 blocks")


def test_workspace_too_small_is_rejected():
    w = workloads.make("gqa8k", B=2, Hkv=8, Hq=64, seq_lens=[64, 64], seed=33)
    cache = new_cache(w)
    with pytest.raises(uq.UqError) as e:
        _run(w, cache, w.q(), ws=torch.empty(256, dtype=torch.uint8, device=DEV))
    assert e.value.status == 4


def test_out_of_range_sequence_length_is_reported():
    w = workloads.make("gqa8k", B=1, Hkv=1, Hq=8, seq_lens=[32], seed=34, n_outlier=2, outlier_channels=None)
    cache = new_cache(w)
    fill_cache(w, [cache])
    bt = torch.from_numpy(w.block_table).to(DEV)
    sl = torch.tensor([10 ** 6], dtype=torch.int32, device=DEV)  # clamped to the table, recorded
    uq.uq_decode_attention(w.q().to(DEV), cache, bt, sl)
    assert uq.uq_check_device_status() == 7


@pytest.mark.parametrize("dtype", [uq.FP8_E4M3, uq.BF16])
@pytest.mark.parametrize("G", [4, 8])
def test_anchor_decode(dtype, G):
    w = workloads.make("gqa8k", B=3, Hkv=2, Hq=2 * G, seq_lens=[1000, 31, 2048], seed=40 + G, n_outlier=3,
                       outlier_channels=None)
    ks, vs = (0.5, 2.0) if dtype == uq.FP8_E4M3 else (1.0, 1.0)
    cache = new_cache(w, dtype, k_scale=ks, v_scale=vs) if dtype == uq.FP8_E4M3 else new_cache(w, dtype)
    fill_cache(w, [cache])
    q = w.q()
    assert_close(_run(w, cache, q), _ref(w, [0, 1, 2], q, dtype, ks, vs), "anchor %d" % dtype)


@pytest.mark.parametrize("dtype", [uq.FP8_E4M3, uq.BF16])
def test_anchor_decode_gqa8k(dtype):
    w = workloads.make("gqa8k")
    cache = new_cache(w, dtype)
    fill_cache(w, [cache])
    q = w.q()
    rng = np.random.default_rng(14)
    seqs = sorted(rng.choice(w.B, 3, replace=False).tolist())
    assert_close(_run(w, cache, q)[seqs], _ref(w, seqs, q, dtype), "anchor gqa8k")


@pytest.mark.parametrize("dtype", [uq.FP4_UE8M0, uq.FP8_E4M3, uq.BF16])
def test_head_dim_256(dtype):
    w = workloads.make("gqa8k", B=3, Hkv=2, Hq=16, D=256, ps=16, seq_lens=[900, 33, 2000], seed=44, n_outlier=4,
                       outlier_channels=None)
    cache = new_cache(w, dtype)
    fill_cache(w, [cache])
    q = w.q()
    assert_close(_run(w, cache, q), _ref(w, [0, 1, 2], q, dtype), "d=256 kind %d" % dtype)


def test_head_dim_256_unbuilt_paths_are_unsupported():
    """At D = 256 the fused append, chunked prefill, cascade, TQ4 and c calibration are not built."""
    w = workloads.make("gqa8k", B=1, Hkv=1, Hq=8, D=256, ps=16, seq_lens=[64], seed=45)
    cache = new_cache(w)
    fill_cache(w, [cache])
    bt = torch.from_numpy(w.block_table).to(DEV)
    sl = torch.tensor([64], dtype=torch.int32, device=DEV)
    q = w.q().to(DEV)
    k, v = w.kv(0, 63, 1, device=DEV)
    slots = torch.from_numpy(w.slots(0, 63, 1)).to(DEV)
    calls = [
        lambda: uq.uq_decode_attention_append(q, k, v, slots, cache, bt, sl),
        lambda: uq.uq_prefill_attention(q, torch.tensor([0, 1], dtype=torch.int32, device=DEV), cache, bt, sl),
        lambda: uq.uq_cascade_decode_attention(q, cache, bt, sl, torch.tensor([0, 1], dtype=torch.int32, device=DEV),
                                               torch.tensor([32], dtype=torch.int32, device=DEV), 32, min_rows=0),
        lambda: uq.uq_calibrate_c(torch.zeros((4, 256), device=DEV), [0.156]),
        lambda: uq.uq_quantize_append(k, v, slots, new_cache(w, uq.TQ4)),
    ]
    for f in calls:
        with pytest.raises(uq.UqError) as e:
            f()
        assert e.value.status == 2  # UQ_ERR_UNSUPPORTED
