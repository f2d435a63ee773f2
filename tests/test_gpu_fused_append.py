"""Fused append + decode (one decode step in one launch): the cache bytes it
writes and the attention it returns must equal, bit for bit, the separate
uq_quantize_append + uq_decode_attention of the same step, and match the
oracle within the decode tolerance."""
import numpy as np
import pytest
import torch

import oracle
import ue8m0_kv_cache_gb300 as uq
import workloads
from gpu_helpers import assert_close, bits, fill_cache, new_cache

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _step_inputs(w, fp32, with_new, seed=21):
    """New-token rows for every sequence and their slots (-1 where with_new is False)."""
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    dt = torch.float32 if fp32 else torch.bfloat16
    k = (torch.randn((w.B, w.Hkv, w.D), generator=g, device=DEV) * 2).to(dt)
    v = torch.randn((w.B, w.Hkv, w.D), generator=g, device=DEV).to(dt)
    slots = []
    for b in range(w.B):
        pos = w.seq_lens[b] - 1
        slots.append(int(w.block_table[b, pos // w.ps]) * w.ps + pos % w.ps if with_new[b] else -1)
    return k, v, torch.tensor(slots, dtype=torch.int64, device=DEV)


def _caches(w, upto):
    """Two caches holding every sequence's first upto[b] tokens."""
    a, b_ = new_cache(w, fill=0), new_cache(w, fill=0)
    for b in range(w.B):
        if upto[b] == 0:
            continue
        k, v = w.kv(b, 0, upto[b], device=DEV)
        sl = torch.from_numpy(w.slots(b, 0, upto[b])).to(DEV)
        for c in (a, b_):
            uq.uq_quantize_append(k, v, sl, c)
    torch.cuda.synchronize()
    return a, b_


@pytest.mark.parametrize("d,ps,fp32", [(128, 16, False), (128, 32, True), (64, 16, False)])
def test_fused_equals_separate(d, ps, fp32):
    lens = [300, 17, 1, 129, 4000, 64]
    w = workloads.make("gqa8k", B=len(lens), Hkv=2, Hq=16, D=d, ps=ps, seq_lens=lens, seed=31)
    with_new = [True, True, True, False, True, True]
    upto = [L - 1 if n else L for L, n in zip(lens, with_new)]
    ca, cb = _caches(w, upto)
    k, v, slots = _step_inputs(w, fp32, with_new)
    k[0, 1, 5] = float("nan")  # a non-finite row takes the 0xFF scale byte on both paths
    bt = torch.from_numpy(w.block_table).to(DEV)
    sl = torch.tensor(lens, dtype=torch.int32, device=DEV)
    q = w.q().to(DEV)

    keep = slots >= 0
    uq.uq_quantize_append(k[keep].contiguous(), v[keep].contiguous(), slots[keep].contiguous(), ca)
    ref = uq.uq_decode_attention(q, ca, bt, sl)
    got = uq.uq_decode_attention_append(q, k, v, slots, cb, bt, sl)
    assert uq.uq_check_device_status() == 0
    for name in ("k_codes", "k_scales", "v_codes", "v_scales"):
        assert torch.equal(getattr(ca, name), getattr(cb, name)), name
    # sequence 0 head 1 holds the NaN row: its outputs are NaN on both paths
    assert torch.equal(torch.nan_to_num(got, nan=7.0), torch.nan_to_num(ref, nan=7.0))


def test_fused_matches_oracle():
    w = workloads.make("gqa8k", B=3, Hkv=2, Hq=16, seq_lens=[1000, 33, 257], seed=32)
    upto = [L - 1 for L in w.seq_lens]
    _, cb = _caches(w, upto)
    k, v, slots = _step_inputs(w, False, [True] * w.B)
    bt = torch.from_numpy(w.block_table).to(DEV)
    sl = torch.tensor(w.seq_lens, dtype=torch.int32, device=DEV)
    q = w.q().to(DEV)
    got = uq.uq_decode_attention_append(q, k, v, slots, cb, bt, sl).cpu().numpy()
    assert uq.uq_check_device_status() == 0
    oc = oracle.Cache(oracle.KIND_FP4, w.num_pages, w.Hkv, w.ps, w.D)
    for b in range(w.B):
        kk, vv = w.kv(b, 0, upto[b], device=DEV)
        oc.append(bits(kk), bits(vv), w.slots(b, 0, upto[b]))
        oc.append(bits(k[b:b + 1]), bits(v[b:b + 1]), np.array([int(slots[b])]))
    ref = oc.decode(bits(q), w.block_table, np.array(w.seq_lens, np.int32))
    assert_close(got, ref, "fused append + decode")


def test_slot_disagreeing_with_block_table_is_recorded():
    w = workloads.make("gqa8k", B=2, Hkv=2, Hq=16, seq_lens=[40, 50], seed=33)
    _, cb = _caches(w, [39, 49])
    k, v, slots = _step_inputs(w, False, [True, True])
    wrong = int(w.block_table[1, 0]) * w.ps + 3  # a slot of sequence 1, not where token 39 of sequence 0 lives
    before = cb.k_codes.clone()
    slots[0] = wrong
    bt = torch.from_numpy(w.block_table).to(DEV)
    sl = torch.tensor(w.seq_lens, dtype=torch.int32, device=DEV)
    uq.uq_decode_attention_append(w.q().to(DEV), k, v, slots, cb, bt, sl)
    assert uq.uq_check_device_status() == 7  # UQ_ERR_DEVICE_BOUNDS
    page, off = divmod(wrong, w.ps)
    assert torch.equal(cb.k_codes[page, :, off], before[page, :, off])  # nothing written there


def test_anchor_cache_is_unsupported():
    w = workloads.make("gqa8k", B=1, Hkv=1, Hq=8, seq_lens=[16], seed=34)
    c = new_cache(w, uq.FP8_E4M3)
    k, v, slots = _step_inputs(w, False, [True])
    bt = torch.from_numpy(w.block_table).to(DEV)
    sl = torch.tensor(w.seq_lens, dtype=torch.int32, device=DEV)
    with pytest.raises(uq.UqError):
        uq.uq_decode_attention_append(w.q().to(DEV), k, v, slots, c, bt, sl)
