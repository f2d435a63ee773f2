"""The device-side failure path, exercised without a GPU fault.

uq_test_arm_decode_timeout makes one warp of one block of the next decode
launch wait, with a short budget, on a shared-memory barrier that nothing
arrives at. That bounded wait runs out and the kernel takes its timeout path:
it records UQ_ERR_DEVICE_TIMEOUT in the device status word, waits (bounded)
for the warp's own copies in flight, and the block stops. The host reads the
status; the context stays usable; the next call, with nothing armed, gives
the same bytes as a clean call (the decode's work split is static, so it is
reproducible bit for bit)."""
import pytest
import torch

import ue8m0_kv_cache_gb300 as uq
import workloads
from gpu_helpers import fill_cache, new_cache

pytestmark = pytest.mark.gpu

UQ_ERR_DEVICE_TIMEOUT = 6
BUDGET = 2_000_000  # SM clock cycles, ~1 ms


@pytest.mark.parametrize("dtype", [uq.FP4_UE8M0, uq.BF16])
def test_injected_decode_timeout_is_reported_and_the_next_call_is_clean(dtype):
    dev = torch.device("cuda")
    w = workloads.make("gqa8k", B=4, Hkv=8, Hq=64, seq_lens=[3000, 2048, 4096, 1500], seed=91)
    cache = new_cache(w, dtype=dtype)
    fill_cache(w, [cache])
    q = w.q().to(dev)
    bt = torch.from_numpy(w.block_table).to(dev)
    sl = torch.tensor(w.seq_lens, dtype=torch.int32, device=dev)
    ref = uq.uq_decode_attention(q, cache, bt, sl)
    assert uq.uq_check_device_status() == 0
    for cta in (0, 5):
        uq.uq_test_arm_decode_timeout(cta, BUDGET)
        uq.uq_decode_attention(q, cache, bt, sl)  # its output is undefined
        assert uq.uq_check_device_status() == UQ_ERR_DEVICE_TIMEOUT
        again = uq.uq_decode_attention(q, cache, bt, sl)
        assert uq.uq_check_device_status() == 0
        assert torch.equal(again, ref), "cta %d" % cta



def test_injected_timeout_in_the_fused_step_then_the_same_step_clean():
    """The bench's step (fused append + decode): after a timed-out call, running the
    same step again leaves the cache and the output exactly as one clean call does
    (the timed-out call may or may not have written each new token: same bytes)."""
    dev = torch.device("cuda")
    lens = [3000, 2048, 4096, 1500]
    w = workloads.make("gqa8k", B=4, Hkv=8, Hq=64, seq_lens=lens, seed=92)
    clean, hit = new_cache(w, fill=0), new_cache(w, fill=0)
    for b in range(w.B):
        k, v = w.kv(b, 0, lens[b] - 1, device=dev)
        sl_b = torch.from_numpy(w.slots(b, 0, lens[b] - 1)).to(dev)
        for c in (clean, hit):
            uq.uq_quantize_append(k, v, sl_b, c)
    g = torch.Generator(device=dev)
    g.manual_seed(93)
    k_new = torch.randn((w.B, w.Hkv, w.D), generator=g, device=dev).to(torch.bfloat16)
    v_new = torch.randn((w.B, w.Hkv, w.D), generator=g, device=dev).to(torch.bfloat16)
    slots = torch.tensor([int(w.block_table[b, (L - 1) // w.ps]) * w.ps + (L - 1) % w.ps for b, L in enumerate(lens)],
                         dtype=torch.int64, device=dev)
    q = w.q().to(dev)
    bt = torch.from_numpy(w.block_table).to(dev)
    sl = torch.tensor(lens, dtype=torch.int32, device=dev)
    ref = uq.uq_decode_attention_append(q, k_new, v_new, slots, clean, bt, sl)
    assert uq.uq_check_device_status() == 0
    uq.uq_test_arm_decode_timeout(0, BUDGET)
    uq.uq_decode_attention_append(q, k_new, v_new, slots, hit, bt, sl)  # its output is undefined
    assert uq.uq_check_device_status() == UQ_ERR_DEVICE_TIMEOUT
    again = uq.uq_decode_attention_append(q, k_new, v_new, slots, hit, bt, sl)
    assert uq.uq_check_device_status() == 0
    for name in ("k_codes", "k_scales", "v_codes", "v_scales"):
        assert torch.equal(getattr(clean, name), getattr(hit, name)), name
    assert torch.equal(again, ref)
