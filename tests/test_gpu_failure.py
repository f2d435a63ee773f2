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

