"""uq_decode_attention_noalloc: the decode for callers that cannot allocate
device memory (its scratch is a static array inside the library).  Called
through the C ABI several times in a row with different inputs -- including a
call over the same sequences with other lengths, so that the split boundaries
move and the previous call's partials sit where this call's are read -- and
checked against the allocating entry point within the parity tolerance.  Kept
in a file that runs last."""
import ctypes as C

import numpy as np
import pytest
import torch

import ue8m0_kv_cache_gb300 as uq
import workloads
from gpu_helpers import MAX_ABS, REL_L2, errors, fill_cache, new_cache

pytestmark = pytest.mark.gpu


def _noalloc(q, cache, bt, sl, out):
    lib = C.CDLL(uq.LIB_PATH)
    fn = lib.uq_decode_attention_noalloc
    fn.restype = C.c_int
    fn.argtypes = [C.c_void_p, C.POINTER(uq.UqCacheStruct), C.c_void_p, C.c_int32, C.c_void_p, C.c_int32,
                   C.c_int32, C.c_float, C.c_void_p, C.c_void_p]
    return fn(q.data_ptr(), C.byref(cache.struct), bt.data_ptr(), bt.shape[1], sl.data_ptr(), q.shape[0],
              q.shape[1], 0.0, out.data_ptr(), torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_allocating_decode_on_successive_calls():
    dev = torch.device("cuda")
    w = workloads.make("gqa8k", B=6, Hkv=8, Hq=64, seq_lens=[3000, 17, 1, 4096, 250, 999], seed=77)
    cache = new_cache(w)
    fill_cache(w, [cache])
    bt = torch.from_numpy(w.block_table).to(dev)
    calls = ((([0, 1, 2, 3, 4, 5], 0), None), (([3, 0, 5], 1), None),
             (([0, 1, 2, 3, 4, 5], 2), [1500, 17, 1, 4000, 249, 64]))
    for call, ((seqs, qstep), lens) in enumerate(calls):
        q = w.q(qstep).to(dev)[seqs].contiguous()
        lens = [w.seq_lens[b] for b in seqs] if lens is None else lens
        sl = torch.tensor(lens, dtype=torch.int32, device=dev)
        btc = bt[seqs].contiguous()
        ref = uq.uq_decode_attention(q, cache, btc, sl).cpu().numpy()
        out = torch.full((len(seqs), w.Hq, w.D), float("nan"), dtype=torch.float32, device=dev)
        assert _noalloc(q, cache, btc, sl, out) == uq.UQ_OK
        assert uq.uq_check_device_status() == 0
        got = out.cpu().numpy()
        assert np.all(np.isfinite(got)), "call %d" % call
        ma, rl = errors(got, ref)
        assert ma <= MAX_ABS and rl <= REL_L2, "call %d: max_abs %.3g rel_l2 %.3g" % (call, ma, rl)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    dev = torch.device("cuda")
    cache = uq.KVCache(uq.FP4_UE8M0, 4, 8, 16, 128, device=dev)
    B = 4096  # 32768 (sequence, kv head) pairs need far more than the static scratch
    q = torch.zeros((B, 64, 128), dtype=torch.bfloat16, device=dev)
    bt = torch.zeros((B, 1), dtype=torch.int32, device=dev)
    sl = torch.zeros((B,), dtype=torch.int32, device=dev)
    out = torch.empty((B, 64, 128), dtype=torch.float32, device=dev)
    assert _noalloc(q, cache, bt, sl, out) == 4  # UQ_ERR_WORKSPACE
    big = 4097  # above the decode's batch limit: rejected before any size arithmetic
    qb = torch.zeros((big, 64, 128), dtype=torch.bfloat16, device=dev)
    btb = torch.zeros((big, 1), dtype=torch.int32, device=dev)
    slb = torch.zeros((big,), dtype=torch.int32, device=dev)
    outb = torch.empty((big, 64, 128), dtype=torch.float32, device=dev)
    assert _noalloc(qb, cache, btb, slb, outb) == 2  # UQ_ERR_UNSUPPORTED
