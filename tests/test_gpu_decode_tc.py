"""The tensor-memory FP4 decode (tcgen05: block-scaled QK^T, P.V into tensor
memory), selected with UQ_FP4_DECODE=tc, which the library reads once per
process: the checks run in a child process.  Same parity bar as the default
decode: the oracle's fp64 decode within the decode tolerance, and the fused
append's cache bytes identical to a separate append."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import sys
import numpy as np
import torch
sys.path.insert(0, ROOT)
sys.path.insert(0, ROOT + "/tests")
import oracle
import ue8m0_kv_cache_gb300 as uq
import workloads
from gpu_helpers import assert_close, bits, fill_cache, new_cache, oracle_from_device
DEV = torch.device("cuda")

# several tiles, segment boundaries inside tiles, ragged tails, an empty sequence,
# G = 4 (heads padded to the 8-head block) and G = 16 (two head blocks)
for G, lens, seed in [(8, [3000, 17, 0, 129, 2048 + 5], 501), (4, [700, 1], 502), (16, [1500, 260], 503)]:
    w = workloads.make("gqa8k", B=len(lens), Hkv=2, Hq=2 * G, seq_lens=lens, seed=seed, n_outlier=3,
                       outlier_channels=None)
    cache = new_cache(w)
    fill_cache(w, [cache])
    q = w.q()
    got = uq.uq_decode_attention(q.to(DEV), cache, torch.from_numpy(w.block_table).to(DEV),
                                 torch.tensor(w.seq_lens, dtype=torch.int32, device=DEV)).cpu().numpy()
    assert uq.uq_check_device_status() == 0
    ref = oracle_from_device(cache).decode(bits(q), w.block_table, np.array(w.seq_lens, np.int32))
    ma, rl = assert_close(got, ref, "tc decode G=%d" % G)
    print("G=%d max_abs %.2e rel_l2 %.2e" % (G, ma, rl))

# page sizes above 16 (a tile's units then share pages) and the shared-prefix path, whose
# per-sequence part runs through this decode from unit S_g / 16
for ps, seed in [(32, 505), (128, 506)]:
    w = workloads.make("gqa8k", B=3, Hkv=2, Hq=16, ps=ps, seq_lens=[2100, 640, 33], seed=seed)
    cache = new_cache(w)
    fill_cache(w, [cache])
    q = w.q()
    got = uq.uq_decode_attention(q.to(DEV), cache, torch.from_numpy(w.block_table).to(DEV),
                                 torch.tensor(w.seq_lens, dtype=torch.int32, device=DEV)).cpu().numpy()
    assert uq.uq_check_device_status() == 0
    ref = oracle_from_device(cache).decode(bits(q), w.block_table, np.array(w.seq_lens, np.int32))
    ma, rl = assert_close(got, ref, "tc decode ps=%d" % ps)
    print("ps=%d max_abs %.2e rel_l2 %.2e" % (ps, ma, rl))
lens = [4096 + 300, 4096 + 17, 4096 + 1000, 4096 + 64]
w = workloads.make("gqa8k", B=4, Hkv=2, Hq=64, seq_lens=lens, seed=507, shared_prefix=4096)
cache = new_cache(w)
fill_cache(w, [cache])
q = w.q()
t32 = lambda x: torch.tensor(x, dtype=torch.int32, device=DEV)
got = uq.uq_cascade_decode_attention(q.to(DEV), cache, torch.from_numpy(w.block_table).to(DEV), t32(lens),
                                     t32([0, 4]), t32([4096]), 4096, min_rows=0).cpu().numpy()
assert uq.uq_check_device_status() == 0
ref = oracle_from_device(cache).decode(bits(q), w.block_table, np.array(lens, np.int32))
ma, rl = assert_close(got, ref, "tc decode under the cascade")
print("cascade max_abs %.2e rel_l2 %.2e" % (ma, rl))

# fused append: the cache bytes equal a separate append, the output the plain decode's
w = workloads.make("gqa8k", B=3, Hkv=2, Hq=16, seq_lens=[1000, 33, 257], seed=504)
ca, cb = new_cache(w), new_cache(w)
upto = [L - 1 for L in w.seq_lens]
for b in range(w.B):
    kk, vv = w.kv(b, 0, upto[b], device=DEV)
    sl_b = torch.from_numpy(w.slots(b, 0, upto[b])).to(DEV)
    for c in (ca, cb):
        uq.uq_quantize_append(kk, vv, sl_b, c)
k = torch.stack([w.kv(b, upto[b], 1, device=DEV)[0][0] for b in range(w.B)]).contiguous()
v = torch.stack([w.kv(b, upto[b], 1, device=DEV)[1][0] for b in range(w.B)]).contiguous()
slots = torch.tensor([int(w.slots(b, upto[b], 1)[0]) for b in range(w.B)], dtype=torch.int64, device=DEV)
bt = torch.from_numpy(w.block_table).to(DEV)
sl = torch.tensor(w.seq_lens, dtype=torch.int32, device=DEV)
q = w.q().to(DEV)
uq.uq_quantize_append(k, v, slots, ca)
ref = uq.uq_decode_attention(q, ca, bt, sl)
got = uq.uq_decode_attention_append(q, k, v, slots, cb, bt, sl)
assert uq.uq_check_device_status() == 0
for name in ("k_codes", "k_scales", "v_codes", "v_scales"):
    assert torch.equal(getattr(ca, name), getattr(cb, name)), name
assert torch.equal(got, ref)
print("tc fused append ok")
'''


def test_tensor_memory_decode_parity():
    env = dict(os.environ, UQ_FP4_DECODE="tc")
    r = subprocess.run([sys.executable, "-c", "ROOT = %r\n" % ROOT + CHILD], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    print(r.stdout)
