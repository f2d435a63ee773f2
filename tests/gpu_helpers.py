"""Helpers shared by the GPU parity tests: fill a device cache through the
library's append entry point, rebuild the same sequences on the oracle side
from the same seeded inputs, and measure errors."""
import numpy as np
import torch

import oracle
import ue8m0_kv_cache_gb300 as uq
import workloads

MAX_ABS = 2e-3   # attention tolerance vs the fp64 oracle on the same dequantised K/V and E4M3 query
REL_L2 = 1e-3

KIND = {uq.FP4_UE8M0: oracle.KIND_FP4, uq.FP8_E4M3: oracle.KIND_FP8, uq.BF16: oracle.KIND_BF16,
        uq.TQ4: oracle.KIND_TQ4}


def bits(t: torch.Tensor) -> np.ndarray:
    """Host numpy copy; bf16 as uint16 bit patterns."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def new_cache(w: workloads.Workload, dtype=uq.FP4_UE8M0, fill=0xFF, k_scale=1.0, v_scale=1.0, fp4_c=0.0):
    return uq.KVCache(dtype, w.num_pages, w.Hkv, w.ps, w.D, k_scale=k_scale, v_scale=v_scale,
                      fill=fill if dtype != uq.BF16 else 0x7FC0, fp4_c=fp4_c)


def fill_cache(w, caches, block=8192, upto=None):
    """Append every sequence's tokens (in blocks) into each device cache."""
    dev = torch.device("cuda")
    for b in range(w.B):
        L = w.seq_lens[b] if upto is None else min(upto, w.seq_lens[b])
        start = w.shared_prefix if (b > 0 and w.shared_prefix) else 0
        for t0 in range(start, L, block):
            n = min(block, L - t0)
            k, v = w.kv(b, t0, n, device=dev)
            slots = torch.from_numpy(w.slots(b, t0, n)).to(dev)
            for c in caches:
                uq.uq_quantize_append(k, v, slots, c)
    torch.cuda.synchronize()


def oracle_for(w, seqs, dtype=uq.FP4_UE8M0, k_scale=1.0, v_scale=1.0, seed=uq.DEFAULT_SEED, c=None):
    """Oracle cache holding only sequences `seqs` (identity page layout), built
    from the same seeded K/V; returns (cache, block_table, seq_lens)."""
    lens = [w.seq_lens[b] for b in seqs]
    pages = [(L + w.ps - 1) // w.ps for L in lens]
    maxp = max(max(pages), 1)
    bt = np.zeros((len(seqs), maxp), np.int32)
    nxt = 0
    for i, p in enumerate(pages):
        bt[i, :p] = np.arange(nxt, nxt + p)
        nxt += p
    oc = oracle.Cache(KIND[dtype], max(nxt, 1), w.Hkv, w.ps, w.D, k_scale=k_scale, v_scale=v_scale, seed=seed, c=c)
    dev = torch.device("cuda")
    for i, b in enumerate(seqs):
        for t0 in range(0, lens[i], 16384):
            n = min(16384, lens[i] - t0)
            k, v = w.kv(b, t0, n, device=dev)
            j = np.arange(t0, t0 + n)
            slots = bt[i, j // w.ps].astype(np.int64) * w.ps + j % w.ps
            oc.append(bits(k), bits(v), slots)
    return oc, bt, np.array(lens, np.int32)


def oracle_from_device(cache, seed=uq.DEFAULT_SEED):
    """Oracle cache holding a copy of a device cache's bytes (same pages, same
    layout): the decode oracle then attends to exactly the values the kernel
    reads."""
    kind = KIND[cache.dtype]
    oc = oracle.Cache(kind, cache.num_pages, cache.num_kv_heads, cache.page_size, cache.head_dim,
                      k_scale=cache.struct.k_scale, v_scale=cache.struct.v_scale, seed=seed)
    host = lambda t, like: t.detach().cpu().contiguous().view(torch.uint8).numpy().view(like.dtype).reshape(like.shape)
    oc.kc, oc.vc = host(cache.k_codes, oc.kc), host(cache.v_codes, oc.vc)
    if oc.ks is not None:
        oc.ks, oc.vs = host(cache.k_scales, oc.ks), host(cache.v_scales, oc.vs)
    return oc


def errors(got: np.ndarray, ref: np.ndarray):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    max_abs = float(np.max(np.abs(got - ref))) if got.size else 0.0
    den = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(got - ref) / den) if den > 0 else float(np.linalg.norm(got - ref))
    return max_abs, rel


def assert_close(got, ref, what=""):
    ma, rl = errors(got, ref)
    assert np.all(np.isfinite(got)), what + ": non-finite output"
    assert ma <= MAX_ABS and rl <= REL_L2, "%s: max_abs %.3g rel_l2 %.3g" % (what, ma, rl)
    return ma, rl


def unquantised_attention(w, b, q_bf16):
    """fp64 attention of sequence b on the original (unquantised) K/V -- for
    the reported, ungated error of the 4-bit cache."""
    k, v = w.kv(b, 0, w.seq_lens[b], device=torch.device("cuda"))
    K = k.double().cpu().numpy()
    V = v.double().cpu().numpy()
    q = q_bf16[b].double().cpu().numpy()
    out = np.zeros((w.Hq, w.D))
    for h in range(w.Hq):
        kv = h // w.G
        s = K[:, kv] @ q[h] / np.sqrt(w.D)
        p = np.exp(s - s.max())
        out[h] = (p @ V[:, kv]) / p.sum()
    return out
