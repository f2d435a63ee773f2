"""Per-layer precision policy: the boundary layers hold BF16 caches and the
inner ones FP4; one decode step over all layers (eager or CUDA-graph replay)
gives every layer the result of its own format's single-layer path, and that
matches the oracle."""
import numpy as np
import pytest
import torch

import oracle
import ue8m0_kv_cache_gb300 as uq
import workloads
from gpu_helpers import assert_close, bits, oracle_for
from ue8m0_kv_cache_gb300.policy import LayeredKVCache, LayerPolicy, layered_workspace

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")
LENS = [300, 45, 777]


def _layers(n):
    """Per-layer workloads: the same page layout (layer 0's), each its own K/V and q."""
    return [workloads.make("gqa8k", B=3, Hkv=2, Hq=16, seq_lens=LENS, seed=200 + l, n_outlier=3,
                           outlier_channels=None, extra_tokens=16) for l in range(n)]


def _fill(lc, ws_):
    w0 = ws_[0]
    for l, w in enumerate(ws_):
        for b in range(w.B):
            k, v = w.kv(b, 0, LENS[b] - 1, device=DEV)
            lc.append(l, k, v, torch.from_numpy(w0.slots(b, 0, LENS[b] - 1)).to(DEV))


def _step_inputs(ws_):
    w0 = ws_[0]
    q = [w.q().to(DEV) for w in ws_]
    kn = [torch.stack([w.kv(b, LENS[b] - 1, 1, device=DEV)[0][0] for b in range(3)]) for w in ws_]
    vn = [torch.stack([w.kv(b, LENS[b] - 1, 1, device=DEV)[1][0] for b in range(3)]) for w in ws_]
    slots = torch.from_numpy(np.array([w0.slots(b, LENS[b] - 1, 1)[0] for b in range(3)])).to(DEV)
    bt = torch.from_numpy(w0.block_table).to(DEV)
    sl = torch.tensor(LENS, dtype=torch.int32, device=DEV)
    out = [torch.empty((3, 16, 128), dtype=torch.float32, device=DEV) for _ in ws_]
    return q, kn, vn, slots, bt, sl, out


def test_step_matches_single_layer_paths_and_oracle():
    n = 6
    pol = LayerPolicy(n, boundary=2, fp4_c=[0, 0, 0.156, 0.195, 0, 0])
    assert pol.dtypes == [uq.BF16, uq.BF16, uq.FP4_UE8M0, uq.FP4_UE8M0, uq.BF16, uq.BF16]
    ws_ = _layers(n)
    w0 = ws_[0]
    lc = LayeredKVCache(pol, w0.num_pages, 2, w0.ps, 128, fill=0)
    _fill(lc, ws_)
    q, kn, vn, slots, bt, sl, out = _step_inputs(ws_)
    wsp = layered_workspace(3, 16, 2, 128)
    lc.decode_step(q, kn, vn, slots, bt, sl, out, wsp)
    assert uq.uq_check_device_status() == 0
    for l in range(n):
        single = uq.KVCache(pol.dtype(l), w0.num_pages, 2, w0.ps, 128, fill=0, fp4_c=pol.fp4_c(l))
        for b in range(3):
            k, v = ws_[l].kv(b, 0, LENS[b], device=DEV)
            uq.uq_quantize_append(k, v, torch.from_numpy(w0.slots(b, 0, LENS[b])).to(DEV), single)
        fn = uq.uq_decode_attention_bf16 if pol.dtype(l) == uq.BF16 else uq.uq_decode_attention
        ref = fn(q[l], single, bt, sl).cpu().numpy()
        got = out[l].cpu().numpy()
        if pol.dtype(l) == uq.BF16:
            assert np.array_equal(got, ref), l
        else:
            assert np.max(np.abs(got - ref)) < 1e-5, l  # fused append + decode vs append, then decode
    # the oracle, for one layer of each format (own page layout, same values)
    for l in (1, 3):
        w = ws_[l]
        oc, obt, ol = oracle_for(w, [0, 1, 2], pol.dtype(l), c=pol.fp4_c(l) or None)
        assert_close(out[l].cpu().numpy(), oc.decode(bits(q[l].cpu()), obt, ol), "layer %d" % l)


def test_graph_replay_equals_eager():
    n = 5
    pol = LayerPolicy(n, boundary=1)
    ws_ = _layers(n)
    w0 = ws_[0]
    eager = LayeredKVCache(pol, w0.num_pages, 2, w0.ps, 128, fill=0)
    graph = LayeredKVCache(pol, w0.num_pages, 2, w0.ps, 128, fill=0)
    _fill(eager, ws_)
    _fill(graph, ws_)
    q, kn, vn, slots, bt, sl, out_e = _step_inputs(ws_)
    out_g = [torch.empty_like(o) for o in out_e]
    wsp_e, wsp_g = layered_workspace(3, 16, 2, 128), layered_workspace(3, 16, 2, 128)
    eager.decode_step(q, kn, vn, slots, bt, sl, out_e, wsp_e)
    graph.capture_step(q, kn, vn, slots, bt, sl, out_g, wsp_g)
    for o in out_g:
        o.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert uq.uq_check_device_status() == 0
    for a, b in zip(out_e, out_g):
        assert torch.equal(a, b)
    for a, b in zip(eager.layers, graph.layers):
        assert torch.equal(a.k_codes, b.k_codes) and torch.equal(a.v_codes, b.v_codes)
