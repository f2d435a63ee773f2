"""Cascade (shared-prefix) decode parity: sequences grouped over a shared
prefix are attended by the shared-prefix kernel (all the group's queries at
once) plus the per-sequence decode for the rest; the result must match the
oracle's fp64 decode of every sequence over its own block table, within the
decode tolerance, and agree with the plain decode on the same cache."""
import numpy as np
import pytest
import torch

import ue8m0_kv_cache_gb300 as uq
import workloads
from gpu_helpers import assert_close, bits, fill_cache, new_cache, oracle_for

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _setup(B, G, lens, shared, d=128, ps=16, seed=80):
    w = workloads.make("gqa8k", B=B, Hkv=2, Hq=2 * G, D=d, ps=ps, seq_lens=lens, seed=seed, shared_prefix=shared,
                       n_outlier=3, outlier_channels=None)
    cache = new_cache(w)
    fill_cache(w, [cache])
    return w, cache


def _t(x):
    return torch.tensor(x, dtype=torch.int32, device=DEV)


def _cascade(w, cache, q, cu, prefix, max_prefix, min_rows=0):
    bt = torch.from_numpy(w.block_table).to(DEV)
    sl = _t(w.seq_lens)
    out = uq.uq_cascade_decode_attention(q.to(DEV), cache, bt, sl, _t(cu), _t(prefix), max_prefix,
                                         min_rows=min_rows)
    status = uq.uq_check_device_status()
    return out.cpu().numpy(), status


def _plain(w, cache, q):
    bt = torch.from_numpy(w.block_table).to(DEV)
    out = uq.uq_decode_attention(q.to(DEV), cache, bt, _t(w.seq_lens))
    assert uq.uq_check_device_status() == 0
    return out.cpu().numpy()


def _ref(w, seqs, q):
    oc, bt, ol = oracle_for(w, seqs)
    return oc.decode(bits(q[seqs]), bt, ol)


def test_groups_ragged_prefixes_and_ungrouped_sequences():
    # all six share their first 2048 tokens; group 0 = seqs 0-2 over the whole
    # prefix, group 1 = seqs 3-4 over 1995 keys (cut to 1984 for the shared
    # kernel), seq 5 in no group; seq 2 ends exactly at the prefix (no own keys)
    lens = [2048 + 300, 2048 + 17, 2048, 2048 + 1000, 2048 + 5, 2048 + 64]
    w, cache = _setup(6, 8, lens, 2048)
    q = w.q()
    got, st = _cascade(w, cache, q, [0, 3, 5], [2048, 1995], 2048)
    assert st == 0
    assert_close(got, _ref(w, list(range(6)), q), "cascade")
    assert np.max(np.abs(got - _plain(w, cache, q))) < 1e-4


def test_group_wider_than_one_row_tile():
    # 20 sequences x 8 heads = 160 query rows per kv head: two row tiles
    lens = [4096 + 37 * i for i in range(20)]
    w, cache = _setup(20, 8, lens, 4096, seed=81)
    q = w.q()
    got, st = _cascade(w, cache, q, [0, 20], [4096], 4096)
    assert st == 0
    seqs = [0, 7, 15, 16, 19]
    assert_close(got[seqs], _ref(w, seqs, q), "two row tiles")
    assert np.max(np.abs(got - _plain(w, cache, q))) < 1e-4


@pytest.mark.parametrize("G,d,ps", [(4, 64, 32), (16, 128, 64), (1, 128, 16)])
def test_shapes(G, d, ps):
    lens = [2048 + 100, 2048 + 33, 2048 + 260, 2048 + 1]
    w, cache = _setup(4, G, lens, 2048, d=d, ps=ps, seed=82 + G)
    q = w.q()
    got, st = _cascade(w, cache, q, [0, 4], [2048], 2048)
    assert st == 0
    assert_close(got, _ref(w, [0, 1, 2, 3], q), "G=%d d=%d ps=%d" % (G, d, ps))


def test_small_groups_run_as_plain_decode():
    lens = [2048 + 100, 2048 + 33, 2048 + 260]
    w, cache = _setup(3, 8, lens, 2048, seed=85)
    q = w.q()
    got, st = _cascade(w, cache, q, [0, 3], [2048], 2048, min_rows=64)  # 24 rows < 64
    assert st == 0
    assert np.array_equal(got, _plain(w, cache, q))


def test_prefix_cut_by_max_prefix_len():
    lens = [4096 + 10, 4096 + 500, 4096 + 3]
    w, cache = _setup(3, 8, lens, 4096, seed=86)
    q = w.q()
    got, st = _cascade(w, cache, q, [0, 3], [4096], 1000)  # shared kernel takes 992 keys, decode the rest
    assert st == 0
    assert_close(got, _ref(w, [0, 1, 2], q), "cut")


def test_max_prefix_far_above_the_prefixes():
    """The shared-prefix kernel sizes its key splits from the prefixes present, not from
    max_prefix_len: a bound 32x the longest prefix, and two groups of unequal prefixes."""
    lens = [2048 + 200, 2048 + 9, 2048 + 77, 2048 + 300, 2048 + 1]  # all share 2048; group 1 claims 1024
    w, cache = _setup(5, 8, lens, 2048, seed=89)
    q = w.q()
    got, st = _cascade(w, cache, q, [0, 3, 5], [2048, 1024], 65536)
    assert st == 0
    assert_close(got, _ref(w, list(range(5)), q), "bound far above")
    assert np.max(np.abs(got - _plain(w, cache, q))) < 1e-4


def test_prefix_longer_than_a_member_is_reported():
    lens = [2048 + 300, 2048 + 17]
    w, cache = _setup(2, 8, lens, 2048, seed=87)
    _, st = _cascade(w, cache, w.q(), [0, 2], [2048 + 100], 4096)
    assert st == 7  # UQ_ERR_DEVICE_BOUNDS


def test_nan_in_shared_prefix_poisons_the_group():
    lens = [2048 + 40, 2048 + 40, 2048 + 40]
    w = workloads.make("gqa8k", B=3, Hkv=1, Hq=8, seq_lens=lens, seed=88, shared_prefix=2048)
    cache = new_cache(w, fill=0)
    for b in range(3):
        t0 = 0 if b == 0 else 2048
        k, v = w.kv(b, t0, lens[b] - t0, device=DEV)
        if b == 0:
            v[100, 0, 5] = float("nan")
        uq.uq_quantize_append(k, v, torch.from_numpy(w.slots(b, t0, lens[b] - t0)).to(DEV), cache)
    got, st = _cascade(w, cache, w.q(), [0, 2], [2048], 2048)
    assert st == 0
    assert np.all(np.isnan(got))  # seq 2 is in no group but its table shares the poisoned page too


@pytest.mark.parametrize("B", [4, 16])
def test_full_size_prefix128k_sampled(B):
    """The bench's cascade workload: 131072-token sequences sharing their first 98304 tokens;
    every sequence through the shared-prefix kernel (min_rows 0); sampled sequences against
    the oracle."""
    base = workloads.make("prefix128k")
    w = workloads.make("prefix128k", B=B, seq_lens=[base.seq_lens[0]] * B)
    cache = new_cache(w)
    fill_cache(w, [cache])
    q = w.q()
    got, st = _cascade(w, cache, q, [0, B], [w.shared_prefix], w.shared_prefix)
    assert st == 0
    seqs = [0, B - 1]
    assert_close(got[seqs], _ref(w, seqs, q), "prefix128k B=%d" % B)


def test_full_size_prefix128k_every_row():
    """The prefix128k workload itself (4 sequences of 131072 tokens sharing 98304) through
    the shared-prefix kernel (min_rows 0, quarter-full row tiles): every output row against
    the oracle's fp64 decode of the device's own cache bytes."""
    from gpu_helpers import oracle_from_device
    from test_gpu_full_size import _oracle_decode
    w = workloads.make("prefix128k")
    cache = new_cache(w)
    fill_cache(w, [cache])
    q = w.q()
    got, st = _cascade(w, cache, q, [0, w.B], [w.shared_prefix], w.shared_prefix)
    assert st == 0
    ref = _oracle_decode(oracle_from_device(cache), bits(q), w.block_table, np.array(w.seq_lens, np.int32))
    ma, rl = assert_close(got, ref, "prefix128k every row")
    print("\nprefix128k cascade, every row: max_abs %.2e rel_l2 %.2e" % (ma, rl))
