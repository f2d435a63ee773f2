"""Pins of the oracle's FP8 E4M3 and bf16 rounding (against PyTorch's own
conversions, a library routine) and of its fp64 attention (against a dense
brute-force restatement, closed forms and page-layout invariances)."""
import numpy as np
import pytest
import scipy.special
import torch

import oracle
import workloads


def test_e4m3_value_table_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_value(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_e4m3_rounding_all_bf16_inputs():
    """All 65536 bf16 bit patterns: RNE to E4M3 must agree with torch's
    conversion wherever torch does not overflow, and saturate to +-448 above."""
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    x = bits.to(torch.float32)
    got = oracle.e4m3_codes(x.numpy())
    finite = torch.isfinite(x)
    small = finite & (x.abs() < 464.0)          # 464 = midpoint of 448 and 480
    ref = x[small].to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got[small.numpy()], ref)
    big = (finite & (x.abs() >= 464.0)).numpy()
    assert np.all((got[big] & 0x7F) == 0x7E)
    assert np.all(got[torch.isnan(x).numpy()] == 0x7F)


def test_e4m3_rounding_dense_fp32():
    rng = np.random.default_rng(9)
    x = np.concatenate([rng.standard_normal(200000) * 3, rng.uniform(-460, 460, 50000),
                        rng.uniform(-0.02, 0.02, 50000)]).astype(np.float32)
    got = oracle.e4m3_codes(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(10)
    x = np.concatenate([rng.standard_normal(20000) * 100, [0.0, -0.0, 1e-40, 3.4e38]]).astype(np.float32)
    got = oracle.f32_to_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------- attention
def _hadamard(d):
    i = np.arange(d)
    pc = np.vectorize(lambda v: bin(v).count("1"))(i[:, None] & i[None, :])
    return np.where(pc % 2 == 0, 1.0, -1.0)


# ---------------------------------------------------------------- query (R4) and the FP8 anchor's scale
def _bf16_of(x):
    return torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("k", [0, 5, 77, 127])
def test_query_fp8_of_a_basis_vector_by_hand(k):
    # R e_k = s_k (column k of H) / sqrt(128): every coordinate is +-0.0883883,
    # whose nearest E4M3 value is 1.375 * 2^-4 (exponent field 3, mantissa 3):
    # byte 0x1B, with bit 7 where s_k H[i][k] < 0
    d = 128
    q = np.zeros(d, np.float32)
    q[k] = 1.0
    got = oracle.query_fp8(_bf16_of(q)[None])[0]
    s = oracle.signs(oracle.DEFAULT_SEED, d)
    neg = (s[k] * _hadamard(d)[:, k]) < 0
    assert np.array_equal(got, np.where(neg, 0x9B, 0x1B).astype(np.uint8))


def test_query_fp8_two_hot_by_hand():
    # q = 2 e_0 + 3 e_5: R q = (2 s_0 H[:,0] + 3 s_5 H[:,5]) / sqrt(128), exact
    # integers +-5, +-1 before the scale; 5 / sqrt(128) = 0.4419 -> 1.75 * 2^-2
    # (byte 0x2E), 1 / sqrt(128) -> 0x1B
    d = 128
    q = np.zeros(d, np.float32)
    q[0], q[5] = 2.0, 3.0
    got = oracle.query_fp8(_bf16_of(q)[None])[0]
    s = oracle.signs(oracle.DEFAULT_SEED, d)
    H = _hadamard(d)
    u = 2 * s[0] * H[:, 0] + 3 * s[5] * H[:, 5]
    want = np.where(np.abs(u) == 5, 0x2E, 0x1B) | np.where(u < 0, 0x80, 0)
    assert np.array_equal(got, want.astype(np.uint8))


@pytest.mark.parametrize("d", [64, 128, 256])
def test_query_fp8_is_e4m3_of_the_rotated_query(d):
    # R4 composes two separately pinned stages: R1 and E4M3 rounding
    q = _bf16_bits(torch.randn(40, d, generator=torch.Generator().manual_seed(d)).to(torch.bfloat16) * 7)
    qf = (q.astype(np.uint32) << 16).view(np.float32)
    want = oracle.e4m3_codes(oracle.rotate_fp32(qf)).reshape(q.shape)
    assert np.array_equal(oracle.query_fp8(q), want)


def test_fp8_append_divides_by_the_tensor_scale():
    # e4m3(x / k_scale): 3 / 0.5 = 6 -> 0x4C, -3 / 0.5 -> 0xCC, 300 / 0.5 = 600 saturates
    # to 448 (0x7E); v: 3 / 2 = 1.5 -> 0x3C
    d, ps = 64, 16
    cache = oracle.Cache(oracle.KIND_FP8, 1, 1, ps, d, k_scale=0.5, v_scale=2.0)
    k = np.full((3, 1, d), 3.0, np.float32)
    k[1] = -3.0
    k[2] = 300.0
    v = np.full((3, 1, d), 3.0, np.float32)
    cache.append(k, v, np.array([0, 1, 2], np.int64))
    assert np.all(cache.kc[0] == 0x4C) and np.all(cache.kc[1] == 0xCC) and np.all(cache.kc[2] == 0x7E)
    assert np.all(cache.vc[:3] == 0x3C)


def _e2m1(code):
    s, e, m = (code >> 3) & 1, (code >> 1) & 3, code & 1
    v = np.where(e == 0, m * 0.5, 2.0 ** (e - 1) * (1 + m / 2))
    return np.where(s == 1, -v, v)


def _dequant_dense(codes, scales):
    """[rows][d/2] codes, [rows][d/32] scales -> [rows][d] fp64 (bit-field
    decode written independently of the oracle)."""
    rows, half = codes.shape
    d = half * 2
    vals = np.empty((rows, d))
    vals[:, 0::2] = _e2m1(codes & 15)
    vals[:, 1::2] = _e2m1(codes >> 4)
    return vals * np.repeat(2.0 ** (scales.astype(np.float64) - 127), 32, axis=1)


def _k_natural(kc):
    """Undo the cache's group-interleaved word order of K rows (include/uq.h):
    word w of group g sits at word position (d/32)*w + g."""
    rows, half = kc.shape
    ng = half // 16
    words = kc.reshape(rows, 4, ng, 4)            # [row][w][g][byte]
    return words.transpose(0, 2, 1, 3).reshape(rows, half)


def test_k_row_word_order():
    """Literal word order of a K row in the cache for head_dim 64 and 128."""
    want64 = ["g0w0", "g1w0", "g0w1", "g1w1", "g0w2", "g1w2", "g0w3", "g1w3"]
    want128 = ["g0w0", "g1w0", "g2w0", "g3w0", "g0w1", "g1w1", "g2w1", "g3w1",
               "g0w2", "g1w2", "g2w2", "g3w2", "g0w3", "g1w3", "g2w3", "g3w3"]
    for d, want in ((64, want64), (128, want128)):
        got = [None] * (d // 8)
        for j in range(0, d // 2, 4):
            g, w = j // 16, (j % 16) // 4
            got[oracle.kbyte_pos(j, d) // 4] = "g%dw%d" % (g, w)
        assert got == want
        # and a cache row: quantise a vector with distinct codes per word, append, compare
        rng = np.random.default_rng(d)
        x = rng.standard_normal((1, 1, d)).astype(np.float32)
        cache = oracle.Cache(oracle.KIND_FP4, 1, 1, 16, d)
        cache.append(x, x, np.array([0]))
        nat, _ = oracle.quantize_vectors(x.reshape(1, d))
        assert np.array_equal(_k_natural(cache.kc[:1]), nat)
        assert np.array_equal(cache.vc[:1], nat)


def _bf16_bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _small(B=3, Hkv=2, Hq=8, d=64, ps=16, lens=(37, 16, 70), shuffled=True, seed=5):
    w = workloads.make("gqa8k", B=B, Hkv=Hkv, Hq=Hq, D=d, ps=ps, seq_lens=list(lens), seed=seed,
                       shuffled=shuffled, n_outlier=3, outlier_channels=None)
    cache = oracle.Cache(oracle.KIND_FP4, w.num_pages, Hkv, ps, d)
    for b in range(B):
        k, v = w.kv(b, 0, lens[b])
        cache.append(_bf16_bits(k), _bf16_bits(v), w.slots(b, 0, lens[b]))
    return w, cache


def test_attention_matches_dense_brute_force():
    w, cache = _small()
    q = _bf16_bits(w.q())
    out = cache.decode(q, w.block_table, np.array(w.seq_lens, np.int32))
    d, G = w.D, w.G
    s = oracle.signs(oracle.DEFAULT_SEED, d).astype(np.float64)
    H = _hadamard(d)
    qt = np.vectorize(oracle.e4m3_value)(oracle.query_fp8(q))  # pinned separately
    K = _dequant_dense(_k_natural(cache.kc), cache.ks)
    V = _dequant_dense(cache.vc, cache.vs)
    for b in range(w.B):
        L = w.seq_lens[b]
        j = np.arange(L)
        for h in range(w.Hq):
            rows = (w.block_table[b, j // w.ps].astype(np.int64) * w.Hkv + h // G) * w.ps + j % w.ps
            logits = K[rows] @ qt[b, h] / np.sqrt(d)
            p = scipy.special.softmax(logits)
            o = p @ V[rows]
            ref = s * (H @ o) / np.sqrt(d)
            assert np.allclose(out[b, h], ref, rtol=1e-12, atol=1e-12)


def test_single_token_closed_form():
    """ctx = 1: softmax weight 1, output = inverse rotation of v^_0."""
    w, cache = _small(B=1, lens=(1,))
    q = _bf16_bits(w.q())
    out = cache.decode(q, w.block_table, np.array([1], np.int32))
    d = w.D
    s = oracle.signs(oracle.DEFAULT_SEED, d).astype(np.float64)
    for h in range(w.Hq):
        row = (w.block_table[0, 0] * w.Hkv + h // w.G) * w.ps
        v0 = _dequant_dense(cache.vc[row:row + 1], cache.vs[row:row + 1])[0]
        assert np.allclose(out[0, h], s * (_hadamard(d) @ v0) / np.sqrt(d), atol=1e-12)


def test_identical_keys_give_mean_of_values():
    d, L = 64, 40
    cache = oracle.Cache(oracle.KIND_FP4, 4, 1, 16, d)
    rng = np.random.default_rng(11)
    k = np.repeat(rng.standard_normal((1, 1, d)), L, axis=0).astype(np.float32)
    v = rng.standard_normal((L, 1, d)).astype(np.float32)
    cache.append(k, v, np.arange(L))
    q = _bf16_bits(torch.randn(1, 2, d).to(torch.bfloat16))
    out = cache.decode(q, np.arange(4, dtype=np.int32)[None], np.array([L], np.int32))
    V = _dequant_dense(cache.vc[:L], cache.vs[:L])
    ref = oracle.inverse_rotate_f64(V.mean(0))
    assert np.allclose(out[0, 0], ref, atol=1e-12) and np.allclose(out[0, 1], ref, atol=1e-12)


def test_page_permutation_invariance():
    w1, c1 = _small(shuffled=False)
    w2, c2 = _small(shuffled=True)
    q = _bf16_bits(w1.q())
    o1 = c1.decode(q, w1.block_table, np.array(w1.seq_lens, np.int32))
    o2 = c2.decode(q, w2.block_table, np.array(w2.seq_lens, np.int32))
    assert not np.array_equal(w1.block_table, w2.block_table)
    assert np.array_equal(o1, o2)


def test_shared_prefix_equals_copied_prefix():
    """A prefix shared through the block table gives the same result as the
    same tokens stored in every sequence's own pages."""
    kw = dict(B=2, Hkv=1, Hq=2, D=64, ps=16, seq_lens=[4096 + 48, 4096 + 80], seed=8, n_outlier=2,
              outlier_channels=None)
    shared = workloads.make("prefix128k", shared_prefix=4096, **kw)
    copied = workloads.make("prefix128k", shared_prefix=0, **kw)
    outs = []
    for w, share in ((shared, True), (copied, False)):
        cache = oracle.Cache(oracle.KIND_FP4, w.num_pages, w.Hkv, w.ps, w.D)
        for b in range(w.B):
            start = 4096 if (share and b > 0) else 0
            k, v = shared.kv(b, start, w.seq_lens[b] - start)
            cache.append(_bf16_bits(k), _bf16_bits(v), w.slots(b, start, w.seq_lens[b] - start))
        outs.append(cache.decode(_bf16_bits(shared.q()), w.block_table, np.array(w.seq_lens, np.int32)))
    assert shared.num_pages < copied.num_pages
    assert np.array_equal(outs[0], outs[1])


def test_empty_sequence_gives_zero():
    w, cache = _small(lens=(0, 5, 16))
    out = cache.decode(_bf16_bits(w.q()), w.block_table, np.array([0, 5, 16], np.int32))
    assert np.all(out[0] == 0) and np.all(np.isfinite(out[1:]))


@pytest.mark.parametrize("kind", [oracle.KIND_FP8, oracle.KIND_BF16])
def test_anchor_attention_matches_dense(kind):
    B, Hkv, Hq, d, ps, L = 2, 2, 4, 64, 16, 50
    rng = np.random.default_rng(12)
    k = (rng.standard_normal((B, L, Hkv, d)) * 3).astype(np.float32)
    v = rng.standard_normal((B, L, Hkv, d)).astype(np.float32)
    pages = (L + ps - 1) // ps
    bt = np.arange(B * pages, dtype=np.int32).reshape(B, pages)
    ks, vs = (0.5, 2.0) if kind == oracle.KIND_FP8 else (1.0, 1.0)
    cache = oracle.Cache(kind, B * pages, Hkv, ps, d, k_scale=ks, v_scale=vs)
    for b in range(B):
        cache.append(k[b], v[b], bt[b, np.arange(L) // ps].astype(np.int64) * ps + np.arange(L) % ps)
    q = _bf16_bits(torch.randn(B, Hq, d).to(torch.bfloat16))
    out = cache.decode(q, bt, np.array([L, L], np.int32))
    qf = q.astype(np.uint32) << 16
    qf = qf.view(np.float32).astype(np.float64)
    if kind == oracle.KIND_FP8:
        Kd = torch.from_numpy(cache.kc).view(torch.float8_e4m3fn).double().numpy() * ks
        Vd = torch.from_numpy(cache.vc).view(torch.float8_e4m3fn).double().numpy() * vs
    else:
        Kd = torch.from_numpy(cache.kc.view(np.int16)).view(torch.bfloat16).double().numpy()
        Vd = torch.from_numpy(cache.vc.view(np.int16)).view(torch.bfloat16).double().numpy()
    for b in range(B):
        j = np.arange(L)
        for h in range(Hq):
            rows = (bt[b, j // ps].astype(np.int64) * Hkv + h // (Hq // Hkv)) * ps + j % ps
            p = scipy.special.softmax(Kd[rows] @ qf[b, h] / np.sqrt(d))
            assert np.allclose(out[b, h], p @ Vd[rows], rtol=1e-12, atol=1e-12)

