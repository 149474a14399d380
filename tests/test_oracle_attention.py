"""Pins for the oracle's attention and split merge (CPU only).

The attention result has a plain definition (softmax(scale * q K^T) V with its log-sum-exp); the
oracle is checked against 50-digit brute force, closed forms (one token, identical keys),
invariants (weights sum to 1, page permutation, GQA = repeated MHA), the split-result merge of
ZipFusion §IV.B, and the dense KV-bytes formula of the FlashSVD v1.5 review (Eq. 8) together with
the AttSVD dense-cache sizes (Table 1).
"""
import math

import mpmath
import numpy as np
import pytest

from decode_attention_compressed_gb300 import inputs as I
from decode_attention_compressed_gb300.accounting import dense_kv_bytes
from oracle import zf_oracle as O


def to_bits(x):
    x = np.asarray(x, np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)   # round to nearest even


def rand_bits(rng, shape, std=1.0):
    return to_bits(rng.standard_normal(shape) * std)


def test_empty_context():
    out, lse, w = O.attention_one(np.ones(4), np.zeros((0, 4)), np.zeros((0, 4)), 0.5)
    assert (out == 0).all() and lse == -math.inf and w.size == 0


def test_one_token_returns_v_exactly():
    rng = np.random.default_rng(0)
    for _ in range(20):
        q, k, v = (O.bf16_to_f64(rand_bits(rng, (128,))) for _ in range(3))
        out, lse, w = O.attention_one(q, k[None], v[None], 1 / math.sqrt(128))
        assert (out == v).all()
        assert lse == (1 / math.sqrt(128)) * float(k @ q)
        assert (w == 1.0).all()


def test_weights_sum_to_one_and_are_ordered_by_score():
    rng = np.random.default_rng(1)
    q = O.bf16_to_f64(rand_bits(rng, (128,)))
    K = O.bf16_to_f64(rand_bits(rng, (333, 128), 3.0))
    V = O.bf16_to_f64(rand_bits(rng, (333, 128)))
    _, _, w = O.attention_one(q, K, V, 1 / math.sqrt(128))
    assert abs(w.sum() - 1.0) < 1e-12
    s = K @ q
    assert (np.argsort(w, kind="stable") == np.argsort(s, kind="stable")).all()


def test_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(2)
    q = O.bf16_to_f64(rand_bits(rng, (128,)))
    k = O.bf16_to_f64(rand_bits(rng, (128,), 4.0))
    V = O.bf16_to_f64(rand_bits(rng, (77, 128)))
    out, lse, _ = O.attention_one(q, np.tile(k, (77, 1)), V, 0.125)
    assert np.abs(out - V.mean(axis=0)).max() < 1e-12
    assert abs(lse - (0.125 * float(k @ q) + math.log(77))) < 1e-12


def _mp_attention(q, K, V, scale):
    mpmath.mp.dps = 50
    s = [mpmath.mpf(scale) * mpmath.fsum(mpmath.mpf(float(a)) * mpmath.mpf(float(b)) for a, b in zip(q, k)) for k in K]
    z = mpmath.fsum(mpmath.e ** x for x in s)
    out = [mpmath.fsum(mpmath.e ** s[t] * mpmath.mpf(float(V[t][c])) for t in range(len(K))) / z for c in range(len(V[0]))]
    return out, mpmath.log(z)


@pytest.mark.parametrize("T,D", [(1, 4), (3, 8), (8, 8), (5, 3)])
def test_brute_force_50_digits(T, D):
    rng = np.random.default_rng(T * 10 + D)
    q = O.bf16_to_f64(rand_bits(rng, (D,), 2.0))
    K = O.bf16_to_f64(rand_bits(rng, (T, D), 2.0))
    V = O.bf16_to_f64(rand_bits(rng, (T, D)))
    scale = 0.37
    out, lse, _ = O.attention_one(q, K, V, scale)
    mo, ml = _mp_attention(q, K, V, scale)
    assert abs(lse - float(ml)) <= 1e-13 * max(1.0, abs(lse))
    for c in range(D):
        assert abs(out[c] - float(mo[c])) <= 1e-13


def test_split_merge_equals_unsplit():
    """ZipFusion §IV.B: split-KV partial results are combined by the split-result merge."""
    rng = np.random.default_rng(3)
    q = O.bf16_to_f64(rand_bits(rng, (128,)))
    K = O.bf16_to_f64(rand_bits(rng, (1000, 128), 2.0))
    V = O.bf16_to_f64(rand_bits(rng, (1000, 128)))
    out, lse, _ = O.attention_one(q, K, V, 0.1)
    for cuts in ([0, 1000], [0, 1, 1000], [0, 64, 128, 999, 1000], list(range(0, 1001, 100))):
        parts = [O.attention_one(q, K[a:b], V[a:b], 0.1) for a, b in zip(cuts[:-1], cuts[1:])]
        mo, ml = O.merge_partials([p[0] for p in parts], [p[1] for p in parts])
        assert np.abs(mo - out).max() < 1e-12 and abs(ml - lse) < 1e-12
    mo, ml = O.merge_partials(np.zeros((2, 128)), [-math.inf, -math.inf])
    assert (mo == 0).all() and ml == -math.inf


def _small_paged(seed=5, B=3, Hq=8, Hkv=2, P=16, lens=(37, 16, 70), pool="random"):
    w = I.Workload("t", B, Hq, Hkv, P, max(lens), pool=pool, seed=seed)
    L = I.make_layer(w, seq_lens=list(lens))
    npg = L.num_pages
    cache = O.Cache(num_pages=npg, num_kv_heads=Hkv, page_size=P, num_raw=npg)
    k = L.k_pages.numpy().view(np.uint16)
    v = L.v_pages.numpy().view(np.uint16)
    O.encode_pages(cache, k, v, list(range(npg)), L.n_valid.numpy(), list(range(npg)))
    return L, cache, k, v


def test_paged_attention_equals_dense_attention():
    L, cache, k, v = _small_paged()
    q = L.q.numpy().view(np.uint16)
    table, lens = L.page_table.numpy(), L.seq_lens.numpy()
    out, lse = O.decode_attention(q, cache, table, lens, L.scale)
    P = cache.page_size
    kseq, vseq = [], []
    for b in range(q.shape[0]):
        n = int(lens[b])
        pages = table[b, : -(-n // P)]
        kseq.append(np.concatenate([k[p].transpose(1, 0, 2) for p in pages])[:n])
        vseq.append(np.concatenate([v[p].transpose(1, 0, 2) for p in pages])[:n])
    ref, ref_lse = O.attention_dense(q, kseq, vseq, L.scale)
    assert (out == ref).all() and (lse == ref_lse).all()
    sub, sub_lse = O.decode_attention(q, cache, table, lens, L.scale, pairs=[(2, 5), (0, 0)])
    assert (sub[2, 5] == out[2, 5]).all() and sub_lse[0, 0] == lse[0, 0]
    assert (sub[1] == 0).all() and np.isneginf(sub_lse[1]).all()


def test_page_permutation_invariance():
    L, cache, k, v = _small_paged(seed=6)
    q = L.q.numpy().view(np.uint16)
    table, lens = L.page_table.numpy(), L.seq_lens.numpy()
    out, lse = O.decode_attention(q, cache, table, lens, L.scale)
    npg = cache.num_pages
    perm = np.random.default_rng(9).permutation(npg)      # new id of old page i is perm[i]
    moved = O.Cache(num_pages=npg, num_kv_heads=cache.num_kv_heads, page_size=cache.page_size, num_raw=npg)
    O.encode_pages(moved, k, v, list(perm), L.n_valid.numpy(), list(perm))
    table2 = np.where(table >= 0, perm[np.maximum(table, 0)], -1)
    out2, lse2 = O.decode_attention(q, moved, table2, lens, L.scale)
    assert (out2 == out).all() and (lse2 == lse).all()


def test_gqa_equals_mha_with_repeated_heads():
    rng = np.random.default_rng(8)
    B, Hq, Hkv, T = 2, 6, 2, 41
    q = rand_bits(rng, (B, Hq, 128))
    ks = [rand_bits(rng, (T, Hkv, 128), 2.0) for _ in range(B)]
    vs = [rand_bits(rng, (T, Hkv, 128)) for _ in range(B)]
    out, lse = O.attention_dense(q, ks, vs, 0.2)
    rep = Hq // Hkv
    out2, lse2 = O.attention_dense(q, [np.repeat(k, rep, axis=1) for k in ks], [np.repeat(v, rep, axis=1) for v in vs], 0.2)
    assert (out == out2).all() and (lse == lse2).all()
    # and the mapping is h // group, not h % Hkv
    assert (out[:, 1] == O.attention_dense(q[:, 1:2], [k[:, 0:1] for k in ks], [v[:, 0:1] for v in vs], 0.2)[0][:, 0]).all()


def test_dense_kv_bytes_formula():
    """FlashSVD v1.5 review, Eq. 8: LLaMA-7B (32 heads, d_h 128, 32 layers, BF16) holds
    524,288 bytes per token; AttSVD Table 1: dense caches of 4.500 GiB (Qwen3-8B: 36 layers,
    8 KV heads) and 6.250 GiB (Phi-4-14B: 40 layers, 10 KV heads) at 32K tokens."""
    for T in (1, 512, 8192):
        assert dense_kv_bytes(32, 128, 32, T) == 524_288 * T
    assert dense_kv_bytes(32, 128, 32, 8192) == 4 * 2 ** 30
    assert dense_kv_bytes(8, 128, 36, 32768) / 2 ** 30 == 4.5
    assert dense_kv_bytes(10, 128, 40, 32768) / 2 ** 30 == 6.25


# ---- several new tokens per request (speculative verification): token t of T at position
# L - T + t attends to positions 0 .. L - T + t (the causal rule, one token's decode per prefix)
def _multi_q(rng, B, T, Hq):
    return rand_bits(rng, (B, T, Hq, 128))


def test_multi_token_with_one_token_is_the_decode():
    L, cache, k, v = _small_paged(seed=11)
    q = L.q.numpy().view(np.uint16)
    table, lens = L.page_table.numpy(), L.seq_lens.numpy()
    out, lse = O.decode_attention(q, cache, table, lens, L.scale)
    mout, mlse = O.decode_attention_multi(q[:, None], cache, table, lens, L.scale)
    assert (mout[:, 0] == out).all() and (mlse[:, 0] == lse).all()


def test_multi_token_identical_keys_give_mean_of_the_visible_values():
    """Closed form: with every key of a head equal, token t's weights are uniform over the
    L - T + t + 1 positions it sees, so out is the mean of those V rows and lse is
    scale * q.k + ln(count)."""
    rng = np.random.default_rng(12)
    B, Hq, Hkv, P, T = 2, 4, 2, 16, 5
    lens = (37, 5)
    w = I.Workload("t", B, Hq, Hkv, P, max(lens), seed=12)
    lay = I.make_layer(w, seq_lens=list(lens))
    k = lay.k_pages.numpy().view(np.uint16).copy()
    v = lay.v_pages.numpy().view(np.uint16)
    krow = rand_bits(rng, (Hkv, 128), 2.0)
    k[:] = krow[None, :, None, :]
    npg = lay.num_pages
    cache = O.Cache(num_pages=npg, num_kv_heads=Hkv, page_size=P, num_raw=npg)
    O.encode_pages(cache, k, v, list(range(npg)), lay.n_valid.numpy(), list(range(npg)))
    q = _multi_q(rng, B, T, Hq)
    table = lay.page_table.numpy()
    out, lse = O.decode_attention_multi(q, cache, table, np.array(lens), 0.125)
    for b in range(B):
        Lb = lens[b]
        vseq = np.concatenate([v[p].transpose(1, 0, 2) for p in table[b, : -(-Lb // P)]])[:Lb]
        for t in range(T):
            n = Lb - T + t + 1
            for h in range(Hq):
                g = h // (Hq // Hkv)
                if n <= 0:
                    assert (out[b, t, h] == 0).all() and np.isneginf(lse[b, t, h])
                    continue
                mean = O.bf16_to_f64(vseq[:n, g]).mean(axis=0)
                assert np.abs(out[b, t, h] - mean).max() < 1e-12
                s = 0.125 * float(O.bf16_to_f64(krow[g]) @ O.bf16_to_f64(q[b, t, h]))
                assert abs(lse[b, t, h] - (s + math.log(n))) < 1e-12


def test_multi_token_each_token_is_a_single_token_decode_of_its_prefix():
    L, cache, k, v = _small_paged(seed=13, lens=(37, 16, 70))
    rng = np.random.default_rng(13)
    T = 4
    q = _multi_q(rng, 3, T, 8)
    table, lens = L.page_table.numpy(), L.seq_lens.numpy()
    out, lse = O.decode_attention_multi(q, cache, table, lens, L.scale)
    for t in range(T):
        ref, ref_lse = O.decode_attention(q[:, t], cache, table, lens - (T - 1 - t), L.scale)
        assert (out[:, t] == ref).all() and (lse[:, t] == ref_lse).all()
    sub, sub_lse = O.decode_attention_multi(q, cache, table, lens, L.scale, pairs=[(2, 3, 5), (0, 1, 0)])
    assert (sub[2, 3, 5] == out[2, 3, 5]).all() and sub_lse[0, 1, 0] == lse[0, 1, 0]
    assert (sub[1] == 0).all() and np.isneginf(sub_lse[1]).all()
