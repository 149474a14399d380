"""GPU parity of zf_encode_pages / zf_decompress against the oracle: bit-exact bytes, directory and
status on the workloads' distributions and on adversarial blocks; decompress returns every
source bit."""
import numpy as np
import pytest
import torch

from decode_attention_compressed_gb300 import inputs as I
from oracle import zf_oracle as O
from tests import helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def zf():
    return H.zf_module()


SMALL = {
    "tiny": I.WORKLOADS["tiny"],
    "llama7b_mha": I.scaled(I.WORKLOADS["llama7b_mha_512"], ctx=128),
    "llama3_8b_batched": I.scaled(I.WORKLOADS["llama3_8b_batched"], batch=4, ctx=300, ctx_min=40),
    "qwen2_7b_maxbatch": I.scaled(I.WORKLOADS["qwen2_7b_maxbatch"], batch=3, ctx=600),
    "long_ctx": I.scaled(I.WORKLOADS["long_ctx"], batch=2, ctx=400),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_encode_matches_oracle_bit_exactly(zf, name):
    layer = I.make_layer(SMALL[name])
    gc = H.gpu_cache_from(layer, zf)
    oc = H.oracle_cache_from(layer, O)
    H.assert_caches_equal(gc, oc)
    # the distributions exercise both kinds of storage and the escape list
    assert (oc.dir == -1).any()
    if name in ("llama3_8b_batched", "long_ctx"):
        assert (oc.dir >= 0).any()          # partial tail pages stay raw


@pytest.mark.parametrize("name", sorted(SMALL))
def test_decompress_returns_every_bit(zf, name):
    layer = I.make_layer(SMALL[name])
    gc = H.gpu_cache_from(layer, zf)
    k, v = zf.decompress(gc, list(range(layer.num_pages)))
    torch.cuda.synchronize()
    assert torch.equal(k.cpu(), layer.k_pages) and torch.equal(v.cpu(), layer.v_pages)
    assert gc.status_word() == 0


def _pattern(s, e, f):
    return (s << 15) | (e << 7) | f


def adversarial_pages(seed=0, hkv=2, P=16):
    """Pages whose blocks cover: all 65,536 BF16 patterns inside a window, escapes of every
    pattern class, exactly 6 and 7 escapes, window boundaries, NaN/Inf/zero/subnormal blocks."""
    rng = np.random.default_rng(seed)
    blocks = []
    for E in range(0, 256, 2):                              # every pattern, compressed
        vals = np.array([_pattern(s, e, f) for s in (0, 1) for e in (E, E + 1) for f in range(128)])
        blocks.append(rng.permutation(vals))
    filler = np.array([_pattern(s, e, f) for s in (0, 1) for e in range(240, 256) for f in range(128)])
    low = rng.permutation(np.array([_pattern(s, e, f) for e in range(240) for s in (0, 1) for f in range(128)]))
    for i in range(0, 6 * 40, 6):                           # 6 escapes (base/2 = 120)
        v = np.concatenate([low[i:i + 6], rng.choice(filler, 506, replace=False)])
        v[-1] = _pattern(1, 255, 3)
        blocks.append(rng.permutation(v))
    seven = np.full(512, _pattern(0, 127, 0))
    seven[:7] = _pattern(0, 20, 1)                           # 7 escapes: the page must stay raw
    blocks.append(rng.permutation(seven))
    b = np.full(512, _pattern(0, 110, 5))
    b[:3] = _pattern(0, 101, 1)
    b[3] = _pattern(1, 116, 9)                               # odd minimum, range 15 -> 3 escapes
    blocks.append(rng.permutation(b))
    b = np.full(512, _pattern(0, 100, 5))
    b[0] = _pattern(1, 115, 0)                               # range 15 from an even minimum
    blocks.append(rng.permutation(b))
    for sp in (0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0xFFFF, 0x0001, 0x807F):
        blocks.append(np.full(512, sp))
    zero_base = rng.integers(0, 128, 512) | (rng.integers(0, 2, 512) << 15)   # exponents 0 (subnormals)
    blocks.append(zero_base)
    per_page = hkv * 2 * (P // 4)
    while len(blocks) % per_page:
        blocks.append(rng.integers(0, 65536, 512))        # random patterns (mostly raw-bound)
    blocks = np.stack(blocks).astype(np.uint16).reshape(-1, hkv, 2, P // 16, 4, 16, 32)
    # -> [n][hkv][K|V][tile][group][16][32] -> natural pages [n][hkv][P][128]
    pages = blocks.transpose(0, 1, 2, 3, 5, 4, 6).reshape(-1, hkv, 2, P, 128)
    return pages[:, :, 0], pages[:, :, 1]


@pytest.mark.parametrize("P", [16, 64])
def test_adversarial_blocks(zf, P):
    k, v = adversarial_pages(hkv=2, P=P)
    n = k.shape[0]
    kt = torch.from_numpy(k.view(np.int16).copy()).cuda()
    vt = torch.from_numpy(v.view(np.int16).copy()).cuda()
    gc = zf.Cache(n, 2, P, n)
    zf.encode_pages(gc, kt, vt, list(range(n)), [P] * n, list(range(n)))
    oc = O.Cache(num_pages=n, num_kv_heads=2, page_size=P, num_raw=n)
    O.encode_pages(oc, k, v, list(range(n)), [P] * n, list(range(n)))
    torch.cuda.synchronize()
    H.assert_caches_equal(gc, oc)
    assert (oc.dir == -1).sum() > 0 and (oc.dir >= 0).sum() > 0
    dk, dv = zf.decompress(gc, list(range(n)))
    torch.cuda.synchronize()
    assert torch.equal(dk, kt) and torch.equal(dv, vt)


def test_page_lifecycle_and_status(zf):
    """ZipFusion §III.D on the GPU: partial pages raw, full pages compressed under their id,
    missing raw slots and bad ids reported in the status word, forced raw storage."""
    w = I.scaled(I.WORKLOADS["llama3_8b_batched"], batch=2, ctx=90, ctx_min=20)
    layer = I.make_layer(w)
    n = layer.num_pages
    ids = list(reversed(range(n)))                       # page i of the call gets id n-1-i
    perm = np.random.default_rng(0).permutation(n + 2)
    raw = [(-1 if i % 3 == 0 else int(perm[i])) for i in range(n)]   # distinct slots
    gc = H.gpu_cache_from(layer, zf, raw_slots=raw, page_ids=ids, extra_raw=2)
    oc = H.oracle_cache_from(layer, O, raw_slots=raw, page_ids=ids, extra_raw=2)
    H.assert_caches_equal(gc, oc)
    # bad page id and bad n_valid
    gc2 = zf.Cache(4, w.num_kv_heads, w.page_size, 4)
    src = layer.k_pages[:3].cuda()
    zf.encode_pages(gc2, src, src, [0, 9, 2], [16, 16, 17], [0, 1, 2])
    torch.cuda.synchronize()
    assert gc2.status_word() == (zf.DEV_BAD_PAGE_ID | zf.DEV_BAD_N_VALID)
    d = gc2.dir.cpu().numpy()
    assert (d[0] == -1).all() and (d[2] == -2).all() and (d[1] == -2).all()
    # forced raw
    gc3 = H.gpu_cache_from(layer, zf, force_raw=True)
    oc3 = H.oracle_cache_from(layer, O, force_raw=True)
    H.assert_caches_equal(gc3, oc3)
    assert (oc3.dir >= 0).all()


def test_decompress_of_invalid_entries(zf):
    gc = zf.Cache(3, 2, 16, 1)
    k, v = zf.decompress(gc, [0, 2, 7])
    torch.cuda.synchronize()
    assert (k == 0).all() and (v == 0).all()
    assert gc.status_word() == (zf.DEV_BAD_DIR | zf.DEV_BAD_PAGE_ID)


@pytest.mark.parametrize("name", ["qwen2_7b_maxbatch", "long_ctx"])
def test_decompress_to_raw_matches_a_raw_encode_and_attends(zf, name):
    """Restore-then-attend baseline: pages decompressed into a dense cache's raw layout are the
    bytes a force-raw encode of the source writes, and dense attention over them matches the
    oracle."""
    layer = I.make_layer(SMALL[name])
    gc = H.gpu_cache_from(layer, zf)
    n = layer.num_pages
    dense = zf.Cache(n, gc.num_kv_heads, gc.page_size, n, compressed=False)
    zf.decompress_to_raw(gc, list(range(n)), dense)
    want = H.gpu_cache_from(layer, zf, force_raw=True)
    torch.cuda.synchronize()
    assert gc.status_word() == 0
    assert torch.equal(dense.k_raw, want.k_raw[:n]) and torch.equal(dense.v_raw, want.v_raw[:n])
    dev = torch.device("cuda")
    out, lse = zf.dense_decode_attn(dense, layer.q.to(dev), layer.page_table.to(dev), layer.seq_lens.to(dev),
                                    layer.scale)
    torch.cuda.synchronize()
    oc = H.oracle_cache_from(layer, O)
    ref_out, ref_lse = O.decode_attention(H.np_bits(layer.q), oc, layer.page_table.numpy(), layer.seq_lens.numpy(),
                                          layer.scale)
    H.compare_attention(out, lse, ref_out, ref_lse)


@pytest.mark.parametrize("P", [16, 64])
def test_append_tokens_matches_oracle_bit_exactly(zf, P):
    """zf_append_tokens against the oracle: pages filled one token per call (the adversarial pages
    above plus two normal ones; two pages start as partial pages written by zf_encode_pages, the
    rest from stale slot contents), compared bit for bit — every raw slot, the compressed slots the
    directory points at, directory and status — at the first, middle and last token."""
    rng = np.random.default_rng(200 + P)
    hkv = 2
    ak, av = adversarial_pages(seed=P, hkv=hkv, P=P)
    nk = ((rng.standard_normal((2, hkv, P, 128)).astype(np.float32).view(np.uint32) + 0x8000) >> 16).astype(np.uint16)
    nvv = ((rng.standard_normal((2, hkv, P, 128)).astype(np.float32).view(np.uint32) + 0x8000) >> 16).astype(np.uint16)
    k = np.concatenate([ak, nk])
    v = np.concatenate([av, nvv])
    n = k.shape[0]
    ids = [int(x) for x in rng.permutation(n + 2)[:n]]
    slots = [int(x) for x in rng.permutation(n + 1)[:n]]
    gc = zf.Cache(n + 2, hkv, P, n + 1)
    oc = O.Cache(num_pages=n + 2, num_kv_heads=hkv, page_size=P, num_raw=n + 1)
    oc.k_raw[:] = rng.integers(0, 1 << 16, oc.k_raw.shape, dtype=np.uint16)
    oc.v_raw[:] = rng.integers(0, 1 << 16, oc.v_raw.shape, dtype=np.uint16)
    gc.k_raw.copy_(torch.from_numpy(oc.k_raw.view(np.int16).reshape(gc.k_raw.shape)))
    gc.v_raw.copy_(torch.from_numpy(oc.v_raw.view(np.int16).reshape(gc.v_raw.shape)))
    kt = torch.from_numpy(k.view(np.int16).copy()).cuda()
    vt = torch.from_numpy(v.view(np.int16).copy()).cuda()
    start = {0: 3, n - 1: P // 2}                           # call index -> tokens already encoded
    for i, t0 in start.items():
        zf.encode_pages(gc, kt[i:i + 1], vt[i:i + 1], [ids[i]], [t0], [slots[i]])
        O.encode_pages(oc, k[i:i + 1], v[i:i + 1], [ids[i]], [t0], [slots[i]])
    for t in range(P):
        sel = [i for i in range(n) if t >= start.get(i, 0)]
        zf.append_tokens(gc, kt[sel, :, t], vt[sel, :, t], [ids[i] for i in sel], [t] * len(sel),
                         [slots[i] for i in sel])
        O.append_tokens(oc, k[sel][:, :, t], v[sel][:, :, t], [ids[i] for i in sel], [t] * len(sel),
                        [slots[i] for i in sel])
        if t in (0, P // 2, P - 1):
            torch.cuda.synchronize()
            H.assert_caches_equal(gc, oc)
            assert (H.np_bits(gc.k_raw) == oc.k_raw.reshape(gc.k_raw.shape)).all()
            assert (H.np_bits(gc.v_raw) == oc.v_raw.reshape(gc.v_raw.shape)).all()
    assert (oc.dir[ids] == O.DIR_COMPRESSED).any() and (oc.dir[ids] >= 0).any()
    dk, dv = zf.decompress(gc, ids)
    torch.cuda.synchronize()
    assert torch.equal(dk, kt) and torch.equal(dv, vt)


def test_append_tokens_reports_bad_entries(zf):
    P, hkv = 16, 2
    gc = zf.Cache(3, hkv, P, 2)
    gc.k_raw.zero_()
    gc.v_raw.zero_()
    oc = O.Cache(num_pages=3, num_kv_heads=hkv, page_size=P, num_raw=2)
    tok = np.arange(4 * hkv * 128, dtype=np.uint16).reshape(4, hkv, 128)
    tt = torch.from_numpy(tok.view(np.int16).copy()).cuda()
    ids, pos, slots = [0, 7, 1, 2], [0, 0, P, 5], [1, 0, 0, 2]   # good, bad id, bad position, bad slot
    zf.append_tokens(gc, tt, tt, ids, pos, slots)
    O.append_tokens(oc, tok, tok, ids, pos, slots)
    torch.cuda.synchronize()
    assert gc.status_word() == oc.status == (O.ST_BAD_PAGE_ID | O.ST_BAD_N_VALID | O.ST_BAD_RAW_SLOT)
    H.assert_caches_equal(gc, oc)
    assert (oc.dir[0] == 1).all() and (oc.dir[1:] == O.DIR_INVALID).all()


def test_validate_pages_flags_exactly_the_damaged_pages(zf):
    """zf_validate_pages after damage to stored metadata: random header / escape bytes of some
    compressed slots, a code that would carry, a directory entry pointing past the raw slots, and
    an id out of range.  The pages flagged are exactly those with a slot the oracle's decoder
    rejects or a bad directory entry; the status word names the kinds."""
    layer = I.make_layer(SMALL["llama3_8b_batched"])
    gc = H.gpu_cache_from(layer, zf)
    n = layer.num_pages
    bad = zf.validate_pages(gc, list(range(n)) + [n + 5])
    torch.cuda.synchronize()
    assert bad[:n].sum().item() == 0 and bad[n].item() == 1 and gc.status_word() == zf.DEV_BAD_PAGE_ID
    gc.status.zero_()
    d = gc.dir.cpu().numpy()
    comp, raw = np.argwhere(d == -1), np.argwhere(d >= 0)
    assert len(comp) > 10 and len(raw) > 0
    rng = np.random.default_rng(5)
    nblk = gc.page_size // 4
    for p, h in comp[rng.choice(len(comp), 8, replace=False)]:
        pool = gc.k_comp if rng.integers(2) else gc.v_comp
        at = int(rng.integers(nblk)) * 784 + int(rng.integers(768, 784))
        pool[p, h, at] = int(rng.integers(256))
    p, h = comp[rng.integers(len(comp))]
    gc.k_comp[p, h, 768] = 127                             # b/2 = 127: any nonzero offset carries
    gc.k_comp[p, h, 512] = 0x01
    p, h = raw[0]
    gc.dir[p, h] = gc.num_raw_slots + 3
    bad = zf.validate_pages(gc, list(range(n)))
    torch.cuda.synchronize()
    kc, vc, dd = gc.k_comp.cpu().numpy(), gc.v_comp.cpu().numpy(), gc.dir.cpu().numpy()
    want = np.zeros(n, np.int32)
    kinds = 0
    for pid in range(n):
        for hh in range(gc.num_kv_heads):
            e = dd[pid, hh]
            if e == -1:
                for rec in (kc[pid, hh], vc[pid, hh]):
                    for b in range(nblk):
                        try:
                            O.decode_block(rec[b * 784:(b + 1) * 784], "k")
                        except ValueError:
                            want[pid] = 1
                            kinds |= zf.DEV_BAD_SLOT
            elif not 0 <= e < gc.num_raw_slots:
                want[pid] = 1
                kinds |= zf.DEV_BAD_DIR
    assert want.sum() >= 3 and kinds == zf.DEV_BAD_SLOT | zf.DEV_BAD_DIR
    assert (bad.cpu().numpy() == want).all()
    assert gc.status_word() == kinds
