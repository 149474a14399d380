"""Pins for the oracle's block codec (CPU only).

Each check ties the oracle to something other than itself: the format rules of ZipFusion §III.B
(eligibility window, 12-bit value code, 768-byte payload), hand-derived golden blocks, exhaustive
enumeration of all 65,536 BF16 patterns, and the no-carry property of ZipFusion §III.C.
"""
import glob
import os

import numpy as np
import pytest

from oracle import zf_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bits(x):
    """float32 values that are exactly representable in BF16 -> BF16 bit patterns."""
    return (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def pattern(s, e, f):
    return np.uint16((s << 15) | (e << 7) | f)


# ----------------------------------------------------------------------------- storage order
def test_storage_order_is_a_bijection():
    for role in "kv":
        assert sorted(O.storage_order(role).ravel()) == list(range(512))


def test_fragment_cells_match_hand_listed_ptx_table():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "mma_a_fragment.txt")) if l.strip() and not l.startswith("#")]
    assert len(rows) == 24
    for lane, r, row, col in (map(int, x) for x in rows):
        assert O.fragment_cell(lane, r) == (row, col)


def test_raw_order_is_the_half_major_storage_order():
    x = np.arange(512, dtype=np.uint16)
    r = O.to_raw_order(x)
    for lane in (0, 5, 31):
        for half in (0, 1):
            assert (r[256 * half + 8 * lane:256 * half + 8 * lane + 8] == x[16 * lane + 8 * half:16 * lane + 8 * half + 8]).all()
    assert (O.from_raw_order(r) == x).all()


def test_key_and_value_orders_differ_and_transpose():
    k, v = O.storage_order("k"), O.storage_order("v")
    assert (k != v).any()
    # within a 16x16 half the value order is the key order of the transposed tile
    for half in range(2):
        kh = k[:, 16 * half:16 * half + 16]
        vh = v[:, 16 * half:16 * half + 16]
        assert (vh.T == kh).all()


# ----------------------------------------------------------------------------- golden blocks
def _load_golden(path):
    role, fill, sets, exp = None, None, [], {"lo": {}, "codes": {}, "escape": {}}
    for line in open(path):
        line = line.split("#")[0].strip()
        if not line:
            continue
        w = line.split()
        if w[0] == "role":
            role = w[1]
        elif w[0] == "fill":
            fill = int(w[1], 16)
        elif w[0] == "set":
            sets.append((int(w[1]), int(w[2]), int(w[3], 16)))
        elif w[0] == "expect":
            if w[1] == "raw":
                exp["raw"] = True
            elif w[1] == "header":
                exp["header"] = int(w[2], 16)
            elif w[2] == "fill":
                exp[w[1] + "_fill"] = int(w[3], 16)
            else:
                exp[w[1]][int(w[2])] = int(w[3], 16)
    block = np.full((16, 32), fill, np.uint16)
    for t, g, v in sets:
        block[t, g] = v
    return role, block, exp


GOLDEN_BLOCKS = sorted(glob.glob(os.path.join(GOLDEN, "block_*.txt")))


@pytest.mark.parametrize("path", GOLDEN_BLOCKS, ids=os.path.basename)
def test_golden_block(path):
    role, block, exp = _load_golden(path)
    slot = O.encode_block(block, role)
    if exp.get("raw"):
        assert slot is None
        return
    assert slot is not None
    want = np.zeros(784, np.uint8)
    want[0:512] = exp.get("lo_fill", 0)
    for p, v in exp["lo"].items():
        want[p] = v
    want[512:768] = exp.get("codes_fill", 0)
    for i, v in exp["codes"].items():
        want[512 + i] = v
    want[768:772] = np.frombuffer(exp["header"].to_bytes(4, "little"), np.uint8)
    for i, v in exp["escape"].items():
        want[772 + 2 * i:774 + 2 * i] = np.frombuffer(v.to_bytes(2, "little"), np.uint8)
    assert (slot == want).all(), np.nonzero(slot != want)
    assert (O.decode_block(slot, role) == block).all()


# ----------------------------------------------------------------------------- format rules
def test_eligible_block_payload_is_768_of_1024_bytes():
    """ZipFusion §III.B / Fig. 2: an eligible 512-value block takes 768 bytes instead of 1024
    (75%), excluding metadata: 512 retained low bytes followed by 256 bytes of packed codes."""
    assert O.BLOCK_VALUES == 512
    assert O.CODES_AT - O.LOW_AT == 512 and O.HEADER_AT - O.CODES_AT == 256
    assert O.HEADER_AT == 768 == 1024 * 3 // 4
    assert O.SLOT_BYTES == 768 + 4 + 2 * O.MAX_ESCAPES


def _random_blocks(seed, n):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        kind = i % 4
        if kind == 0:      # narrow window, any start
            e0 = int(rng.integers(0, 241))
            e = rng.integers(e0, e0 + 16, (16, 32))
        elif kind == 1:    # window of width 15..17
            e0 = int(rng.integers(0, 238))
            e = rng.integers(e0, e0 + int(rng.integers(15, 18)), (16, 32))
        elif kind == 2:    # Gaussian values with per-channel scales (the workloads' shape)
            x = (rng.standard_normal((16, 32)) * np.exp(0.5 * rng.standard_normal(32))).astype(np.float32)
            out.append((x.view(np.uint32) >> 16).astype(np.uint16))
            continue
        else:              # wide window: escapes
            e = rng.integers(0, 256, (16, 32))
        s = rng.integers(0, 2, (16, 32))
        f = rng.integers(0, 128, (16, 32))
        out.append(((s << 15) | (np.minimum(e, 255) << 7) | f).astype(np.uint16))
    return out


def test_window_rule_of_the_pages_when_it_fits():
    """When every exponent is in [b, b+15] with b = min rounded down to even, the block is encoded
    with exactly that base and no escapes; when it is not, escapes are used (or it is raw)."""
    for blk in _random_blocks(1, 400):
        _, e, _ = O.bf16_fields(blk)
        b = int(e.min()) & ~1
        fits = int(e.max()) <= b + 15
        for role in "kv":
            slot = O.encode_block(blk, role)
            if fits:
                assert slot is not None
                half, n_esc, _ = O.parse_header(slot)
                assert (half, n_esc) == (b // 2, 0)
            elif slot is not None:
                assert O.parse_header(slot)[1] > 0
            if slot is not None:
                assert (O.decode_block(slot, role) == blk).all()


def test_window_boundaries():
    blk = np.full((16, 32), pattern(0, 100, 5), np.uint16)
    blk[3, 7] = pattern(1, 115, 9)                 # range 15 from an even minimum: fits
    assert O.parse_header(O.encode_block(blk, "k"))[:2] == (50, 0)
    blk[:] = pattern(0, 110, 5)
    blk[0, 0:3] = pattern(0, 101, 1)               # range 15 from an odd minimum: b0 = 100 and
    blk[3, 7] = pattern(1, 116, 9)                 # 116 > 115, so the window moves up to [102, 117]
    half, n_esc, esc = O.parse_header(O.encode_block(blk, "k"))
    assert (half, n_esc) == (51, 3) and all(eh == 50 for _, eh in esc)
    assert (O.decode_block(O.encode_block(blk, "k"), "k") == blk).all()
    blk[:] = pattern(0, 108, 5)
    blk[5, 5] = pattern(0, 100, 0)                 # range 16 from an even minimum
    blk[0, 0] = pattern(0, 116, 0)
    half, n_esc, esc = O.parse_header(O.encode_block(blk, "v"))
    assert (half, n_esc) == (51, 1) and esc[0][1] == 50
    assert (O.decode_block(O.encode_block(blk, "v"), "v") == blk).all()
    blk[:] = pattern(0, 100, 5)
    blk[0, 0] = pattern(0, 116, 0)                 # 511 values below the moved window: raw
    assert O.encode_block(blk, "k") is None


def test_escape_count_limit():
    blk = np.full((16, 32), bits(1.0), np.uint16)
    for i in range(6):
        blk[i, i] = bits(2.0 ** -100)
    slot = O.encode_block(blk, "v")
    assert slot is not None and O.parse_header(slot)[1] == 6
    assert (O.decode_block(slot, "v") == blk).all()
    blk[6, 6] = bits(2.0 ** -90)
    assert O.encode_block(blk, "v") is None


# ----------------------------------------------------------------------------- exhaustive
def test_every_bf16_pattern_round_trips_in_window():
    """All 65,536 patterns: the 512 patterns with exponent in {E, E+1} (E even) fill one block
    exactly, which satisfies the pages' window rule with b = E."""
    rng = np.random.default_rng(7)
    seen = 0
    for E in range(0, 256, 2):
        vals = np.array([pattern(s, e, f) for s in (0, 1) for e in (E, E + 1) for f in range(128)], np.uint16)
        blk = rng.permutation(vals).reshape(16, 32)
        role = "kv"[(E // 2) % 2]
        slot = O.encode_block(blk, role)
        assert slot is not None
        assert O.parse_header(slot)[:2] == (E // 2, 0)
        assert (O.decode_block(slot, role) == blk).all()
        seen += len(np.unique(vals))
    assert seen == 65536


def test_every_low_exponent_pattern_round_trips_as_escape():
    """Every pattern with exponent < 240 also round-trips as one of 6 escapes of a block whose
    other values (exponents 240..255, including Inf/NaN patterns) fix the window at [240, 255]."""
    rng = np.random.default_rng(11)
    pats = np.array([pattern(s, e, f) for e in range(240) for s in (0, 1) for f in range(128)], np.uint16)
    pats = rng.permutation(pats)
    filler = np.array([pattern(s, e, f) for s in (0, 1) for e in range(240, 256) for f in range(128)], np.uint16)
    for i in range(0, len(pats), 6):
        chunk = pats[i:i + 6]
        vals = np.concatenate([chunk, rng.choice(filler, 512 - len(chunk), replace=False)])
        vals[-1] = pattern(0, 255, 1)          # keep the top exponent at 255
        blk = rng.permutation(vals).reshape(16, 32)
        role = "kv"[(i // 6) % 2]
        slot = O.encode_block(blk, role)
        half, n_esc, _ = O.parse_header(slot)
        assert half == 120 and n_esc == len(chunk)
        assert (O.decode_block(slot, role) == blk).all()


def test_special_values():
    specials = [0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0xFFFF, 0x0001, 0x807F, 0x7F7F]
    for sp in specials:
        blk = np.full((16, 32), sp, np.uint16)
        for role in "kv":
            slot = O.encode_block(blk, role)
            assert slot is not None and (O.decode_block(slot, role) == blk).all()
    zero = np.zeros((16, 32), np.uint16)
    assert O.parse_header(O.encode_block(zero, "k"))[:2] == (0, 0)
    neg_zero = np.full((16, 32), 0x8000, np.uint16)
    assert (O.decode_block(O.encode_block(neg_zero, "k"), "k") == 0x8000).all()


def test_high_byte_addition_never_carries():
    """ZipFusion §III.C: a 32-bit add of the replicated base restores four high bytes with no
    carry across bytes.  Exhaustive over b/2 in 0..127 and all 4-tuples of codes whose exponent
    high bits (b/2 + offset) stay a 7-bit field."""
    nib = np.arange(16, dtype=np.uint32)
    a, b, c, d = np.meshgrid(nib, nib, nib, nib, indexing="ij")
    quads = np.stack([a.ravel(), b.ravel(), c.ravel(), d.ravel()], axis=1)        # 65536 x 4
    byte = ((quads >> 3) << 7) | (quads & 7)                                      # sign | offset
    word = byte[:, 0] | (byte[:, 1] << 8) | (byte[:, 2] << 16) | (byte[:, 3] << 24)
    checked = 0
    for half in range(128):
        ok = ((quads & 7) + half <= 127).all(axis=1)
        w = word[ok] + np.uint32(half * 0x01010101)
        want = byte[ok] + half                                                    # per-byte sums
        got = np.stack([(w >> (8 * i)) & 0xFF for i in range(4)], axis=1)
        assert (got == want).all()
        assert ((got >> 7) == (quads[ok] >> 3)).all()                             # sign bit kept
        checked += int(ok.sum())
    assert checked > 8_000_000


def test_encoded_offsets_respect_the_no_carry_bound():
    for blk in _random_blocks(3, 200):
        for role in "kv":
            slot = O.encode_block(blk, role)
            if slot is None:
                continue
            half, _, _ = O.parse_header(slot)
            codes = np.concatenate([slot[512:768] & 0xF, slot[512:768] >> 4])
            assert ((codes & 7).astype(int) + half <= 127).all()


def test_malformed_headers_are_rejected():
    slot = O.encode_block(np.full((16, 32), bits(1.0), np.uint16), "k")
    for bad in (0x0100003F | 0x80, 0x0100003F | 0x0800, 0x0200003F, 0x0100073F):
        s = slot.copy()
        s[768:772] = np.frombuffer(bad.to_bytes(4, "little"), np.uint8)
        with pytest.raises(ValueError):
            O.decode_block(s, "k")


# ----------------------------------------------------------------------------- pages
def _page(rng, P, wide=False):
    x = rng.standard_normal((P, 128)).astype(np.float32)
    if wide:
        x[0, 0] = 2.0 ** 60
        x[1:8, 0] = 2.0 ** -60
    return ((x.view(np.uint32) + 0x8000) >> 16).astype(np.uint16)


@pytest.mark.parametrize("P", [16, 64])
def test_page_lifecycle(P):
    """ZipFusion §III.D: partial pages stay raw; a full page is compressed under the same page id;
    a page that cannot be encoded stays raw; raw storage needs a raw slot."""
    rng = np.random.default_rng(P)
    H = 2
    cache = O.Cache(num_pages=6, num_kv_heads=H, page_size=P, num_raw=3)
    src_k = np.stack([np.stack([_page(rng, P, wide=(i == 3 and h == 1)) for h in range(H)]) for i in range(5)])
    src_v = np.stack([np.stack([_page(rng, P) for h in range(H)]) for i in range(5)])
    page_ids = [4, 0, 2, 5, 1]
    n_valid = [P, P - 3, P, P, 1]
    raw_slots = [-1, 2, -1, 0, -1]
    O.encode_pages(cache, src_k, src_v, page_ids, n_valid, raw_slots)
    assert (cache.dir[4] == O.DIR_COMPRESSED).all()
    assert (cache.dir[0] == 2).all()                  # partial -> raw slot 2
    assert (cache.dir[2] == O.DIR_COMPRESSED).all()
    assert cache.dir[5, 0] == O.DIR_COMPRESSED and cache.dir[5, 1] == 0   # head 1 not encodable
    assert (cache.dir[1] == O.DIR_INVALID).all()      # partial with no raw slot
    assert cache.status == O.ST_BAD_RAW_SLOT
    assert (cache.dir[3] == O.DIR_INVALID).all()      # never written
    k, v = O.decompress(cache, page_ids)
    for i, pid in enumerate(page_ids):
        if pid == 1:
            assert (k[i] == 0).all()
            continue
        assert (k[i] == src_k[i]).all() and (v[i] == src_v[i]).all()
    forced = O.Cache(num_pages=6, num_kv_heads=H, page_size=P, num_raw=6)
    O.encode_pages(forced, src_k, src_v, page_ids, [P] * 5, list(range(5)), force_raw=True)
    assert (forced.dir[page_ids] == np.arange(5)[:, None]).all()


@pytest.mark.parametrize("P", [16, 64])
def test_appending_a_page_token_by_token_equals_encoding_it(P):
    """ZipFusion §III.D: a page fills uncompressed, a token at a time, and is compressed once
    full.  Appending its tokens one by one into a raw slot (starting from stale slot contents, or
    from a partial page that encode_pages stored raw) must leave exactly what encode_pages leaves
    for the same tokens: the first t tokens readable after t appends, and when full the same
    compressed slots (or the same raw record, for a page that cannot be encoded)."""
    rng = np.random.default_rng(100 + P)
    H = 2
    src_k = np.stack([np.stack([_page(rng, P, wide=(i == 2 and h == 0)) for h in range(H)]) for i in range(3)])
    src_v = np.stack([np.stack([_page(rng, P) for h in range(H)]) for i in range(3)])
    ref = O.Cache(num_pages=4, num_kv_heads=H, page_size=P, num_raw=3)
    O.encode_pages(ref, src_k, src_v, [3, 0, 1], [P, P, P], [0, 1, 2])
    app = O.Cache(num_pages=4, num_kv_heads=H, page_size=P, num_raw=3)
    app.k_raw[:] = rng.integers(0, 1 << 16, app.k_raw.shape, dtype=np.uint16)   # stale slot contents
    app.v_raw[:] = rng.integers(0, 1 << 16, app.v_raw.shape, dtype=np.uint16)
    k_start = 5                                         # page 0 starts as a 5-token partial page
    O.encode_pages(app, src_k[1:2], src_v[1:2], [0], [k_start], [1])
    assert (app.dir[0] == 1).all()
    for t in range(P):
        sel = [i for i in range(3) if not (i == 1 and t < k_start)]
        O.append_tokens(app, src_k[sel][:, :, t], src_v[sel][:, :, t], [[3, 0, 1][i] for i in sel], [t] * len(sel),
                        [[0, 1, 2][i] for i in sel])
        for i, pid in enumerate([3, 0, 1]):
            kv = O.read_page_head(app, pid, 0)
            assert (kv[0][: t + 1] == src_k[i, 0, : t + 1]).all() and (kv[1][: t + 1] == src_v[i, 0, : t + 1]).all()
            if t < P - 1:
                assert (app.dir[pid] == [0, 1, 2][i]).all()
    assert app.status == 0
    assert (app.dir == ref.dir).all()
    assert app.dir[1, 0] == 2 and app.dir[3, 0] == O.DIR_COMPRESSED     # the wide page head stays raw
    comp = ref.dir == O.DIR_COMPRESSED
    assert (app.k_comp[comp] == ref.k_comp[comp]).all() and (app.v_comp[comp] == ref.v_comp[comp]).all()
    assert (app.k_raw[2, 0] == ref.k_raw[2, 0]).all() and (app.v_raw[2, 0] == ref.v_raw[2, 0]).all()


def test_append_errors():
    P, H = 16, 2
    c = O.Cache(num_pages=2, num_kv_heads=H, page_size=P, num_raw=1)
    tok = np.zeros((1, H, 128), np.uint16)
    O.append_tokens(c, tok, tok, [2], [0], [0])
    assert c.status == O.ST_BAD_PAGE_ID and (c.dir == O.DIR_INVALID).all()
    c.dir[:] = 0
    O.append_tokens(c, tok, tok, [1], [P], [0])
    assert c.status & O.ST_BAD_N_VALID and (c.dir[1] == O.DIR_INVALID).all() and (c.dir[0] == 0).all()
    c.dir[:] = 0
    O.append_tokens(c, tok, tok, [0], [3], [1])
    assert c.status & O.ST_BAD_RAW_SLOT and (c.dir[0] == O.DIR_INVALID).all() and (c.dir[1] == 0).all()


def test_offsets_that_would_carry_are_rejected():
    """ZipFusion §III.C: high bytes are rebuilt by adding b/2 to 3-bit offsets with no carry into
    the sign bit, so b/2 + offset <= 127 for every code.  Exponents {254, 255} give b/2 = 127 with
    offset 0 only; a code with offset 1 there would carry and cannot come from any BF16 value."""
    top = O.encode_block(np.full((16, 32), pattern(0, 255, 5), np.uint16), "k")
    assert O.parse_header(top)[0] == 127
    s = top.copy()
    s[512 + 7] |= 0x10                                   # offset 1 in one high nibble
    with pytest.raises(ValueError):
        O.decode_block(s, "k")
    low = O.encode_block(np.full((16, 32), pattern(1, 200, 5), np.uint16), "k")
    s = low.copy()
    s[512:768] = 0x77                                    # offset 7 everywhere: 100 + 7 fits
    assert O.decode_block(s, "k").shape == (16, 32)
