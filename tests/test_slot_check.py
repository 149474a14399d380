"""zf_slot_is_valid (host entry of the metadata check zf_validate_pages runs on the device)
against the oracle's block decoder: both accept exactly the same slots, over encoded blocks and
thousands of random corruptions of their header, escape and code bytes.  CPU only."""
import numpy as np
import pytest

from oracle import zf_oracle as O
from tests import helpers as H
from tests.test_oracle_codec import _random_blocks


@pytest.fixture(scope="module")
def zf():
    return H.zf_module()


def _oracle_ok(slot):
    try:
        O.decode_block(slot, "k")
        return True
    except ValueError:
        return False


def test_host_slot_check_agrees_with_the_oracle(zf):
    rng = np.random.default_rng(11)
    slots = [s for s in (O.encode_block(b, "kv"[i % 2]) for i, b in enumerate(_random_blocks(3, 60))) if s is not None]
    assert len(slots) > 20
    n_ok = n_bad = 0
    for _ in range(4000):
        s = slots[rng.integers(len(slots))].copy()
        kind = rng.integers(6)
        if kind == 0:                                   # one random header byte
            s[768 + rng.integers(4)] = rng.integers(256)
        elif kind == 1:                                 # one header bit
            bit = int(rng.integers(32))
            s[768 + bit // 8] ^= 1 << (bit % 8)
        elif kind == 2:                                 # escape count and entries
            s[769] = rng.integers(8)
            s[772:784] = rng.integers(0, 256, 12)
        elif kind == 3:                                 # ascending escapes, count matching
            k = int(rng.integers(0, 7))
            pos = np.sort(rng.choice(512, k, replace=False))
            if k and rng.integers(2):
                pos[-1] = pos[0]                        # a repeat
            s[769] = k
            s[772:784] = 0
            for j, p in enumerate(pos):
                e = (int(p) << 7) | int(rng.integers(128))
                s[772 + 2 * j:774 + 2 * j] = [e & 0xFF, e >> 8]
        elif kind == 4:                                 # high base, random codes: carries
            s[768] = rng.integers(118, 128)
            s[512:768] = rng.integers(0, 256, 256) & rng.integers(0, 256, 256) & 0x33
        want = _oracle_ok(s)
        assert zf.slot_is_valid(s.tobytes()) == want, (kind, s[768:784])
        n_ok += want
        n_bad += not want
    assert n_ok > 500 and n_bad > 500
