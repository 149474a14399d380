"""The pins have teeth: plant a plausible mistake in the oracle (on the CPU, via monkeypatch) and
check that at least one pin fails."""
import math

import numpy as np
import pytest

import tests.test_oracle_attention as TA
import tests.test_oracle_codec as TC
from oracle import zf_oracle as O


def _fails(fn, *args):
    with pytest.raises((AssertionError, ValueError, TypeError, IndexError)):
        fn(*args)


def test_base_not_rounded_to_even_is_caught(monkeypatch):
    def bad_base(e):
        emin, emax = int(e.min()), int(e.max())
        b = emin if emax <= emin + 15 else emax - 15
        return b, np.nonzero(e < b)[0]
    monkeypatch.setattr(O, "block_base", bad_base)
    _fails(TC.test_window_rule_of_the_pages_when_it_fits)


def test_swapped_nibble_pairing_is_caught(monkeypatch):
    real = O.encode_block

    def bad_encode(block, role):
        slot = real(block, role)
        if slot is not None:
            c = slot[512:768].copy()
            slot[512:768] = ((c & 0xF) << 4) | (c >> 4)
        return slot
    monkeypatch.setattr(O, "encode_block", bad_encode)
    _fails(TC.test_golden_block, [p for p in TC.GOLDEN_BLOCKS if "block_k_escape" in p][0])


def test_transposed_value_order_is_caught(monkeypatch):
    monkeypatch.setitem(O._ORDER, "v", O.storage_order("k"))
    _fails(TC.test_golden_block, [p for p in TC.GOLDEN_BLOCKS if "block_v" in p][0])


def test_dropped_escape_patch_is_caught(monkeypatch):
    real = O.parse_header
    monkeypatch.setattr(O, "parse_header", lambda slot: real(slot)[:2] + ([],))
    _fails(TC.test_every_low_exponent_pattern_round_trips_as_escape)


def test_log2_lse_is_caught(monkeypatch):
    real = O.attention_one

    def bad(q, K, V, scale):
        out, lse, w = real(q, K, V, scale)
        return out, lse / math.log(2), w
    monkeypatch.setattr(O, "attention_one", bad)
    _fails(TA.test_brute_force_50_digits, 3, 8)


def test_missing_scale_is_caught(monkeypatch):
    real = O.attention_one
    monkeypatch.setattr(O, "attention_one", lambda q, K, V, scale: real(q, K, V, 1.0))
    _fails(TA.test_brute_force_50_digits, 5, 3)


def test_keys_used_as_values_is_caught(monkeypatch):
    real = O.attention_one
    monkeypatch.setattr(O, "attention_one", lambda q, K, V, scale: real(q, K, K, scale))
    _fails(TA.test_one_token_returns_v_exactly)


def test_wrong_gqa_mapping_is_caught(monkeypatch):
    def bad_dense(q_bits, k_seqs, v_seqs, scale):
        B, Hq, D = q_bits.shape
        q = O.bf16_to_f64(q_bits)
        out = np.zeros((B, Hq, D))
        lse = np.zeros((B, Hq))
        for b in range(B):
            K, V = O.bf16_to_f64(k_seqs[b]), O.bf16_to_f64(v_seqs[b])
            for h in range(Hq):
                g = h % K.shape[1]
                out[b, h], lse[b, h], _ = O.attention_one(q[b, h], K[:, g], V[:, g], scale)
        return out, lse
    monkeypatch.setattr(O, "attention_dense", bad_dense)
    _fails(TA.test_gqa_equals_mha_with_repeated_heads)


def test_merge_without_renormalisation_is_caught(monkeypatch):
    def bad_merge(outs, lses):
        return np.mean(np.asarray(outs), axis=0), float(np.max(lses))
    monkeypatch.setattr(O, "merge_partials", bad_merge)
    _fails(TA.test_split_merge_equals_unsplit)


def test_multi_token_off_by_one_is_caught(monkeypatch):
    """Token t seeing one position fewer than its own (a causal limit of L - T + t, exclusive)."""
    real = O.attention_one

    def drop_last(q, K, V, scale):
        return real(q, K[:-1], V[:-1], scale) if len(K) else real(q, K, V, scale)

    def bad_multi(q_bits, cache, page_table, seq_lens, scale, pairs=None):
        monkeypatch.setattr(O, "attention_one", drop_last)
        try:
            return real_multi(q_bits, cache, page_table, seq_lens, scale, pairs)
        finally:
            monkeypatch.setattr(O, "attention_one", real)
    real_multi = O.decode_attention_multi
    monkeypatch.setattr(O, "decode_attention_multi", bad_multi)
    _fails(TA.test_multi_token_identical_keys_give_mean_of_the_visible_values)


def test_append_with_swapped_k_and_v_is_caught(monkeypatch):
    real = O.append_tokens
    monkeypatch.setattr(O, "append_tokens", lambda c, k, v, *rest: real(c, v, k, *rest))
    _fails(TC.test_appending_a_page_token_by_token_equals_encoding_it, 16)


def test_append_that_never_compresses_is_caught(monkeypatch):
    real = O.encode_page_head
    monkeypatch.setattr(O, "append_tokens", _append_without_step_2(real))
    _fails(TC.test_appending_a_page_token_by_token_equals_encoding_it, 16)


def _append_without_step_2(encode_page_head):
    def bad(cache, k_tok, v_tok, page_ids, positions, raw_slots):
        P = cache.page_size
        for i, pid in enumerate(page_ids):
            pos, slot = int(positions[i]), int(raw_slots[i])
            for h in range(cache.num_kv_heads):
                k, v = O.decode_page_head("raw", cache.k_raw[slot, h], cache.v_raw[slot, h], P)
                k[pos], v[pos] = k_tok[i, h], v_tok[i, h]
                _, cache.k_raw[slot, h], cache.v_raw[slot, h] = encode_page_head(k, v, pos + 1, force_raw=True)
                cache.dir[int(pid), h] = slot
    return bad


def test_sign_dropping_bf16_widening_is_caught(monkeypatch):
    """A widening that loses the sign bit passes every attention pin (both sides of each go through
    it); the BF16 pins catch it."""
    import tests.test_oracle_bf16 as TB
    real = O.bf16_to_f64
    monkeypatch.setattr(O, "bf16_to_f64", lambda x: real(np.asarray(x, dtype=np.uint16) & np.uint16(0x7FFF)))
    _fails(TB.test_hand_listed_patterns)
    _fails(TB.test_every_pattern_matches_an_independent_field_decode)


def test_bf16_widening_with_a_shifted_exponent_is_caught(monkeypatch):
    import tests.test_oracle_bf16 as TB
    real = O.bf16_to_f64
    monkeypatch.setattr(O, "bf16_to_f64", lambda x: real(x) * 2.0)
    _fails(TB.test_hand_listed_patterns)
