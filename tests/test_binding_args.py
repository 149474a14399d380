"""The Python binding's argument checks (CPU only, no kernel is launched): the C ABI receives bare
pointers, so dtype, device, shape and layout of every tensor are checked before a call reaches it,
and a mismatch raises instead of letting a kernel read the wrong bytes."""
import pytest
import torch

from tests import helpers as H


@pytest.fixture(scope="module")
def zf():
    return H.zf_module()


def _attn_inputs():
    q = torch.zeros(3, 8, 128, dtype=torch.int16)
    table = torch.zeros(3, 4, dtype=torch.int32)
    lens = torch.zeros(3, dtype=torch.int32)
    return q, table, lens


@pytest.mark.parametrize("entry", ["decode_attn", "dense_decode_attn", "decode_attn_static"])
def test_attention_arguments_are_checked(zf, entry):
    c = zf.Cache(8, 2, 16, 8, device="cpu")
    f = getattr(zf, entry)
    q, table, lens = _attn_inputs()
    cases = [
        ((q.float(), table, lens), {}, "q: dtype"),
        ((q[..., :64], table, lens), {}, "q: shape"),
        ((q.to("meta"), table, lens), {}, "q is on meta"),
        ((q, table.long(), lens), {}, "page_table: dtype"),
        ((q, table[:2], lens), {}, "page_table: 2 rows"),
        ((q, table[0], lens), {}, "page_table: shape"),
        ((q, table, lens[:2]), {}, "seq_lens: 2 rows"),
        ((q, table, lens.long()), {}, "seq_lens: dtype"),
        ((q, table, lens), dict(out=torch.zeros(3, 8, 64)), "out: shape"),
        ((q, table, lens), dict(out=torch.zeros(3, 128, 8).transpose(1, 2)), "contiguous"),
        ((q, table, lens), dict(lse=torch.zeros(3, 8, dtype=torch.float64)), "lse: dtype"),
        ((q, table, lens), dict(lse=torch.zeros(3, 9)), "lse: shape"),
    ]
    for args, kw, msg in cases:
        with pytest.raises(ValueError, match=msg):
            f(c, *args, 0.1, **kw)
    with pytest.raises(TypeError):
        f(c, q.numpy(), table, lens, 0.1)


def test_multi_token_attention_arguments_are_checked(zf):
    c = zf.Cache(8, 2, 16, 8, device="cpu")
    q = torch.zeros(3, 2, 8, 128, dtype=torch.int16)
    _, table, lens = _attn_inputs()
    with pytest.raises(ValueError, match="q: shape"):
        zf.decode_attn_multi(c, q[:, 0], table, lens, 0.1)
    with pytest.raises(ValueError, match="page_table: 2 rows"):
        zf.decode_attn_multi(c, q, table[:2], lens, 0.1)
    with pytest.raises(ValueError, match="out: shape"):
        zf.decode_attn_multi(c, q, table, lens, 0.1, out=torch.zeros(3, 8, 128))
    with pytest.raises(ValueError, match="lse: shape"):
        zf.decode_attn_multi(c, q, table, lens, 0.1, lse=torch.zeros(3, 8, 2))


def test_encode_and_append_arguments_are_checked(zf):
    c = zf.Cache(8, 2, 16, 8, device="cpu")
    src = torch.zeros(2, 2, 16, 128, dtype=torch.int16)
    with pytest.raises(ValueError, match="src_k: shape"):
        zf.encode_pages(c, torch.zeros(2, 3, 16, 128, dtype=torch.int16), src, [0, 1], [16, 16])
    with pytest.raises(ValueError, match="src_k: shape"):
        zf.encode_pages(c, torch.zeros(2, 2, 32, 128, dtype=torch.int16), src, [0, 1], [16, 16])
    with pytest.raises(ValueError, match="src_v: shape"):
        zf.encode_pages(c, src, src[:1], [0, 1], [16, 16])
    with pytest.raises(ValueError, match="src_v: dtype"):
        zf.encode_pages(c, src, src.float(), [0, 1], [16, 16])
    with pytest.raises(ValueError, match="page_ids: 1 entries"):
        zf.encode_pages(c, src, src, [0], [16, 16])
    with pytest.raises(ValueError, match="n_valid: 3 entries"):
        zf.encode_pages(c, src, src, [0, 1], torch.tensor([16, 16, 16]))
    with pytest.raises(ValueError, match="raw_slots: 1 entries"):
        zf.encode_pages(c, src, src, [0, 1], [16, 16], [0])
    tok = torch.zeros(2, 2, 128, dtype=torch.int16)
    with pytest.raises(ValueError, match="k_tok: shape"):
        zf.append_tokens(c, torch.zeros(2, 2, 64, dtype=torch.int16), tok, [0, 1], [0, 0], [0, 1])
    with pytest.raises(ValueError, match="v_tok: shape"):
        zf.append_tokens(c, tok, tok[:1], [0, 1], [0, 0], [0, 1])
    with pytest.raises(ValueError, match="positions: 1 entries"):
        zf.append_tokens(c, tok, tok, [0, 1], [0], [0, 1])
    with pytest.raises(ValueError, match="k_tok is on meta"):
        zf.append_tokens(c, tok.to("meta"), tok, [0, 1], [0, 0], [0, 1])
