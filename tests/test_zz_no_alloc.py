"""zf_decode_attn_static: decode attention for callers that cannot allocate device memory (for
example a plugin inside an engine that owns all device memory and offers no scratch hook).  It uses
the library's static scratch array instead of a caller workspace; its results must match
zf_decode_attn's.  This file is collected last on purpose."""
import numpy as np
import pytest
import torch

from decode_attention_compressed_gb300 import inputs as I
from tests import helpers as H

pytestmark = pytest.mark.gpu


def _close(a_out, a_lse, b_out, b_lse):
    a_out, b_out = a_out.cpu().double().numpy(), b_out.cpu().double().numpy()
    a_lse, b_lse = a_lse.cpu().double().numpy(), b_lse.cpu().double().numpy()
    assert (np.isneginf(a_lse) == np.isneginf(b_lse)).all()
    d = np.abs(a_out - b_out)
    finite = ~np.isneginf(b_lse)
    dl = np.abs(a_lse[finite] - b_lse[finite]) if finite.any() else np.zeros(1)
    assert d.max() <= H.MAX_ABS and d.mean() <= H.MEAN_ABS and dl.max() <= H.LSE_ABS


def test_static_scratch_entry_point_matches_the_workspace_one():
    zf = H.zf_module()
    cases = [
        (I.scaled(I.WORKLOADS["qwen2_7b_maxbatch"], batch=6, ctx=900), None),
        (I.scaled(I.WORKLOADS["llama3_8b_batched"], batch=5, ctx=700, ctx_min=1), [700, 0, 33, 512, 1]),
    ]
    runs = []
    for w, lens in cases:
        layer = I.make_layer(w, seq_lens=lens)
        cache = H.gpu_cache_from(layer, zf)
        q, table, sl = layer.q.cuda(), layer.page_table.cuda(), layer.seq_lens.cuda()
        ref = zf.decode_attn(cache, q, table, sl, layer.scale)
        runs.append((cache, q, table, sl, layer.scale, ref))
    torch.cuda.synchronize()
    # two calls in a row through the C ABI, each checked against zf_decode_attn
    outs = [zf.decode_attn_static(c, q, t, s, sc) for c, q, t, s, sc, _ in runs]
    torch.cuda.synchronize()
    for (c, *_, ref), got in zip(runs, outs):
        _close(got[0], got[1], ref[0], ref[1])
        assert c.status_word() == 0


def test_sizes_beyond_the_static_scratch_are_rejected():
    zf = H.zf_module()
    cache = zf.Cache(4, 1, 16, 4)
    B, Hq, max_pages = 4096, 64, 4                    # partials need > 32 MiB
    assert zf.workspace_size(B, Hq, 1, 16, max_pages) > zf.STATIC_WORKSPACE_BYTES
    q = torch.zeros((B, Hq, 128), dtype=torch.int16, device="cuda")
    table = torch.zeros((B, max_pages), dtype=torch.int32, device="cuda")
    lens = torch.zeros(B, dtype=torch.int32, device="cuda")
    with pytest.raises(zf.ZfError, match="static workspace"):
        zf.decode_attn_static(cache, q, table, lens)
