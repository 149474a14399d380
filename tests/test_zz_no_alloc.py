"""zf_decode_attn_static: decode attention for callers that cannot allocate device memory (for
example a plugin inside an engine that owns all device memory through its own pool and offers no
scratch hook, or a latency-critical path where cudaMalloc's implicit synchronisation is not
allowed).  It uses the library's static scratch array instead of a caller workspace; its results
must equal zf_decode_attn's bit for bit and meet the oracle's bars.

The file name sorts last so that a `pytest -x` run which stops at a failure here has already run
every other test.  Nothing here depends on that order: the first case runs in a fresh process, where
the static call is the process's first attention call (so its address lookup is the one that loads
the library's device code), and the cases in this process pass whether or not other tests ran
before them."""
import os
import subprocess
import sys
import textwrap

import pytest
import torch

from decode_attention_compressed_gb300 import inputs as I
from oracle import zf_oracle as O
from tests import helpers as H

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CASES = [
    (I.scaled(I.WORKLOADS["qwen2_7b_maxbatch"], batch=6, ctx=900), None),
    (I.scaled(I.WORKLOADS["llama3_8b_batched"], batch=5, ctx=700, ctx_min=1), [700, 0, 33, 512, 1]),
]


def test_static_call_first_in_a_fresh_process():
    """A new process whose first attention call is the static one: the address lookup loads the
    module there.  Two static calls in a row, each bit-identical to zf_decode_attn."""
    H.zf_module()                  # build here, so the child only loads the library
    code = textwrap.dedent("""
        import sys, torch
        sys.path.insert(0, %r)
        from decode_attention_compressed_gb300 import inputs as I, zf
        from tests import helpers as H
        w = I.scaled(I.WORKLOADS["qwen2_7b_maxbatch"], batch=3, ctx=500)
        layer = I.make_layer(w)
        cache = H.gpu_cache_from(layer, zf)
        q, t, s = layer.q.cuda(), layer.page_table.cuda(), layer.seq_lens.cuda()
        a = zf.decode_attn_static(cache, q, t, s, layer.scale)
        b = zf.decode_attn_static(cache, q, t, s, layer.scale)
        ref = zf.decode_attn(cache, q, t, s, layer.scale)
        torch.cuda.synchronize()
        ok = all(torch.equal(x[0], ref[0]) and torch.equal(x[1], ref[1]) for x in (a, b))
        print("OK" if ok and cache.status_word() == 0 else "MISMATCH")
    """ % ROOT)
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    assert res.stdout.strip().endswith("OK"), res.stdout[-2000:]


def test_static_scratch_entry_point_matches_the_workspace_one():
    zf = H.zf_module()
    runs = []
    for w, lens in CASES:
        layer = I.make_layer(w, seq_lens=lens)
        cache = H.gpu_cache_from(layer, zf)
        q, table, sl = layer.q.cuda(), layer.page_table.cuda(), layer.seq_lens.cuda()
        ref = zf.decode_attn(cache, q, table, sl, layer.scale)
        runs.append((layer, cache, q, table, sl, ref))
    torch.cuda.synchronize()
    # two calls in a row through the C ABI (the second finds the first one's partials in the
    # array), each equal to zf_decode_attn bit for bit and within the oracle's bars
    outs = [zf.decode_attn_static(c, q, t, s, lay.scale) for lay, c, q, t, s, _ in runs]
    torch.cuda.synchronize()
    for (layer, c, *_, ref), got in zip(runs, outs):
        assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])
        assert c.status_word() == 0
        oc = H.oracle_cache_from(layer, O)
        ref_out, ref_lse = O.decode_attention(H.np_bits(layer.q), oc, layer.page_table.numpy(),
                                              layer.seq_lens.numpy(), layer.scale)
        H.compare_attention(got[0], got[1], ref_out, ref_lse)


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
