"""GPU parity of zf_decode_attn and zf_dense_decode_attn against the float64 oracle.

Bars (float32 kernel vs float64 oracle on the same BF16 inputs): max-abs 4e-3 and mean-abs 5e-4
on `out`, 1e-3 on `lse`; empty contexts give out = 0 and lse = -inf exactly.
Small cases compare every output; the full-size workloads, run in the benchmark's launch
configuration, compare sampled (request, head) outputs that the oracle computes one by one.
"""
import math

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


def W(B, hq, hkv, P, ctx, **kw):
    return I.Workload("case", B, hq, hkv, P, ctx, **kw)


CASES = {
    "one_token": (W(1, 8, 2, 16, 1), [1]),
    "ragged_gqa4": (W(2, 8, 2, 16, 67, pool="random", seed=3), [17, 67]),
    "mha": (W(3, 4, 4, 16, 33, seed=4), [33, 16, 5]),
    "gqa7_spikes": (W(3, 14, 2, 16, 300, pool="random", k_sigma=0.7, n_outlier=0, spike_prob=0.02,
                      v_std=0.5, seed=5), [300, 48, 1]),
    "gqa8": (W(2, 16, 2, 16, 200, seed=6), [200, 129]),
    "gqa12_two_slices": (W(2, 24, 2, 16, 150, pool="random", seed=7), [150, 31]),
    "gqa1_page64": (W(3, 2, 2, 64, 260, pool="random", seed=8), [260, 65, 7]),
    "page64_gqa4": (W(2, 16, 4, 64, 700, pool="random", seed=9), [700, 129]),
    "empty_requests": (W(4, 8, 2, 16, 40, seed=10), [0, 40, 0, 3]),
    "long_chunked": (W(1, 8, 1, 16, 3000, seed=11), [3000]),
    # more (request, kv head) pairs than SMs: the planner takes balanced page ranges, so ranges
    # cross request boundaries and skip empty requests
    "balanced_ragged": (W(40, 8, 4, 16, 1024, pool="random", seed=12),
                        [0 if i in (3, 17) else 1024 if i == 5 else (37 * i * i + 11 * i) % 1025 for i in range(40)]),
    # GQA 16 (two 8-head slices per kv head) with balanced ranges
    "balanced_two_slices": (W(48, 32, 2, 16, 1024, pool="random", seed=16),
                            [0 if i % 11 == 4 else (53 * i * i + 7 * i + 1) % 1025 for i in range(48)]),
    # other page sizes: 2, 3 and 8 tiles per page (items cut at 128, 85 and 32 pages)
    "page32_ragged": (W(5, 8, 2, 32, 900, pool="random", seed=13), [900, 0, 33, 511, 64]),
    "page48_gqa2": (W(3, 4, 2, 48, 500, pool="random", seed=14), [500, 47, 49]),
    "page128_gqa16": (W(2, 32, 2, 128, 1000, pool="random", seed=15), [1000, 129]),
}


def _run(zf, layer, cache, dense=False):
    dev = torch.device("cuda")
    q = layer.q.to(dev)
    table = layer.page_table.to(dev)
    lens = layer.seq_lens.to(dev)
    out, lse = (zf.dense_decode_attn if dense else zf.decode_attn)(cache, q, table, lens, layer.scale)
    torch.cuda.synchronize()
    return out, lse


def _oracle(layer):
    oc = H.oracle_cache_from(layer, O)
    return O.decode_attention(H.np_bits(layer.q), oc, layer.page_table.numpy(), layer.seq_lens.numpy(), layer.scale)


@pytest.mark.parametrize("name", sorted(CASES))
def test_small_cases(zf, name):
    w, lens = CASES[name]
    layer = I.make_layer(w, seq_lens=lens)
    ref_out, ref_lse = _oracle(layer)
    gc = H.gpu_cache_from(layer, zf)
    out, lse = _run(zf, layer, gc)
    H.compare_attention(out, lse, ref_out, ref_lse)
    assert gc.status_word() == 0
    # each compressed kernel on its own, whichever the call would pick (the tensor-memory kernel
    # also for a single column per kv head: one of 16 MMA columns used)
    dev = torch.device("cuda")
    for kernel in ("warp_mma", "tcgen05"):
        o, l = zf.decode_attn(gc, layer.q.to(dev), layer.page_table.to(dev), layer.seq_lens.to(dev), layer.scale,
                              kernel=kernel)
        torch.cuda.synchronize()
        H.compare_attention(o, l, ref_out, ref_lse)
        assert gc.status_word() == 0, kernel
    dc = H.gpu_cache_from(layer, zf, force_raw=True)
    dout, dlse = _run(zf, layer, dc, dense=True)
    H.compare_attention(dout, dlse, ref_out, ref_lse)
    assert dc.status_word() == 0


def test_mixed_raw_and_compressed_pages(zf):
    """Full pages forced raw next to compressed ones and raw partial tails, in one request."""
    w = W(2, 12, 3, 16, 250, pool="random", seed=12)
    layer = I.make_layer(w, seq_lens=[250, 181])
    gc = H.gpu_cache_from(layer, zf)
    some = list(range(0, layer.num_pages, 3))
    zf.encode_pages(gc, layer.k_pages[some].cuda(), layer.v_pages[some].cuda(), some, [16] * len(some), some,
                    force_raw=True)
    torch.cuda.synchronize()
    d = gc.dir.cpu().numpy()
    assert (d == -1).any() and (d >= 0).any()
    ref_out, ref_lse = _oracle(layer)
    out, lse = _run(zf, layer, gc)
    H.compare_attention(out, lse, ref_out, ref_lse)


@pytest.mark.parametrize("kernel", ["warp_mma", "tcgen05"])
def test_deterministic(zf, kernel):
    for name in ("gqa7_spikes", "balanced_two_slices"):
        w, lens = CASES[name]
        layer = I.make_layer(w, seq_lens=lens)
        gc = H.gpu_cache_from(layer, zf)
        dev = torch.device("cuda")
        args = (gc, layer.q.to(dev), layer.page_table.to(dev), layer.seq_lens.to(dev), layer.scale)
        a = zf.decode_attn(*args, kernel=kernel)
        b = zf.decode_attn(*args, kernel=kernel)
        torch.cuda.synchronize()
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_one_workspace_across_calls_of_different_shapes(zf):
    """One workspace serves calls of different lengths and batch sizes (its contents between calls
    do not matter) and gives the same bits as fresh ones."""
    cases = [(W(3, 8, 2, 16, 900, pool="random", seed=21), [900, 333, 17]),
             (W(2, 14, 2, 16, 2000, pool="random", seed=22), [2000, 1999]),
             (W(3, 8, 2, 16, 900, pool="random", seed=21), [900, 333, 17])]
    ws = zf.new_workspace(max(zf.workspace_size(w.batch, w.num_q_heads, w.num_kv_heads, w.page_size, w.max_pages)
                              for w, _ in cases))
    for w, lens in cases:
        layer = I.make_layer(w, seq_lens=lens)
        gc = H.gpu_cache_from(layer, zf)
        q, t, sl = layer.q.cuda(), layer.page_table.cuda(), layer.seq_lens.cuda()
        shared = zf.decode_attn(gc, q, t, sl, layer.scale, workspace=ws)
        fresh = zf.decode_attn(gc, q, t, sl, layer.scale)
        torch.cuda.synchronize()
        assert torch.equal(shared[0], fresh[0]) and torch.equal(shared[1], fresh[1])
        ref_out, ref_lse = _oracle(layer)
        H.compare_attention(shared[0], shared[1], ref_out, ref_lse)


def test_bad_page_ids_are_reported_not_faulted(zf):
    w = W(2, 8, 2, 16, 64, seed=13)
    layer = I.make_layer(w, seq_lens=[64, 40])
    gc = H.gpu_cache_from(layer, zf)
    table = layer.page_table.clone()
    table[0, 1] = 10 ** 6
    table[1, 0] = -5
    out, lse = zf.decode_attn(gc, layer.q.cuda(), table.cuda(), layer.seq_lens.cuda(), layer.scale)
    torch.cuda.synchronize()
    assert gc.status_word() & zf.DEV_BAD_PAGE_ID
    assert torch.isfinite(out).all()
    lens = torch.tensor([64, 10 ** 6], dtype=torch.int32)
    gc.status.zero_()
    zf.decode_attn(gc, layer.q.cuda(), layer.page_table.cuda(), lens.cuda(), layer.scale)
    torch.cuda.synchronize()
    assert gc.status_word() & zf.DEV_BAD_SEQ_LEN


SMALL_WORKLOADS = {
    "tiny": (I.WORKLOADS["tiny"], None),
    "llama7b_mha": (I.scaled(I.WORKLOADS["llama7b_mha_512"], ctx=256), None),
    "llama3_8b_batched": (I.scaled(I.WORKLOADS["llama3_8b_batched"], batch=5, ctx=700, ctx_min=100), None),
    "qwen2_7b_maxbatch": (I.scaled(I.WORKLOADS["qwen2_7b_maxbatch"], batch=3, ctx=800), None),
    "long_ctx": (I.scaled(I.WORKLOADS["long_ctx"], batch=2, ctx=1500), [1500, 1473]),
}


@pytest.mark.parametrize("name", sorted(SMALL_WORKLOADS))
def test_workload_shapes_small(zf, name):
    w, lens = SMALL_WORKLOADS[name]
    layer = I.make_layer(w, seq_lens=lens)
    ref_out, ref_lse = _oracle(layer)
    gc = H.gpu_cache_from(layer, zf)
    out, lse = _run(zf, layer, gc)
    H.compare_attention(out, lse, ref_out, ref_lse)
    dc = H.gpu_cache_from(layer, zf, force_raw=True)
    H.compare_attention(*_run(zf, layer, dc, dense=True), ref_out, ref_lse)


# ------------------------------------------------------------------ full-size workloads, sampled
FULL = ["tiny", "llama7b_mha_512", "llama7b_mha_2048", "llama7b_mha_8192", "llama3_8b_batched",
        "qwen2_7b_maxbatch", "long_ctx"]


def sampled_reference(layer, pairs):
    """Oracle outputs for the sampled (request, query head) pairs, one by one, from the BF16
    source pages of that request and kv head."""
    w = layer.workload
    P, group = w.page_size, w.group
    table = layer.page_table.cpu().numpy()
    lens = layer.seq_lens.cpu().numpy()
    q = H.np_bits(layer.q)
    out = np.zeros((w.batch, w.num_q_heads, 128))
    lse = np.full((w.batch, w.num_q_heads), -math.inf)
    for b, h in pairs:
        L = int(lens[b])
        pages = torch.as_tensor(table[b, : -(-L // P)], dtype=torch.long, device=layer.k_pages.device)
        g = h // group
        K = H.np_bits(layer.k_pages[pages, g].reshape(-1, 128))[:L]
        V = H.np_bits(layer.v_pages[pages, g].reshape(-1, 128))[:L]
        out[b, h], lse[b, h], _ = O.attention_one(O.bf16_to_f64(q[b, h]), O.bf16_to_f64(K), O.bf16_to_f64(V),
                                                  layer.scale)
    return out, lse


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(zf, name):
    w = I.WORKLOADS[name]
    layer = I.make_layer(w, layer=0, device="cuda")
    npg = layer.num_pages
    # encode exactly as the benchmark does: page i keeps id i and may fall back to raw slot i
    gc = zf.Cache(npg, w.num_kv_heads, w.page_size, npg)
    zf.encode_pages(gc, layer.k_pages, layer.v_pages, list(range(npg)), layer.n_valid, list(range(npg)))
    out, lse = zf.decode_attn(gc, layer.q, layer.page_table, layer.seq_lens, layer.scale)
    torch.cuda.synchronize()
    assert gc.status_word() == 0
    # every request's first and last query head (the ends of its pairs' page ranges), plus 64 random
    # (request, head) rows: at least 64 rows, across the CTA ranges of the balanced split
    rng = np.random.default_rng(0)
    rows = w.batch * w.num_q_heads
    picked = rng.choice(rows, size=min(64, rows), replace=False)
    pairs = sorted({(int(i) // w.num_q_heads, int(i) % w.num_q_heads) for i in picked}
                   | {(b, h) for b in range(w.batch) for h in (0, w.num_q_heads - 1)})
    assert len(pairs) >= min(64, rows)
    ref_out, ref_lse = sampled_reference(layer, pairs)
    H.compare_attention(out, lse, ref_out, ref_lse, pairs=pairs)
    # properties at any size: finite, |out| bounded by max |v| of the request's head
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    # the dense comparator on the same inputs, same launch configuration
    dc = zf.Cache(npg, w.num_kv_heads, w.page_size, npg, compressed=False)
    zf.encode_pages(dc, layer.k_pages, layer.v_pages, list(range(npg)), layer.n_valid, list(range(npg)),
                    force_raw=True)
    dout, dlse = zf.dense_decode_attn(dc, layer.q, layer.page_table, layer.seq_lens, layer.scale)
    torch.cuda.synchronize()
    assert dc.status_word() == 0
    H.compare_attention(dout, dlse, ref_out, ref_lse, pairs=pairs)
    del dc, dout, dlse
    # the sampled pages decompress to their source bits
    sample_pages = sorted({int(x) for x in rng.integers(0, npg, 16)})
    k, v = zf.decompress(gc, sample_pages)
    idx = torch.as_tensor(sample_pages, device="cuda")
    assert torch.equal(k, layer.k_pages[idx]) and torch.equal(v, layer.v_pages[idx])


def test_back_to_back_calls_with_inputs_changed_between_them(zf):
    """Consecutive calls on one stream whose page table and lengths are rewritten in place between
    them (a shape where each call plans and prefetches its first tiles before the previous grid
    has finished): each call sees its own inputs."""
    w = W(2, 32, 32, 16, 2048, pool="random", seed=23)
    layer = I.make_layer(w, seq_lens=[2048, 2048])
    gc = H.gpu_cache_from(layer, zf)
    dev = torch.device("cuda")
    q = layer.q.to(dev)
    table_a, lens_a = layer.page_table.clone(), layer.seq_lens.clone()
    table_b = torch.flip(layer.page_table, dims=[0]).contiguous()   # the requests swap their pages
    lens_b = torch.tensor([1500, 77], dtype=lens_a.dtype)
    table_dev, lens_dev = table_a.to(dev), lens_a.to(dev)
    ws = zf.new_workspace(zf.workspace_size(w.batch, w.num_q_heads, w.num_kv_heads, w.page_size, w.max_pages))
    outs = []
    for table, lens in ((table_a, lens_a), (table_b, lens_b), (table_a, lens_a)):
        table_dev.copy_(table.to(dev), non_blocking=True)
        lens_dev.copy_(lens.to(dev), non_blocking=True)
        o, l = zf.decode_attn(gc, q, table_dev, lens_dev, layer.scale, workspace=ws)
        outs.append((o.clone(), l.clone()))
    torch.cuda.synchronize()
    assert gc.status_word() == 0
    oc = H.oracle_cache_from(layer, O)
    for (o, l), (table, lens) in zip(outs, ((table_a, lens_a), (table_b, lens_b), (table_a, lens_a))):
        ref_out, ref_lse = O.decode_attention(H.np_bits(layer.q), oc, table.numpy(), lens.numpy(), layer.scale)
        H.compare_attention(o, l, ref_out, ref_lse)
    assert torch.equal(outs[0][0], outs[2][0]) and torch.equal(outs[0][1], outs[2][1])


@pytest.mark.parametrize("tokens", [1, 4])
@pytest.mark.parametrize("dense", [False, True])
@pytest.mark.parametrize("change", ["lengths_and_table", "table_only", "nothing"])
def test_inputs_written_by_the_preceding_grid_after_it_lets_the_call_start(zf, change, dense, tokens):
    """A kernel ahead of the call lets it start at once and rewrites the page table (and lengths)
    about 200 us later: the call plans its first item from the old values while that kernel runs,
    and must compute from the new ones (the plan is dropped when anything it read has changed).
    With four new tokens per request the same holds for zf_decode_attn_multi."""
    w = W(2, 32, 32, 16, 2048, pool="random", seed=29)
    layer = I.make_layer(w, seq_lens=[2048, 2048])
    gc = H.gpu_cache_from(layer, zf, force_raw=dense)
    dev = torch.device("cuda")
    q_host = I.make_multi_queries(w, tokens) if tokens > 1 else layer.q
    q = q_host.to(dev)
    table_a, lens_a = layer.page_table.clone(), layer.seq_lens.clone()
    table_b, lens_b = table_a.clone(), lens_a.clone()
    if change != "nothing":
        table_b = torch.flip(table_a, dims=[0]).contiguous()      # the requests swap their pages
    if change == "lengths_and_table":
        lens_b = torch.tensor([1500, 77], dtype=lens_a.dtype)
    table_dev, lens_dev = table_a.to(dev), lens_a.to(dev)
    new_table, new_lens = table_b.to(dev), lens_b.to(dev)
    ws = zf.new_workspace(zf.workspace_size_multi(w.batch, tokens, w.num_q_heads, w.num_kv_heads, w.page_size,
                                                  w.max_pages))
    late_copy = H.late_writer()
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    assert late_copy(new_table.data_ptr(), table_dev.data_ptr(), table_dev.numel(), new_lens.data_ptr(),
                     lens_dev.data_ptr(), lens_dev.numel(), 200_000, stream.cuda_stream) == 0
    call = zf.decode_attn_multi if tokens > 1 else zf.decode_attn
    o, l = call(gc, q, table_dev, lens_dev, layer.scale, workspace=ws, dense=dense)
    torch.cuda.synchronize()
    assert gc.status_word() == 0
    oc = H.oracle_cache_from(layer, O, force_raw=dense)
    ref = O.decode_attention_multi if tokens > 1 else O.decode_attention
    ref_out, ref_lse = ref(H.np_bits(q_host), oc, table_b.numpy(), lens_b.numpy(), layer.scale)
    H.compare_attention(o, l, ref_out, ref_lse)


# ---- several new tokens per request (zf_decode_attn_multi): token t of T sees positions up to
# seq_len - T + t
MULTI_CASES = {
    "mha_t4": (W(2, 8, 8, 16, 300, pool="random", seed=41), [300, 77], 4),
    "gqa4_t2": (W(3, 8, 2, 16, 200, pool="random", seed=42), [200, 33, 17], 2),
    "gqa4_t3_two_slices": (W(2, 8, 2, 16, 180, seed=43), [180, 90], 3),
    "gqa7_t2_spikes": (W(2, 14, 2, 16, 250, pool="random", k_sigma=0.7, n_outlier=0, spike_prob=0.02, v_std=0.5,
                          seed=44), [250, 40], 2),
    "page64_t8": (W(2, 4, 4, 64, 400, pool="random", seed=45), [400, 129], 8),
    "tokens_that_see_nothing": (W(3, 4, 2, 16, 10, seed=46), [3, 1, 10], 4),
    "one_token": (W(2, 8, 2, 16, 100, seed=47), [100, 31], 1),
    # 32 columns per kv head (GQA 16 x 2 tokens): one tensor-memory pass, four warp-MMA passes
    "gqa16_t2": (W(3, 32, 2, 16, 700, pool="random", seed=48), [700, 129, 5], 2),
    # 16 columns from MHA x 16 tokens, 64-token pages, ragged
    "mha_t16_page64": (W(2, 2, 2, 64, 530, pool="random", seed=49), [530, 200], 16),
    # 40 columns: a 32-column slice and an 8-column slice
    "gqa20_t2_two_slices": (W(2, 40, 2, 16, 300, pool="random", seed=50), [300, 250], 2),
    # one new token, GQA 12: 12 columns, which AUTO gives the tensor-memory kernel
    "gqa12_t1": (W(2, 24, 2, 16, 333, pool="random", seed=51), [333, 50], 1),
}


@pytest.mark.parametrize("kernel", ["auto", "warp_mma", "tcgen05", "dense"])
@pytest.mark.parametrize("name", sorted(MULTI_CASES))
def test_multi_token_cases(zf, name, kernel):
    w, lens, T = MULTI_CASES[name]
    dense = kernel == "dense"
    layer = I.make_layer(w, seq_lens=lens)
    gc = H.gpu_cache_from(layer, zf, force_raw=dense)
    q = I.make_multi_queries(w, T)
    dev = torch.device("cuda")
    out, lse = zf.decode_attn_multi(gc, q.to(dev), layer.page_table.to(dev), layer.seq_lens.to(dev), layer.scale,
                                    dense=dense, kernel="auto" if dense else kernel)
    torch.cuda.synchronize()
    assert gc.status_word() == 0
    oc = H.oracle_cache_from(layer, O, force_raw=dense)
    ref_out, ref_lse = O.decode_attention_multi(H.np_bits(q), oc, layer.page_table.numpy(), layer.seq_lens.numpy(),
                                                layer.scale)
    H.compare_attention(out, lse, ref_out, ref_lse)
    if T == 1:   # the same bits as the single-token entry point
        o1, l1 = zf.decode_attn(gc, q[:, 0].contiguous().to(dev), layer.page_table.to(dev),
                                layer.seq_lens.to(dev), layer.scale, dense=dense,
                                kernel="auto" if dense else kernel)
        torch.cuda.synchronize()
        assert torch.equal(o1, out[:, 0]) and torch.equal(l1, lse[:, 0])


def test_multi_token_full_size_sampled(zf):
    """Four new tokens per request on the LLaMA-7B MHA 8K shape (one layer), in the benchmark's
    launch configuration; sampled (request, token, head) outputs against the float64 attention."""
    w = I.WORKLOADS["llama7b_mha_8192"]
    T = 4
    layer = I.make_layer(w, layer=0, device="cuda")
    npg = layer.num_pages
    gc = zf.Cache(npg, w.num_kv_heads, w.page_size, npg)
    zf.encode_pages(gc, layer.k_pages, layer.v_pages, list(range(npg)), layer.n_valid, list(range(npg)))
    q = I.make_multi_queries(w, T, device="cuda")
    out, lse = zf.decode_attn_multi(gc, q, layer.page_table, layer.seq_lens, layer.scale)
    torch.cuda.synchronize()
    assert gc.status_word() == 0
    picks = [(0, t, h) for t in range(T) for h in (0, 13, 31)]
    qn, table, lens = H.np_bits(q), layer.page_table.cpu().numpy(), layer.seq_lens.cpu().numpy()
    ref_out = np.zeros(tuple(out.shape))
    ref_lse = np.full(tuple(lse.shape), -math.inf)
    for b, t, h in picks:
        L = int(lens[b]) - T + t + 1
        pages = torch.as_tensor(table[b, : -(-L // w.page_size)], dtype=torch.long, device="cuda")
        K = H.np_bits(layer.k_pages[pages, h].reshape(-1, 128))[:L]
        V = H.np_bits(layer.v_pages[pages, h].reshape(-1, 128))[:L]
        ref_out[b, t, h], ref_lse[b, t, h], _ = O.attention_one(O.bf16_to_f64(qn[b, t, h]), O.bf16_to_f64(K),
                                                                O.bf16_to_f64(V), layer.scale)
    H.compare_attention(out, lse, ref_out, ref_lse, pairs=picks)


@pytest.mark.parametrize("name, kernel", [("gqa16_t2", "tcgen05"), ("gqa20_t2_two_slices", "tcgen05"),
                                          ("gqa7_t2_spikes", "tcgen05"), ("mha_t16_page64", "tcgen05"),
                                          ("gqa12_t1", "tcgen05"), ("gqa4_t2", "warp_mma"), ("page64_t8", "warp_mma")])
def test_auto_kernel_choice(zf, name, kernel):
    """ZF_KERNEL_AUTO runs the tensor-memory kernel above 8 columns per kv head and the warp-MMA
    kernel up to 8: its results are bit for bit those of the kernel it picks."""
    w, lens, T = MULTI_CASES[name]
    layer = I.make_layer(w, seq_lens=lens)
    gc = H.gpu_cache_from(layer, zf)
    q = I.make_multi_queries(w, T).cuda()
    table, sl = layer.page_table.cuda(), layer.seq_lens.cuda()
    auto = zf.decode_attn_multi(gc, q, table, sl, layer.scale)
    picked = zf.decode_attn_multi(gc, q, table, sl, layer.scale, kernel=kernel)
    torch.cuda.synchronize()
    assert torch.equal(auto[0], picked[0]) and torch.equal(auto[1], picked[1])


def test_batch_beyond_the_tensor_memory_kernel(zf):
    """A batch whose request lengths do not fit the tensor-memory kernel's shared memory (more than
    1379 requests at 16 columns): asked for by name it is refused before any launch; AUTO runs the
    warp-MMA kernel instead, bit for bit, and both match the oracle."""
    w = W(1500, 32, 2, 16, 40, ctx_min=1, pool="random", seed=52)        # 16 query heads per kv head
    layer = I.make_layer(w)
    gc = H.gpu_cache_from(layer, zf)
    q, table, sl = layer.q.cuda(), layer.page_table.cuda(), layer.seq_lens.cuda()
    with pytest.raises(zf.ZfError, match="unsupported"):
        zf.decode_attn(gc, q, table, sl, layer.scale, kernel="tcgen05")
    auto = zf.decode_attn(gc, q, table, sl, layer.scale)
    mma = zf.decode_attn(gc, q, table, sl, layer.scale, kernel="warp_mma")
    torch.cuda.synchronize()
    assert gc.status_word() == 0
    assert torch.equal(auto[0], mma[0]) and torch.equal(auto[1], mma[1])
    oc = H.oracle_cache_from(layer, O)
    ref_out, ref_lse = O.decode_attention(H.np_bits(layer.q), oc, layer.page_table.numpy(), layer.seq_lens.numpy(),
                                          layer.scale)
    H.compare_attention(auto[0], auto[1], ref_out, ref_lse)


@pytest.mark.parametrize("hq, limit", [(32, 1379), (64, 1363)])
def test_tensor_memory_kernel_batch_limit(zf, hq, limit):
    """The largest batch whose request lengths fit the tensor-memory kernel's shared memory: 1379
    requests at 16 columns per kv head, 1363 at 32.  At the limit the kernel runs (AUTO picks it, bit
    for bit) and matches the oracle; one request more is refused by name before any launch."""
    w = W(limit + 1, hq, 2, 16, 24, ctx_min=1, pool="random", seed=53)
    layer = I.make_layer(w)
    gc = H.gpu_cache_from(layer, zf)
    q, table, sl = layer.q.cuda(), layer.page_table.cuda(), layer.seq_lens.cuda()
    with pytest.raises(zf.ZfError, match="unsupported"):
        zf.decode_attn(gc, q, table, sl, layer.scale, kernel="tcgen05")
    q, table, sl = q[:limit], table[:limit], sl[:limit]
    tc = zf.decode_attn(gc, q, table, sl, layer.scale, kernel="tcgen05")
    auto = zf.decode_attn(gc, q, table, sl, layer.scale)
    torch.cuda.synchronize()
    assert gc.status_word() == 0
    assert torch.equal(auto[0], tc[0]) and torch.equal(auto[1], tc[1])
    oc = H.oracle_cache_from(layer, O)
    ref_out, ref_lse = O.decode_attention(H.np_bits(layer.q[:limit]), oc, layer.page_table[:limit].numpy(),
                                          layer.seq_lens[:limit].numpy(), layer.scale)
    H.compare_attention(tc[0], tc[1], ref_out, ref_lse)


@pytest.mark.parametrize("T", [2, 4])
def test_tcgen05_full_size_sampled(zf, T):
    """Two or four new tokens per request on the Qwen2-7B max-batch shape (GQA 7: 14 or 28
    columns per kv head, one 16- or 32-column pass), one layer in the benchmark's launch
    configuration: the tensor-memory kernel on sampled (request, token, head) outputs against
    float64 attention, and every output against the warp-MMA kernel."""
    w = I.WORKLOADS["qwen2_7b_maxbatch"]
    layer = I.make_layer(w, layer=0, device="cuda")
    npg = layer.num_pages
    gc = zf.Cache(npg, w.num_kv_heads, w.page_size, npg)
    zf.encode_pages(gc, layer.k_pages, layer.v_pages, list(range(npg)), layer.n_valid, list(range(npg)))
    q = I.make_multi_queries(w, T, device="cuda")
    ws = zf.new_workspace(zf.workspace_size_multi(w.batch, T, w.num_q_heads, w.num_kv_heads, w.page_size,
                                                  w.max_pages))
    out, lse = zf.decode_attn_multi(gc, q, layer.page_table, layer.seq_lens, layer.scale, workspace=ws,
                                    kernel="tcgen05")
    mo, ml = zf.decode_attn_multi(gc, q, layer.page_table, layer.seq_lens, layer.scale, workspace=ws,
                                  kernel="warp_mma")
    torch.cuda.synchronize()
    assert gc.status_word() == 0
    d = (out - mo).abs()
    assert float(d.max()) <= 2 * H.MAX_ABS and float(d.mean()) <= H.MEAN_ABS
    assert float((lse - ml).abs().max()) <= 2 * H.LSE_ABS
    rng = np.random.default_rng(7)
    picks = sorted({(int(rng.integers(w.batch)), t, int(rng.integers(w.num_q_heads))) for t in range(T) for _ in range(24)}
                   | {(0, 0, 0), (w.batch - 1, T - 1, w.num_q_heads - 1)})
    qn, table, lens = H.np_bits(q), layer.page_table.cpu().numpy(), layer.seq_lens.cpu().numpy()
    ref_out = np.zeros(tuple(out.shape))
    ref_lse = np.full(tuple(lse.shape), -math.inf)
    for b, t, h in picks:
        L = int(lens[b]) - T + t + 1
        pages = torch.as_tensor(table[b, : -(-L // w.page_size)], dtype=torch.long, device="cuda")
        g = h // w.group
        K = H.np_bits(layer.k_pages[pages, g].reshape(-1, 128))[:L]
        V = H.np_bits(layer.v_pages[pages, g].reshape(-1, 128))[:L]
        ref_out[b, t, h], ref_lse[b, t, h], _ = O.attention_one(O.bf16_to_f64(qn[b, t, h]), O.bf16_to_f64(K),
                                                                O.bf16_to_f64(V), layer.scale)
    H.compare_attention(out, lse, ref_out, ref_lse, pairs=picks)


def test_decode_loop_through_the_page_manager(zf):
    """A serving loop driven by zf_kv over two layers whose caches share one raw-slot pool: three
    prompts admitted (their pages written by zf_encode_pages, per layer), 24 decode steps that each
    append one token per request with zf_append_tokens (written in place into the raw tail page,
    which is compressed when it fills), raw slots reclaimed layer by layer from the directories
    after every step, one request released and another admitted mid-way.  Layer 1's keys carry a spike every 24 tokens, so the
    pages holding one stay raw in layer 1 only and their layer-0 slots go back to the pool for
    either layer to reuse.  At several steps each layer's attention over the exported page table
    matches the float64 attention over each request's token stream."""
    P, Hkv, Hq, D, NL = 16, 2, 8, 128, 2
    dev = torch.device("cuda")
    gen = torch.Generator().manual_seed(61)
    max_len = 160
    streams_k, streams_v = [], []
    for layer in range(NL):
        ks, vs = [], []
        for _ in range(4):
            k = torch.randn(max_len, Hkv, D, generator=gen).mul(torch.exp(0.5 * torch.randn(D, generator=gen)))
            if layer == 1:
                k[7::24, 0, 5:13] *= 2.0 ** -30             # 8 escapes: that page-head stays raw
            ks.append(k.to(torch.bfloat16).view(torch.int16))
            vs.append(torch.randn(max_len, Hkv, D, generator=gen).to(torch.bfloat16).view(torch.int16))
        streams_k.append(ks)
        streams_v.append(vs)
    num_raw = 20
    kv = zf.KvManager(num_pages=40, num_raw_slots=num_raw, page_size=P, max_requests=4, max_pages_per_req=10,
                      num_layers=NL)
    caches = [zf.Cache(40, Hkv, P, num_raw, device=dev)]
    caches.append(zf.Cache(40, Hkv, P, num_raw, device=dev, raw_pool=caches[0]))
    stream_of = {}
    kept_seen = []

    def write(req, ids, nv, rs):
        s = stream_of[req]
        length = int(kv.export()[1][req])
        first = -(-length // P) - len(ids)                   # index of the first listed page
        for layer in range(NL):
            pages_k = torch.zeros(len(ids), Hkv, P, D, dtype=torch.int16)
            pages_v = torch.zeros_like(pages_k)
            for j in range(len(ids)):
                lo = (first + j) * P
                hi = lo + nv[j]
                pages_k[j, :, : nv[j]] = streams_k[layer][s][lo:hi].transpose(0, 1)
                pages_v[j, :, : nv[j]] = streams_v[layer][s][lo:hi].transpose(0, 1)
            zf.encode_pages(caches[layer], pages_k.to(dev), pages_v.to(dev), ids, nv, rs[layer])

    def reclaim():            # only once every page listed as pending has been encoded in every layer
        kv.reclaim_from(caches)
        st = kv.stats()
        kept_seen.append((st["raw_full_pages"], st["raw_full_slots"]))

    def check():
        table, lens = kv.export()
        for layer in range(NL):
            q = torch.randn(4, Hq, D, generator=gen).to(torch.bfloat16).view(torch.int16)
            out, lse = zf.decode_attn(caches[layer], q.to(dev), table.to(dev), lens.to(dev), 0.125)
            torch.cuda.synchronize()
            assert caches[layer].status_word() == 0
            ref_out = np.zeros((4, Hq, D))
            ref_lse = np.full((4, Hq), -math.inf)
            for req, s in stream_of.items():
                L = int(lens[req])
                for h in range(Hq):
                    g = h // (Hq // Hkv)
                    ref_out[req, h], ref_lse[req, h], _ = O.attention_one(
                        O.bf16_to_f64(H.np_bits(q[req, h])), O.bf16_to_f64(H.np_bits(streams_k[layer][s][:L, g])),
                        O.bf16_to_f64(H.np_bits(streams_v[layer][s][:L, g])), 0.125)
            H.compare_attention(out, lse, ref_out, ref_lse)

    for req, length in ((0, 37), (1, 16), (2, 70)):
        stream_of[req] = req
        ids, nv, rs = kv.admit(req, length)
        write(req, ids, nv, rs)
        reclaim()
    check()
    for step in range(24):
        if step == 10:                                       # request 1 leaves, request 3 arrives
            kv.release(1)
            del stream_of[1]
            stream_of[3] = 3
            ids, nv, rs = kv.admit(3, 50)
            write(3, ids, nv, rs)
            reclaim()
        reqs = sorted(stream_of)
        ids, nv, rs = kv.append(reqs)
        lens = kv.export()[1]
        for layer in range(NL):             # the new token of each request, written in place
            k_tok = torch.stack([streams_k[layer][stream_of[q]][int(lens[q]) - 1] for q in reqs])
            v_tok = torch.stack([streams_v[layer][stream_of[q]][int(lens[q]) - 1] for q in reqs])
            zf.append_tokens(caches[layer], k_tok.to(dev), v_tok.to(dev), ids, [f - 1 for f in nv], rs[layer])
        reclaim()
        if step % 6 == 5:
            check()
    st = kv.stats()
    assert st["pending_pages"] == 0 and st["tokens"] == int(kv.export()[1].sum())
    # full pages with a spike stayed raw in layer 1 only: one kept slot each, none in layer 0
    assert any(p > 0 for p, _ in kept_seen) and all(p == n for p, n in kept_seen), kept_seen
    table, lens = kv.export()
    full = [int(table[q, i]) for q in range(4) for i in range(int(lens[q]) // P)]
    d0, d1 = caches[0].dir.cpu()[full], caches[1].dir.cpu()[full]
    assert (d0 == zf.DIR_COMPRESSED).all()
    raw_pages = int((d1 >= 0).any(dim=1).sum())
    assert raw_pages > 0 and st["raw_full_pages"] == raw_pages == st["raw_full_slots"]
