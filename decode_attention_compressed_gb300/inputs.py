"""Seeded synthetic decode workloads: shapes and value distributions of the five decode
configurations this library is measured on.

This module only draws random numbers and lays out pages; it contains no compression and no
attention arithmetic, so both the CUDA path's tests/benchmark and the CPU oracle can consume
exactly the same arrays.  All values are BF16 bit patterns stored as int16 tensors.

Value recipe (one layer):
  s_c    = exp(sigma * N(0,1))                per channel c (shared by all heads and tokens)
  s_c   *= 10 for channels 0..n_outlier-1     (outlier channels)
  K[t,h,c] = N(0,1) * s_c                     (+ spikes: with probability spike_prob a
                                               (token, head) gets one uniform channel x spike_mult)
  V[t,h,c] = N(0, v_std^2);  q = N(0,1);  scale = 1/sqrt(128);  every value rounded to BF16 (RNE)
Page layout: request b owns ceil(L_b / P) pages; "ordered" pools give request b the pages
right after request b-1's, "random" pools hand out a random permutation of the shared pool.
Seeds: a workload's seed * 1000 + layer.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch

HEAD_DIM = 128


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    page_size: int
    ctx: int                      # context length (upper bound when ragged)
    ctx_min: int | None = None    # ragged: per-request length uniform in [ctx_min, ctx]
    layers: int = 1
    pool: str = "ordered"         # "ordered" | "random"
    k_sigma: float = 0.5
    n_outlier: int = 4
    spike_prob: float = 0.0
    spike_mult: float = 50.0
    v_std: float = 1.0
    seed: int = 0
    note: str = ""

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def max_pages(self) -> int:
        return -(-self.ctx // self.page_size)


# The decode configurations (tiny, LLaMA-7B MHA, Llama-3-8B batched, Qwen2-7B max batch, long
# context, and the batch-64 shape of the pages' kernel figure).  LLaMA-7B MHA is one workload per
# context length.
WORKLOADS = {
    "tiny": Workload("tiny", 1, 32, 8, 16, 512, seed=0,
                     note="batch 1, 32/8 heads, ctx 512, page 16, pages in order"),
    "llama7b_mha_512": Workload("llama7b_mha_512", 1, 32, 32, 16, 512, layers=32, seed=1),
    "llama7b_mha_2048": Workload("llama7b_mha_2048", 1, 32, 32, 16, 2048, layers=32, seed=1),
    "llama7b_mha_8192": Workload("llama7b_mha_8192", 1, 32, 32, 16, 8192, layers=32, seed=1,
                                 note="32 layers, batch 1, 32/32 heads, ctx 8192, page 16"),
    "llama3_8b_batched": Workload("llama3_8b_batched", 64, 32, 8, 16, 8192, ctx_min=1024,
                                  pool="random", seed=2,
                                  note="batch 64, 32/8 heads, ctx U[1024,8192], page 16, random pool"),
    "qwen2_7b_maxbatch": Workload("qwen2_7b_maxbatch", 128, 28, 4, 16, 8192, pool="random",
                                  k_sigma=0.7, n_outlier=0, spike_prob=0.02, v_std=0.5, seed=3,
                                  note="batch 128, 28/4 heads (GQA 7), ctx 8192, page 16, random pool, "
                                       "2% (token, head) one-channel x50 spikes"),
    "long_ctx": Workload("long_ctx", 4, 32, 8, 64, 131072, pool="random", seed=4,
                         note="batch 4, 32/8 heads, ctx 131072, page 64, random pool"),
    # the shape the ZipFusion attention-kernel figure (§IV.B, Fig. 4) times: an 8B model with 32
    # query and 8 kv heads, batch 64, contexts 2048 and 8192, 16-token pages
    "batch64_gqa4_2048": Workload("batch64_gqa4_2048", 64, 32, 8, 16, 2048, pool="random", seed=5,
                                  note="batch 64, 32/8 heads, ctx 2048, page 16, random pool"),
    "batch64_gqa4_8192": Workload("batch64_gqa4_8192", 64, 32, 8, 16, 8192, pool="random", seed=6,
                                  note="batch 64, 32/8 heads, ctx 8192, page 16, random pool"),
}


def scaled(w: Workload, **kw) -> Workload:
    """A copy of a workload with some fields replaced (smaller parity-test variants)."""
    return replace(w, **kw)


@dataclass
class LayerInputs:
    workload: Workload
    layer: int
    seq_lens: torch.Tensor        # [B] int32
    page_table: torch.Tensor      # [B][max_pages] int32, -1 past each request's pages
    n_valid: torch.Tensor         # [num_pages] int32 tokens filled in each pool page
    k_pages: torch.Tensor         # [num_pages][Hkv][P][128] int16 (BF16 bits), natural layout
    v_pages: torch.Tensor
    q: torch.Tensor               # [B][Hq][128] int16 (BF16 bits)
    scale: float = field(default=1.0 / math.sqrt(HEAD_DIM))

    @property
    def num_pages(self) -> int:
        return int(self.k_pages.shape[0])


def _bits(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.bfloat16).view(torch.int16)


def make_multi_queries(w: Workload, tokens: int, layer: int = 0, device="cpu") -> torch.Tensor:
    """Queries of `tokens` new tokens per request, N(0, 1) cast to BF16: [batch][tokens][q heads][128]
    BF16 bits (int16)."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(w.seed * 1000 + 500 + layer)
    return _bits(torch.randn(w.batch, tokens, w.num_q_heads, HEAD_DIM, generator=gen, device=dev))


def make_layer(w: Workload, layer: int = 0, device="cpu", seq_lens=None) -> LayerInputs:
    """Generate one layer's pages, page table and query for workload `w`."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(w.seed * 1000 + layer)
    B, Hkv, P, D = w.batch, w.num_kv_heads, w.page_size, HEAD_DIM

    s = torch.exp(w.k_sigma * torch.randn(D, generator=gen, device=dev))
    s[: w.n_outlier] *= 10.0
    if seq_lens is None:
        if w.ctx_min is None:
            lens = torch.full((B,), w.ctx, dtype=torch.int64, device=dev)
        else:
            lens = torch.randint(w.ctx_min, w.ctx + 1, (B,), generator=gen, device=dev)
    else:
        lens = torch.as_tensor(seq_lens, dtype=torch.int64, device=dev)
    lens_cpu = lens.cpu()
    npages = [(int(L) + P - 1) // P for L in lens_cpu]
    total = sum(npages)
    max_pages = max([w.max_pages] + npages)
    if w.pool == "random":
        perm = torch.randperm(total, generator=gen, device=dev).cpu()
    else:
        perm = torch.arange(total)
    counts = torch.tensor(npages, dtype=torch.int64)
    req = torch.repeat_interleave(torch.arange(B), counts)                 # request of each pool slot
    first = torch.cumsum(counts, 0) - counts
    idx_in_req = torch.arange(total) - torch.repeat_interleave(first, counts)
    table = torch.full((B, max_pages), -1, dtype=torch.int32)
    table[req, idx_in_req] = perm.to(torch.int32)
    n_valid = torch.zeros(total, dtype=torch.int32)
    n_valid[perm] = torch.clamp(lens_cpu[req] - idx_in_req * P, max=P).to(torch.int32)

    K = torch.randn(total, Hkv, P, D, generator=gen, device=dev) * s
    if w.spike_prob > 0:
        hit = torch.rand(total, Hkv, P, generator=gen, device=dev) < w.spike_prob
        chan = torch.randint(0, D, (total, Hkv, P), generator=gen, device=dev)
        onehot = torch.nn.functional.one_hot(chan, D).to(torch.bool) & hit[..., None]
        K = torch.where(onehot, K * w.spike_mult, K)
        del hit, chan, onehot
    k_bits = _bits(K)
    del K
    v_bits = _bits(torch.randn(total, Hkv, P, D, generator=gen, device=dev) * w.v_std)
    q_bits = _bits(torch.randn(B, w.num_q_heads, D, generator=gen, device=dev))
    return LayerInputs(w, layer, lens.to(torch.int32), table.to(dev), n_valid.to(dev),
                       k_bits, v_bits, q_bits)

