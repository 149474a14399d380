"""Byte accounting for the decode path (host-side arithmetic used by the benchmark's roofline).

Compressed slot sizes follow the block format: a 512-value block (16 tokens x 32 channels) takes
784 bytes when compressed (768 payload bytes, ZipFusion §III.B, plus 16 metadata bytes) and
1024 bytes raw.
"""
from __future__ import annotations

HEAD_DIM = 128
SLOT_BYTES = 784
RAW_BLOCK_BYTES = 1024
BLOCKS_PER_TILE = 4            # 128 channels / 32
TILE_TOKENS = 16


def dense_kv_bytes(num_kv_heads: int, head_dim: int, layers: int, tokens: int, elem_bytes: int = 2) -> int:
    """Dense K+V cache bytes: 2 (K and V) x heads x head_dim x layers x tokens x element size
    (FlashSVD v1.5 review, "Memory Budget", Eq. 8)."""
    return 2 * num_kv_heads * head_dim * layers * tokens * elem_bytes


def compressed_bytes_per_token_head() -> int:
    """K+V bytes one token of one KV head occupies when its page is compressed: 2 x 784 / 16 x 4 / 4."""
    return 2 * SLOT_BYTES * BLOCKS_PER_TILE // TILE_TOKENS


def dense_bytes_per_token_head() -> int:
    return 2 * HEAD_DIM * 2


def page_head_bytes(page_size: int, compressed: bool) -> int:
    """K+V bytes of one page of one KV head as the attention kernel copies it."""
    per_block = SLOT_BYTES if compressed else RAW_BLOCK_BYTES
    return 2 * (page_size // TILE_TOKENS) * BLOCKS_PER_TILE * per_block
