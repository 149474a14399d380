"""Thin Python binding over libzf.so (C ABI in include/zf.h).

Argument marshalling only: torch tensors provide device memory and the current CUDA stream; every
step of encoding, decompression and attention runs in the library's CUDA kernels.  The library is
loaded on first use and a missing library raises: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libzf.so")

HEAD_DIM = 128
SLOT_BYTES = 784
RAW_BLOCK_BYTES = 1024
DIR_COMPRESSED = -1
DIR_INVALID = -2
ENCODE_FORCE_RAW = 1
DEV_BAD_PAGE_ID, DEV_BAD_RAW_SLOT, DEV_BAD_N_VALID = 0x1, 0x2, 0x4
DEV_BAD_SEQ_LEN, DEV_BAD_DIR, DEV_TIMEOUT, DEV_BAD_SLOT = 0x8, 0x10, 0x20, 0x40

_c_int32, _c_void_p, _c_size_t, _c_float = ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_float


class ZfCacheDesc(ctypes.Structure):
    _fields_ = [
        ("num_pages", _c_int32), ("num_kv_heads", _c_int32), ("head_dim", _c_int32),
        ("page_size", _c_int32), ("num_raw_slots", _c_int32), ("reserved", _c_int32),
        ("k_comp", _c_void_p), ("v_comp", _c_void_p), ("k_raw", _c_void_p), ("v_raw", _c_void_p),
        ("dir", _c_void_p), ("status", _c_void_p),
    ]


class ZfKvStats(ctypes.Structure):
    _fields_ = [
        ("tokens", ctypes.c_int64), ("free_pages", _c_int32), ("free_raw_slots", _c_int32),
        ("active_requests", _c_int32), ("partial_pages", _c_int32), ("pending_pages", _c_int32),
        ("raw_full_pages", _c_int32), ("compressed_pages", _c_int32), ("new_page_capacity", _c_int32),
        ("raw_full_slots", _c_int32),
    ]


_P32 = ctypes.POINTER(_c_int32)

# name -> (restype, argtypes), mirroring include/zf.h
SIGNATURES = {
    "zf_status_string": (ctypes.c_char_p, [_c_int32]),
    "zf_page_head_bytes": (_c_size_t, [_c_int32, _c_int32]),
    "zf_encode_pages": (_c_int32, [ctypes.POINTER(ZfCacheDesc), _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                   _c_void_p, _c_int32, _c_int32, _c_void_p]),
    "zf_append_tokens": (_c_int32, [ctypes.POINTER(ZfCacheDesc), _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                    _c_void_p, _c_int32, _c_void_p]),
    "zf_validate_pages": (_c_int32, [ctypes.POINTER(ZfCacheDesc), _c_void_p, _c_int32, _c_void_p, _c_void_p]),
    "zf_slot_is_valid": (_c_int32, [_c_void_p]),
    "zf_decompress": (_c_int32, [ctypes.POINTER(ZfCacheDesc), _c_void_p, _c_int32, _c_void_p, _c_void_p, _c_void_p]),
    "zf_decompress_to_raw": (_c_int32, [ctypes.POINTER(ZfCacheDesc), _c_void_p, _c_int32, _c_void_p, _c_void_p,
                                        _c_void_p]),
    "zf_decode_attn_workspace_size": (_c_size_t, [_c_int32, _c_int32, _c_int32, _c_int32, _c_int32]),
    "zf_decode_attn": (_c_int32, [ctypes.POINTER(ZfCacheDesc), _c_void_p, _c_int32, _c_int32, _c_void_p, _c_int32,
                                  _c_void_p, _c_float, _c_void_p, _c_void_p, _c_void_p, _c_size_t, _c_void_p]),
    "zf_dense_decode_attn": (_c_int32, [ctypes.POINTER(ZfCacheDesc), _c_void_p, _c_int32, _c_int32, _c_void_p,
                                        _c_int32, _c_void_p, _c_float, _c_void_p, _c_void_p, _c_void_p, _c_size_t,
                                        _c_void_p]),
    "zf_decode_attn_static": (_c_int32, [ctypes.POINTER(ZfCacheDesc), _c_void_p, _c_int32, _c_int32, _c_void_p,
                                         _c_int32, _c_void_p, _c_float, _c_void_p, _c_void_p, _c_void_p]),
    "zf_decode_attn_multi_workspace_size": (_c_size_t, [_c_int32, _c_int32, _c_int32, _c_int32, _c_int32, _c_int32]),
    "zf_decode_attn_multi": (_c_int32, [ctypes.POINTER(ZfCacheDesc), _c_void_p, _c_int32, _c_int32, _c_int32,
                                        _c_void_p, _c_int32, _c_void_p, _c_float, _c_void_p, _c_void_p, _c_void_p,
                                        _c_size_t, _c_void_p]),
    "zf_decode_attn_multi_kernel": (_c_int32, [ctypes.POINTER(ZfCacheDesc), _c_void_p, _c_int32, _c_int32, _c_int32,
                                               _c_void_p, _c_int32, _c_void_p, _c_float, _c_void_p, _c_void_p,
                                               _c_void_p, _c_size_t, _c_int32, _c_void_p]),
    "zf_decode_attn_wait_test": (_c_int32, [ctypes.POINTER(ZfCacheDesc), _c_void_p, _c_int32, _c_int32, _c_int32,
                                            _c_void_p, _c_int32, _c_void_p, _c_float, _c_void_p, _c_void_p,
                                            _c_void_p, _c_size_t, _c_int32, ctypes.c_uint64, ctypes.c_uint64,
                                            _c_void_p]),
    "zf_dense_decode_attn_multi": (_c_int32, [ctypes.POINTER(ZfCacheDesc), _c_void_p, _c_int32, _c_int32, _c_int32,
                                              _c_void_p, _c_int32, _c_void_p, _c_float, _c_void_p, _c_void_p,
                                              _c_void_p, _c_size_t, _c_void_p]),
    "zf_kv_create": (_c_int32, [_c_int32, _c_int32, _c_int32, _c_int32, _c_int32, _c_int32, ctypes.POINTER(_c_void_p)]),
    "zf_kv_destroy": (None, [_c_void_p]),
    "zf_kv_admit": (_c_int32, [_c_void_p, _c_int32, _c_int32, _P32, _P32, _P32, _P32]),
    "zf_kv_append": (_c_int32, [_c_void_p, _P32, _c_int32, _P32, _P32, _P32]),
    "zf_kv_pending": (_c_int32, [_c_void_p, _P32, _P32, _c_int32, _P32]),
    "zf_kv_reclaim": (_c_int32, [_c_void_p, _P32, _P32, _c_int32]),
    "zf_kv_release": (_c_int32, [_c_void_p, _c_int32]),
    "zf_kv_export": (_c_int32, [_c_void_p, _P32, _P32]),
    "zf_kv_get_stats": (_c_int32, [_c_void_p, ctypes.POINTER(ZfKvStats)]),
    "zf_kv_plan_pages": (_c_int32, [ctypes.c_int64, _c_int32, _c_int32, _c_int32, _P32, _P32]),
}

_LIB = None


class ZfError(RuntimeError):
    pass


def lib() -> ctypes.CDLL:
    """The loaded libzf.so (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise ZfError(f"{LIB_PATH} is missing: build it with `python -m decode_attention_compressed_gb300.build`")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype, fn.argtypes = res, args
        _LIB = handle
    return _LIB


def status_string(code: int) -> str:
    return lib().zf_status_string(code).decode()


def _check(name: str, code: int):
    if code != 0:
        raise ZfError(f"{name}: {status_string(code)} ({code})")


def _stream(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dev_i32(x, device):
    return torch.as_tensor(x, dtype=torch.int32, device=device).contiguous()


_BITS16 = (torch.int16, torch.bfloat16)      # BF16 bit patterns, either view


def _count(x) -> int:
    return int(x.numel()) if isinstance(x, torch.Tensor) else len(x)


def _arg(t, name, cache, dtypes, shape=None, min_rows=None):
    """Checks the C ABI cannot make (it sees bare pointers): dtype, device, shape.  `shape` entries
    of None match any size; min_rows bounds the first dimension from below."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype not in dtypes:
        raise ValueError(f"{name}: dtype {t.dtype}, expected {' or '.join(str(d) for d in dtypes)}")
    if t.device != cache.device:
        raise ValueError(f"{name} is on {t.device}, the cache on {cache.device}")
    if shape is not None and (t.dim() != len(shape) or
                              any(w is not None and h != w for h, w in zip(t.shape, shape))):
        want = "[" + "][".join("*" if w is None else str(w) for w in shape) + "]"
        raise ValueError(f"{name}: shape {list(t.shape)}, expected {want}")
    if min_rows is not None and (t.dim() < 1 or t.shape[0] < min_rows):
        raise ValueError(f"{name}: {t.shape[0] if t.dim() else 0} rows, at least {min_rows} needed")
    return t.contiguous()


def _result(t, name, cache, shape):
    """An output the kernels write in place: float32, contiguous, exactly `shape`."""
    _arg(t, name, cache, (torch.float32,), shape)
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (it is written in place)")
    return t


def _attn_args(cache, q, page_table, seq_lens, B):
    page_table = _arg(page_table, "page_table", cache, (torch.int32,), (None, None), min_rows=B)
    seq_lens = _arg(seq_lens, "seq_lens", cache, (torch.int32,), (None,), min_rows=B)
    return page_table, seq_lens


class Cache:
    """One layer's paged cache in device memory, laid out as include/zf.h describes.

    k_comp/v_comp: [num_pages][Hkv][P/4 * 784] uint8; k_raw/v_raw: [num_raw][Hkv][P/4 * 512] int16
    (BF16 bits); dir: [num_pages][Hkv] int32; status: one int32 device word.  raw_pool=another
    Cache makes this layer use that cache's raw arrays (one raw pool for all layers, as KvManager
    with num_layers > 1 hands out slots).
    """

    def __init__(self, num_pages, num_kv_heads, page_size, num_raw_slots, device="cuda", compressed=True,
                 raw_pool=None):
        nblk = page_size // 4
        self.num_pages, self.num_kv_heads, self.page_size = num_pages, num_kv_heads, page_size
        self.num_raw_slots = num_raw_slots
        dev = torch.device(device)
        if raw_pool is not None:                   # share another cache's raw arrays (one pool for all layers)
            if (raw_pool.num_kv_heads, raw_pool.page_size, raw_pool.num_raw_slots) != (num_kv_heads, page_size,
                                                                                      num_raw_slots):
                raise ValueError("a shared raw pool must match the kv heads, page size and raw slot count")
        if compressed:
            self.k_comp = torch.empty((num_pages, num_kv_heads, nblk * SLOT_BYTES), dtype=torch.uint8, device=dev)
            self.v_comp = torch.empty_like(self.k_comp)
        else:
            self.k_comp = self.v_comp = None       # dense cache: raw slots only (zf_dense_decode_attn)
        self.dir = torch.full((num_pages, num_kv_heads), DIR_INVALID, dtype=torch.int32, device=dev)
        if raw_pool is not None:
            self.k_raw, self.v_raw = raw_pool.k_raw, raw_pool.v_raw
        else:
            self.k_raw = torch.empty((num_raw_slots, num_kv_heads, nblk * 512), dtype=torch.int16, device=dev)
            self.v_raw = torch.empty_like(self.k_raw)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

    @property
    def device(self):
        return self.status.device

    def desc(self) -> ZfCacheDesc:
        return ZfCacheDesc(self.num_pages, self.num_kv_heads, HEAD_DIM, self.page_size, self.num_raw_slots, 0,
                           _ptr(self.k_comp), _ptr(self.v_comp), _ptr(self.k_raw), _ptr(self.v_raw),
                           _ptr(self.dir), _ptr(self.status))

    def status_word(self) -> int:
        return int(self.status.item())

    def stored_bytes(self, num_pages=None) -> int:
        """Bytes the first `num_pages` pages actually occupy (synchronises): every page head costs
        its compressed record or its raw record, plus its directory entry."""
        n = self.num_pages if num_pages is None else num_pages
        nblk = self.page_size // 4
        if self.k_comp is None:
            return n * self.num_kv_heads * 2 * nblk * RAW_BLOCK_BYTES
        d = self.dir[:n].cpu()
        comp = int((d == DIR_COMPRESSED).sum())
        raw = int((d >= 0).sum())
        return 2 * nblk * (comp * SLOT_BYTES + raw * RAW_BLOCK_BYTES) + d.numel() * 4


def encode_pages(cache: Cache, src_k, src_v, page_ids, n_valid, raw_slots=None, force_raw=False, stream=None):
    """Compress (or store raw) pages: src_k/src_v [n][Hkv][P][128] int16 BF16 bits on the device."""
    dev = cache.device
    shape = (None, cache.num_kv_heads, cache.page_size, HEAD_DIM)
    src_k = _arg(src_k, "src_k", cache, _BITS16, shape)
    src_v = _arg(src_v, "src_v", cache, _BITS16, tuple(src_k.shape))
    n = int(src_k.shape[0])
    for name, x in (("page_ids", page_ids), ("n_valid", n_valid), ("raw_slots", raw_slots)):
        if x is not None and _count(x) != n:
            raise ValueError(f"{name}: {_count(x)} entries for {n} pages")
    ids = _dev_i32(page_ids, dev)
    nv = _dev_i32(n_valid, dev)
    rs = _dev_i32(raw_slots, dev) if raw_slots is not None else _dev_i32([-1] * n, dev)
    d = cache.desc()
    code = lib().zf_encode_pages(ctypes.byref(d), _ptr(src_k), _ptr(src_v), _ptr(ids), _ptr(nv), _ptr(rs), n,
                                 ENCODE_FORCE_RAW if force_raw else 0, _stream(stream))
    _check("zf_encode_pages", code)
    return ids, nv, rs          # keep them alive until the stream has consumed them


def append_tokens(cache: Cache, k_tok, v_tok, page_ids, positions, raw_slots, stream=None):
    """zf_append_tokens: k_tok/v_tok [n][Hkv][128] int16 BF16 bits on the device; entry i is token
    positions[i] of page page_ids[i], written into raw slot raw_slots[i] (the page is compressed
    when that token fills it).  Returns the index tensors (keep them alive until the stream has
    consumed them)."""
    dev = cache.device
    k_tok = _arg(k_tok, "k_tok", cache, _BITS16, (None, cache.num_kv_heads, HEAD_DIM))
    v_tok = _arg(v_tok, "v_tok", cache, _BITS16, tuple(k_tok.shape))
    n = int(k_tok.shape[0])
    for name, x in (("page_ids", page_ids), ("positions", positions), ("raw_slots", raw_slots)):
        if _count(x) != n:
            raise ValueError(f"{name}: {_count(x)} entries for {n} tokens")
    ids, pos, rs = _dev_i32(page_ids, dev), _dev_i32(positions, dev), _dev_i32(raw_slots, dev)
    d = cache.desc()
    _check("zf_append_tokens", lib().zf_append_tokens(ctypes.byref(d), _ptr(k_tok), _ptr(v_tok), _ptr(ids), _ptr(pos),
                                                       _ptr(rs), n, _stream(stream)))
    return ids, pos, rs


def validate_pages(cache: Cache, page_ids, stream=None):
    """zf_validate_pages: an int32 device tensor, 1 for each listed page whose stored form has a
    problem (the cache's status word says which kind)."""
    dev = cache.device
    ids = _dev_i32(page_ids, dev)
    bad = torch.zeros(int(ids.numel()), dtype=torch.int32, device=dev)
    d = cache.desc()
    _check("zf_validate_pages", lib().zf_validate_pages(ctypes.byref(d), _ptr(ids), int(ids.numel()), _ptr(bad),
                                                         _stream(stream)))
    return bad


def slot_is_valid(slot) -> bool:
    """zf_slot_is_valid on one 784-byte compressed slot held in host memory (bytes or uint8 array)."""
    buf = (ctypes.c_uint8 * SLOT_BYTES).from_buffer_copy(bytes(slot)[:SLOT_BYTES].ljust(SLOT_BYTES, b"\0"))
    return bool(lib().zf_slot_is_valid(ctypes.addressof(buf)))


def decompress(cache: Cache, page_ids, stream=None):
    dev = cache.device
    ids = _dev_i32(page_ids, dev)
    n = int(ids.numel())
    k = torch.empty((n, cache.num_kv_heads, cache.page_size, HEAD_DIM), dtype=torch.int16, device=dev)
    v = torch.empty_like(k)
    d = cache.desc()
    _check("zf_decompress", lib().zf_decompress(ctypes.byref(d), _ptr(ids), n, _ptr(k), _ptr(v), _stream(stream)))
    return k, v


def decompress_to_raw(cache: Cache, page_ids, dense: Cache, stream=None):
    """zf_decompress_to_raw: page_ids[i] of `cache` into raw slot i of the dense cache `dense`
    (same kv heads and page size, at least len(page_ids) raw slots).  Returns the id tensor (keep it
    alive until the stream has consumed it)."""
    dev = cache.device
    ids = _dev_i32(page_ids, dev)
    n = int(ids.numel())
    if dense.num_kv_heads != cache.num_kv_heads or dense.page_size != cache.page_size or dense.num_raw_slots < n:
        raise ValueError("the dense cache must match the kv heads and page size and hold n raw slots")
    d = cache.desc()
    _check("zf_decompress_to_raw", lib().zf_decompress_to_raw(ctypes.byref(d), _ptr(ids), n, _ptr(dense.k_raw),
                                                               _ptr(dense.v_raw), _stream(stream)))
    return ids


def workspace_size(batch, num_q_heads, num_kv_heads, page_size, max_pages) -> int:
    return int(lib().zf_decode_attn_workspace_size(batch, num_q_heads, num_kv_heads, page_size, max_pages))


def new_workspace(nbytes, device="cuda"):
    """A workspace buffer for zf_decode_attn (any contents are fine)."""
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


# attention kernels of zf_decode_attn_multi_kernel
KERNELS = {"auto": 0, "warp_mma": 1, "tcgen05": 2}


def _kernel_code(kernel, dense):
    if kernel not in KERNELS:
        raise ValueError(f"kernel must be one of {sorted(KERNELS)}")
    if dense and kernel != "auto":
        raise ValueError("the dense comparator has one kernel (warp MMA)")
    return KERNELS[kernel]


def decode_attn(cache: Cache, q, page_table, seq_lens, scale=None, out=None, lse=None, workspace=None,
                stream=None, dense=False, kernel="auto"):
    """Decode attention over the cache.  q [B][Hq][128] int16 (BF16 bits), page_table [B][max_pages]
    int32, seq_lens [B] int32, all on the device.  Returns (out [B][Hq][128] f32, lse [B][Hq] f32).
    dense=True runs zf_dense_decode_attn on the raw pool (page id = raw slot).  kernel: "auto"
    (zf_decode_attn), or "warp_mma" / "tcgen05" (zf_decode_attn_multi_kernel with one new token)."""
    code = _kernel_code(kernel, dense)
    if code:
        o, l = decode_attn_multi(cache, q[:, None], page_table, seq_lens, scale,
                                 out=None if out is None else out[:, None], lse=None if lse is None else lse[:, None],
                                 workspace=workspace, stream=stream, kernel=kernel)
        return o[:, 0], l[:, 0]
    q = _arg(q, "q", cache, _BITS16, (None, None, HEAD_DIM))
    B, Hq, _ = q.shape
    page_table, seq_lens = _attn_args(cache, q, page_table, seq_lens, B)
    max_pages = int(page_table.shape[1])
    scale = 1.0 / math.sqrt(HEAD_DIM) if scale is None else scale
    dev = cache.device
    out = torch.empty((B, Hq, HEAD_DIM), dtype=torch.float32, device=dev) if out is None else \
        _result(out, "out", cache, (B, Hq, HEAD_DIM))
    lse = torch.empty((B, Hq), dtype=torch.float32, device=dev) if lse is None else _result(lse, "lse", cache, (B, Hq))
    need = workspace_size(B, Hq, cache.num_kv_heads, cache.page_size, max_pages)
    if workspace is None:
        workspace = new_workspace(need, dev)
    d = cache.desc()
    fn = lib().zf_dense_decode_attn if dense else lib().zf_decode_attn
    code = fn(ctypes.byref(d), _ptr(q), B, Hq, _ptr(page_table), max_pages, _ptr(seq_lens), scale, _ptr(out),
              _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    _check("zf_dense_decode_attn" if dense else "zf_decode_attn", code)
    return out, lse


def dense_decode_attn(cache: Cache, q, page_table, seq_lens, scale=None, **kw):
    return decode_attn(cache, q, page_table, seq_lens, scale, dense=True, **kw)


def workspace_size_multi(batch, tokens, num_q_heads, num_kv_heads, page_size, max_pages) -> int:
    return int(lib().zf_decode_attn_multi_workspace_size(batch, tokens, num_q_heads, num_kv_heads, page_size,
                                                         max_pages))


def decode_attn_multi(cache: Cache, q, page_table, seq_lens, scale=None, out=None, lse=None, workspace=None,
                      stream=None, dense=False, kernel="auto"):
    """zf_decode_attn_multi: T new tokens per request.  q [B][T][Hq][128] int16 (BF16 bits); token t
    of request b attends to positions 0 .. seq_lens[b] - T + t.  Returns (out [B][T][Hq][128] f32,
    lse [B][T][Hq] f32).  dense=True runs zf_dense_decode_attn_multi.  kernel: "auto", "warp_mma" or
    "tcgen05" (zf_decode_attn_multi_kernel)."""
    code = _kernel_code(kernel, dense)
    q = _arg(q, "q", cache, _BITS16, (None, None, None, HEAD_DIM))
    B, T, Hq, _ = q.shape
    page_table, seq_lens = _attn_args(cache, q, page_table, seq_lens, B)
    max_pages = int(page_table.shape[1])
    scale = 1.0 / math.sqrt(HEAD_DIM) if scale is None else scale
    dev = cache.device
    out = torch.empty((B, T, Hq, HEAD_DIM), dtype=torch.float32, device=dev) if out is None else \
        _result(out, "out", cache, (B, T, Hq, HEAD_DIM))
    lse = torch.empty((B, T, Hq), dtype=torch.float32, device=dev) if lse is None else \
        _result(lse, "lse", cache, (B, T, Hq))
    if workspace is None:
        workspace = new_workspace(workspace_size_multi(B, T, Hq, cache.num_kv_heads, cache.page_size, max_pages), dev)
    d = cache.desc()
    args = (ctypes.byref(d), _ptr(q), B, T, Hq, _ptr(page_table), max_pages, _ptr(seq_lens), scale, _ptr(out),
            _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size())
    if code:
        name = "zf_decode_attn_multi_kernel"
        status = lib().zf_decode_attn_multi_kernel(*args, code, _stream(stream))
    else:
        name = "zf_dense_decode_attn_multi" if dense else "zf_decode_attn_multi"
        status = getattr(lib(), name)(*args, _stream(stream))
    _check(name, status)
    return out, lse


def decode_attn_wait_test(cache: Cache, q, page_table, seq_lens, scale=None, kernel="warp_mma", wait_limit_ns=1000000,
                          publish_delay_ns=0, stream=None):
    """zf_decode_attn_wait_test (tests of the failure path): one new token per request, the
    kernel's waits for its metadata warp's items limited to wait_limit_ns and that warp's first
    item published publish_delay_ns late.  Returns (out, lse); with the delay above the limit
    the outputs are not meaningful and the cache's status word gets DEV_TIMEOUT."""
    q = _arg(q, "q", cache, _BITS16, (None, None, HEAD_DIM))
    B, Hq, _ = q.shape
    page_table, seq_lens = _attn_args(cache, q, page_table, seq_lens, B)
    max_pages = int(page_table.shape[1])
    scale = 1.0 / math.sqrt(HEAD_DIM) if scale is None else scale
    dev = cache.device
    out = torch.empty((B, Hq, HEAD_DIM), dtype=torch.float32, device=dev)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    workspace = new_workspace(workspace_size(B, Hq, cache.num_kv_heads, cache.page_size, max_pages), dev)
    d = cache.desc()
    _check("zf_decode_attn_wait_test",
           lib().zf_decode_attn_wait_test(ctypes.byref(d), _ptr(q), B, 1, Hq, _ptr(page_table), max_pages,
                                          _ptr(seq_lens), scale, _ptr(out), _ptr(lse), _ptr(workspace),
                                          workspace.numel() * workspace.element_size(), _kernel_code(kernel, False),
                                          int(wait_limit_ns), int(publish_delay_ns), _stream(stream)))
    return out, lse


STATIC_WORKSPACE_BYTES = 32 << 20
ERR_STATIC_WORKSPACE_EXCEEDED = -5
ERR_STATIC_WORKSPACE_UNAVAILABLE = -7


def decode_attn_static(cache: Cache, q, page_table, seq_lens, scale=None, out=None, lse=None, stream=None):
    """zf_decode_attn_static: the same attention without a caller-provided workspace, for callers
    that cannot allocate device memory (the library's 32 MiB static scratch array is used).
    Calls must not overlap on the GPU; the first call on a device must precede any stream capture."""
    q = _arg(q, "q", cache, _BITS16, (None, None, HEAD_DIM))
    B, Hq, _ = q.shape
    page_table, seq_lens = _attn_args(cache, q, page_table, seq_lens, B)
    scale = 1.0 / math.sqrt(HEAD_DIM) if scale is None else scale
    dev = cache.device
    out = torch.empty((B, Hq, HEAD_DIM), dtype=torch.float32, device=dev) if out is None else \
        _result(out, "out", cache, (B, Hq, HEAD_DIM))
    lse = torch.empty((B, Hq), dtype=torch.float32, device=dev) if lse is None else _result(lse, "lse", cache, (B, Hq))
    d = cache.desc()
    code = lib().zf_decode_attn_static(ctypes.byref(d), _ptr(q), B, Hq, _ptr(page_table), int(page_table.shape[1]),
                                       _ptr(seq_lens), scale, _ptr(out), _ptr(lse), _stream(stream))
    _check("zf_decode_attn_static", code)
    return out, lse


# --------------------------------------------------------------------------------- page manager
ERR_CAPACITY = -6


def _i32(values):
    arr = (_c_int32 * max(len(values), 1))(*values)
    return arr


class KvManager:
    """zf_kv: host-side page manager (page ids for all layers, one raw-slot pool shared by
    num_layers layers).  admit/append return the write list (page_ids, n_valid, raw_slots) with
    raw_slots[l] the slot list of layer l's call: encode_pages for a prompt, append_tokens
    (positions n_valid - 1) for a decode step."""

    def __init__(self, num_pages, num_raw_slots, page_size, max_requests, max_pages_per_req, num_layers=1):
        self.page_size, self.max_requests, self.max_pages = page_size, max_requests, max_pages_per_req
        self.num_layers = num_layers
        h = _c_void_p()
        _check("zf_kv_create", lib().zf_kv_create(num_pages, num_raw_slots, num_layers, page_size, max_requests,
                                                   max_pages_per_req, ctypes.byref(h)))
        self._h = h

    def close(self):
        if self._h:
            lib().zf_kv_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _layers(self, flat, n):
        return [list(flat[l * n:(l + 1) * n]) for l in range(self.num_layers)]

    def admit(self, req, length):
        n_max = max(-(-length // self.page_size), 1)
        ids, nv, n = (_c_int32 * n_max)(), (_c_int32 * n_max)(), _c_int32()
        rs = (_c_int32 * (n_max * self.num_layers))()
        _check("zf_kv_admit", lib().zf_kv_admit(self._h, req, length, ids, nv, rs, ctypes.byref(n)))
        k = n.value
        return list(ids[:k]), list(nv[:k]), self._layers(rs, k)

    def append(self, reqs):
        n = len(reqs)
        ids, nv = (_c_int32 * max(n, 1))(), (_c_int32 * max(n, 1))()
        rs = (_c_int32 * max(n * self.num_layers, 1))()
        _check("zf_kv_append", lib().zf_kv_append(self._h, _i32(reqs), n, ids, nv, rs))
        return list(ids[:n]), list(nv[:n]), self._layers(rs, n)

    def pending(self):
        """(page ids, raw slots per layer) of the full pages awaiting reclaim, ascending id."""
        n = _c_int32()
        code = lib().zf_kv_pending(self._h, None, None, 0, ctypes.byref(n))
        if code not in (0, -1):
            _check("zf_kv_pending", code)
        k = n.value
        ids, rs = (_c_int32 * max(k, 1))(), (_c_int32 * max(k * self.num_layers, 1))()
        _check("zf_kv_pending", lib().zf_kv_pending(self._h, ids, rs, k, ctypes.byref(n)))
        return list(ids[:k]), self._layers(rs, k)

    def reclaim(self, page_ids, kept_raw):
        """kept_raw[l][i]: page_ids[i] has a page-head stored raw in layer l (keeps that layer's slot)."""
        n = len(page_ids)
        if len(kept_raw) != self.num_layers or any(len(row) != n for row in kept_raw):
            raise ValueError("kept_raw needs one row of len(page_ids) flags per layer")
        flat = [int(bool(x)) for row in kept_raw for x in row]
        _check("zf_kv_reclaim", lib().zf_kv_reclaim(self._h, _i32(page_ids), _i32(flat), n))

    def reclaim_from(self, caches):
        """Reclaim every pending page from the directories of `caches`.  With num_layers layers,
        caches[l] is layer l (each layer keeps or returns its own slot); with num_layers == 1, any
        number of caches addressed by the same slots (a page keeps its slot if it is raw in any)."""
        ids, _ = self.pending()
        if not ids:
            return 0
        if self.num_layers > 1 and len(caches) != self.num_layers:
            raise ValueError("one cache per layer")
        idx = torch.as_tensor(ids, dtype=torch.long)
        raw = [(c.dir.index_select(0, idx.to(c.dir.device)).cpu() >= 0).any(dim=1) for c in caches]
        if self.num_layers == 1:
            kept = [torch.stack(raw).any(dim=0).tolist()]
        else:
            kept = [r.tolist() for r in raw]
        self.reclaim(ids, kept)
        return len(ids)

    def release(self, req):
        _check("zf_kv_release", lib().zf_kv_release(self._h, req))

    def export(self):
        """(page_table [max_requests][max_pages_per_req], seq_lens [max_requests]) int32 CPU tensors."""
        table = torch.empty((self.max_requests, self.max_pages), dtype=torch.int32)
        lens = torch.empty(self.max_requests, dtype=torch.int32)
        _check("zf_kv_export", lib().zf_kv_export(self._h, ctypes.cast(table.data_ptr(), _P32),
                                                   ctypes.cast(lens.data_ptr(), _P32)))
        return table, lens

    def stats(self) -> dict:
        st = ZfKvStats()
        _check("zf_kv_get_stats", lib().zf_kv_get_stats(self._h, ctypes.byref(st)))
        return {name: getattr(st, name) for name, _ in ZfKvStats._fields_}


def kv_plan_pages(bytes_per_layer, num_kv_heads, page_size, num_raw_slots):
    """(page ids, dense pages) that bytes_per_layer holds (zf_kv_plan_pages)."""
    a, b = _c_int32(), _c_int32()
    _check("zf_kv_plan_pages", lib().zf_kv_plan_pages(int(bytes_per_layer), num_kv_heads, page_size, num_raw_slots,
                                                       ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value
