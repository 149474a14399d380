"""The C ABI without a GPU: libzf.so builds, loads, exports every function include/zf.h declares,
and rejects bad arguments on the host before launching anything."""
import ctypes
import os
import re

import pytest

from decode_attention_compressed_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "zf.h")


@pytest.fixture(scope="module")
def zf():
    B.build()
    from decode_attention_compressed_gb300 import zf as Z
    Z.lib()
    return Z


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(zf_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(zf):
    names = declared_functions()
    assert set(names) == set(zf.SIGNATURES), names
    handle = zf.lib()
    for n in names:
        assert getattr(handle, n) is not None


def test_status_strings(zf):
    assert zf.status_string(0) == "ok"
    assert zf.status_string(-1) == "invalid argument"
    assert zf.status_string(-3) == "workspace too small"
    assert zf.status_string(-7).startswith("no device memory left")
    assert zf.status_string(12345) == "unknown status"


def test_page_head_bytes(zf):
    f = zf.lib().zf_page_head_bytes
    assert f(16, 1) == 4 * 784 and f(16, 0) == 4 * 1024
    assert f(64, 1) == 16 * 784 and f(128, 0) == 32 * 1024
    assert f(8, 1) == 0 and f(24, 1) == 0 and f(256, 1) == 0


def _desc(zf, **kw):
    d = dict(num_pages=4, num_kv_heads=2, head_dim=128, page_size=16, num_raw_slots=2, reserved=0,
             k_comp=0x1000, v_comp=0x2000, k_raw=0x3000, v_raw=0x4000, dir=0x5000, status=None)
    d.update(kw)
    return zf.ZfCacheDesc(**d)


def _encode(zf, desc, n=1, src=0x10000, flags=0, ids=0x20000):
    return zf.lib().zf_encode_pages(ctypes.byref(desc) if desc is not None else None, src, src, ids, 0x30000,
                                    0x40000, n, flags, None)


def test_encode_rejects_bad_arguments_before_launch(zf):
    assert _encode(zf, None) == -1
    assert _encode(zf, _desc(zf, head_dim=64)) == -1
    assert _encode(zf, _desc(zf, page_size=24)) == -1
    assert _encode(zf, _desc(zf, page_size=256)) == -2
    assert _encode(zf, _desc(zf, reserved=1)) == -1
    assert _encode(zf, _desc(zf, k_comp=0x1008)) == -1            # misaligned pool
    assert _encode(zf, _desc(zf, dir=None)) == -1
    assert _encode(zf, _desc(zf), src=0x10002) == -1             # misaligned source
    assert _encode(zf, _desc(zf), ids=None) == -1
    assert _encode(zf, _desc(zf), n=-1) == -1
    assert _encode(zf, _desc(zf), flags=4) == -1
    assert _encode(zf, _desc(zf), n=0) == 0                      # nothing to do, nothing launched
    assert _encode(zf, _desc(zf, k_comp=None), n=0) == -1
    assert _encode(zf, _desc(zf, k_comp=None), n=0, flags=1) == 0  # forced raw needs no compressed pools


def test_decompress_rejects_bad_arguments(zf):
    f = zf.lib().zf_decompress
    d = _desc(zf)
    assert f(None, 0x1000, 1, 0x2000, 0x3000, None) == -1
    assert f(ctypes.byref(d), None, 1, 0x2000, 0x3000, None) == -1
    assert f(ctypes.byref(d), 0x1000, 1, 0x2001, 0x3000, None) == -1
    assert f(ctypes.byref(d), 0x1000, 0, 0x2000, 0x3000, None) == 0
    # every pool the descriptor sizes must be present: the directory may point into any of them
    for pool in ("k_comp", "v_comp", "k_raw", "v_raw", "dir"):
        bad = _desc(zf, **{pool: None})
        for g in (zf.lib().zf_decompress, zf.lib().zf_decompress_to_raw):
            assert g(ctypes.byref(bad), 0x1000, 1, 0x2000, 0x3000, None) == -1, pool
    assert zf.lib().zf_decompress_to_raw(ctypes.byref(d), 0x1000, 1, 0x2000, 0x3008, None) == -1


def test_append_rejects_bad_arguments_before_launch(zf):
    f = zf.lib().zf_append_tokens

    def call(desc, n=1, tok=0x10000, ids=0x20000, pos=0x30000, slots=0x40000):
        return f(ctypes.byref(desc) if desc is not None else None, tok, tok, ids, pos, slots, n, None)
    assert call(None) == -1
    assert call(_desc(zf, k_raw=None)) == -1                     # needs the raw pools
    assert call(_desc(zf, k_comp=None)) == -1                    # and the compressed ones
    assert call(_desc(zf, v_raw=0x4008)) == -1                   # misaligned raw pool
    assert call(_desc(zf), tok=None) == -1
    assert call(_desc(zf), pos=None) == -1
    assert call(_desc(zf), slots=None) == -1
    assert call(_desc(zf), n=-1) == -1
    assert call(_desc(zf), n=0) == 0                             # nothing to do, nothing launched


def test_validate_rejects_bad_arguments_before_launch(zf):
    f = zf.lib().zf_validate_pages
    d = _desc(zf)
    assert f(None, 0x1000, 1, 0x2000, None) == -1
    assert f(ctypes.byref(_desc(zf, k_comp=None)), 0x1000, 1, 0x2000, None) == -1
    assert f(ctypes.byref(d), None, 1, 0x2000, None) == -1
    assert f(ctypes.byref(d), 0x1000, 1, 0x2002, None) == -1       # misaligned flag array
    assert f(ctypes.byref(d), 0x1000, -1, 0x2000, None) == -1
    assert f(ctypes.byref(d), 0x1000, 0, 0x2000, None) == 0
    assert zf.lib().zf_slot_is_valid(None) == 0


def _attn(zf, desc, batch=2, hq=8, max_pages=4, q=0x10000, out=0x20000, lse=0x30000, ws=0x40000, ws_bytes=1 << 20,
          dense=False, scale=0.1):
    f = zf.lib().zf_dense_decode_attn if dense else zf.lib().zf_decode_attn
    return f(ctypes.byref(desc), q, batch, hq, 0x50000, max_pages, 0x60000, scale, out, lse, ws, ws_bytes, None)


@pytest.mark.parametrize("dense", [False, True])
def test_attention_rejects_bad_arguments(zf, dense):
    d = _desc(zf)
    assert _attn(zf, d, batch=4097, dense=dense) == -1                  # above ZF_MAX_BATCH
    assert _attn(zf, d, hq=7, dense=dense) == -1                        # 7 query heads over 2 kv heads
    assert _attn(zf, d, hq=1, dense=dense) == -1                        # fewer query heads than kv heads
    assert _attn(zf, d, max_pages=0, dense=dense) == -1
    assert _attn(zf, d, q=None, dense=dense) == -1
    assert _attn(zf, d, q=0x10004, dense=dense) == -1
    assert _attn(zf, d, out=0x20008, dense=dense) == -1
    assert _attn(zf, d, lse=0x30002, dense=dense) == -1
    assert _attn(zf, d, ws=None, dense=dense) == -1
    assert _attn(zf, d, scale=float("nan"), dense=dense) == -1
    assert _attn(zf, _desc(zf, head_dim=96), dense=dense) == -1
    assert _attn(zf, d, batch=0, dense=dense) == 0                      # empty batch: no launch


def test_compressed_attention_needs_a_directory(zf):
    assert _attn(zf, _desc(zf, dir=None)) == -1
    assert _attn(zf, _desc(zf, k_comp=None)) == -1


def test_python_binding_has_no_fallback(zf, monkeypatch, tmp_path):
    monkeypatch.setattr(zf, "_LIB", None)
    monkeypatch.setattr(zf, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(zf.ZfError):
        zf.lib()


@pytest.mark.parametrize("dense", [False, True])
def test_multi_token_attention_rejects_bad_token_counts(zf, dense):
    d = _desc(zf)
    f = zf.lib().zf_dense_decode_attn_multi if dense else zf.lib().zf_decode_attn_multi

    def call(tokens, hq=8):
        return f(ctypes.byref(d), 0x10000, 2, tokens, hq, 0x50000, 4, 0x60000, 0.1, 0x20000, 0x30000, 0x40000,
                 1 << 20, None)
    assert call(0) == -1
    assert call(-3) == -1
    assert call(65) == -1                                            # above ZF_MAX_TOKENS
    assert call(2, hq=7) == -1                                       # heads still a multiple of kv heads
    assert zf.lib().zf_decode_attn_multi_workspace_size(1, 0, 8, 2, 16, 4) == 0
    assert zf.lib().zf_decode_attn_multi_workspace_size(1, 2, 7, 2, 16, 4) == 0


def test_kernel_choice_is_checked(zf):
    """zf_decode_attn_multi_kernel rejects an unknown kernel before anything is launched."""
    f = zf.lib().zf_decode_attn_multi_kernel
    d = _desc(zf)
    for bad in (-1, 3, 99):
        assert f(ctypes.byref(d), 0x1000, 1, 1, 4, 0x2000, 4, 0x3000, 0.1, 0x4000, 0x5000, 0x6000, 1 << 20, bad,
                 None) == -1
    assert zf.KERNELS == {"auto": 0, "warp_mma": 1, "tcgen05": 2}


def test_product_path_never_touches_the_oracle():
    """The library and its binding neither import nor read anything under oracle/ (the oracle is
    test infrastructure; a product path through it would be a CPU fallback)."""
    pkg = os.path.join(ROOT, "decode_attention_compressed_gb300")
    offenders = []
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                if re.search(r"^\s*(from|import)\s+oracle\b|zf_oracle|[\"']oracle[/\"']", text, flags=re.M):
                    offenders.append(f)
    assert offenders == []
