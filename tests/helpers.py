"""Shared helpers for the GPU parity tests: build the same cache with the CUDA library and with
the oracle from one set of seeded inputs, and compare."""
import numpy as np
import torch

from decode_attention_compressed_gb300 import build as B
from decode_attention_compressed_gb300 import inputs as I

# correctness bars for attention (float32 kernel vs float64 oracle)
MAX_ABS = 4e-3
MEAN_ABS = 5e-4
LSE_ABS = 1e-3


def zf_module():
    B.build()
    from decode_attention_compressed_gb300 import zf
    zf.lib()
    return zf


def late_writer():
    """The test-only kernel of late_writer.cu (built on first use into tests/_build): late_copy(src0,
    dst0, n0, src1, dst1, n1, delay_ns, stream) lets the next grid start at once and copies the
    int32 arrays about delay_ns later."""
    import ctypes
    import os
    import subprocess
    here = os.path.dirname(os.path.abspath(__file__))
    out_dir = os.path.join(here, "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, "liblate_writer.so")
    src = os.path.join(here, "late_writer.cu")
    if not os.path.exists(so) or os.path.getmtime(so) < os.path.getmtime(src):
        subprocess.run([B.nvcc(), *B.ARCH, "-O2", "-shared", "-Xcompiler", "-fPIC", src, "-o", so], check=True)
    lib = ctypes.CDLL(so)
    fn = lib.late_copy
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                   ctypes.c_longlong, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


def np_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().view(np.uint16)


def gpu_cache_from(layer: I.LayerInputs, zf, raw_slots=None, force_raw=False, page_ids=None, extra_raw=0):
    """Encode every pool page of `layer` on the GPU (page i of the pool keeps id i unless page_ids
    says otherwise).  Raw slot i is offered to page i by default."""
    npg = layer.num_pages
    ids = list(range(npg)) if page_ids is None else list(page_ids)
    rs = list(range(npg)) if raw_slots is None else list(raw_slots)
    cache = zf.Cache(npg, layer.workload.num_kv_heads, layer.workload.page_size, npg + extra_raw)
    dev = torch.device("cuda")
    zf.encode_pages(cache, layer.k_pages.to(dev), layer.v_pages.to(dev), ids, layer.n_valid.cpu().tolist(), rs,
                    force_raw=force_raw)
    torch.cuda.synchronize()
    return cache


def oracle_cache_from(layer: I.LayerInputs, O, raw_slots=None, force_raw=False, page_ids=None, extra_raw=0):
    npg = layer.num_pages
    ids = list(range(npg)) if page_ids is None else list(page_ids)
    rs = list(range(npg)) if raw_slots is None else list(raw_slots)
    cache = O.Cache(num_pages=npg, num_kv_heads=layer.workload.num_kv_heads, page_size=layer.workload.page_size,
                    num_raw=npg + extra_raw)
    O.encode_pages(cache, np_bits(layer.k_pages), np_bits(layer.v_pages), ids, layer.n_valid.cpu().numpy(), rs,
                   force_raw=force_raw)
    return cache


def assert_caches_equal(gc, oc):
    """Bit-exact comparison of the GPU cache against the oracle cache: directory, status, and the
    bytes of every slot the directory points at."""
    gdir = gc.dir.cpu().numpy()
    assert (gdir == oc.dir).all(), np.argwhere(gdir != oc.dir)[:10]
    assert gc.status_word() == oc.status
    kc, vc = gc.k_comp.cpu().numpy(), gc.v_comp.cpu().numpy()
    kr, vr = np_bits(gc.k_raw), np_bits(gc.v_raw)
    comp = np.argwhere(oc.dir == -1)
    if len(comp):
        p, h = comp[:, 0], comp[:, 1]
        assert (kc[p, h] == oc.k_comp[p, h]).all()
        assert (vc[p, h] == oc.v_comp[p, h]).all()
    raw = np.argwhere(oc.dir >= 0)
    if len(raw):
        p, h = raw[:, 0], raw[:, 1]
        s = oc.dir[p, h]
        assert (kr[s, h] == oc.k_raw[s, h]).all()
        assert (vr[s, h] == oc.v_raw[s, h]).all()


def compare_attention(out, lse, ref_out, ref_lse, pairs=None):
    """Apply the correctness bars; returns (max_abs, mean_abs, max_lse_abs)."""
    out = out.detach().cpu().numpy().astype(np.float64)
    lse = lse.detach().cpu().numpy().astype(np.float64)
    if pairs is not None:
        idx = tuple(np.array(pairs).T)
        out, lse, ref_out, ref_lse = out[idx], lse[idx], ref_out[idx], ref_lse[idx]
    empty = np.isneginf(ref_lse)
    assert (np.isneginf(lse) == empty).all()
    assert (out[empty] == 0).all()
    d = np.abs(out - ref_out)
    dl = np.abs(lse[~empty] - ref_lse[~empty]) if (~empty).any() else np.zeros(1)
    stats = (float(d.max()), float(d.mean()), float(dl.max()))
    assert stats[0] <= MAX_ABS and stats[1] <= MEAN_ABS and stats[2] <= LSE_ABS, stats
    return stats
