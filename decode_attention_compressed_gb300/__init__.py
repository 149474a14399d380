"""Decode attention over a losslessly compressed BF16 paged KV cache, for GB300 (sm_103a).

The compute lives in the CUDA library ``libzf.so`` (C ABI declared in ``include/zf.h``);
``decode_attention_compressed_gb300.zf`` is a thin ctypes binding over it.  Importing this package
does not load the library; the binding loads it on first use and raises if it is missing.
"""
