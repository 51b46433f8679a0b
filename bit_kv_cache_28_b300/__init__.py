"""bitkv: softmax attention over a 2-bit / mixed-precision quantised KV cache on B300 (sm_103a).

The compute path is ``libbitkv.so`` (CUDA kernels behind a C ABI, declared in
``include/bitkv.h``); :mod:`bit_kv_cache_28_b300.bitkv` is a thin ctypes binding
with the same call names.  Importing this package does not load the library;
the first call through the binding does, and raises if it is missing.
"""

__all__ = ["bitkv", "synth"]
