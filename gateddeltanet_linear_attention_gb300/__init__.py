"""GB300 (sm_103a) GatedDeltaNet mixer: hand-written CUDA kernels behind a C ABI.

The C ABI is declared in include/gdn.h; ``gateddeltanet_linear_attention_gb300.gdn``
is the thin ctypes binding with the same entry-point names, ``.inputs`` the
seeded synthetic-input generator and ``.build_lib`` the in-tree nvcc build.
The compiled library is loaded on first use and the binding raises if it is
missing: there is no CPU fallback.
"""
__all__ = ["gdn", "inputs", "build_lib"]
