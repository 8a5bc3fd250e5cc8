"""cross_context_kv_gb300 -- repair of reused KV-cache chunks on one NVIDIA GB300.

The compute lives in libkvfix.so (hand-written CUDA for sm_103a, C ABI in
include/kvfix.h); `kvfix` is its thin ctypes binding and `synth` the seeded synthetic
workloads.  Build the library with `cross_context_kv_gb300.build.build()`.
"""
__all__ = ["kvfix", "synth", "build"]
