"""Batch-invariant MoE prefill numerics for one GB300 (sm_103a).

The product is the C-ABI library libbi.so (include/bi.h), built from
csrc/ for sm_103a.  `binding` is its thin ctypes binding; `synth` holds the
seeded synthetic input generators shared by tests and the benchmark.
Importing this package loads nothing: call `binding.load()`.
"""
__all__ = ["binding", "synth", "build"]
