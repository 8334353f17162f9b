"""GB300 (sm_103a) DeepSeek-V4 DSA indexer hot path: indexer score, fused top-k and the
paged mxfp4 gather, as a C-ABI CUDA library (include/dsa.h) with a thin ctypes binding.

Submodules: ``dsa`` (the binding), ``device`` (torch-owned device buffers for a batch),
``synth`` (seeded synthetic workloads), ``build`` (nvcc build of the library).
"""
__all__ = ["dsa", "device", "synth", "build"]
