"""group_affine_bit_gb300: a GB300 (sm_103a) library for the MLX-style
group-affine quantized linear projection, y = bf16(x . bf16(s*q + b)^T).

The compute path is libaffqmm.so (C ABI in include/affqmm.h, CUDA kernels in
csrc/); ``api`` is its thin Python binding and ``synth`` draws seeded
synthetic inputs.  Build the library with ``build.build()``.
"""

__all__ = ["api", "build", "synth"]
