"""CSA2 global-attention step over an FP4 (E2M1) main KV cache on B300.

The compute lives in libcsa2.so (CUDA kernels for sm_103a behind the C ABI
in include/csa2.h); `csa2` is its Python binding and `synth` draws the
seeded synthetic workloads.
"""
