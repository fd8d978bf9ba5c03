"""Top-k Mixture-of-Experts FFN forward pass for NVIDIA B300 (sm_103a).

The compute lives in libmoe.so (CUDA kernels behind the C ABI in include/moe.h); the
binding is `mixture_experts_sparse_02_b300.moe`.  Build the library with
`python -m mixture_experts_sparse_02_b300.build`.
"""
