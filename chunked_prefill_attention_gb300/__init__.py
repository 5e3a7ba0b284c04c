"""Chunked Q8_0-KV causal prefill attention for NVIDIA GB300 (sm_103a).

The compute path is the C-ABI library libq8attn.so (kernels in csrc/, ABI in
include/q8attn.h); `q8attn` is its Python binding.  `workloads` draws the
seeded synthetic inputs.  Importing the package does not load the library;
the first call does, and fails loudly when it is missing.
"""

__all__ = ["q8attn", "workloads"]
