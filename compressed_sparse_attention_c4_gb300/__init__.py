"""GB300 (sm_103a) library for DeepSeek-V4-style compressed sparse attention.

The compute lives in the C-ABI shared library ``libdsv4sa.so`` (CUDA kernels
for sm_103a); ``compressed_sparse_attention_c4_gb300.dsv4sa`` is a thin ctypes
binding that passes torch tensors to it as raw pointers.  ``workloads`` builds
the seeded synthetic inputs.
"""
__all__ = ["dsv4sa", "workloads"]
