"""GB300-native INT8-KV decode attention.

``kvq8`` is the Python binding of the C-ABI library ``libkvq8.so`` (CUDA
kernels for sm_103a); ``workloads`` draws the seeded synthetic inputs.
Importing the package loads nothing: the library is opened on first use,
and every entry point raises if it cannot be opened (there is no CPU path).
"""
__all__ = ["kvq8", "workloads"]
