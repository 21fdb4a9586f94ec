"""GB300-native dense GEMM: D = alpha * op(A) @ op(B) + beta * C on sm_103a.

The compute path is a C-ABI shared library built from ``csrc/`` (TMA,
tcgen05 tensor cores, tensor memory); ``gemm`` below is its thin ctypes
binding.  Importing this package does not load the library; the first use
of ``gemm`` does, and raises if it has not been built.
"""

__all__ = ["gemm", "gemm_status_string", "gemm_poll_device_error", "inputs"]


def __getattr__(name):
    if name in ("gemm", "gemm_status_string", "gemm_poll_device_error", "GemmError",
                "library", "load_library"):
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
