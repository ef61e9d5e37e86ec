"""GB300-native split-KV paged-attention decode.

``binding``    -- ctypes binding of libpa_decode.so (the C ABI in include/pa_decode.h)
``workloads``  -- seeded synthetic decode inputs (no attention arithmetic)
``build``      -- nvcc build of the library for sm_103a

The binding is imported lazily so that the workload generators can be used
without the compiled library.
"""
__all__ = ["binding", "workloads", "build"]
