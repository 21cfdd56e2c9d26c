"""GB300-native tensor-parallel Llama decoder forward, t ranks emulated as
shard buffers on one GPU.  The compute path is the C ABI in include/tp.h
(CUDA kernels for sm_103a); this package holds its build script and thin
Python bindings."""
from . import binding  # noqa: F401

__all__ = ["binding", "runtime", "build"]
