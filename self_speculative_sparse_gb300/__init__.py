"""Vegas verification-guided sparse self-speculative decoding: the GB300 hot path.

The compute lives in ``libvg.so`` (CUDA for sm_103a behind the C ABI of
``include/vg.h``); ``binding`` marshals arguments to it and ``runtime`` holds the
device-resident workload (KV cache slot pool, workspace, outputs) around it.
Importing this package does not load the library; the first call does, and fails
loudly if it has not been built.
"""
from . import binding  # noqa: F401

__all__ = ["binding"]
__version__ = "0.1.0"
