"""Kimi Delta Attention (KDA) on one GB300: a C-ABI CUDA library and its Python binding.

``kda_chunk_fwd``   chunk-parallel prefill of the gated delta-rule layer.
``kda_decode_step`` single-token recurrent decode, state updated in place.

The compiled library (``csrc/`` -> ``libkda.so``) is loaded lazily on first
use; importing this package does not require a GPU.
"""
from .binding import (  # noqa: F401
    KdaError,
    build,
    kda_chunk_fwd,
    kda_decode_step,
    kda_get_device_error,
    library_path,
    load,
)

__all__ = ["KdaError", "build", "kda_chunk_fwd", "kda_decode_step",
           "kda_get_device_error", "library_path", "load"]
