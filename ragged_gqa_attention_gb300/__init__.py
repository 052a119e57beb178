"""Ragged GQA fused attention for GB300 (sm_103a).

The compute lives in the CUDA library ``lib/librga.so`` (C ABI:
``include/rga.h``); this package is its Python binding plus the seeded input
generators used by the tests and the benchmark.
"""
from .binding import (RgaError, device_status, load, trt_attention,  # noqa: F401
                      trt_quantized_attention)
from .buildlib import build  # noqa: F401
