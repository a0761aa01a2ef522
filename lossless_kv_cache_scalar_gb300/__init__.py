"""GB300-native speculative KV coding: lossless entropy coding of KV-cache
scalars against a predictor (mu, sigma) under the three-component mixture of
the Speculative KV Coding wiki. The work runs in libskv.so (include/skv.h);
this package is its binding and the seeded synthetic workloads.
"""
from ._binding import SKVError, SKV_BF16, SKV_E4M3, STATUS_NAMES, lib  # noqa: F401
from .api import (Coder, HostCoder, Layout, calibrate_sigma, cdf_eval, decode,  # noqa: F401
                  decode_chunks, encode, histogram, requantize)

__all__ = ["Coder", "HostCoder", "Layout", "SKVError", "calibrate_sigma", "cdf_eval", "decode",
           "decode_chunks", "encode", "histogram", "lib", "requantize"]
