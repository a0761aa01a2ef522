"""ctypes binding of libskv.so with the C ABI's own names (include/skv.h).

Argument marshalling only: every step of the coder runs in the library's
CUDA kernels. The library is loaded on first use; if it is missing or does
not load, the call raises -- there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libskv.so")

SKV_BF16, SKV_E4M3 = 0, 1
SKV_FORMAT_VERSION = 1
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "CUDA", 3: "NONFINITE_MU", 4: "BAD_SIGMA",
                5: "EMPTY_MARGINAL", 6: "CAPACITY", 7: "CORRUPT", 8: "TIMEOUT"}


class skv_layout(C.Structure):
    _fields_ = [("version", C.c_uint32), ("dtype", C.c_uint32), ("n_layers", C.c_uint32),
                ("n_kv", C.c_uint32), ("n_heads", C.c_uint32), ("head_dim", C.c_uint32),
                ("n_tokens", C.c_uint64), ("tokens_per_chunk", C.c_uint32),
                ("streams_per_chunk", C.c_uint32), ("w_narrow", C.c_uint32),
                ("w_wide", C.c_uint32), ("w_marginal", C.c_uint32),
                ("sigma_block_tokens", C.c_uint32)]


# name -> (restype, argtypes); the exported symbols of include/skv.h
_u32, _u64, _i32, _vp = C.c_uint32, C.c_uint64, C.c_int32, C.c_void_p
_LP = C.POINTER(skv_layout)
SIGNATURES = {
    "skv_version": (_u32, []),
    "skv_status_string": (C.c_char_p, [_i32]),
    "skv_layout_init": (_i32, [_LP, _u32, _u32, _u32, _u32, _u32, _u64]),
    "skv_layout_check": (_i32, [_LP]),
    "skv_num_chunks": (_i32, [_LP, C.POINTER(_u64)]),
    "skv_max_encoded_bytes": (_i32, [_LP, C.POINTER(_u64)]),
    "skv_workspace_bytes": (_i32, [_LP, _i32, C.POINTER(_u64)]),
    "skv_encode": (_i32, [_LP, _vp, _vp, _vp, _vp, _vp, _u64, _vp, _vp, _vp, _u64, _vp]),
    "skv_decode": (_i32, [_LP, _vp, _u64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _u64, _vp]),
    "skv_decode_chunks": (_i32, [_LP, _vp, _u64, _vp, _vp, _vp, _vp, _vp, _u32, _vp, _vp, _vp,
                                 _u64, _vp]),
    "skv_cdf_eval": (_i32, [_LP, _vp, _u64, _vp, _vp, _vp, _vp, _vp, _vp, _u64, _vp]),
    "skv_decode_noalloc": (_i32, [_LP, _vp, _u64, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "skv_decode_prepare": (_i32, [_LP, _vp, _vp, _vp, _vp, _u64, _vp]),
    "skv_decode_chunks_prepared": (_i32, [_LP, _vp, _u64, _vp, _vp, _vp, _u32, _vp, _vp, _vp, _u64, _vp]),
    "skv_histogram": (_i32, [_u32, _vp, _u64, _vp, _i32, _vp]),
    "skv_decode_offload": (_i32, [_LP, _vp, _u64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _u64, _vp,
                                  _u64, _vp, _vp]),
    "skv_requantize": (_i32, [_u32, _u32, _vp, _u64, _vp, _vp, _vp, _u64, _vp]),
    "skv_host_staging_bytes": (_i32, [_LP, _u32, _i32, C.POINTER(_u64)]),
    "skv_encode_host": (_i32, [_LP, _vp, _vp, _vp, _vp, _vp, _u64, _vp, _vp, _vp, _u64, _u32, _vp, _vp, _vp]),
    "skv_decode_host": (_i32, [_LP, _vp, _u64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _u64, _u32, _vp, _vp, _vp]),
    "skv_search_eval": (_i32, [_LP, _vp, _u64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _u64, _vp]),
    "skv_peak_probe": (_i32, [_i32, _u32, _vp, C.POINTER(_u64), _vp]),
    "skv_op_table": (_i32, [_i32, C.POINTER(_u32), C.POINTER(_u32), _u32]),
    "skv_decode_pages_host": (_i32, [_LP, _vp, _u64, _vp, _vp, _vp, _u32, _vp, _vp, _vp, _u64, _vp, _u64, _vp,
                                     _vp]),
    "skv_offload_plan": (_i32, [_vp, _u64, _u64, _u64, _vp, _u64, C.POINTER(_u64)]),
    "skv_calibrate_sigma": (_i32, [_LP, _vp, _vp, _vp, _u64, _vp, _vp]),
}

_lib = None


class SKVError(RuntimeError):
    def __init__(self, where: str, status: int):
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")
        self.status = status
        self.name = STATUS_NAMES.get(status, str(status))


def lib():
    """The loaded library; builds it in-tree first if it is absent or stale."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH) or os.environ.get("SKV_NO_AUTOBUILD") != "1":
            from . import build as _build
            _build.build()
        try:
            L = C.CDLL(LIB_PATH)
        except OSError as e:
            raise RuntimeError(f"the SKV CUDA library {LIB_PATH} does not load: {e}") from e
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def check(where: str, rc: int):
    if rc != 0:
        raise SKVError(where, rc)
