"""ctypes wrapper of the CPU oracle (oracle/skv_oracle.c).

TEST INFRASTRUCTURE: the oracle checks the CUDA library; it is not part of it.
Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg (and its
`--impl reference` arm) import this module. It never imports the library
package and the library never imports it.

Arrays are numpy: codes as uint16 (bf16) or uint8 (e4m3) in the canonical
[n_layers][n_kv][T][H][D] order, sigma as float32 [n_layers][n_kv][H][D],
counts as uint64 [N] indexed by code.
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass

import numpy as np

from . import build as _build

BF16, E4M3 = 0, 1
STATUS = {0: "OK", 1: "INVALID_ARG", 3: "NONFINITE_MU", 4: "BAD_SIGMA",
          5: "EMPTY_MARGINAL", 6: "CAPACITY", 7: "CORRUPT", 9: "NOMEM"}


class OracleError(RuntimeError):
    def __init__(self, status: int):
        super().__init__(f"oracle status {status} ({STATUS.get(status, '?')})")
        self.status = status
        self.name = STATUS.get(status, "?")


class _Layout(C.Structure):
    _fields_ = [("dtype", C.c_uint32), ("n_layers", C.c_uint32), ("n_kv", C.c_uint32),
                ("n_heads", C.c_uint32), ("head_dim", C.c_uint32), ("n_tokens", C.c_uint64),
                ("tokens_per_chunk", C.c_uint32), ("streams_per_chunk", C.c_uint32),
                ("w_n", C.c_uint32), ("w_w", C.c_uint32), ("w_h", C.c_uint32),
                ("sigma_block", C.c_uint32)]


@dataclass
class Layout:
    dtype: int
    n_layers: int
    n_kv: int
    n_heads: int
    head_dim: int
    n_tokens: int
    tokens_per_chunk: int = 256
    streams_per_chunk: int = 64
    w_n: int = 95
    w_w: int = 3
    w_h: int = 2
    sigma_block: int = 0       # tokens per sigma block (0: one sigma per channel)

    def c(self) -> _Layout:
        return _Layout(self.dtype, self.n_layers, self.n_kv, self.n_heads, self.head_dim,
                       self.n_tokens, self.tokens_per_chunk, self.streams_per_chunk,
                       self.w_n, self.w_w, self.w_h, self.sigma_block)

    @property
    def n_sigma_blocks(self) -> int:
        return -(-self.n_tokens // self.sigma_block) if self.sigma_block else 1

    @property
    def sigma_shape(self) -> tuple:
        if self.sigma_block:
            return (self.n_layers, self.n_kv, self.n_sigma_blocks, self.n_heads, self.head_dim)
        return (self.n_layers, self.n_kv, self.n_heads, self.head_dim)

    @property
    def n_codes(self) -> int:
        return 65536 if self.dtype == BF16 else 256

    @property
    def code_dtype(self):
        return np.uint16 if self.dtype == BF16 else np.uint8

    @property
    def n_elems(self) -> int:
        return self.n_layers * self.n_kv * self.n_tokens * self.n_heads * self.head_dim


_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        u32, u64, f32, vp = C.c_uint32, C.c_uint64, C.c_float, C.c_void_p
        L.oracle_ord.restype = u32
        L.oracle_ord.argtypes = [u32, u32]
        L.oracle_code.restype = u32
        L.oracle_code.argtypes = [u32, u32]
        L.oracle_value.restype = f32
        L.oracle_value.argtypes = [u32, u32]
        L.oracle_edge.restype = f32
        L.oracle_edge.argtypes = [u32, u32]
        L.oracle_phi_q.restype = u32
        L.oracle_phi_q.argtypes = [C.c_int32]
        L.oracle_phi_table.argtypes = [vp]
        L.oracle_cdf_all.argtypes = [u32, u32, f32, u32, u32, u32, vp, vp]
        L.oracle_cdf_eval.argtypes = [u32, u32, u32, u32, vp, u64, vp, vp, vp, vp]
        L.oracle_find_symbols.argtypes = [u32, u32, f32, u32, u32, u32, vp, u64, vp, vp]
        L.oracle_num_chunks.argtypes = [C.POINTER(_Layout), C.POINTER(u64)]
        L.oracle_max_encoded_bytes.argtypes = [C.POINTER(_Layout), C.POINTER(u64)]
        L.oracle_encode_chunks.argtypes = [C.POINTER(_Layout), vp, vp, vp, vp, vp, u64, vp, u64,
                                           vp, u32]
        L.oracle_decode.argtypes = [C.POINTER(_Layout), vp, u64, vp, vp, vp, vp, vp, u32]
        L.oracle_decode_pages.argtypes = [C.POINTER(_Layout), vp, u64, vp, vp, vp, vp, vp, u64,
                                          vp, u32]
        L.oracle_ideal_bits.restype = C.c_double
        L.oracle_ideal_bits.argtypes = [C.POINTER(_Layout), vp, vp, vp, vp]
        L.oracle_model_bits.restype = C.c_double
        L.oracle_model_bits.argtypes = [C.POINTER(_Layout), vp, vp, vp, vp]
        L.oracle_histogram.argtypes = [u32, vp, u64, vp, C.c_int]
        L.oracle_calibrate_sigma.argtypes = [C.POINTER(_Layout), vp, vp, vp, u64, vp]
        L.oracle_requantize.argtypes = [u32, u32, vp, u64, vp, vp, vp, vp, u64]
        _lib = L
    return _lib


def _p(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _check(st: int):
    if st != 0:
        raise OracleError(st)


def threads() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


# ------------------------------------------------------------ scalar pieces

def ord_(dtype: int, code: int) -> int:
    return lib().oracle_ord(dtype, code)


def code(dtype: int, o: int) -> int:
    return lib().oracle_code(dtype, o)


def value(dtype: int, code_: int) -> float:
    return lib().oracle_value(dtype, code_)


def edge(dtype: int, o: int) -> float:
    return lib().oracle_edge(dtype, o)


def phi_q(zq: int) -> int:
    return lib().oracle_phi_q(zq)


def phi_table() -> np.ndarray:
    t = np.zeros(4097, np.uint32)
    lib().oracle_phi_table(_p(t))
    return t


def _counts_arg(dtype: int, counts):
    n = 65536 if dtype == BF16 else 256
    if counts is None:
        counts = np.zeros(n, np.uint64)
    return np.ascontiguousarray(counts, np.uint64)


def cdf_all(dtype: int, mu_code: int, sigma: float, weights=(95, 3, 2), counts=None) -> np.ndarray:
    """C(o) for o = 0..N for one (mu, sigma)."""
    n = 65536 if dtype == BF16 else 256
    counts = _counts_arg(dtype, counts)
    out = np.zeros(n + 1, np.uint64)
    _check(lib().oracle_cdf_all(dtype, mu_code, float(sigma), *weights, _p(counts), _p(out)))
    return out


def cdf_eval(dtype: int, mu_codes, sigmas, ords, weights=(95, 3, 2), counts=None) -> np.ndarray:
    counts = _counts_arg(dtype, counts)
    mu_codes = np.ascontiguousarray(mu_codes, np.uint32)
    sigmas = np.ascontiguousarray(sigmas, np.float32)
    ords = np.ascontiguousarray(ords, np.uint32)
    out = np.zeros(len(ords), np.uint64)
    _check(lib().oracle_cdf_eval(dtype, *weights, _p(counts), len(ords), _p(mu_codes),
                                 _p(sigmas), _p(ords), _p(out)))
    return out


def find_symbols(dtype: int, mu_code: int, sigma: float, slots, weights=(95, 3, 2),
                 counts=None) -> np.ndarray:
    counts = _counts_arg(dtype, counts)
    slots = np.ascontiguousarray(slots, np.uint64)
    out = np.zeros(len(slots), np.uint32)
    _check(lib().oracle_find_symbols(dtype, mu_code, float(sigma), *weights, _p(counts),
                                     len(slots), _p(slots), _p(out)))
    return out


# ------------------------------------------------------------ whole streams

def num_chunks(lay: Layout) -> int:
    n = C.c_uint64()
    _check(lib().oracle_num_chunks(C.byref(lay.c()), C.byref(n)))
    return n.value


def max_encoded_bytes(lay: Layout) -> int:
    n = C.c_uint64()
    _check(lib().oracle_max_encoded_bytes(C.byref(lay.c()), C.byref(n)))
    return n.value


def _inputs(lay, kv, mu, sigma, counts):
    cd = lay.code_dtype
    kv = None if kv is None else np.ascontiguousarray(kv).view(cd).reshape(-1)
    mu = np.ascontiguousarray(mu).view(cd).reshape(-1)
    sigma = np.ascontiguousarray(sigma, np.float32).reshape(-1)
    if sigma.size != int(np.prod(lay.sigma_shape)):
        raise ValueError(f"sigma has {sigma.size} entries, the layout needs {lay.sigma_shape}")
    if mu.size != lay.n_elems or (kv is not None and kv.size != lay.n_elems):
        raise ValueError("kv / mu sizes do not match the layout")
    counts = _counts_arg(lay.dtype, counts)
    return kv, mu, sigma, counts


def encode(lay: Layout, kv, mu, sigma, counts, chunk_ids=None, nthreads: int | None = None):
    """Encode all chunks (or the listed ones). Returns (bitstream uint8, offsets uint64)."""
    kv, mu, sigma, counts = _inputs(lay, kv, mu, sigma, counts)
    cap = max_encoded_bytes(lay)
    ids = None
    n_ids = num_chunks(lay)
    if chunk_ids is not None:
        ids = np.ascontiguousarray(chunk_ids, np.uint64)
        n_ids = len(ids)
    out = np.zeros(max(cap, 16), np.uint8)
    offs = np.zeros(n_ids + 1, np.uint64)
    st = lib().oracle_encode_chunks(C.byref(lay.c()), _p(kv), _p(mu), _p(sigma), _p(counts),
                                    _p(ids), n_ids, _p(out), cap, _p(offs),
                                    nthreads or threads())
    _check(st)
    return out[: int(offs[-1])].copy(), offs


def decode(lay: Layout, stream, offsets, mu, sigma, counts, nthreads: int | None = None):
    _, mu, sigma, counts = _inputs(lay, None, mu, sigma, counts)
    stream = np.ascontiguousarray(stream, np.uint8)
    offsets = np.ascontiguousarray(offsets, np.uint64)
    out = np.zeros(lay.n_elems, lay.code_dtype)
    st = lib().oracle_decode(C.byref(lay.c()), _p(stream), stream.size, _p(offsets), _p(mu),
                             _p(sigma), _p(counts), _p(out), nthreads or threads())
    _check(st)
    return out


def decode_pages(lay: Layout, stream, offsets, mu, sigma, counts, chunk_ids,
                 nthreads: int | None = None):
    _, mu, sigma, counts = _inputs(lay, None, mu, sigma, counts)
    stream = np.ascontiguousarray(stream, np.uint8)
    offsets = np.ascontiguousarray(offsets, np.uint64)
    ids = np.ascontiguousarray(chunk_ids, np.uint64)
    page = lay.tokens_per_chunk * lay.n_heads * lay.head_dim
    out = np.zeros(len(ids) * page, lay.code_dtype)
    st = lib().oracle_decode_pages(C.byref(lay.c()), _p(stream), stream.size, _p(offsets),
                                   _p(mu), _p(sigma), _p(counts), _p(ids), len(ids), _p(out),
                                   nthreads or threads())
    _check(st)
    return out.reshape(len(ids), page)


def ideal_bits(lay: Layout, kv, mu, sigma, counts) -> float:
    kv, mu, sigma, counts = _inputs(lay, kv, mu, sigma, counts)
    return lib().oracle_ideal_bits(C.byref(lay.c()), _p(kv), _p(mu), _p(sigma), _p(counts))


def model_bits(lay: Layout, kv, mu, sigma, counts) -> float:
    kv, mu, sigma, counts = _inputs(lay, kv, mu, sigma, counts)
    return lib().oracle_model_bits(C.byref(lay.c()), _p(kv), _p(mu), _p(sigma), _p(counts))


# ------------------------------------------------- model inputs: p_hat, sigma

def histogram(dtype: int, codes, counts=None) -> np.ndarray:
    """Counts of every code bit pattern (uint64[N]); adds to `counts` if given."""
    n = 65536 if dtype == BF16 else 256
    codes = np.ascontiguousarray(codes, np.uint16 if dtype == BF16 else np.uint8).reshape(-1)
    acc = counts is not None
    out = np.ascontiguousarray(counts, np.uint64).copy() if acc else np.zeros(n, np.uint64)
    _check(lib().oracle_histogram(dtype, _p(codes), codes.size, _p(out), int(acc)))
    return out


def calibrate_sigma(lay: Layout, kv: np.ndarray, mu: np.ndarray, t_cal: int,
                    mask: np.ndarray | None = None) -> np.ndarray:
    """Frozen per-channel sigma (float32 [n_layers][n_kv][H][D], or per sigma block
    [n_layers][n_kv][n_blocks][H][D]) from the first t_cal tokens (of each block)."""
    cd = lay.code_dtype
    kv = np.ascontiguousarray(kv).view(cd)
    mu = np.ascontiguousarray(mu).view(cd)
    if mask is not None:
        mask = np.ascontiguousarray(mask).view(np.uint8)
    out = np.zeros(lay.sigma_shape, np.float32)
    _check(lib().oracle_calibrate_sigma(C.byref(lay.c()), _p(kv), _p(mu), _p(mask), int(t_cal),
                                        _p(out)))
    return out


# ------------------------------------- context page: 2b-bit -> b-bit codes

RQ_ERS, RQ_DRS, RQ_MRS = 0, 1, 2


def requantize(mode: int, b: int, packed_in: np.ndarray, n: int, scale_in, group: int, zero_in=None):
    """(packed b-bit codes uint8[n b / 8], new scales float32[n_groups]) from
    packed 2b-bit codes (PM-KVQ section: ERS / DRS / MRS)."""
    packed_in = np.ascontiguousarray(packed_in, np.uint8).reshape(-1)
    scale_in = np.ascontiguousarray(scale_in, np.float32).reshape(-1)
    n_groups = -(-n // group)
    if packed_in.size * 8 < n * 2 * b or scale_in.size < n_groups:
        raise ValueError("inputs shorter than n codes / n_groups scales")
    if zero_in is not None:
        zero_in = np.ascontiguousarray(zero_in, np.float32).reshape(-1)
    out = np.zeros(max(n * b // 8, 1), np.uint8)
    sc = np.zeros(max(n_groups, 1), np.float32)
    _check(lib().oracle_requantize(mode, b, _p(packed_in), n, _p(out), _p(scale_in), _p(zero_in),
                                   _p(sc), group))
    return out[: n * b // 8], sc[:n_groups]
