"""PyTorch-facing wrapper of the C ABI: device buffers, streams and status words.

PyTorch only provides device memory and streams here; encoding and decoding
run in libskv.so's kernels (skv_encode / skv_decode / skv_decode_chunks /
skv_cdf_eval), called through the ctypes binding with raw device pointers.
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass

import torch

from . import _binding as B

_DT = {"bf16": B.SKV_BF16, "e4m3": B.SKV_E4M3}


@dataclass
class Layout:
    """Shape and coding parameters (the skv_layout struct of include/skv.h)."""
    dtype: str
    n_layers: int
    n_kv: int
    n_heads: int
    head_dim: int
    n_tokens: int
    tokens_per_chunk: int = 256
    streams_per_chunk: int = 64
    weights: tuple = (95, 3, 2)
    sigma_block_tokens: int = 0   # 0: one sigma per channel; else tokens per sigma block

    def c(self) -> B.skv_layout:
        w = self.weights
        return B.skv_layout(B.SKV_FORMAT_VERSION, _DT[self.dtype], self.n_layers, self.n_kv,
                            self.n_heads, self.head_dim, self.n_tokens, self.tokens_per_chunk,
                            self.streams_per_chunk, w[0], w[1], w[2], self.sigma_block_tokens)

    @property
    def n_sigma_blocks(self) -> int:
        b = self.sigma_block_tokens
        return -(-self.n_tokens // b) if b else 1

    @property
    def sigma_shape(self) -> tuple:
        if self.sigma_block_tokens:
            return (self.n_layers, self.n_kv, self.n_sigma_blocks, self.n_heads, self.head_dim)
        return (self.n_layers, self.n_kv, self.n_heads, self.head_dim)

    @property
    def n_codes(self) -> int:
        return 65536 if self.dtype == "bf16" else 256

    @property
    def bytes_per_code(self) -> int:
        return 2 if self.dtype == "bf16" else 1

    @property
    def n_elems(self) -> int:
        return self.n_layers * self.n_kv * self.n_tokens * self.n_heads * self.head_dim

    @property
    def page_elems(self) -> int:
        return self.tokens_per_chunk * self.n_heads * self.head_dim

    def _q(self, fn, *extra) -> int:
        v = C.c_uint64()
        B.check(fn.__name__, fn(C.byref(self.c()), *extra, C.byref(v)))
        return v.value

    @property
    def n_chunks(self) -> int:
        return self._q(B.lib().skv_num_chunks)

    @property
    def max_encoded_bytes(self) -> int:
        return self._q(B.lib().skv_max_encoded_bytes)

    def workspace_bytes(self, encode: bool, fast: bool = True) -> int:
        """Workspace of skv_encode (encode=True) or of the decoders; fast=True
        includes the outlier inverse tables (op 2), fast=False is the minimum."""
        op = 1 if encode else (2 if fast else 0)
        return self._q(B.lib().skv_workspace_bytes, op)

    @classmethod
    def for_tensor(cls, kv: torch.Tensor, dtype: str | None = None, **kw) -> "Layout":
        L, K, T, H, D = kv.shape
        if dtype is None:
            dtype = "bf16" if kv.element_size() == 2 else "e4m3"
        return cls(dtype, L, K, H, D, T, **kw)


def _ptr(t: torch.Tensor | None):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream_handle(stream: torch.cuda.Stream | None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def _check_model_inputs(lay: Layout, sigma: torch.Tensor, counts: torch.Tensor | None):
    """sigma and counts must be device tensors of the layout's sizes (the C ABI
    takes bare pointers, so a short table would be read past its end)."""
    n_sig = 1
    for d in lay.sigma_shape:
        n_sig *= d
    if not sigma.is_cuda or not sigma.is_contiguous() or sigma.dtype != torch.float32 \
            or sigma.numel() != n_sig:
        raise ValueError(f"sigma must be a contiguous float32 CUDA tensor of shape {lay.sigma_shape}")
    if counts is not None and (not counts.is_cuda or counts.dtype != torch.int64
                               or counts.numel() != lay.n_codes or not counts.is_contiguous()):
        raise ValueError(f"counts must be a contiguous int64 CUDA tensor of {lay.n_codes} entries")


def _check_dev(t, what: str, dtype=None, numel=None, min_numel=None, elem_size=None):
    """A device buffer handed to the C ABI as a bare pointer: contiguous, on the
    GPU, of the given dtype or element size, and large enough."""
    if t is None or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{what} must be a contiguous CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{what} must be {dtype}")
    if elem_size is not None and t.element_size() != elem_size:
        raise ValueError(f"{what} must have {elem_size}-byte elements")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{what} must have {numel} elements")
    if min_numel is not None and t.numel() < min_numel:
        raise ValueError(f"{what} must have at least {min_numel} elements")


def _check_codes(t: torch.Tensor, lay: Layout, what: str):
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{what} must be a contiguous CUDA tensor")
    if t.element_size() != lay.bytes_per_code or t.numel() != lay.n_elems:
        raise ValueError(f"{what}: expected {lay.n_elems} codes of {lay.bytes_per_code} bytes")


class Coder:
    """Encoder/decoder for one layout, holding its workspace and status word.

    One Coder must not run two calls at once on different streams (they would
    share the workspace).
    """

    def __init__(self, layout: Layout, device: torch.device | str | int = "cuda",
                 encode: bool = True, decode: bool = True, fast_decode: bool = True):
        self.layout = layout
        self.device = torch.device(device)
        self._c = layout.c()
        need = 0
        if encode:
            need = max(need, layout.workspace_bytes(True))
        if decode:
            need = max(need, layout.workspace_bytes(False, fast_decode))
        self.workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=self.device)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.n_chunks = layout.n_chunks

    def _check_stream_and_offsets(self, bitstream, offsets):
        _check_dev(bitstream, "bitstream", torch.uint8)
        _check_dev(offsets, "offsets", torch.int64, numel=self.n_chunks + 1)

    def _check_pages(self, chunk_ids, pages_out):
        _check_dev(chunk_ids, "chunk_ids", torch.int32)
        _check_dev(pages_out, "pages_out", elem_size=self.layout.bytes_per_code,
                   numel=chunk_ids.numel() * self.layout.page_elems)

    # -- status
    def check_status(self, where: str, stream=None):
        (stream or torch.cuda.current_stream()).synchronize()
        st = int(self.status.item())
        if st:
            raise B.SKVError(where, st)

    def alloc_output(self):
        cap = self.layout.max_encoded_bytes
        out = torch.empty(max(cap, 16), dtype=torch.uint8, device=self.device)
        offsets = torch.empty(self.n_chunks + 1, dtype=torch.int64, device=self.device)
        return out, offsets

    # -- encode
    def encode_into(self, kv, mu, sigma, counts, out, offsets, stream=None):
        """Enqueue skv_encode; no synchronisation."""
        lay = self.layout
        _check_codes(kv, lay, "kv")
        _check_codes(mu, lay, "mu")
        _check_model_inputs(lay, sigma, counts)
        _check_dev(out, "out", torch.uint8)
        _check_dev(offsets, "offsets", torch.int64, numel=self.n_chunks + 1)
        rc = B.lib().skv_encode(C.byref(self._c), _ptr(kv), _ptr(mu), _ptr(sigma), _ptr(counts),
                                _ptr(out), out.numel(), _ptr(offsets), _ptr(self.status),
                                _ptr(self.workspace), self.workspace.numel(),
                                _stream_handle(stream))
        B.check("skv_encode", rc)

    def encode(self, kv, mu, sigma, counts, stream=None):
        """Encode and check. Returns (bitstream uint8 tensor, offsets int64 tensor)."""
        out, offsets = self.alloc_output()
        self.encode_into(kv, mu, sigma, counts, out, offsets, stream)
        self.check_status("skv_encode", stream)
        total = int(offsets[-1].item())
        return out[:total], offsets

    # -- decode
    def decode_into(self, bitstream, offsets, mu, sigma, counts, kv_out, stream=None):
        lay = self.layout
        _check_codes(mu, lay, "mu")
        _check_codes(kv_out, lay, "kv_out")
        _check_model_inputs(lay, sigma, counts)
        self._check_stream_and_offsets(bitstream, offsets)
        rc = B.lib().skv_decode(C.byref(self._c), _ptr(bitstream), bitstream.numel(),
                                _ptr(offsets), _ptr(mu), _ptr(sigma), _ptr(counts), _ptr(kv_out),
                                _ptr(self.status), _ptr(self.workspace), self.workspace.numel(),
                                _stream_handle(stream))
        B.check("skv_decode", rc)

    def decode(self, bitstream, offsets, mu, sigma, counts, stream=None):
        kv = torch.empty_like(mu)
        self.decode_into(bitstream, offsets, mu, sigma, counts, kv, stream)
        self.check_status("skv_decode", stream)
        return kv

    def decode_chunks_into(self, bitstream, offsets, mu, sigma, counts, chunk_ids, pages_out,
                           stream=None):
        lay = self.layout
        ids = chunk_ids
        self._check_pages(ids, pages_out)
        self._check_stream_and_offsets(bitstream, offsets)
        _check_codes(mu, lay, "mu")
        _check_model_inputs(lay, sigma, counts)
        rc = B.lib().skv_decode_chunks(C.byref(self._c), _ptr(bitstream), bitstream.numel(),
                                       _ptr(offsets), _ptr(mu), _ptr(sigma), _ptr(counts), _ptr(ids),
                                       ids.numel(), _ptr(pages_out), _ptr(self.status),
                                       _ptr(self.workspace), self.workspace.numel(),
                                       _stream_handle(stream))
        B.check("skv_decode_chunks", rc)

    def prepare_decode(self, sigma, counts, stream=None, check: bool = True):
        """Build the decoder tables once (skv_decode_prepare) for decode_chunks_prepared."""
        _check_model_inputs(self.layout, sigma, counts)
        rc = B.lib().skv_decode_prepare(C.byref(self._c), _ptr(sigma), _ptr(counts), _ptr(self.status),
                                        _ptr(self.workspace), self.workspace.numel(),
                                        _stream_handle(stream))
        B.check("skv_decode_prepare", rc)
        if check:
            self.check_status("skv_decode_prepare", stream)

    def decode_chunks_prepared_into(self, bitstream, offsets, mu, chunk_ids, pages_out, stream=None):
        lay = self.layout
        self._check_pages(chunk_ids, pages_out)
        self._check_stream_and_offsets(bitstream, offsets)
        _check_codes(mu, lay, "mu")
        rc = B.lib().skv_decode_chunks_prepared(C.byref(self._c), _ptr(bitstream), bitstream.numel(),
                                                _ptr(offsets), _ptr(mu), _ptr(chunk_ids),
                                                chunk_ids.numel(), _ptr(pages_out), _ptr(self.status),
                                                _ptr(self.workspace), self.workspace.numel(),
                                                _stream_handle(stream))
        B.check("skv_decode_chunks_prepared", rc)

    def decode_offload_into(self, host_bitstream, host_offsets, offsets, mu, sigma, counts, kv_out,
                            staging, stream=None, copy_stream=None):
        """Enqueue skv_decode_offload: decode from a (pinned) host bitstream through
        a two-half device staging buffer, copies on `copy_stream` overlapping decode
        on `stream`. host_offsets is the CPU int64 copy of `offsets`."""
        lay = self.layout
        if host_bitstream.is_cuda or host_offsets.is_cuda:
            raise ValueError("host_bitstream and host_offsets must be CPU tensors")
        if host_offsets.dtype != torch.int64 or host_offsets.numel() != self.n_chunks + 1 \
                or not host_offsets.is_contiguous() or not host_bitstream.is_contiguous():
            raise ValueError("host_offsets must be a contiguous int64 CPU tensor of n_chunks + 1")
        _check_dev(offsets, "offsets", torch.int64, numel=self.n_chunks + 1)
        if not staging.is_cuda or staging.dtype != torch.uint8 or not staging.is_contiguous():
            raise ValueError("staging must be a contiguous uint8 CUDA tensor")
        _check_codes(mu, lay, "mu")
        _check_codes(kv_out, lay, "kv_out")
        _check_model_inputs(lay, sigma, counts)
        st = _stream_handle(stream)
        cs = copy_stream if copy_stream is not None else torch.cuda.Stream(device=mu.device)
        rc = B.lib().skv_decode_offload(C.byref(self._c), C.c_void_p(host_bitstream.data_ptr()),
                                        host_bitstream.numel() * host_bitstream.element_size(),
                                        C.c_void_p(host_offsets.data_ptr()), _ptr(offsets), _ptr(mu),
                                        _ptr(sigma), _ptr(counts), _ptr(kv_out), _ptr(self.status),
                                        _ptr(self.workspace), self.workspace.numel(), _ptr(staging),
                                        staging.numel(), st, C.c_void_p(cs.cuda_stream))
        B.check("skv_decode_offload", rc)
        return cs

    def decode_pages_host_into(self, host_bitstream, host_offsets, mu, host_ids, pages_out, staging,
                               stream=None, copy_stream=None):
        """Enqueue skv_decode_pages_host: the listed pages, read from a (pinned) host
        bitstream, decoded with the tables of prepare_decode. host_ids: CPU int32."""
        lay = self.layout
        if host_bitstream.is_cuda or host_offsets.is_cuda or host_ids.is_cuda:
            raise ValueError("host_bitstream, host_offsets and host_ids must be CPU tensors")
        if host_ids.dtype != torch.int32 or not host_ids.is_contiguous():
            raise ValueError("host_ids must be a contiguous int32 CPU tensor")
        if host_offsets.dtype != torch.int64 or host_offsets.numel() != self.n_chunks + 1 \
                or not host_offsets.is_contiguous() or not host_bitstream.is_contiguous():
            raise ValueError("host_offsets must be the contiguous int64 CPU offsets (n_chunks + 1)")
        _check_dev(pages_out, "pages_out", elem_size=lay.bytes_per_code, numel=host_ids.numel() * lay.page_elems)
        _check_dev(staging, "staging", torch.uint8)
        _check_codes(mu, lay, "mu")
        cs = copy_stream if copy_stream is not None else torch.cuda.Stream(device=mu.device)
        rc = B.lib().skv_decode_pages_host(C.byref(self._c), C.c_void_p(host_bitstream.data_ptr()),
                                           host_bitstream.numel() * host_bitstream.element_size(),
                                           C.c_void_p(host_offsets.data_ptr()), _ptr(mu),
                                           C.c_void_p(host_ids.data_ptr()), host_ids.numel(), _ptr(pages_out),
                                           _ptr(self.status), _ptr(self.workspace), self.workspace.numel(),
                                           _ptr(staging), staging.numel(), _stream_handle(stream),
                                           C.c_void_p(cs.cuda_stream))
        B.check("skv_decode_pages_host", rc)
        return cs

    def decode_chunks(self, bitstream, offsets, mu, sigma, counts, chunk_ids, stream=None):
        lay = self.layout
        pages = torch.zeros((chunk_ids.numel(), lay.page_elems), dtype=mu.dtype, device=mu.device)
        self.decode_chunks_into(bitstream, offsets, mu, sigma, counts, chunk_ids, pages, stream)
        self.check_status("skv_decode_chunks", stream)
        return pages


def _check_query(layout: Layout, counts, n: int, **bufs):
    """Per-query arrays of cdf_eval / search_eval: n 4-byte entries each."""
    if counts is not None:
        _check_dev(counts, "counts", torch.int64, numel=layout.n_codes)
    elif layout.weights[2]:
        raise ValueError("counts are needed when the marginal weight is nonzero")
    for name, t in bufs.items():
        _check_dev(t, name, elem_size=4, numel=n)


def cdf_eval(layout: Layout, counts, mu_codes, sigmas, ords, stream=None) -> torch.Tensor:
    """C(o) per query via skv_cdf_eval (uint32 results as int64 tensor)."""
    dev = mu_codes.device
    n = ords.numel()
    _check_query(layout, counts, n, mu_codes=mu_codes, sigmas=sigmas, ords=ords)
    ws = torch.empty(max(layout.workspace_bytes(False), 256), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.empty(n, dtype=torch.int32, device=dev)
    rc = B.lib().skv_cdf_eval(C.byref(layout.c()), _ptr(counts), n, _ptr(mu_codes), _ptr(sigmas),
                              _ptr(ords), _ptr(out), _ptr(status), _ptr(ws), ws.numel(),
                              _stream_handle(stream))
    B.check("skv_cdf_eval", rc)
    (stream or torch.cuda.current_stream()).synchronize()
    st = int(status.item())
    if st:
        raise B.SKVError("skv_cdf_eval", st)
    return out.to(torch.int64) & 0xFFFFFFFF


def encode(layout: Layout, kv, mu, sigma, counts, stream=None):
    return Coder(layout, kv.device, decode=False).encode(kv, mu, sigma, counts, stream)


def decode(layout: Layout, bitstream, offsets, mu, sigma, counts, stream=None):
    return Coder(layout, mu.device, encode=False).decode(bitstream, offsets, mu, sigma, counts, stream)


def decode_chunks(layout: Layout, bitstream, offsets, mu, sigma, counts, chunk_ids, stream=None):
    return Coder(layout, mu.device, encode=False).decode_chunks(bitstream, offsets, mu, sigma,
                                                                counts, chunk_ids, stream)


def histogram(codes: torch.Tensor, dtype: str | None = None, counts: torch.Tensor | None = None,
              stream=None) -> torch.Tensor:
    """Code histogram (skv_histogram): int64 [N] counts of every bit pattern.

    `codes` is any contiguous CUDA tensor of 2-byte (bf16) or 1-byte (e4m3)
    codes; with `counts` given, the histogram is added to it in place.
    """
    if not codes.is_cuda or not codes.is_contiguous():
        raise ValueError("codes must be a contiguous CUDA tensor")
    if dtype is None:
        dtype = "bf16" if codes.element_size() == 2 else "e4m3"
    n_codes = 65536 if dtype == "bf16" else 256
    if codes.element_size() != (2 if dtype == "bf16" else 1):
        raise ValueError(f"{dtype} codes must be {2 if dtype == 'bf16' else 1}-byte elements")
    acc = counts is not None
    if acc:
        if counts.dtype != torch.int64 or counts.numel() != n_codes or not counts.is_cuda:
            raise ValueError(f"counts must be an int64 CUDA tensor of {n_codes} entries")
    else:
        counts = torch.empty(n_codes, dtype=torch.int64, device=codes.device)
    rc = B.lib().skv_histogram(_DT[dtype], _ptr(codes), codes.numel(), _ptr(counts), int(acc),
                               _stream_handle(stream))
    B.check("skv_histogram", rc)
    return counts


def calibrate_sigma(layout: Layout, kv: torch.Tensor, mu: torch.Tensor, t_cal: int,
                    mask: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Frozen per-(layer, kv, head, channel) sigma from tokens < t_cal (skv_calibrate_sigma).

    `mask` (bool or uint8, the layout of kv) keeps only the elements it marks.
    Returns float32 [n_layers][n_kv][n_heads][head_dim], or with sigma blocks
    [n_layers][n_kv][n_blocks][n_heads][head_dim] (each block from its own first
    t_cal tokens).
    """
    _check_codes(kv, layout, "kv")
    _check_codes(mu, layout, "mu")
    if mask is not None:
        if not mask.is_cuda or not mask.is_contiguous() or mask.element_size() != 1 \
                or mask.numel() != layout.n_elems:
            raise ValueError("mask must be a contiguous 1-byte CUDA tensor shaped like kv")
    sigma = torch.empty(layout.sigma_shape, dtype=torch.float32, device=kv.device)
    rc = B.lib().skv_calibrate_sigma(C.byref(layout.c()), _ptr(kv), _ptr(mu), _ptr(mask), int(t_cal),
                                     _ptr(sigma), _stream_handle(stream))
    B.check("skv_calibrate_sigma", rc)
    return sigma


def offload_plan(host_offsets, batch_bytes: int, max_chunks: int = 0) -> list:
    """skv_offload_plan: first chunk of each batch (plus n_chunks at the end)."""
    import numpy as np
    offs = np.ascontiguousarray(np.asarray(host_offsets), dtype=np.uint64)
    n = offs.size - 1
    nb = C.c_uint64()
    p = offs.ctypes.data_as(C.c_void_p)
    B.check("skv_offload_plan", B.lib().skv_offload_plan(p, n, batch_bytes, max_chunks, None, 0,
                                                         C.byref(nb)))
    out = np.zeros(nb.value + 1, np.uint64)
    B.check("skv_offload_plan", B.lib().skv_offload_plan(p, n, batch_bytes, max_chunks,
                                                         out.ctypes.data_as(C.c_void_p), out.size,
                                                         C.byref(nb)))
    return [int(v) for v in out]


RQ_MODES = {"ers": 0, "drs": 1, "mrs": 2}


def requantize(codes: torch.Tensor, n: int, b: int, scale: torch.Tensor, group: int, mode: str = "ers",
               stream=None):
    """skv_requantize: packed 2b-bit codes (uint8 CUDA tensor) -> (packed b-bit codes,
    new scales). mode "ers" (Equivalent Right Shift), "drs" or "mrs"."""
    if not codes.is_cuda or codes.dtype != torch.uint8 or not codes.is_contiguous():
        raise ValueError("codes must be a contiguous uint8 CUDA tensor")
    if codes.numel() * 8 < n * 2 * b:
        raise ValueError("codes holds fewer than n codes of 2b bits")
    n_groups = -(-n // group)
    if scale.dtype != torch.float32 or not scale.is_cuda or not scale.is_contiguous() or scale.numel() < n_groups:
        raise ValueError("scale must be a float32 CUDA tensor with one entry per group")
    out = torch.empty(max(n * b // 8, 16), dtype=torch.uint8, device=codes.device)
    s_out = torch.empty(max(n_groups, 1), dtype=torch.float32, device=codes.device)
    rc = B.lib().skv_requantize(RQ_MODES[mode], b, _ptr(codes), n, _ptr(out), _ptr(scale), _ptr(s_out), group,
                                _stream_handle(stream))
    B.check("skv_requantize", rc)
    return out[: n * b // 8], s_out[:n_groups]


class HostCoder:
    """skv_encode_host / skv_decode_host: the cache and the bitstream live in
    (page-locked) host memory; batches of `layers_per_batch` layers stream
    through a device staging buffer with copies overlapping the kernels."""

    def __init__(self, layout: Layout, device="cuda", layers_per_batch: int | None = None,
                 fast_decode: bool = True):
        """layers_per_batch None: four batches (each fills most of the GPU on
        caches of Qwen3-8B size, and copies of three of them overlap compute)."""
        self.layout = layout
        self.device = torch.device(device)
        self.lpb = int(layers_per_batch) if layers_per_batch else max(1, -(-layout.n_layers // 4))
        self._c = layout.c()
        need = 0
        for op in (1, 2 if fast_decode else 0):
            v = C.c_uint64()
            B.check("skv_host_staging_bytes", B.lib().skv_host_staging_bytes(C.byref(self._c), self.lpb, op, C.byref(v)))
            need = max(need, v.value)
        self.staging = torch.empty(max(need, 256), dtype=torch.uint8, device=self.device)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.copy_stream = torch.cuda.Stream(device=self.device)       # host to device
        self.copy_out_stream = torch.cuda.Stream(device=self.device)   # device to host
        self.n_chunks = layout.n_chunks

    def _check_host(self, t, what, nbytes=None):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{what} must be a contiguous CPU tensor (page-locked for overlap)")
        if nbytes is not None and t.numel() * t.element_size() < nbytes:
            raise ValueError(f"{what} is smaller than {nbytes} bytes")

    def check_status(self, where):
        torch.cuda.synchronize(self.device)
        st = int(self.status.item())
        if st:
            raise B.SKVError(where, st)

    def encode_into(self, kv, mu, sigma, counts, out, offsets, stream=None):
        """kv, mu: host codes (canonical layout); out: host uint8 buffer; offsets: host
        int64 [n_chunks + 1] (written). Returns the stream's byte count."""
        lay = self.layout
        raw = lay.n_elems * lay.bytes_per_code
        self._check_host(kv, "kv", raw)
        self._check_host(mu, "mu", raw)
        self._check_host(out, "out")
        self._check_host(offsets, "offsets", 8 * (self.n_chunks + 1))
        _check_model_inputs(lay, sigma, counts)
        rc = B.lib().skv_encode_host(C.byref(self._c), C.c_void_p(kv.data_ptr()), C.c_void_p(mu.data_ptr()),
                                     _ptr(sigma), _ptr(counts), C.c_void_p(out.data_ptr()),
                                     out.numel() * out.element_size(), C.c_void_p(offsets.data_ptr()),
                                     _ptr(self.status), _ptr(self.staging), self.staging.numel(), self.lpb,
                                     _stream_handle(stream), C.c_void_p(self.copy_stream.cuda_stream),
                                     C.c_void_p(self.copy_out_stream.cuda_stream))
        B.check("skv_encode_host", rc)
        return int(offsets[-1])

    def decode_into(self, bits, nbytes, offsets, mu, sigma, counts, kv_out, stream=None):
        lay = self.layout
        raw = lay.n_elems * lay.bytes_per_code
        self._check_host(bits, "bits", nbytes)
        self._check_host(offsets, "offsets", 8 * (self.n_chunks + 1))
        self._check_host(mu, "mu", raw)
        self._check_host(kv_out, "kv_out", raw)
        _check_model_inputs(lay, sigma, counts)
        rc = B.lib().skv_decode_host(C.byref(self._c), C.c_void_p(bits.data_ptr()), nbytes,
                                     C.c_void_p(offsets.data_ptr()), C.c_void_p(mu.data_ptr()), _ptr(sigma),
                                     _ptr(counts), C.c_void_p(kv_out.data_ptr()), _ptr(self.status),
                                     _ptr(self.staging), self.staging.numel(), self.lpb, _stream_handle(stream),
                                     C.c_void_p(self.copy_stream.cuda_stream),
                                     C.c_void_p(self.copy_out_stream.cuda_stream))
        B.check("skv_decode_host", rc)


def search_eval(layout: Layout, counts, mu_codes, sigmas, slots, fast: bool = True, stream=None):
    """skv_search_eval: the decoder's search for each (mu code, sigma, slot)
    query. Returns (o, C(o), f(o)) as int64 tensors."""
    dev = mu_codes.device
    n = slots.numel()
    _check_query(layout, counts, n, mu_codes=mu_codes, sigmas=sigmas, slots=slots)
    ws = torch.empty(max(layout.workspace_bytes(False, fast), 256), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    outs = [torch.empty(n, dtype=torch.int32, device=dev) for _ in range(3)]
    rc = B.lib().skv_search_eval(C.byref(layout.c()), _ptr(counts), n, _ptr(mu_codes), _ptr(sigmas), _ptr(slots),
                                 _ptr(outs[0]), _ptr(outs[1]), _ptr(outs[2]), _ptr(status), _ptr(ws), ws.numel(),
                                 _stream_handle(stream))
    B.check("skv_search_eval", rc)
    (stream or torch.cuda.current_stream()).synchronize()
    st = int(status.item())
    if st:
        raise B.SKVError("skv_search_eval", st)
    return tuple(o.to(torch.int64) & 0xFFFFFFFF for o in outs)
