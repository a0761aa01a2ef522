"""skv_decode_noalloc: decoding for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc or lend the library a workspace -- a host
program whose memory pool owns all device memory and gives a plugin no
allocator, or a latency-critical path where allocating (and the device-wide
synchronisation that freeing brings) is not allowed. skv_decode_noalloc keeps
its scratch in a fixed array inside the library instead. These tests call it
through the C ABI and check that it gives exactly skv_decode's output, on two
calls in a row, and that it turns away a layout too large for its scratch.

This file runs last (pytest collects files in name order) so that a failure
here, in a run that stops at the first failure, comes after every other test.
"""
import ctypes as C

import pytest
import torch

from lossless_kv_cache_scalar_gb300 import Coder, Layout, synth
from lossless_kv_cache_scalar_gb300 import _binding as B

pytestmark = pytest.mark.gpu


def _noalloc(lay, bits, offs, mu, sigma, counts, out, status):
    s = torch.cuda.current_stream()
    return B.lib().skv_decode_noalloc(C.byref(lay.c()), C.c_void_p(bits.data_ptr()), bits.numel(),
                                      C.c_void_p(offs.data_ptr()), C.c_void_p(mu.data_ptr()),
                                      C.c_void_p(sigma.data_ptr()), C.c_void_p(counts.data_ptr()),
                                      C.c_void_p(out.data_ptr()), C.c_void_p(status.data_ptr()),
                                      C.c_void_p(s.cuda_stream))


@pytest.mark.parametrize("name,kw,sblk", [("tiny", {}, 0), ("fp8_32b", dict(n_layers=2, n_tokens=600), 0),
                                          ("qwen3_0p6b", dict(n_layers=3, n_tokens=1024), 256)])
def test_noalloc_decode_matches_decode_twice(name, kw, sblk):
    cfg = synth.CONFIGS[name].scaled(**kw) if kw else synth.CONFIGS[name]
    w = {k: v.cuda() for k, v in synth.generate(cfg).items()}
    lay = Layout(cfg.dtype, cfg.n_layers, cfg.n_kv, cfg.n_heads, cfg.head_dim, cfg.n_tokens,
                 sigma_block_tokens=sblk)
    if sblk:
        # one sigma row per block of sblk tokens (each block's own RMS)
        from lossless_kv_cache_scalar_gb300 import calibrate_sigma
        w["sigma"] = calibrate_sigma(lay, w["kv"], w["mu"], sblk)
    coder = Coder(lay)
    bits, offs = coder.encode(w["kv"], w["mu"], w["sigma"], w["counts"])
    ref = coder.decode(bits, offs, w["mu"], w["sigma"], w["counts"])
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call in range(2):
        out = torch.full_like(w["mu"], 0x55)        # stale contents must not matter
        rc = _noalloc(lay, bits, offs, w["mu"], w["sigma"], w["counts"], out, status)
        assert rc == 0, f"call {call}: {B.STATUS_NAMES.get(rc, rc)}"
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"call {call}: status {B.STATUS_NAMES.get(int(status.item()))}"
        assert torch.equal(out, ref), f"call {call}: differs from skv_decode"
        assert torch.equal(out, w["kv"])


@pytest.mark.parametrize("layers,tokens,sblk", [(100, 256, 0), (25, 1024, 256)])
def test_noalloc_rejects_layout_beyond_its_scratch(layers, tokens, sblk):
    # 100 planes-pairs x 1,024 channels, or 25 x 4 sigma blocks x 1,024: 800 KiB of
    # sigma entries + the 256 KiB P_hat table > 1 MiB
    lay = Layout("bf16", layers, 2, 8, 128, tokens, sigma_block_tokens=sblk)
    dummy = torch.zeros(16, dtype=torch.int64, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = _noalloc(lay, dummy, dummy, dummy, dummy, dummy, dummy, status)
    assert B.STATUS_NAMES[rc] == "INVALID_ARG"
