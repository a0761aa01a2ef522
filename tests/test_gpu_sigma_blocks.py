"""GPU parity of the position-aware sigma (one sigma per block of B tokens,
the variant the 推测性KV编码 blog's limitations section leaves to future
work): bitstreams, offsets and decoded codes bit-equal to the CPU oracle's,
page decodes included, and the per-block calibration bit-equal too.
"""
import numpy as np
import pytest
import torch

from lossless_kv_cache_scalar_gb300 import Coder, Layout, SKVError, calibrate_sigma, synth
from oracle import oracle as O
from tests import _skvtest as H

pytestmark = pytest.mark.gpu


def _o(lay: Layout) -> O.Layout:
    o = H.o_layout(lay)
    o.sigma_block = lay.sigma_block_tokens
    return o


def _workload(name, layers, tokens, B, Tc=256, W=64, t_cal=None):
    cfg = synth.CONFIGS[name].scaled(n_layers=layers, n_tokens=tokens)
    w = synth.generate(cfg, "cuda", with_mask=True)
    lay = Layout(cfg.dtype, cfg.n_layers, cfg.n_kv, cfg.n_heads, cfg.head_dim, cfg.n_tokens,
                 tokens_per_chunk=Tc, streams_per_chunk=W, sigma_block_tokens=B)
    mask = w["mask"].view(torch.uint8)
    sigma = calibrate_sigma(lay, w["kv"], w["mu"], t_cal or min(B or tokens, tokens), mask=mask)
    return lay, w, sigma


@pytest.mark.parametrize("name,layers,tokens,B,Tc,W", [
    ("tiny", 1, 256, 256, 256, 64),          # one block = the static case
    ("tiny", 1, 700, 200, 100, 32),          # ragged last block and page
    ("qwen3_0p6b", 2, 1024, 256, 256, 64),
    ("qwen3_0p6b", 2, 1000, 512, 128, 96),
    ("fp8_32b", 2, 600, 300, 100, 64),       # e4m3
    ("paged_14b", 1, 1300, 1024, 256, 256),  # block longer than several pages
])
def test_sigma_blocks_stream_parity(name, layers, tokens, B, Tc, W):
    lay, w, sigma = _workload(name, layers, tokens, B, Tc, W)
    assert tuple(sigma.shape) == lay.sigma_shape
    c = Coder(lay, "cuda")
    s, offs = c.encode(w["kv"], w["mu"], sigma, w["counts"])
    h = synth.to_numpy(w)
    so, oo = O.encode(_o(lay), h["kv"], h["mu"], sigma.cpu().numpy(), h["counts"])
    assert np.array_equal(offs.cpu().numpy().astype(np.uint64), oo)
    assert np.array_equal(s.cpu().numpy(), so)
    back = c.decode(s, offs, w["mu"], sigma, w["counts"])
    assert torch.equal(back, w["kv"])
    # random pages, with and without the prepared tables
    n = lay.n_chunks
    ids = torch.tensor(sorted({0, n - 1, n // 2, n // 3}), dtype=torch.int32, device="cuda")
    pages = c.decode_chunks(s, offs, w["mu"], sigma, w["counts"], ids)
    ref = O.decode_pages(_o(lay), so, oo, h["mu"], sigma.cpu().numpy(), h["counts"],
                         ids.cpu().numpy())
    assert np.array_equal(pages.cpu().numpy().view(ref.dtype).reshape(ref.shape), ref)
    c.prepare_decode(sigma, w["counts"])
    out = torch.zeros_like(pages)
    c.decode_chunks_prepared_into(s, offs, w["mu"], ids, out)
    c.check_status("prepared")
    assert torch.equal(out, pages)


@pytest.mark.parametrize("name,tokens,B,t_cal", [("tiny", 700, 200, 200), ("tiny", 700, 200, 37),
                                                  ("fp8_32b", 600, 300, 300),
                                                  ("qwen3_0p6b", 1024, 500, 100)])
def test_sigma_blocks_calibration_parity(name, tokens, B, t_cal):
    cfg = synth.CONFIGS[name].scaled(n_layers=2, n_tokens=tokens)
    w = synth.generate(cfg, "cuda", with_mask=True)
    lay = Layout(cfg.dtype, cfg.n_layers, cfg.n_kv, cfg.n_heads, cfg.head_dim, cfg.n_tokens,
                 tokens_per_chunk=100, sigma_block_tokens=B)
    for mask in (None, w["mask"].view(torch.uint8)):
        got = calibrate_sigma(lay, w["kv"], w["mu"], t_cal, mask=mask).cpu().numpy()
        h = synth.to_numpy(w)
        ref = O.calibrate_sigma(_o(lay), h["kv"], h["mu"], t_cal,
                                mask=None if mask is None else mask.cpu().numpy())
        assert got.shape == ref.shape == lay.sigma_shape
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_sigma_blocks_argument_checks():
    cfg = synth.CONFIGS["tiny"]
    w = synth.generate(cfg, "cuda")
    # B not a multiple of the page length is not a valid layout
    bad = Layout("bf16", 1, 2, 8, 128, 256, tokens_per_chunk=100, sigma_block_tokens=150)
    with pytest.raises(SKVError):
        bad.n_chunks
    lay = Layout("bf16", 1, 2, 8, 128, 256, tokens_per_chunk=64, sigma_block_tokens=128)
    with pytest.raises(SKVError):                     # t_cal above the block length
        calibrate_sigma(lay, w["kv"], w["mu"], 129)
    # a static sigma table is too small for a blocked layout: refused before the call
    with pytest.raises(ValueError):
        Coder(lay, "cuda").encode(w["kv"], w["mu"], w["sigma"], w["counts"])
    # the workspace grows by the blocked sigma table only
    static = Layout("bf16", 1, 2, 8, 128, 256, tokens_per_chunk=64)
    assert lay.workspace_bytes(False, False) - static.workspace_bytes(False, False) >= 4 * 2 * 1024
