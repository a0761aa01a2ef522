"""GPU tests of the offload decode (skv_decode_offload): a bitstream kept in
pinned host memory, copied in batches through a two-half staging buffer on
a copy stream while the previous batch decodes. The decoded cache must equal
the encoder's input and the oracle's decode, for every staging size from one
chunk per batch to the whole stream in one batch."""
import numpy as np
import pytest
import torch

from lossless_kv_cache_scalar_gb300 import Coder, Layout, SKVError, calibrate_sigma, synth
from lossless_kv_cache_scalar_gb300.api import offload_plan
from oracle import oracle as O
from tests import _skvtest as H

pytestmark = pytest.mark.gpu


def _encoded(name, layers, tokens, **kw):
    cfg = synth.CONFIGS[name].scaled(n_layers=layers, n_tokens=tokens)
    w = synth.generate(cfg, "cuda")
    lay = Layout(cfg.dtype, cfg.n_layers, cfg.n_kv, cfg.n_heads, cfg.head_dim, cfg.n_tokens, **kw)
    c = Coder(lay, "cuda")
    s, offs = c.encode(w["kv"], w["mu"], w["sigma"], w["counts"])
    host = torch.empty(s.numel(), dtype=torch.uint8).pin_memory()
    host.copy_(s)
    return lay, w, c, s, offs, host, offs.cpu()


def _staging_sizes(host_offs):
    o = host_offs.numpy().astype(np.int64)
    biggest = int(np.diff(o).max())
    total = int(o[-1])
    return [2 * biggest, 2 * (biggest * 3 + 16), 2 * (total // 5 + biggest), 2 * total + 64]


@pytest.mark.parametrize("name,layers,tokens,kw", [
    ("tiny", 1, 256, dict(tokens_per_chunk=64)),
    ("qwen3_0p6b", 3, 1024, {}),
    ("fp8_32b", 2, 700, dict(tokens_per_chunk=100, streams_per_chunk=96)),
    ("paged_14b", 1, 2048, dict(streams_per_chunk=256)),
])
def test_offload_decode_equals_input(name, layers, tokens, kw):
    lay, w, c, s, offs, host, host_offs = _encoded(name, layers, tokens, **kw)
    for size in _staging_sizes(host_offs):
        staging = torch.empty(size, dtype=torch.uint8, device="cuda")
        out = torch.full_like(w["kv"], 0x55)
        stream = torch.cuda.current_stream()
        c.decode_offload_into(host, host_offs, offs, w["mu"], w["sigma"], w["counts"], out, staging,
                              stream=stream)
        c.check_status("offload", stream)
        assert torch.equal(out, w["kv"]), size
        n_batches = len(offload_plan(host_offs.numpy(), (size // 2) & ~15)) - 1
        assert n_batches >= 1
    # and the oracle decodes the same host bytes to the same cache
    if name == "tiny":
        h = synth.to_numpy(w)
        ref = O.decode(H.o_layout(lay), host.numpy(), host_offs.numpy().astype(np.uint64), h["mu"],
                       h["sigma"], h["counts"])
        assert np.array_equal(out.cpu().numpy().view(ref.dtype).reshape(-1), ref)


def test_offload_with_sigma_blocks():
    cfg = synth.CONFIGS["qwen3_0p6b"].scaled(n_layers=2, n_tokens=1024)
    w = synth.generate(cfg, "cuda", with_mask=True)
    lay = Layout("bf16", 2, 2, 8, 128, 1024, sigma_block_tokens=512)
    sigma = calibrate_sigma(lay, w["kv"], w["mu"], 512, mask=w["mask"].view(torch.uint8))
    c = Coder(lay, "cuda")
    s, offs = c.encode(w["kv"], w["mu"], sigma, w["counts"])
    host = s.cpu().pin_memory()
    staging = torch.empty(2 * (int(offs[-1]) // 3 + 1024 * 1024), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(w["kv"])
    c.decode_offload_into(host, offs.cpu(), offs, w["mu"], sigma, w["counts"], out, staging)
    c.check_status("offload")
    assert torch.equal(out, w["kv"])


def test_offload_rejects_small_staging_and_bad_offsets():
    lay, w, c, s, offs, host, host_offs = _encoded("tiny", 1, 256, tokens_per_chunk=64)
    biggest = int(np.diff(host_offs.numpy()).max())
    out = torch.empty_like(w["kv"])
    small = torch.empty(2 * biggest - 32, dtype=torch.uint8, device="cuda")
    with pytest.raises(SKVError) as e:
        c.decode_offload_into(host, host_offs, offs, w["mu"], w["sigma"], w["counts"], out, small)
    assert e.value.name == "INVALID_ARG"
    bad = host_offs.clone()
    bad[2] = int(host_offs[1]) - 16                      # offsets[2] < offsets[1]
    staging = torch.empty(4 * biggest, dtype=torch.uint8, device="cuda")
    with pytest.raises(SKVError) as e:
        c.decode_offload_into(host, bad, offs, w["mu"], w["sigma"], w["counts"], out, staging)
    assert e.value.name == "CORRUPT"
    # device offsets that disagree with the staged bytes are caught by the decoder
    dev_bad = offs.clone()
    dev_bad[1] += 16
    c.decode_offload_into(host, host_offs, dev_bad, w["mu"], w["sigma"], w["counts"], out, staging)
    with pytest.raises(SKVError) as e:
        c.check_status("offload")
    assert e.value.name == "CORRUPT"


@pytest.mark.parametrize("name,layers,tokens,kw", [
    ("qwen3_0p6b", 2, 1024, {}),
    ("fp8_32b", 2, 700, dict(tokens_per_chunk=100, streams_per_chunk=96)),
    ("paged_14b", 1, 2048, dict(streams_per_chunk=256)),
])
def test_pages_from_host_equal_device_pages(name, layers, tokens, kw):
    """skv_decode_pages_host: listed pages read from the host bitstream decode
    to the same pages as skv_decode_chunks on the device stream, in list order,
    duplicates and the last (shorter) page included."""
    lay, w, c, s, offs, host, host_offs = _encoded(name, layers, tokens, **kw)
    c.prepare_decode(w["sigma"], w["counts"])
    rng = np.random.default_rng(11)
    n = lay.n_chunks
    ids = np.concatenate([rng.integers(0, n, 9), [n - 1, 0, n - 1]]).astype(np.int32)
    sizes = np.diff(host_offs.numpy())
    staging = torch.empty(int(sizes[ids].sum()) + 4096, dtype=torch.uint8, device="cuda")
    pages = torch.zeros((ids.size, lay.page_elems), dtype=w["mu"].dtype, device="cuda")
    c.decode_pages_host_into(host, host_offs, w["mu"], torch.from_numpy(ids), pages, staging)
    c.check_status("pages from host")
    want = c.decode_chunks(s, offs, w["mu"], w["sigma"], w["counts"], torch.from_numpy(ids).cuda())
    assert torch.equal(pages, want)
    # a staging buffer one page short is refused before anything is copied
    short = torch.empty(int(sizes[ids].sum()) - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(SKVError):
        c.decode_pages_host_into(host, host_offs, w["mu"], torch.from_numpy(ids), pages, short)
    with pytest.raises(SKVError):
        bad = torch.tensor([0, n], dtype=torch.int32)
        c.decode_pages_host_into(host, host_offs, w["mu"], bad, pages[:2], staging)
