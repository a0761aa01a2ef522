"""GPU tests of the host-buffer pipelines (skv_encode_host / skv_decode_host):
the cache and the bitstream in host memory, batches of layers streamed through
device staging with copies overlapping the kernels. The bitstream and offsets
must equal skv_encode's byte for byte for every batch size, and decoding must
restore the cache exactly."""
import numpy as np
import pytest
import torch

from lossless_kv_cache_scalar_gb300 import Coder, HostCoder, Layout, SKVError, calibrate_sigma, synth

pytestmark = pytest.mark.gpu


def _case(name, layers, tokens, **kw):
    cfg = synth.CONFIGS[name].scaled(n_layers=layers, n_tokens=tokens)
    w = synth.generate(cfg, "cuda", with_mask=True)
    lay = Layout(cfg.dtype, cfg.n_layers, cfg.n_kv, cfg.n_heads, cfg.head_dim, cfg.n_tokens, **kw)
    sigma = w["sigma"]
    if lay.sigma_block_tokens:
        sigma = calibrate_sigma(lay, w["kv"], w["mu"], lay.sigma_block_tokens, mask=w["mask"].view(torch.uint8))
    return lay, w, sigma


@pytest.mark.parametrize("name,layers,tokens,kw,lpbs", [
    ("tiny", 1, 256, {}, [1]),
    ("qwen3_0p6b", 5, 512, {}, [1, 2, 3, 5, 8]),
    ("fp8_32b", 3, 300, dict(tokens_per_chunk=100, streams_per_chunk=96), [1, 2]),
    ("qwen3_0p6b", 3, 1024, dict(sigma_block_tokens=512), [2]),
])
@pytest.mark.parametrize("pinned", [True, False])
def test_host_pipeline_matches_device_coder(name, layers, tokens, kw, lpbs, pinned):
    lay, w, sigma = _case(name, layers, tokens, **kw)
    ref_bits, ref_offs = Coder(lay, "cuda").encode(w["kv"], w["mu"], sigma, w["counts"])
    kv_h, mu_h = w["kv"].cpu(), w["mu"].cpu()
    if pinned:
        kv_h, mu_h = kv_h.pin_memory(), mu_h.pin_memory()
    for lpb in lpbs:
        hc = HostCoder(lay, "cuda", layers_per_batch=lpb)
        out = torch.zeros(lay.max_encoded_bytes, dtype=torch.uint8)
        offs = torch.zeros(lay.n_chunks + 1, dtype=torch.int64)
        if pinned:
            out, offs = out.pin_memory(), offs.pin_memory()
        n = hc.encode_into(kv_h, mu_h, sigma, w["counts"], out, offs)
        hc.check_status("encode_host")
        assert n == ref_bits.numel()
        assert torch.equal(offs, ref_offs.cpu()), lpb
        assert torch.equal(out[:n], ref_bits.cpu()), lpb
        back = torch.full_like(kv_h, 0x11)
        hc.decode_into(out, n, offs, mu_h, sigma, w["counts"], back)
        hc.check_status("decode_host")
        assert torch.equal(back, kv_h), lpb


def test_host_pipeline_errors():
    lay, w, sigma = _case("qwen3_0p6b", 2, 512)
    hc = HostCoder(lay, "cuda", layers_per_batch=1)
    kv_h, mu_h = w["kv"].cpu(), w["mu"].cpu()
    offs = torch.zeros(lay.n_chunks + 1, dtype=torch.int64)
    small = torch.zeros(1024, dtype=torch.uint8)
    with pytest.raises(SKVError) as e:
        hc.encode_into(kv_h, mu_h, sigma, w["counts"], small, offs)
    assert e.value.name == "CAPACITY"
    out = torch.zeros(lay.max_encoded_bytes, dtype=torch.uint8)
    n = hc.encode_into(kv_h, mu_h, sigma, w["counts"], out, offs)
    bad = offs.clone()
    bad[3] = bad[2] - 16
    with pytest.raises(SKVError) as e:
        hc.decode_into(out, n, bad, mu_h, sigma, w["counts"], torch.empty_like(kv_h))
    assert e.value.name == "CORRUPT"
    with pytest.raises(SKVError) as e:                      # offsets past the stream's end
        hc.decode_into(out, n - 16, offs, mu_h, sigma, w["counts"], torch.empty_like(kv_h))
    assert e.value.name == "CORRUPT"
