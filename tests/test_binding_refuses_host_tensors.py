"""The product path has no CPU fallback: every entry point of the Python
binding refuses host (CPU) tensors with an error before anything reaches the
C ABI, here on a machine without a GPU."""
import pytest
import torch

import lossless_kv_cache_scalar_gb300 as skv
from lossless_kv_cache_scalar_gb300 import api


def _lay():
    return skv.Layout("bf16", 1, 2, 8, 128, 256)


def test_histogram_and_calibration_refuse_host_tensors():
    lay = _lay()
    codes = torch.zeros(lay.n_elems, dtype=torch.int16)
    with pytest.raises(ValueError):
        skv.histogram(codes)
    with pytest.raises(ValueError):
        skv.calibrate_sigma(lay, codes.view(2, 256, 8, 128), codes.view(2, 256, 8, 128), 16)


def test_coder_refuses_host_tensors():
    lay = _lay()
    c = skv.Coder(lay, "cpu", decode=False)          # buffers on the host: nothing can run
    kv = torch.zeros(lay.n_elems, dtype=torch.int16)
    sigma = torch.ones(lay.sigma_shape, dtype=torch.float32)
    counts = torch.ones(lay.n_codes, dtype=torch.int64)
    out = torch.empty(lay.max_encoded_bytes, dtype=torch.uint8)
    offs = torch.empty(lay.n_chunks + 1, dtype=torch.int64)
    with pytest.raises(ValueError):
        c.encode_into(kv, kv, sigma, counts, out, offs)
    with pytest.raises(ValueError):
        c.decode_into(out, offs, kv, sigma, counts, kv)


def test_model_queries_refuse_host_tensors():
    lay = _lay()
    q = torch.zeros(4, dtype=torch.int32)
    s = torch.ones(4, dtype=torch.float32)
    counts = torch.ones(lay.n_codes, dtype=torch.int64)
    with pytest.raises(ValueError):
        api.cdf_eval(lay, counts, q, s, q)
    with pytest.raises(ValueError):
        api.search_eval(lay, counts, q, s, q)
    with pytest.raises(ValueError):
        skv.requantize(torch.zeros(64, dtype=torch.uint8), 64, 4, torch.ones(1), 64)


def test_missing_library_raises(monkeypatch):
    """If the CUDA library cannot be loaded the binding raises: it never
    substitutes another implementation."""
    from lossless_kv_cache_scalar_gb300 import _binding as B
    import os
    monkeypatch.setattr(B, "_lib", None)
    monkeypatch.setattr(B, "LIB_PATH", os.path.join(B.HERE, "no_such_library_for_this_test.so"))
    with pytest.raises(RuntimeError):
        B.lib()
    with pytest.raises(RuntimeError):
        _lay().n_chunks                                # any call that needs the library
