"""GPU parity of the model-input kernels (skv_histogram, skv_calibrate_sigma)
through the C ABI against the CPU oracle: bit-exact counts and bit-exact sigma.

Cases span every alignment of the code pointer, ragged lengths, accumulation,
both code types, masks, partial calibration windows, and the full-size
Qwen3-8B-shaped cache (counts against the workload's own bincount; sigma
against the oracle on the calibration tokens).
"""
import numpy as np
import pytest
import torch

from lossless_kv_cache_scalar_gb300 import Layout, SKVError, calibrate_sigma, histogram, synth
from oracle import oracle as O
from tests import _skvtest as H

pytestmark = pytest.mark.gpu


def _codes(dtype, n, seed):
    g = torch.Generator().manual_seed(seed)
    if dtype == "bf16":
        return torch.randint(-32768, 32768, (n,), generator=g, dtype=torch.int32).to(torch.int16)
    return torch.randint(0, 256, (n,), generator=g, dtype=torch.int32).to(torch.uint8)


def _o_dt(dtype):
    return O.BF16 if dtype == "bf16" else O.E4M3


def _host(t):
    a = t.cpu().numpy()
    return a.view(np.uint16) if a.dtype == np.int16 else a


# ---------------------------------------------------------------- histogram

@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("n", [0, 1, 7, 8, 9, 15, 16, 17, 4099, 1_000_003])
def test_histogram_lengths(dtype, n):
    c = _codes(dtype, n, n)
    got = histogram(c.cuda(), dtype).cpu().numpy().view(np.uint64)
    assert np.array_equal(got, O.histogram(_o_dt(dtype), _host(c)))


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_histogram_every_alignment(dtype):
    """Start the view at every offset inside a 16-byte line."""
    base = _codes(dtype, 300_017, 42).cuda()
    per = 8 if dtype == "bf16" else 16
    for off in range(per + 1):
        view = base[off:off + 100_000 - off]
        got = histogram(view, dtype).cpu().numpy().view(np.uint64)
        assert np.array_equal(got, O.histogram(_o_dt(dtype), _host(view))), off


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_histogram_accumulate_and_skewed(dtype):
    """Accumulation adds in place; a heavily skewed input (one code almost
    everywhere) counts exactly despite the colliding atomics."""
    a = _codes(dtype, 50_001, 1).cuda()
    b = torch.zeros(2_000_000, dtype=a.dtype, device="cuda")
    b[::97] = a[: b[::97].numel()]
    counts = histogram(a, dtype)
    histogram(b, dtype, counts=counts)
    ref = O.histogram(_o_dt(dtype), _host(a))
    ref = O.histogram(_o_dt(dtype), _host(b), counts=ref)
    assert np.array_equal(counts.cpu().numpy().view(np.uint64), ref)


@pytest.mark.parametrize("name", ["tiny", "qwen3_0p6b", "fp8_32b"])
def test_histogram_workloads(name):
    cfg = synth.CONFIGS[name]
    if name == "fp8_32b":
        cfg = cfg.scaled(n_layers=2, n_tokens=1024)
    w = synth.generate(cfg, "cuda")
    got = histogram(w["kv"])
    assert torch.equal(got, w["counts"])
    ref = O.histogram(_o_dt(cfg.dtype), synth.to_numpy(w)["kv"])
    assert np.array_equal(got.cpu().numpy().view(np.uint64), ref)


def test_histogram_full_size_qwen3_8b():
    """4.83 GB of bf16 codes: equal to the generator's torch.bincount counts."""
    w = synth.generate(synth.CONFIGS["qwen3_8b"], "cuda")
    got = histogram(w["kv"])
    assert torch.equal(got, w["counts"])
    assert int(got.sum()) == w["kv"].numel()


def test_histogram_rejects_bad_args():
    c = _codes("bf16", 16, 0).cuda()
    with pytest.raises(ValueError):
        histogram(c, "e4m3")
    with pytest.raises(ValueError):
        histogram(c, counts=torch.zeros(10, dtype=torch.int64, device="cuda"))


# ------------------------------------------------------- sigma calibration

def _check_sigma(cfg, t_cal, use_mask):
    w = synth.generate(cfg, "cuda", with_mask=use_mask)
    lay = H.layout_of(cfg)
    mask = w["mask"].view(torch.uint8) if use_mask else None
    got = calibrate_sigma(lay, w["kv"], w["mu"], t_cal, mask=mask).cpu().numpy()
    h = synth.to_numpy(w)
    ref = O.calibrate_sigma(H.o_layout(lay), h["kv"], h["mu"], t_cal,
                            mask=None if mask is None else mask.cpu().numpy())
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    return got, w


@pytest.mark.parametrize("t_cal", [1, 7, 100, 256])
@pytest.mark.parametrize("use_mask", [False, True])
def test_sigma_tiny(t_cal, use_mask):
    _check_sigma(synth.CONFIGS["tiny"], t_cal, use_mask)


@pytest.mark.parametrize("name,layers,tokens", [("qwen3_0p6b", 28, 1024), ("fp8_32b", 3, 2048),
                                                ("paged_14b", 2, 1500)])
def test_sigma_workloads(name, layers, tokens):
    cfg = synth.CONFIGS[name].scaled(n_layers=layers, n_tokens=tokens)
    got, w = _check_sigma(cfg, min(1024, tokens), True)
    if cfg.calibrate:
        # the generator's own calibration (torch float64 sums): within one binary32 step
        ulps = (torch.from_numpy(got).view(torch.int32).long()
                - w["sigma"].cpu().view(torch.int32).long()).abs()
        assert int(ulps.max()) <= 1


def test_sigma_odd_geometry_and_nonfinite():
    """HD not a multiple of the block, NaN / inf codes in the window, an empty mask."""
    lay = Layout("bf16", 3, 2, 3, 40, 50)
    g = torch.Generator().manual_seed(5)
    shape = (3, 2, 50, 3, 40)
    mu = torch.randint(0x3C00, 0x4100, shape, generator=g, dtype=torch.int32)
    kv = mu + torch.randint(-50, 51, shape, generator=g, dtype=torch.int32)
    kv[0, 0, 3, 0, :5] = 0x7FC0
    mu[1, 1, 4, 2, 7:9] = 0xFF80
    kv, mu = kv.to(torch.int16), mu.to(torch.int16)
    mask = (torch.rand(shape, generator=g) < 0.5).to(torch.uint8)
    mask[2, 0, :, 1, :] = 0
    got = calibrate_sigma(lay, kv.cuda(), mu.cuda(), 33, mask=mask.cuda()).cpu().numpy()
    ref = O.calibrate_sigma(H.o_layout(lay), kv.numpy().view(np.uint16), mu.numpy().view(np.uint16),
                            33, mask=mask.numpy())
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    assert np.all(got[2, 0, 1] == 2.0 ** -126)


def test_sigma_full_size_qwen3_8b():
    """All 73,728 channels of the Qwen3-8B-shaped cache from its first 1,024
    tokens, in the launch the calibration step would use; the oracle gets the
    same tokens as a 1,024-token layout."""
    cfg = synth.CONFIGS["qwen3_8b"]
    w = synth.generate(cfg, "cuda", with_mask=True)
    lay = H.layout_of(cfg)
    got = calibrate_sigma(lay, w["kv"], w["mu"], 1024, mask=w["mask"].view(torch.uint8))
    head = {k: w[k][:, :, :1024].contiguous() for k in ("kv", "mu", "mask")}
    gen_sigma = w["sigma"].cpu()
    del w
    # the generator's own calibration of this workload (torch float64 sums): within one step
    ulps = (got.cpu().view(torch.int32).long() - gen_sigma.view(torch.int32).long()).abs()
    assert int(ulps.max()) <= 1
    lay_h = H.layout_of(cfg.scaled(n_tokens=1024))
    ref = O.calibrate_sigma(H.o_layout(lay_h), _host(head["kv"]), _host(head["mu"]), 1024,
                            mask=head["mask"].view(torch.uint8).cpu().numpy())
    assert np.array_equal(got.cpu().numpy().view(np.uint32), ref.view(np.uint32))


def test_sigma_rejects_bad_window():
    cfg = synth.CONFIGS["tiny"]
    w = synth.generate(cfg, "cuda")
    lay = H.layout_of(cfg)
    for t in (0, cfg.n_tokens + 1):
        with pytest.raises(SKVError):
            calibrate_sigma(lay, w["kv"], w["mu"], t)


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_sigma_every_code(dtype):
    """Every code bit pattern as kv (subnormals, zeros, the largest values, NaN
    and infinities), against three predictors: zero, a random code, the code itself."""
    n = 65536 if dtype == "bf16" else 256
    D = 8 if dtype == "bf16" else 16
    T = n // D
    lay = Layout(dtype, 1, 1, 1, D, T)
    allc = torch.arange(n, dtype=torch.int32)
    kv = (allc - 65536 * (allc >= 32768)).to(torch.int16) if dtype == "bf16" else allc.to(torch.uint8)
    g = torch.Generator().manual_seed(17)
    rnd = torch.randint(0, n, (n,), generator=g, dtype=torch.int32)
    rnd = (rnd - 65536 * (rnd >= 32768)).to(torch.int16) if dtype == "bf16" else rnd.to(torch.uint8)
    for mu in (torch.zeros_like(kv), rnd, kv.clone()):
        got = calibrate_sigma(lay, kv.cuda(), mu.cuda(), T).cpu().numpy()
        ref = O.calibrate_sigma(H.o_layout(lay), _host(kv), _host(mu), T)
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
        # one channel holding every value of one exponent column: also per-token windows
        got = calibrate_sigma(lay, kv.cuda(), mu.cuda(), max(1, T // 3)).cpu().numpy()
        ref = O.calibrate_sigma(H.o_layout(lay), _host(kv), _host(mu), max(1, T // 3))
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
