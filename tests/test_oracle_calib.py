"""Pins of the oracle's model inputs: the code histogram behind p_hat (the
Speculative KV Coding wiki, mixture section) and the frozen per-channel sigma
(the wiki's predictor-choice section; the blog's predictor-engineering and
information-theory sections: the optimum Gaussian scale is the residual's
root mean square about mu).

Each pin comes from outside the oracle: numpy's bincount, residual sets whose
root mean square is an exact small integer, invariances (masked, late-token
and non-finite elements do not matter; doubling every value doubles sigma),
the clamp at 2^-126, and the workload generator's own calibration.
"""
import numpy as np
import pytest
import torch

from lossless_kv_cache_scalar_gb300 import synth
from oracle import oracle as O

BF16_ONE, BF16_SEVEN, BF16_ZERO = 0x3F80, 0x40E0, 0x0000
E4M3_ONE, E4M3_SEVEN, E4M3_ZERO = 0x38, 0x4E, 0x00


def _lay(dtype=O.BF16, L=1, K=2, H=2, D=8, T=16):
    return O.Layout(dtype, L, K, H, D, T)


def _shape(lay):
    return (lay.n_layers, lay.n_kv, lay.n_tokens, lay.n_heads, lay.head_dim)


# ---------------------------------------------------------------- histogram

@pytest.mark.parametrize("dtype", [O.BF16, O.E4M3])
def test_histogram_is_bincount(dtype):
    rng = np.random.default_rng(7)
    n_codes = 65536 if dtype == O.BF16 else 256
    codes = rng.integers(0, n_codes, 100_003).astype(np.uint16 if dtype == O.BF16 else np.uint8)
    h = O.histogram(dtype, codes)
    assert h.dtype == np.uint64 and h.size == n_codes
    assert np.array_equal(h, np.bincount(codes, minlength=n_codes).astype(np.uint64))
    assert int(h.sum()) == codes.size


def test_histogram_accumulates_and_counts_nan_codes():
    codes = np.array([0x7FC0, 0xFFFF, 0x7F80, 0x0001, 0x0001], np.uint16)
    h = O.histogram(O.BF16, codes)
    assert h[0x7FC0] == 1 and h[0xFFFF] == 1 and h[0x7F80] == 1 and h[1] == 2
    h2 = O.histogram(O.BF16, codes, counts=h)
    assert np.array_equal(h2, 2 * h)
    assert int(O.histogram(O.BF16, np.zeros(0, np.uint16)).sum()) == 0


# ---------------------------------------------------------- sigma: closed forms

@pytest.mark.parametrize("dtype,zero,one,seven", [(O.BF16, BF16_ZERO, BF16_ONE, BF16_SEVEN),
                                                  (O.E4M3, E4M3_ZERO, E4M3_ONE, E4M3_SEVEN)])
def test_sigma_exact_rms(dtype, zero, one, seven):
    """Residuals 1 and 7 in equal numbers: mean square 25, sigma exactly 5."""
    lay = _lay(dtype)
    cd = lay.code_dtype
    mu = np.full(_shape(lay), zero, cd)
    kv = np.full(_shape(lay), one, cd)
    kv[:, :, 1::2] = seven
    s = O.calibrate_sigma(lay, kv, mu, t_cal=lay.n_tokens)
    assert s.shape == (1, 2, 2, 8) and np.all(s == 5.0)
    # negative residuals (mu above kv) give the same scale
    s2 = O.calibrate_sigma(lay, mu, kv, t_cal=lay.n_tokens)
    assert np.all(s2 == 5.0)


def test_sigma_constant_residual_and_scale():
    """r = one bf16 step above 1 (2^-7) everywhere: sigma = 2^-7; doubling every
    value (exponent + 1) doubles sigma exactly."""
    lay = _lay()
    mu = np.full(_shape(lay), BF16_ONE, np.uint16)
    kv = np.full(_shape(lay), BF16_ONE + 1, np.uint16)
    assert np.all(O.calibrate_sigma(lay, kv, mu, 16) == 2.0 ** -7)
    rng = np.random.default_rng(3)
    mu = (rng.integers(0x3000, 0x4000, _shape(lay))).astype(np.uint16)
    kv = (mu.astype(np.int32) + rng.integers(-40, 41, _shape(lay))).astype(np.uint16)
    s1 = O.calibrate_sigma(lay, kv, mu, 16)
    s2 = O.calibrate_sigma(lay, kv + 0x80, mu + 0x80, 16)
    assert np.array_equal(s2, 2 * s1)


def test_sigma_matches_float64_rms():
    """Against numpy's own float64 mean of squares (a different summation order):
    equal, or one binary32 step apart where the two sums straddle a rounding point."""
    lay = _lay(T=300, H=4, D=32)
    rng = np.random.default_rng(11)
    mu_v = rng.standard_normal(_shape(lay)).astype(np.float32)
    kv_v = mu_v + 0.05 * rng.standard_normal(_shape(lay)).astype(np.float32)
    mu = (torch.from_numpy(mu_v).to(torch.bfloat16).view(torch.int16).numpy()).view(np.uint16)
    kv = (torch.from_numpy(kv_v).to(torch.bfloat16).view(torch.int16).numpy()).view(np.uint16)
    t_cal = 257
    s = O.calibrate_sigma(lay, kv, mu, t_cal)
    val = lambda c: (c.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    r = val(kv[:, :, :t_cal]) - val(mu[:, :, :t_cal])
    ref = np.sqrt(np.mean(r * r, axis=2)).astype(np.float32)
    ulps = np.abs(s.view(np.int32).astype(np.int64) - ref.view(np.int32).astype(np.int64))
    assert ulps.max() <= 1
    assert np.mean(ulps == 0) > 0.99


# ------------------------------------------------------------ sigma: invariances

def _random_pair(lay, seed):
    rng = np.random.default_rng(seed)
    mu = rng.integers(0x3C00, 0x4100, _shape(lay)).astype(np.uint16)
    kv = (mu.astype(np.int32) + rng.integers(-60, 61, _shape(lay))).astype(np.uint16)
    return kv, mu


def test_sigma_ignores_masked_late_and_nonfinite_elements():
    lay = _lay(T=40)
    kv, mu = _random_pair(lay, 5)
    t_cal = 25
    base = O.calibrate_sigma(lay, kv, mu, t_cal)
    # tokens at and after t_cal do not matter
    kv2 = kv.copy()
    kv2[:, :, t_cal:] = 0x7F7F
    assert np.array_equal(O.calibrate_sigma(lay, kv2, mu, t_cal), base)
    # masked-out elements do not matter, whatever their values
    rng = np.random.default_rng(9)
    mask = (rng.random(_shape(lay)) < 0.8).astype(np.uint8)
    with_mask = O.calibrate_sigma(lay, kv, mu, t_cal, mask=mask)
    kv3 = np.where(mask == 1, kv, np.uint16(0x7F00))
    assert np.array_equal(O.calibrate_sigma(lay, kv3, mu, t_cal, mask=mask), with_mask)
    # NaN / infinite codes count as masked out
    kv4 = np.where(mask == 1, kv, np.uint16(0x7FC0))
    mu4 = mu.copy()
    assert np.array_equal(O.calibrate_sigma(lay, kv4, mu4, t_cal), with_mask)
    kv5 = kv.copy()
    mu5 = np.where(mask == 1, mu, np.uint16(0xFF80))
    assert np.array_equal(O.calibrate_sigma(lay, kv5, mu5, t_cal), with_mask)


def test_sigma_clamps_at_least_valid_value():
    lay = _lay()
    kv, mu = _random_pair(lay, 1)
    # zero residuals, and nothing counted, both give 2^-126
    assert np.all(O.calibrate_sigma(lay, mu, mu, 16) == 2.0 ** -126)
    none = np.zeros(_shape(lay), np.uint8)
    assert np.all(O.calibrate_sigma(lay, kv, mu, 16, mask=none) == 2.0 ** -126)
    # largest finite residuals, opposite signs: the RMS overflows binary32 and clamps
    big = np.full(_shape(lay), 0x7F7F, np.uint16)
    s = O.calibrate_sigma(lay, big, big | 0x8000, 16)
    assert np.all(s == np.finfo(np.float32).max)


def test_sigma_rejects_bad_t_cal():
    lay = _lay()
    kv, mu = _random_pair(lay, 2)
    for t in (0, 17):
        with pytest.raises(O.OracleError):
            O.calibrate_sigma(lay, kv, mu, t)


@pytest.mark.parametrize("name", ["tiny", "fp8_32b"])
def test_sigma_matches_generator_calibration(name):
    """The workload generator calibrates sigma the same way (RMS over the first
    tokens, Gaussian-drawn elements only) with torch's float64 sums: the oracle
    given the generator's mask agrees to one binary32 step."""
    cfg = synth.CONFIGS[name].scaled(n_layers=1, n_tokens=384, calibrate=True, calib_tokens=200)
    w = synth.generate(cfg, "cpu", with_mask=True)
    h = synth.to_numpy(w)
    lay = O.Layout(O.BF16 if cfg.dtype == "bf16" else O.E4M3, cfg.n_layers, cfg.n_kv, cfg.n_heads,
                   cfg.head_dim, cfg.n_tokens)
    mask = w["mask"].numpy().astype(np.uint8)
    s = O.calibrate_sigma(lay, h["kv"], h["mu"], cfg.calib_tokens, mask=mask)
    ulps = np.abs(s.view(np.int32).astype(np.int64) - h["sigma"].view(np.int32).astype(np.int64))
    assert ulps.max() <= 1


# ------------------------------------------------------------ sigma blocks

def _encode_chunks(lay, kv, mu, sigma, counts):
    stream, offs = O.encode(lay, kv, mu, sigma, counts)
    return [bytes(stream[offs[k]:offs[k + 1]]) for k in range(len(offs) - 1)]


@pytest.mark.parametrize("dtype", [O.BF16, O.E4M3])
def test_sigma_blocks_equal_per_block_static_coding(dtype):
    """A cache coded with one sigma per block of B tokens gives, chunk for
    chunk, the bytes of each block's tokens coded as a cache of its own with
    that block's sigma as the frozen sigma (chunks are independent, and a
    block is a whole number of pages)."""
    H_, D = (2, 8) if dtype == O.BF16 else (1, 16)
    L, K, T, Tc, B = 2, 2, 700, 100, 300        # blocks of 300, 300, 100 tokens
    lay = O.Layout(dtype, L, K, H_, D, T, Tc, 32, sigma_block=B)
    rng = np.random.default_rng(21)
    cd = lay.code_dtype
    n = 65536 if dtype == O.BF16 else 256
    lo, hi = (0x3C00, 0x4100) if dtype == O.BF16 else (0x30, 0x50)
    mu = rng.integers(lo, hi, (L, K, T, H_, D)).astype(cd)
    kv = (mu.astype(np.int32) + rng.integers(-20, 21, mu.shape)).astype(cd)
    sigma = (0.01 + rng.random(lay.sigma_shape)).astype(np.float32)
    counts = O.histogram(dtype, kv)
    got = _encode_chunks(lay, kv, mu, sigma, counts)
    P = -(-T // Tc)
    for b in range(lay.n_sigma_blocks):
        t0, t1 = b * B, min(T, (b + 1) * B)
        sub = O.Layout(dtype, L, K, H_, D, t1 - t0, Tc, 32)
        ref = _encode_chunks(sub, np.ascontiguousarray(kv[:, :, t0:t1]),
                             np.ascontiguousarray(mu[:, :, t0:t1]),
                             np.ascontiguousarray(sigma[:, :, b]), counts)
        Pb = -(-(t1 - t0) // Tc)
        for p in range(L * K):
            for j in range(Pb):
                assert got[p * P + t0 // Tc + j] == ref[p * Pb + j], (b, p, j)
    # and the whole cache decodes back
    stream, offs = O.encode(lay, kv, mu, sigma, counts)
    assert np.array_equal(O.decode(lay, stream, offs, mu, sigma, counts), kv.reshape(-1))
    # a sigma table of the wrong shape is refused before the C code reads it
    with pytest.raises(ValueError):
        O.encode(lay, kv, mu, sigma[:, :, :2], counts)


def test_sigma_blocks_calibration():
    """Each block's sigma is its own first t_cal tokens' RMS: block 0 holds
    residuals 1 and 7 (sigma 5), block 1 residual 3 (sigma 3), and the short
    last block residual 0.5 (sigma 0.5) -- and equals the static calibration
    of the block's tokens alone."""
    lay = O.Layout(O.BF16, 1, 2, 2, 8, 600, 100, 32, sigma_block=200)
    shape = (1, 2, 600, 2, 8)
    mu = np.zeros(shape, np.uint16)
    kv = np.full(shape, BF16_ONE, np.uint16)
    kv[:, :, 1:200:2] = BF16_SEVEN
    kv[:, :, 200:400] = 0x4040                      # 3.0
    kv[:, :, 400:] = 0x3F00                         # 0.5
    s = O.calibrate_sigma(lay, kv, mu, t_cal=200)
    assert s.shape == (1, 2, 3, 2, 8)
    assert np.all(s[:, :, 0] == 5.0) and np.all(s[:, :, 1] == 3.0) and np.all(s[:, :, 2] == 0.5)
    rng = np.random.default_rng(4)
    kv2, mu2 = _random_pair(O.Layout(O.BF16, 1, 2, 2, 8, 600), 8)
    s2 = O.calibrate_sigma(lay, kv2, mu2, t_cal=150)
    for b in range(3):
        sub = O.Layout(O.BF16, 1, 2, 2, 8, 200)
        ref = O.calibrate_sigma(sub, np.ascontiguousarray(kv2[:, :, 200 * b:200 * (b + 1)]),
                                np.ascontiguousarray(mu2[:, :, 200 * b:200 * (b + 1)]), t_cal=150)
        assert np.array_equal(s2[:, :, b], ref)
    with pytest.raises(O.OracleError):
        O.calibrate_sigma(lay, kv2, mu2, t_cal=201)
    with pytest.raises(O.OracleError):          # B must be a multiple of the page length
        O.calibrate_sigma(O.Layout(O.BF16, 1, 2, 2, 8, 600, 100, 32, sigma_block=150), kv2, mu2, 10)
