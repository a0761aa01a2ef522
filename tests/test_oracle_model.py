"""Pins of the oracle's cumulative frequencies C(o) and its inversion (SKV v1 format §5).

The integer model is compared with the real-valued mixture of the Speculative
KV Coding wiki (mixture section), evaluated in double precision with libm's
erfc; the search with numpy's searchsorted on the full table.
"""
import math

import numpy as np
import pytest

from oracle import oracle as O

M = {O.BF16: 1 << 24, O.E4M3: 1 << 16}
NC = {O.BF16: 65536, O.E4M3: 256}


def _bf16(x: float) -> int:
    import torch
    return int(torch.tensor([x], dtype=torch.float32).to(torch.bfloat16).view(torch.int16).item()) & 0xFFFF


def _e4m3(x: float) -> int:
    import torch
    return int(torch.tensor([x], dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).item())


def _counts(dtype, seed=3):
    rng = np.random.default_rng(seed)
    n = NC[dtype]
    c = rng.integers(0, 50, n).astype(np.uint64)
    c[rng.integers(0, n, n // 3)] = 0
    return c


def _real_cdf(dtype, mu_code, sigma, weights, counts):
    """o + (M - N) * q_cum(E(o)) / 100 with the exact mixture CDF (double, libm)."""
    n = NC[dtype]
    mu = O.value(dtype, mu_code)
    wn, ww, wh = weights
    tot = float(counts.sum())
    cum = np.concatenate([[0.0], np.cumsum([float(counts[O.code(dtype, o)]) for o in range(n)])])
    out = np.zeros(n + 1)
    for o in range(n + 1):
        e = O.edge(dtype, o)
        def phi(x):
            return 0.5 * math.erfc(-x / math.sqrt(2.0))
        zn = (e - mu) / sigma if math.isfinite(e) else e
        pn = phi(zn) if math.isfinite(zn) else (0.0 if zn < 0 else 1.0)
        pw = phi(zn / 3) if math.isfinite(zn) else pn
        ph = cum[o] / tot if tot else 0.0
        out[o] = o + (M[dtype] - n) * (wn * pn + ww * pw + wh * ph) / 100.0
    return out


CASES = [
    (O.BF16, 1.5, 2.0 ** -5), (O.BF16, -0.0731, 0.004), (O.BF16, 0.0, 1e-3),
    (O.BF16, 3.0e-39, 1e-36), (O.BF16, -3.3e38, 1e37), (O.BF16, 12.5, 2.0 ** -126),
    (O.BF16, 0.25, 1e30), (O.BF16, 7.0, 0.031),
    (O.E4M3, 1.0, 0.4), (O.E4M3, -37.0, 3.0), (O.E4M3, 0.0, 0.02), (O.E4M3, 448.0, 100.0),
]


@pytest.mark.parametrize("dtype,mu,sigma", CASES)
@pytest.mark.parametrize("weights", [(95, 3, 2), (100, 0, 0), (0, 0, 100), (50, 30, 20)])
def test_cdf_properties_and_real_mixture(dtype, mu, sigma, weights):
    counts = _counts(dtype)
    mc = _bf16(mu) if dtype == O.BF16 else _e4m3(mu)
    c = O.cdf_all(dtype, mc, sigma, weights, counts).astype(np.int64)
    n = NC[dtype]
    assert c[0] == 0 and c[n] == M[dtype]
    f = np.diff(c)
    assert f.min() >= 1 and f.sum() == M[dtype]
    ref = _real_cdf(dtype, mc, np.float32(sigma).item(), weights, counts)
    # z is quantised to 2^-16 (<= phi(0) 2^-16 of mass) and Phi is linearly
    # interpolated on a 1/256 grid (<= 9 units of 2^-24): in C units this is
    # (M - N) * (0.4 * 2^-16 + 10 * 2^-24), plus 2 for the floors.
    tol = (M[dtype] - n) * (0.4 * 2.0 ** -16 + 10 * 2.0 ** -24) + 2
    err = np.abs(c - ref)
    assert err.max() <= tol, (err.max(), tol, int(err.argmax()))


def test_cdf_eval_matches_full_table():
    rng = np.random.default_rng(11)
    counts = _counts(O.BF16)
    mus = rng.integers(0, 65536, 40)
    mus[(mus >> 7 & 0xFF) == 0xFF] = 0x3F80
    sig = np.exp(rng.normal(-3, 3, 40)).astype(np.float32)
    for i in range(40):
        full = O.cdf_all(O.BF16, int(mus[i]), float(sig[i]), (95, 3, 2), counts)
        ords = rng.integers(0, 65537, 64).astype(np.uint32)
        got = O.cdf_eval(O.BF16, np.full(64, mus[i]), np.full(64, sig[i]), ords, (95, 3, 2), counts)
        assert np.array_equal(got, full[ords])


def test_pure_gaussian_is_symmetric_about_mu():
    # With weights (100,0,0) and mu on a code, mass is symmetric: f(ord(mu)+k) == f(ord(mu)-k)
    # as long as the code spacing is uniform around mu (mid-binade).
    mc = _bf16(1.5)
    c = O.cdf_all(O.BF16, mc, 2.0 ** -5, (100, 0, 0)).astype(np.int64)
    f = np.diff(c)
    o = O.ord_(O.BF16, mc)
    for k in range(1, 30):
        assert abs(int(f[o + k]) - int(f[o - k])) <= 2


@pytest.mark.parametrize("dtype,mu,sigma", [(O.BF16, 1.5, 2.0 ** -5), (O.BF16, 0.0, 1e-3),
                                            (O.BF16, -120.0, 30.0), (O.E4M3, 3.0, 0.7)])
def test_inversion_at_every_boundary(dtype, mu, sigma):
    counts = _counts(dtype)
    mc = _bf16(mu) if dtype == O.BF16 else _e4m3(mu)
    c = O.cdf_all(dtype, mc, sigma, (95, 3, 2), counts).astype(np.uint64)
    n = NC[dtype]
    lows = c[:-1]
    highs = c[1:] - 1
    slots = np.concatenate([lows, highs])
    want = np.concatenate([np.arange(n), np.arange(n)]).astype(np.uint32)
    if dtype == O.E4M3:
        slots = np.arange(M[dtype], dtype=np.uint64)
        want = (np.searchsorted(c, slots, side="right") - 1).astype(np.uint32)
    else:
        rng = np.random.default_rng(2)
        extra = rng.integers(0, M[dtype], 100000).astype(np.uint64)
        slots = np.concatenate([slots, extra])
        want = np.concatenate([want, (np.searchsorted(c, extra, side="right") - 1).astype(np.uint32)])
    got = O.find_symbols(dtype, mc, sigma, slots, (95, 3, 2), counts)
    assert np.array_equal(got, want)


def test_bad_sigma_and_nonfinite_mu_are_reported():
    with pytest.raises(O.OracleError) as e:
        O.cdf_all(O.BF16, 0x3F80, 0.0)
    assert e.value.name == "BAD_SIGMA"
    with pytest.raises(O.OracleError) as e:
        O.cdf_all(O.BF16, 0x3F80, float("inf"))
    assert e.value.name == "BAD_SIGMA"
    with pytest.raises(O.OracleError) as e:
        O.cdf_all(O.BF16, 0x7FC0, 1.0, (100, 0, 0))
    assert e.value.name == "NONFINITE_MU"
    with pytest.raises(O.OracleError) as e:
        O.cdf_all(O.BF16, 0x3F80, 1.0, (95, 3, 2), np.zeros(65536, np.uint64))
    assert e.value.name == "EMPTY_MARGINAL"


@pytest.mark.parametrize("mu,sigma", [(1.5, 2.0 ** -5), (-120.0, 30.0)])
def test_inversion_exhaustive_bf16(mu, sigma):
    """Every one of the 2^24 bf16 slots: the oracle's search returns the o with
    C(o) <= slot < C(o+1), i.e. numpy's searchsorted over the oracle's own C."""
    counts = _counts(O.BF16)
    mc = _bf16(mu)
    c = O.cdf_all(O.BF16, mc, sigma, (95, 3, 2), counts).astype(np.uint64)
    step = 1 << 22
    for s0 in range(0, 1 << 24, step):
        slots = np.arange(s0, s0 + step, dtype=np.uint64)
        want = (np.searchsorted(c, slots, side="right") - 1).astype(np.uint32)
        got = O.find_symbols(O.BF16, mc, sigma, slots, (95, 3, 2), counts)
        assert np.array_equal(got, want), s0
