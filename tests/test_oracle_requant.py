"""Pins of the oracle's 2b -> b bit requantisation (the PM-KVQ section of the
third page: progressive quantisation, Equivalent Right Shift with the new
scale (2^b + 1) S and the zero point kept).

Pins from outside the oracle: the page's own arithmetic ((2^(2b) - 1) /
(2^b - 1) = 2^b + 1, so the new grid's points sit on the old grid's), the
exact rational round(q / (2^b + 1)) for every code q (fractions), the
add-and-shift form the page says it reduces to, numpy shifts for the two
baselines, and a bit-level packing round trip."""
from fractions import Fraction

import numpy as np
import pytest

from oracle import oracle as O


def _pack(codes, w):
    bits = ((np.asarray(codes, np.uint64)[:, None] >> np.arange(w, dtype=np.uint64)) & 1).astype(np.uint8)
    return np.packbits(bits.reshape(-1), bitorder="little")


def _unpack(packed, n, w):
    bits = np.unpackbits(np.asarray(packed, np.uint8), bitorder="little")[: n * w].reshape(n, w)
    return (bits.astype(np.uint64) << np.arange(w, dtype=np.uint64)).sum(1)


@pytest.mark.parametrize("b", [1, 2, 4, 8])
def test_ers_is_exact_rounding_on_every_code(b):
    q = np.arange(2 ** (2 * b))
    q = np.concatenate([q, q]) if b == 1 else q         # n b must fill whole bytes
    n = q.size
    scale = np.full(4, 0.37, np.float32)
    zero = np.full(4, -3.25, np.float32)
    out, s = O.requantize(O.RQ_ERS, b, _pack(q, 2 * b), n, scale, -(-n // 4), zero_in=zero)
    got = _unpack(out, n, b)
    ref = np.array([int(Fraction(int(v), 2 ** b + 1) + Fraction(1, 2)) for v in q])
    assert np.array_equal(got, ref)
    # the page's add-and-shift form: t = q + 2^(b-1), a = t >> b, a - [a > t mod 2^b]
    t = q + 2 ** (b - 1)
    a = t >> b
    assert np.array_equal(got, a - (a > (t & (2 ** b - 1))))
    # (2^(2b) - 1) / (2^b - 1) = 2^b + 1: the scale grows by exactly that factor,
    # and old codes (2^b + 1) k are the new grid's points k
    assert Fraction(2 ** (2 * b) - 1, 2 ** b - 1) == 2 ** b + 1
    assert np.all(s == np.float32(np.float64(2 ** b + 1) * np.float64(np.float32(0.37))))
    k = np.arange(2 ** b)
    assert np.array_equal(got[(2 ** b + 1) * k], k)           # old codes (2^b + 1) k -> k
    assert got.max() == 2 ** b - 1


@pytest.mark.parametrize("b", [1, 2, 4, 8])
def test_shift_baselines(b):
    rng = np.random.default_rng(b)
    n = 8 * 37
    q = rng.integers(0, 2 ** (2 * b), n)
    sc = rng.random(7).astype(np.float32) + 0.1
    drs, s1 = O.requantize(O.RQ_DRS, b, _pack(q, 2 * b), n, sc, 50)
    mrs, s2 = O.requantize(O.RQ_MRS, b, _pack(q, 2 * b), n, sc, 50)
    assert np.array_equal(_unpack(drs, n, b), q >> b)
    assert np.array_equal(_unpack(mrs, n, b), np.minimum((q + 2 ** (b - 1)) >> b, 2 ** b - 1))
    ref = (sc[: len(s1)].astype(np.float64) * 2 ** b).astype(np.float32)
    assert len(s1) == 6 and np.array_equal(s1, ref) and np.array_equal(s1, s2)


def test_ers_error_is_smallest():
    """Reconstruction against the 8-bit values: ERS's error never exceeds half
    its own step and its RMS is below both shifts' (DRS is biased low)."""
    rng = np.random.default_rng(0)
    n = 4096
    q = rng.integers(0, 256, n)
    S = 0.01
    x = S * q
    errs = {}
    for mode in (O.RQ_ERS, O.RQ_DRS, O.RQ_MRS):
        out, s = O.requantize(mode, 4, _pack(q, 8), n, np.full(1, S, np.float32), n)
        xr = _unpack(out, n, 4) * float(s[0])
        errs[mode] = np.sqrt(np.mean((xr - x) ** 2))
        if mode == O.RQ_ERS:
            assert np.max(np.abs(xr - x)) <= 0.5 * float(s[0]) + 1e-9
    assert errs[O.RQ_ERS] < errs[O.RQ_MRS] < errs[O.RQ_DRS]


def test_requantize_rejects_bad_args():
    with pytest.raises(O.OracleError):
        O.requantize(O.RQ_ERS, 3, np.zeros(8, np.uint8), 8, np.ones(1, np.float32), 8)
    with pytest.raises(O.OracleError):
        O.requantize(O.RQ_ERS, 2, np.zeros(8, np.uint8), 6, np.ones(1, np.float32), 8)  # 6 * 2 bits
