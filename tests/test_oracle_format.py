"""Pins of the oracle's alphabet, edges and fixed-point Phi (SKV v1 format §§1-3).

Each check compares the oracle with something other than itself: exact
rational arithmetic on the code values, numpy's own bf16/e4m3 decoding via
torch, libm's erfc, and the table generator's exact regeneration.
"""
import math
import os
import subprocess
import sys
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _values_torch(dtype):
    """All code values decoded by torch (independent of the oracle)."""
    if dtype == O.BF16:
        codes = torch.arange(65536, dtype=torch.int32)
        codes = torch.where(codes >= 32768, codes - 65536, codes).to(torch.int16)
        return codes.view(torch.bfloat16).float().numpy().astype(np.float64)
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).float().numpy().astype(np.float64)


@pytest.mark.parametrize("dtype", [O.BF16, O.E4M3])
def test_values_match_torch_decoding(dtype):
    vals = _values_torch(dtype)
    n = len(vals)
    mine = np.array([O.value(dtype, b) for b in range(n)], np.float64)
    both_nan = np.isnan(vals) & np.isnan(mine)
    assert np.all(both_nan | (vals == mine))


@pytest.mark.parametrize("dtype", [O.BF16, O.E4M3])
def test_order_is_a_value_sort(dtype):
    vals = _values_torch(dtype)
    n = len(vals)
    ords = np.array([O.ord_(dtype, b) for b in range(n)])
    assert sorted(ords) == list(range(n)), "ord is a bijection"
    assert all(O.code(dtype, int(ords[b])) == b for b in range(n))
    fin = np.flatnonzero(np.isfinite(vals))
    by_ord = fin[np.argsort(ords[fin])]
    v = vals[by_ord]
    # finite values strictly increase along ord, except -0 directly below +0
    dv = np.diff(v)
    zero_pair = (v[:-1] == 0) & (v[1:] == 0)
    assert np.all((dv > 0) | zero_pair)
    neg0 = (1 << 15) if dtype == O.BF16 else (1 << 7)
    assert ords[neg0] + 1 == ords[0]
    # non-finite codes sit outside the finite range, negative ones below
    for b in np.flatnonzero(~np.isfinite(vals)):
        neg = b & (n // 2)
        if neg:
            assert ords[b] < ords[fin].min()
        else:
            assert ords[b] > ords[fin].max()


@pytest.mark.parametrize("dtype", [O.BF16, O.E4M3])
def test_edges_are_exact_midpoints(dtype):
    vals = _values_torch(dtype)
    n = len(vals)
    maxc = 0x7F7F if dtype == O.BF16 else 0x7E
    o_lo = O.ord_(dtype, maxc | (n // 2))
    o_hi = O.ord_(dtype, maxc)
    for o in range(n + 1):
        e = O.edge(dtype, o)
        if o <= o_lo:
            assert e == -math.inf
        elif o > o_hi:
            assert e == math.inf
        else:
            a = Fraction(float(vals[O.code(dtype, o - 1)]))
            b = Fraction(float(vals[O.code(dtype, o)]))
            assert Fraction(e) == (a + b) / 2, (o, e)
    # the central edge between -0 and +0 is +0
    assert O.edge(dtype, n // 2) == 0.0
    assert math.copysign(1.0, O.edge(dtype, n // 2)) == 1.0


def test_phi_table_against_libm():
    t = O.phi_table().astype(np.int64)
    assert t.shape == (4097,)
    assert t[0] == 0 and t[2048] == 1 << 23 and t[4096] == 1 << 24
    assert np.all(np.diff(t) >= 0)
    assert np.all(t + t[::-1] == 1 << 24)
    for i in range(4097):
        x = (i - 2048) / 256.0
        ref = (1 << 24) * 0.5 * math.erfc(-x / math.sqrt(2.0))
        frac = ref - math.floor(ref)
        if abs(frac - 0.5) < 1e-6:
            assert abs(t[i] - ref) <= 0.5 + 1e-6
        else:
            assert t[i] == round(ref), (i, t[i], ref)


def test_phi_table_regenerates():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "oracle", "gen_phi_table.py"), "--check"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr


def test_phi_q_grid_saturation_and_accuracy():
    t = O.phi_table().astype(np.int64)
    for j in range(-2048, 2049, 7):
        assert O.phi_q(256 * j) == t[j + 2048]
    assert O.phi_q(-524288) == 0 and O.phi_q(-10 ** 7) == 0
    assert O.phi_q(524288) == 1 << 24 and O.phi_q(10 ** 7) == 1 << 24
    rng = np.random.default_rng(5)
    zs = np.concatenate([rng.integers(-524288, 524288, 4000), np.arange(-1000, 1000)])
    for zq in zs:
        ref = (1 << 24) * 0.5 * math.erfc(-(zq / 65536.0) / math.sqrt(2.0))
        # linear interpolation on a 1/256 grid: |Phi''| <= 0.242 gives <= 7.8 units, plus rounding
        assert abs(O.phi_q(int(zq)) - ref) <= 9.0, zq


def test_phi_q_monotone_dense():
    prev = -1
    for zq in range(-524800, 524800, 37):
        v = O.phi_q(zq)
        assert v >= prev
        prev = v
