"""The C-ABI library builds, loads and exports every symbol include/skv.h declares;
its host-side geometry agrees with the SKV v1 format (checked against the oracle's
sizes). No GPU work is done here.
"""
import ctypes as C
import os
import re
import subprocess
import sys

import pytest

from lossless_kv_cache_scalar_gb300 import _binding as B
from lossless_kv_cache_scalar_gb300 import Layout
from oracle import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "skv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(skv_[a-z_0-9]+)\s*\(", text)))


def test_header_declarations_are_exported():
    names = _declared()
    assert "skv_encode" in names and "skv_decode" in names and "skv_decode_chunks" in names
    lib = B.lib()
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\b(skv_[a-z_0-9]+)\b", out))
    assert set(names) <= exported
    assert set(B.SIGNATURES) == set(names), "binding covers exactly the header"


def test_version_and_status_strings():
    lib = B.lib()
    assert lib.skv_version() == 1
    for code, name in B.STATUS_NAMES.items():
        assert lib.skv_status_string(code).decode() == name
    assert lib.skv_status_string(99).decode() == "UNKNOWN"


def test_layout_init_and_checks():
    lib = B.lib()
    lay = B.skv_layout()
    assert lib.skv_layout_init(C.byref(lay), 0, 36, 2, 8, 128, 32768) == 0
    assert (lay.tokens_per_chunk, lay.streams_per_chunk) == (256, 64)
    assert (lay.w_narrow, lay.w_wide, lay.w_marginal) == (95, 3, 2)
    bad = [dict(streams_per_chunk=48), dict(streams_per_chunk=288), dict(tokens_per_chunk=0),
           dict(w_marginal=3), dict(version=2), dict(dtype=5), dict(n_heads=1, head_dim=4), dict(sigma_block_tokens=100),
           dict(n_tokens=(1 << 40) + 1),                                   # T above 2^40
           dict(n_layers=1 << 20, n_kv=1 << 10),                           # 2^30 planes x 2^15 x 2^10 scalars
           dict(n_layers=0xFFFFFFFF, n_kv=0xFFFFFFFF, n_tokens=0)]         # empty, but 2^64 planes of sigma
    for kw in bad:
        l2 = B.skv_layout()
        C.memmove(C.byref(l2), C.byref(lay), C.sizeof(lay))
        for k, v in kw.items():
            setattr(l2, k, v)
        assert lib.skv_layout_check(C.byref(l2)) == 1, kw
    # e4m3 needs HD % 16 == 0, bf16 HD % 8 == 0
    assert lib.skv_layout_init(C.byref(lay), 1, 1, 1, 1, 8, 4) == 1
    assert lib.skv_layout_init(C.byref(lay), 0, 1, 1, 1, 8, 4) == 0


CASES = [("bf16", 1, 2, 8, 128, 256, 256, 64), ("bf16", 3, 2, 2, 64, 300, 256, 32),
         ("bf16", 2, 1, 1, 1024, 1000, 100, 256), ("e4m3", 2, 2, 2, 64, 96, 64, 64),
         ("bf16", 1, 2, 8, 128, 0, 256, 64), ("e4m3", 1, 1, 1, 16, 7, 3, 96)]


@pytest.mark.parametrize("dt,L,K,H,D,T,Tc,W", CASES)
def test_geometry_matches_oracle(dt, L, K, H, D, T, Tc, W):
    lay = Layout(dt, L, K, H, D, T, tokens_per_chunk=Tc, streams_per_chunk=W)
    ol = O.Layout(O.BF16 if dt == "bf16" else O.E4M3, L, K, H, D, T, tokens_per_chunk=Tc,
                  streams_per_chunk=W)
    assert lay.n_chunks == O.num_chunks(ol)
    assert lay.max_encoded_bytes == O.max_encoded_bytes(ol)
    small = lay.workspace_bytes(False, fast=False)
    assert small < (1 << 20) + 4 * L * K * H * D + 4096
    m = 24 if dt == "bf16" else 16
    # fast adds the two outlier inverse tables and, for bf16, the (edge, P_hat) pairs
    pairs = (8 * 65537 + 255) // 256 * 256 if dt == "bf16" else 0
    assert lay.workspace_bytes(False, fast=True) == small + 2 * (2 << m) + pairs
    if T:
        assert lay.workspace_bytes(True) > 0


def test_library_table_generator_is_independent_and_agrees():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "lossless_kv_cache_scalar_gb300", "csrc",
                                                     "gen_phi_q24.py"), "--check"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    lib_t = [int(x) for x in re.findall(r"(\d+)u", open(os.path.join(
        ROOT, "lossless_kv_cache_scalar_gb300", "csrc", "phi_q24.h")).read().split("*/")[1])]
    assert lib_t == [int(v) for v in O.phi_table()]


def test_host_staging_bytes():
    """skv_host_staging_bytes is host arithmetic: larger batches need more staging,
    the decoder's inverse tables add 2 x 2 x 2^m bytes, and bad arguments are refused."""
    lay = Layout("bf16", 8, 2, 8, 128, 1024)
    lib = B.lib()

    def q(lpb, op):
        v = C.c_uint64()
        rc = lib.skv_host_staging_bytes(C.byref(lay.c()), lpb, op, C.byref(v))
        return rc, v.value

    sizes = [q(l, 1)[1] for l in (1, 2, 4, 8)]
    assert all(a < b for a, b in zip(sizes, sizes[1:]))
    assert q(16, 1) == q(8, 1)                        # capped at the layer count
    rc0, dec = q(2, 0)
    rc2, dec_fast = q(2, 2)
    assert rc0 == 0 and rc2 == 0 and dec_fast - dec >= 2 * (2 << 24)
    assert q(0, 1)[0] == 1 and q(2, 7)[0] == 1
