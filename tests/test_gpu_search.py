"""Exhaustive check of the decoder's slot -> code search (skv_search_eval runs
the decoder's own estimate, exact test and cooperative search): for every one
of the 2^24 bf16 slots (2^16 for e4m3) and a spread of (mu, sigma), the code
equals the one the oracle's cumulative frequencies bracket (numpy
searchsorted over the oracle's C), and C(o), f(o) equal the oracle's, with
the minimum workspace (no search tables) and the full one (pair table and
outlier inverse tables)."""
import numpy as np
import pytest
import torch

from lossless_kv_cache_scalar_gb300 import Layout, synth
from lossless_kv_cache_scalar_gb300.api import search_eval
from oracle import oracle as O

pytestmark = pytest.mark.gpu


def _bf16(x):
    return int(torch.tensor([x]).to(torch.bfloat16).view(torch.int16).item()) & 0xFFFF


def _e4m3(x):
    return int(torch.tensor([x]).to(torch.float8_e4m3fn).view(torch.uint8).item())


@pytest.fixture(scope="module")
def counts_bf16():
    return synth.generate(synth.CONFIGS["tiny"], "cuda")["counts"]


@pytest.mark.parametrize("mu,sigma", [(1.5, 2.0 ** -5), (0.0, 1e-3), (-120.0, 30.0), (3.0e-39, 1e-36),
                                      (1e30, 1e29), (0.25, 1e30), (-0.0731, 0.004)])
@pytest.mark.parametrize("fast", [True, False])
def test_search_every_bf16_slot(counts_bf16, mu, sigma, fast):
    lay = Layout("bf16", 1, 2, 8, 128, 256)
    mc = _bf16(mu)
    C = O.cdf_all(O.BF16, mc, sigma, (95, 3, 2), counts_bf16.cpu().numpy().astype(np.uint64)).astype(np.int64)
    n = 1 << 24
    slots = torch.arange(n, dtype=torch.int32, device="cuda")
    mus = torch.full((n,), mc, dtype=torch.int32, device="cuda")
    sig = torch.full((n,), sigma, dtype=torch.float32, device="cuda")
    o, c, f = search_eval(lay, counts_bf16, mus, sig, slots, fast=fast)
    o = o.cpu().numpy()
    want = np.searchsorted(C, np.arange(n, dtype=np.int64), side="right") - 1
    bad = np.flatnonzero(o != want)
    assert bad.size == 0, f"{bad.size} slots wrong, first {bad[:5]}"
    assert np.array_equal(c.cpu().numpy(), C[want])
    assert np.array_equal(f.cpu().numpy(), C[want + 1] - C[want])


@pytest.mark.parametrize("mu,sigma", [(1.0, 0.4), (-37.0, 3.0), (0.0, 0.02), (448.0, 100.0), (3.0, 1e30)])
@pytest.mark.parametrize("fast", [True, False])
def test_search_every_e4m3_slot(mu, sigma, fast):
    w = synth.generate(synth.CONFIGS["fp8_32b"].scaled(n_layers=1, n_tokens=64), "cuda")
    lay = Layout("e4m3", 1, 2, 8, 128, 64)
    mc = _e4m3(mu)
    C = O.cdf_all(O.E4M3, mc, sigma, (95, 3, 2), w["counts"].cpu().numpy().astype(np.uint64)).astype(np.int64)
    n = 1 << 16
    slots = torch.arange(n, dtype=torch.int32, device="cuda")
    mus = torch.full((n,), mc, dtype=torch.int32, device="cuda")
    sig = torch.full((n,), sigma, dtype=torch.float32, device="cuda")
    o, c, f = search_eval(lay, w["counts"], mus, sig, slots, fast=fast)
    want = np.searchsorted(C, np.arange(n, dtype=np.int64), side="right") - 1
    assert np.array_equal(o.cpu().numpy(), want)
    assert np.array_equal(f.cpu().numpy(), C[want + 1] - C[want])


def test_search_mixed_queries(counts_bf16):
    """Random (mu, sigma, slot) triples in one launch, so neighbouring lanes of a
    warp search different distributions at once."""
    rng = np.random.default_rng(5)
    n = 200_000
    mus = rng.integers(0, 65536, n).astype(np.uint32)
    mus[(mus & 0x7F80) == 0x7F80] &= 0xBFFF                   # finite mu only
    sig = np.exp(rng.uniform(-20, 20, n)).astype(np.float32)
    slots = rng.integers(0, 1 << 24, n).astype(np.uint32)
    lay = Layout("bf16", 1, 2, 8, 128, 256)
    t = lambda a, dt: torch.from_numpy(a.view(dt)).cuda()
    o, c, f = search_eval(lay, counts_bf16, t(mus, np.int32), t(sig, np.float32), t(slots, np.int32))
    cnt = counts_bf16.cpu().numpy().astype(np.uint64)
    # the oracle's C at o and o + 1 for each query
    co = O.cdf_eval(O.BF16, mus, sig, o.cpu().numpy().astype(np.uint32), (95, 3, 2), cnt).astype(np.int64)
    c1 = O.cdf_eval(O.BF16, mus, sig, (o.cpu().numpy() + 1).astype(np.uint32), (95, 3, 2), cnt).astype(np.int64)
    s = slots.astype(np.int64)
    assert np.all(co <= s) and np.all(s < c1)
    assert np.array_equal(c.cpu().numpy(), co) and np.array_equal(f.cpu().numpy(), c1 - co)
