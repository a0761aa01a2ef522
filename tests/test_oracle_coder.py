"""Pins of the oracle's coder (SKV v1 format §§6-7) against what the pages fix.

- Lossless: decode(encode(x)) == x bit for bit (wiki pipeline section: the
  decoder restores KV_full from the bits and (mu, sigma) alone).
- Rate = cross-entropy (wiki core-idea section H(p,q) = H(p) + KL with
  H(p) = 0; blog information-theory section): coded bits track the ideal
  sum of -log2 q(x) of the real-valued mixture.
- Gaussian closed form (blog information-theory section): at the optimal
  sigma the rate is 1/2 log(2 pi e sigma^2), here in bits per code of spacing
  Delta: 1/2 log2(2 pi e (sigma/Delta)^2).
- Predictor limits (wiki predictor-choice table; blog predictor section): the
  target itself as predictor costs ~0 bits, noise ~16 bits per bf16 scalar.
- The p-hat-only model codes at the data's empirical entropy.
"""
import math

import numpy as np
import pytest
import torch

from oracle import oracle as O
from lossless_kv_cache_scalar_gb300 import synth


def _layout(dtype, L, K, T, H, D, **kw):
    return O.Layout(dtype, L, K, H, D, T, **kw)


def _tiny():
    w = synth.to_numpy(synth.generate(synth.CONFIGS["tiny"]))
    lay = _layout(O.BF16, 1, 2, 256, 8, 128)
    return lay, w


def _payload_bits(lay, stream, offsets):
    return 8.0 * float(offsets[-1])


def test_tiny_round_trip_and_rate():
    lay, w = _tiny()
    s, offs = O.encode(lay, w["kv"], w["mu"], w["sigma"], w["counts"])
    assert offs[0] == 0 and np.all(np.diff(offs.astype(np.int64)) % 16 == 0)
    back = O.decode(lay, s, offs, w["mu"], w["sigma"], w["counts"])
    assert np.array_equal(back, w["kv"].reshape(-1))
    n = lay.n_elems
    bits = _payload_bits(lay, s, offs) / n
    ideal = O.ideal_bits(lay, w["kv"], w["mu"], w["sigma"], w["counts"]) / n
    model = O.model_bits(lay, w["kv"], w["mu"], w["sigma"], w["counts"]) / n
    # the coded size is within 1% of the ideal cross-entropy
    assert bits <= 1.01 * ideal, (bits, ideal)
    # and within the flush/header overhead of the integer model's own code length
    n_chunks = O.num_chunks(lay)
    overhead = n_chunks * (8 * 64 + 16 + 2 * 16) * 8 / n
    assert model <= bits <= model * 1.0005 + overhead + 0.001, (model, bits, overhead)
    assert 4.0 < bits < 7.0


def test_encode_is_deterministic_and_chunk_local():
    lay, w = _tiny()
    s1, o1 = O.encode(lay, w["kv"], w["mu"], w["sigma"], w["counts"], nthreads=1)
    s2, o2 = O.encode(lay, w["kv"], w["mu"], w["sigma"], w["counts"], nthreads=4)
    assert np.array_equal(s1, s2) and np.array_equal(o1, o2)
    # encoding a single chunk yields the same bytes as its slice of the full stream
    s3, o3 = O.encode(lay, w["kv"], w["mu"], w["sigma"], w["counts"], chunk_ids=[1])
    assert np.array_equal(s3, s1[int(o1[1]):int(o1[2])])
    pages = O.decode_pages(lay, s1, o1, w["mu"], w["sigma"], w["counts"], [1, 0])
    kv = w["kv"].reshape(2, -1)
    assert np.array_equal(pages[0], kv[1]) and np.array_equal(pages[1], kv[0])


@pytest.mark.parametrize("W,Tc,T", [(32, 256, 300), (64, 100, 257), (128, 7, 20), (256, 256, 1),
                                    (96, 64, 130), (64, 256, 0)])
def test_ragged_geometries_round_trip(W, Tc, T):
    cfg = synth.CONFIGS["tiny"].scaled(n_tokens=max(T, 1), n_heads=2, head_dim=64, seed=77 + W)
    w = synth.to_numpy(synth.generate(cfg))
    if T == 0:
        w["kv"] = w["kv"][:, :, :0]
        w["mu"] = w["mu"][:, :, :0]
    lay = _layout(O.BF16, 1, 2, T, 2, 64, tokens_per_chunk=Tc, streams_per_chunk=W)
    s, offs = O.encode(lay, w["kv"], w["mu"], w["sigma"], w["counts"])
    assert len(offs) == O.num_chunks(lay) + 1
    back = O.decode(lay, s, offs, w["mu"], w["sigma"], w["counts"])
    assert np.array_equal(back, w["kv"].reshape(-1))


def test_every_bit_pattern_round_trips():
    rng = np.random.default_rng(9)
    lay = _layout(O.BF16, 1, 1, 64, 1, 1024)
    kv = rng.integers(0, 65536, lay.n_elems).astype(np.uint16)
    kv[:65536] = np.arange(65536, dtype=np.uint16)        # all codes incl. NaN/inf payloads
    mu = rng.integers(0, 65536, lay.n_elems).astype(np.uint16)
    mu[(mu >> 7 & 0xFF) == 0xFF] = 0x3F80                   # mu must be finite
    sigma = np.exp(rng.normal(0, 4, 1024)).astype(np.float32)
    counts = np.bincount(kv, minlength=65536).astype(np.uint64)
    s, offs = O.encode(lay, kv, mu, sigma, counts)
    assert np.array_equal(O.decode(lay, s, offs, mu, sigma, counts), kv)


def test_e4m3_round_trip_all_codes():
    rng = np.random.default_rng(4)
    lay = _layout(O.E4M3, 2, 2, 96, 2, 64, tokens_per_chunk=64)
    kv = rng.integers(0, 256, lay.n_elems).astype(np.uint8)
    kv[:256] = np.arange(256, dtype=np.uint8)
    mu = rng.integers(0, 256, lay.n_elems).astype(np.uint8)
    mu[(mu & 0x7F) == 0x7F] = 0x38
    sigma = np.exp(rng.normal(0, 2, 2 * 2 * 128)).astype(np.float32)
    counts = np.bincount(kv, minlength=256).astype(np.uint64)
    s, offs = O.encode(lay, kv, mu, sigma, counts)
    assert np.array_equal(O.decode(lay, s, offs, mu, sigma, counts), kv)


def _gauss_layout(T):
    return _layout(O.BF16, 1, 1, T, 1, 1024, w_n=100, w_w=0, w_h=0)


@pytest.mark.parametrize("mu,sigma,delta", [(1.5, 2.0 ** -5, 2.0 ** -7), (192.0, 16.0, 1.0)])
def test_pure_gaussian_closed_form(mu, sigma, delta):
    T = 1024
    lay = _gauss_layout(T)
    g = torch.Generator().manual_seed(12)
    x = (mu + sigma * torch.randn(lay.n_elems, generator=g)).to(torch.bfloat16)
    kv = x.view(torch.int16).numpy().view(np.uint16)
    mu_c = torch.full((lay.n_elems,), mu).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    sig = np.full(1024, sigma, np.float32)
    closed = 0.5 * math.log2(2 * math.pi * math.e * (sigma / delta) ** 2)
    ideal = O.ideal_bits(lay, kv, mu_c, sig, None) / lay.n_elems
    s, offs = O.encode(lay, kv, mu_c, sig, None)
    coded = 8.0 * float(offs[-1]) / lay.n_elems
    assert abs(ideal - closed) < 0.02, (ideal, closed)
    assert abs(coded - closed) < 0.02 + 0.01, (coded, closed)
    assert np.array_equal(O.decode(lay, s, offs, mu_c, sig, None), kv)


def test_phat_only_codes_at_empirical_entropy():
    lay, w = _tiny()
    lay.w_n, lay.w_w, lay.w_h = 0, 0, 100
    c = w["counts"].astype(np.float64)
    p = c[c > 0] / c.sum()
    ent = float(-(p * np.log2(p)).sum())
    s, offs = O.encode(lay, w["kv"], w["mu"], w["sigma"], w["counts"])
    coded = 8.0 * float(offs[-1]) / lay.n_elems
    flush = O.num_chunks(lay) * (64 * 8 + 64) * 8 / lay.n_elems
    # the floor of one count per code costs -log2(1 - N/M) = 0.0056 bits at most
    assert ent - 0.001 <= coded <= ent + 0.0057 + flush + 0.002, (coded, ent)


def test_predictor_equal_to_target_costs_almost_nothing():
    lay, w = _tiny()
    sig = np.full_like(w["sigma"], 2.0 ** -126)
    s, offs = O.encode(lay, w["kv"], w["kv"], sig, w["counts"])
    coded = 8.0 * float(offs[-1]) / lay.n_elems
    assert coded < 0.1, coded
    assert np.array_equal(O.decode(lay, s, offs, w["kv"], sig, w["counts"]), w["kv"].reshape(-1))


def test_noise_costs_sixteen_bits():
    rng = np.random.default_rng(21)
    lay = _layout(O.BF16, 1, 1, 512, 1, 1024, w_n=0, w_w=0, w_h=100)
    kv = rng.integers(0, 65536, lay.n_elems).astype(np.uint16)
    mu = np.full(lay.n_elems, 0x3F80, np.uint16)
    counts = np.ones(65536, np.uint64)              # uniform histogram: f = 256 for every code
    s, offs = O.encode(lay, kv, mu, np.ones(1024, np.float32), counts)
    coded = 8.0 * float(offs[-1]) / lay.n_elems
    flush = O.num_chunks(lay) * (64 * 8 + 16 + 2 * 16) * 8 / lay.n_elems
    assert 16.0 <= coded <= 16.0 + 0.0003 + flush, coded


def test_corruption_is_detected():
    lay, w = _tiny()
    s, offs = O.encode(lay, w["kv"], w["mu"], w["sigma"], w["counts"])
    rng = np.random.default_rng(0)
    hdr = 8 * 64 + 16
    for trial in range(6):
        bad = s.copy()
        pos = int(rng.integers(hdr + 64, int(offs[1]) - 64))
        bad[pos] ^= np.uint8(1 << int(rng.integers(0, 8)))
        with pytest.raises(O.OracleError) as e:
            O.decode(lay, bad, offs, w["mu"], w["sigma"], w["counts"])
        assert e.value.name == "CORRUPT"
    # truncated stream, inconsistent offsets, state out of range
    with pytest.raises(O.OracleError):
        O.decode(lay, s[:-16], offs, w["mu"], w["sigma"], w["counts"])
    bad_off = offs.copy()
    bad_off[1] += 16
    with pytest.raises(O.OracleError):
        O.decode(lay, s, bad_off, w["mu"], w["sigma"], w["counts"])
    bad = s.copy()
    bad[7] = 0xFF
    with pytest.raises(O.OracleError):
        O.decode(lay, bad, offs, w["mu"], w["sigma"], w["counts"])


def test_input_errors():
    lay, w = _tiny()
    sig = w["sigma"].copy()
    sig.reshape(-1)[5] = np.nan
    with pytest.raises(O.OracleError) as e:
        O.encode(lay, w["kv"], w["mu"], sig, w["counts"])
    assert e.value.name == "BAD_SIGMA"
    mu = w["mu"].copy()
    mu.reshape(-1)[100] = 0x7F80
    with pytest.raises(O.OracleError) as e:
        O.encode(lay, w["kv"], mu, w["sigma"], w["counts"])
    assert e.value.name == "NONFINITE_MU"
    with pytest.raises(O.OracleError) as e:
        O.encode(lay, w["kv"], w["mu"], w["sigma"], np.zeros(65536, np.uint64))
    assert e.value.name == "EMPTY_MARGINAL"


# The rate bound on every workload recipe (scaled to a few million scalars so
# the oracle finishes in seconds): coded bits per scalar at most 1% above the
# ideal cross-entropy of the real-valued mixture (blog information-theory
# section: code length = -log2 q), and within the chunk header and flush
# overhead of the integer model's own code length, so that a growth of either
# fails here.
@pytest.mark.parametrize("name,layers,tokens", [("tiny", None, None), ("qwen3_0p6b", 2, 1024),
                                                ("qwen3_8b", 2, 2048), ("fp8_32b", 2, 2048),
                                                ("paged_14b", 1, 2048)])
def test_rate_bound_every_recipe(name, layers, tokens):
    cfg = synth.CONFIGS[name]
    if layers:
        cfg = cfg.scaled(n_layers=layers, n_tokens=tokens)
    w = synth.to_numpy(synth.generate(cfg))
    dt = O.BF16 if cfg.dtype == "bf16" else O.E4M3
    lay = _layout(dt, cfg.n_layers, cfg.n_kv, cfg.n_tokens, cfg.n_heads, cfg.head_dim)
    s, offs = O.encode(lay, w["kv"], w["mu"], w["sigma"], w["counts"])
    n = lay.n_elems
    bits = _payload_bits(lay, s, offs) / n
    ideal = O.ideal_bits(lay, w["kv"], w["mu"], w["sigma"], w["counts"]) / n
    model = O.model_bits(lay, w["kv"], w["mu"], w["sigma"], w["counts"]) / n
    assert bits <= 1.01 * ideal, (name, bits, ideal)
    # per chunk: W final states (8 B), the group word counts padded to 16 B, and
    # at most 12 B of padding per group's word array
    W, G = lay.streams_per_chunk, lay.streams_per_chunk // 32
    header = O.num_chunks(lay) * (8 * W + 16 * ((4 * G + 15) // 16) + 12 * G) * 8 / n
    assert model <= bits <= model + header + 0.002, (name, model, bits, header)
