"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

The bar is bit-exactness everywhere: the model's cumulative frequencies, the
compressed bitstream and offsets, and the decoded KV codes. Inputs are the
seeded synthetic workloads (same recipe as the benchmark) at sizes the oracle
finishes in seconds, spanning several chunks and a ragged tail; the
full-size workloads are checked on sampled chunks (bytes equal to the
oracle's encoding of that chunk alone) and by exact round trip.
"""
import zlib

import numpy as np
import pytest
import torch

from lossless_kv_cache_scalar_gb300 import Coder, Layout, SKVError, cdf_eval, synth
from oracle import oracle as O
from tests import _skvtest as H

pytestmark = pytest.mark.gpu


def _bf16(x):
    return int(torch.tensor([x]).to(torch.bfloat16).view(torch.int16).item()) & 0xFFFF


def _e4m3(x):
    return int(torch.tensor([x]).to(torch.float8_e4m3fn).view(torch.uint8).item())


# ---------------------------------------------------------------- the model

MODEL_CASES = {
    "bf16": [(1.5, 2.0 ** -5), (-0.0731, 0.004), (0.0, 1e-3), (3.0e-39, 1e-36), (-3.3e38, 1e37),
             (12.5, 2.0 ** -126), (0.25, 1e30), (7.0, 0.031), (-2.0e-3, 50.0), (1e-40, 3.0)],
    "e4m3": [(1.0, 0.4), (-37.0, 3.0), (0.0, 0.02), (448.0, 100.0), (-0.015625, 2.0 ** -126),
             (3.0, 1e30)],
}


@pytest.mark.parametrize("dt", ["bf16", "e4m3"])
@pytest.mark.parametrize("weights", [(95, 3, 2), (100, 0, 0), (0, 0, 100), (50, 30, 20)])
def test_cdf_kernel_all_ordinals(dt, weights):
    n = 65536 if dt == "bf16" else 256
    rng = np.random.default_rng(17)
    counts = rng.integers(0, 40, n).astype(np.uint64)
    counts[rng.integers(0, n, n // 3)] = 0
    mus, sigs, ords = [], [], []
    for mu, sg in MODEL_CASES[dt]:
        mc = _bf16(mu) if dt == "bf16" else _e4m3(mu)
        mus.append(np.full(n + 1, mc, np.uint32))
        sigs.append(np.full(n + 1, sg, np.float32))
        ords.append(np.arange(n + 1, dtype=np.uint32))
    # plus random (mu code, sigma) pairs over the whole finite range
    k = 20000
    rmu = rng.integers(0, n, k).astype(np.uint32)
    fin = (rmu & 0x7F80) != 0x7F80 if dt == "bf16" else (rmu & 0x7F) != 0x7F
    rmu[~fin] = 0
    mus.append(rmu)
    sigs.append(np.exp(rng.uniform(-80, 80, k)).astype(np.float32).clip(2.0 ** -126, 3e38))
    ords.append(rng.integers(0, n + 1, k).astype(np.uint32))
    mus, sigs, ords = (np.concatenate(a) for a in (mus, sigs, ords))
    want = O.cdf_eval(O.BF16 if dt == "bf16" else O.E4M3, mus, sigs, ords, weights, counts)
    lay = Layout(dt, 1, 1, 1, 16, 1, weights=weights)
    t = lambda a, d: torch.from_numpy(a.view(d)).cuda()  # noqa: E731
    got = cdf_eval(lay, t(counts, np.int64), t(mus, np.int32), t(sigs, np.float32), t(ords, np.int32))
    got = got.cpu().numpy().astype(np.uint64)
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, (bad[:5], got[bad[:5]], want[bad[:5]], mus[bad[:5]], sigs[bad[:5]], ords[bad[:5]])


# ------------------------------------------------------------- whole streams

def _workload(cfg):
    w = synth.generate(cfg)
    return H.dev(w), H.host(w)


def test_tiny_bitexact():
    cfg = synth.CONFIGS["tiny"]
    wd, wh = _workload(cfg)
    H.assert_same_stream(H.layout_of(cfg), wd, wh)


SCALED = [
    ("qwen3_0p6b", dict(n_layers=2, n_tokens=1024 + 37)),
    ("qwen3_8b", dict(n_layers=1, n_tokens=1100)),
    ("fp8_32b", dict(n_layers=2, n_tokens=600, calib_tokens=512)),
    ("paged_14b", dict(n_layers=1, n_tokens=700, calib_tokens=512)),
]


@pytest.mark.parametrize("name,kw", SCALED, ids=[s[0] for s in SCALED])
def test_config_recipes_bitexact(name, kw):
    cfg = synth.CONFIGS[name].scaled(**kw)
    wd, wh = _workload(cfg)
    H.assert_same_stream(H.layout_of(cfg), wd, wh)


@pytest.mark.parametrize("W,Tc,T", [(32, 256, 300), (96, 100, 257), (256, 7, 20), (128, 1, 3),
                                    (64, 256, 1), (32, 64, 130)])
def test_geometries_bitexact(W, Tc, T):
    cfg = synth.CONFIGS["tiny"].scaled(n_tokens=T, n_heads=2, head_dim=64, seed=300 + W + T)
    wd, wh = _workload(cfg)
    H.assert_same_stream(H.layout_of(cfg, tokens_per_chunk=Tc, streams_per_chunk=W), wd, wh)


@pytest.mark.parametrize("W,Tc,T", [(32, 256, 300), (96, 100, 257), (256, 7, 20), (128, 1, 3),
                                    (256, 256, 513)])
def test_e4m3_geometries_bitexact(W, Tc, T):
    """The same ragged geometries for e4m3 (16 codes per vector; the decoder's
    lane-sliced code tables and per-word 1/sigma loads), against the oracle."""
    cfg = synth.CONFIGS["fp8_32b"].scaled(n_layers=1, n_tokens=T, n_heads=2, head_dim=64, seed=400 + W + T)
    wd, wh = _workload(cfg)
    H.assert_same_stream(H.layout_of(cfg, tokens_per_chunk=Tc, streams_per_chunk=W), wd, wh)


def test_empty_input():
    lay = Layout("bf16", 2, 2, 8, 128, 0)
    c = Coder(lay)
    z = torch.empty((2, 2, 0, 8, 128), dtype=torch.int16, device="cuda")
    sig = torch.ones((2, 2, 8, 128), device="cuda")
    cnt = torch.ones(65536, dtype=torch.int64, device="cuda")
    s, offs = c.encode(z, z, sig, cnt)
    assert s.numel() == 0 and offs.numel() == 1 and int(offs[0]) == 0
    back = c.decode(s, offs, z, sig, cnt)
    assert back.numel() == 0


@pytest.mark.parametrize("weights", [(100, 0, 0), (0, 0, 100), (50, 30, 20), (0, 100, 0)])
def test_weights_bitexact(weights):
    cfg = synth.CONFIGS["tiny"].scaled(n_tokens=300, seed=55)
    wd, wh = _workload(cfg)
    H.assert_same_stream(H.layout_of(cfg, weights=weights), wd, wh)


def test_all_bf16_bit_patterns():
    rng = np.random.default_rng(9)
    lay = Layout("bf16", 1, 1, 1, 1024, 80)
    n = lay.n_elems
    kv = rng.integers(0, 65536, n).astype(np.uint16)
    kv[:65536] = np.arange(65536, dtype=np.uint16)
    mu = rng.integers(0, 65536, n).astype(np.uint16)
    mu[(mu & 0x7F80) == 0x7F80] = 0x3F80
    sigma = np.exp(rng.normal(0, 4, 1024)).astype(np.float32)
    counts = np.bincount(kv, minlength=65536).astype(np.uint64)
    wh = {"kv": kv, "mu": mu, "sigma": sigma, "counts": counts}
    wd = {"kv": torch.from_numpy(kv.view(np.int16)).cuda().view(1, 1, 80, 1, 1024),
          "mu": torch.from_numpy(mu.view(np.int16)).cuda().view(1, 1, 80, 1, 1024),
          "sigma": torch.from_numpy(sigma).cuda(), "counts": torch.from_numpy(counts.view(np.int64)).cuda()}
    H.assert_same_stream(lay, wd, wh)


def test_all_e4m3_codes():
    rng = np.random.default_rng(4)
    lay = Layout("e4m3", 2, 2, 2, 64, 96, tokens_per_chunk=64)
    n = lay.n_elems
    kv = rng.integers(0, 256, n).astype(np.uint8)
    kv[:256] = np.arange(256, dtype=np.uint8)
    mu = rng.integers(0, 256, n).astype(np.uint8)
    mu[(mu & 0x7F) == 0x7F] = 0x38
    sigma = np.exp(rng.normal(0, 2, 2 * 2 * 128)).astype(np.float32)
    counts = np.bincount(kv, minlength=256).astype(np.uint64)
    shp = (2, 2, 96, 2, 64)
    wh = {"kv": kv, "mu": mu, "sigma": sigma, "counts": counts}
    wd = {"kv": torch.from_numpy(kv).cuda().view(shp), "mu": torch.from_numpy(mu).cuda().view(shp),
          "sigma": torch.from_numpy(sigma).cuda(), "counts": torch.from_numpy(counts.view(np.int64)).cuda()}
    H.assert_same_stream(lay, wd, wh)


def test_predictor_equal_to_target():
    cfg = synth.CONFIGS["tiny"]
    wd, wh = _workload(cfg)
    wd["mu"] = wd["kv"].clone()
    wh["mu"] = wh["kv"].copy()
    wd["sigma"] = torch.full_like(wd["sigma"], 2.0 ** -126)
    wh["sigma"] = np.full_like(wh["sigma"], 2.0 ** -126)
    s, offs, _ = H.assert_same_stream(H.layout_of(cfg), wd, wh)
    assert 8.0 * s.numel() / cfg.n_elems < 0.1


@pytest.mark.parametrize("name,kw", [("qwen3_0p6b", dict(n_layers=2, n_tokens=700)),
                                     ("fp8_32b", dict(n_layers=2, n_tokens=300, calib_tokens=256))])
def test_minimum_workspace_decode_is_identical(name, kw):
    # without the outlier inverse tables far outliers are found by bisection
    cfg = synth.CONFIGS[name].scaled(**kw)
    wd, _ = _workload(cfg)
    lay = H.layout_of(cfg)
    s, offs = Coder(lay).encode(wd["kv"], wd["mu"], wd["sigma"], wd["counts"])
    slow = Coder(lay, encode=False, fast_decode=False)
    assert slow.workspace.numel() < lay.workspace_bytes(False, fast=True)
    back = slow.decode(s, offs, wd["mu"], wd["sigma"], wd["counts"])
    assert torch.equal(back, wd["kv"])


# -------------------------------------------------------------- page access

def test_decode_chunks_pages():
    cfg = synth.CONFIGS["paged_14b"].scaled(n_layers=1, n_tokens=1000, calib_tokens=512)
    wd, wh = _workload(cfg)
    lay = H.layout_of(cfg)
    c = Coder(lay)
    s, offs = c.encode(wd["kv"], wd["mu"], wd["sigma"], wd["counts"])
    ids = torch.tensor([5, 0, 3, 7, 3], dtype=torch.int32, device="cuda")
    pages = c.decode_chunks(s, offs, wd["mu"], wd["sigma"], wd["counts"], ids)
    want = O.decode_pages(H.o_layout(lay), s.cpu().numpy(), offs.cpu().numpy().astype(np.uint64),
                          wh["mu"], wh["sigma"], wh["counts"], ids.cpu().numpy().astype(np.uint64))
    got = pages.cpu().numpy().view(np.uint16)
    # chunk 7 is the short last page of plane 1 (1000 = 3 * 256 + 232 tokens)
    for i, k in enumerate(ids.tolist()):
        ntok = 232 if k in (3, 7) else 256
        n = ntok * 1024
        assert np.array_equal(got[i, :n], want[i, :n]), k
        plane, page = divmod(k, 4)
        ref = wh["kv"].reshape(2, 1000 * 1024)[plane, page * 256 * 1024: page * 256 * 1024 + n]
        assert np.array_equal(got[i, :n], ref)


@pytest.mark.parametrize("W", [64, 256])
def test_prepared_page_decode(W):
    cfg = synth.CONFIGS["paged_14b"].scaled(n_layers=2, n_tokens=777, calib_tokens=512)
    wd, _ = _workload(cfg)
    lay = H.layout_of(cfg, streams_per_chunk=W)
    c = Coder(lay)
    s, offs = c.encode(wd["kv"], wd["mu"], wd["sigma"], wd["counts"])
    c.prepare_decode(wd["sigma"], wd["counts"])
    kv = wd["kv"].reshape(lay.n_layers * 2, -1)
    P = -(-lay.n_tokens // lay.tokens_per_chunk)
    rng = np.random.default_rng(W)
    for _ in range(3):
        ids = torch.tensor(rng.integers(0, lay.n_chunks, 5), dtype=torch.int32, device="cuda")
        pages = torch.zeros((5, lay.page_elems), dtype=wd["kv"].dtype, device="cuda")
        c.decode_chunks_prepared_into(s, offs, wd["mu"], ids, pages)
        c.check_status("prepared")
        for i, k in enumerate(ids.tolist()):
            plane, page = divmod(k, P)
            t0 = page * lay.tokens_per_chunk
            n = (min(lay.n_tokens, t0 + lay.tokens_per_chunk) - t0) * 1024
            assert torch.equal(pages[i, :n], kv[plane, t0 * 1024: t0 * 1024 + n])


def test_decode_chunks_rejects_bad_id():
    cfg = synth.CONFIGS["tiny"]
    wd, _ = _workload(cfg)
    c = Coder(H.layout_of(cfg))
    s, offs = c.encode(wd["kv"], wd["mu"], wd["sigma"], wd["counts"])
    ids = torch.tensor([0, 2], dtype=torch.int32, device="cuda")
    with pytest.raises(SKVError) as e:
        c.decode_chunks(s, offs, wd["mu"], wd["sigma"], wd["counts"], ids)
    assert e.value.name == "INVALID_ARG"


def test_binding_rejects_bad_buffers():
    """The C ABI takes bare pointers, so the binding refuses buffers that are too
    short, of the wrong element size or not contiguous before any call."""
    cfg = synth.CONFIGS["tiny"]
    wd, _ = _workload(cfg)
    lay = H.layout_of(cfg)
    c = Coder(lay)
    s, offs = c.encode(wd["kv"], wd["mu"], wd["sigma"], wd["counts"])
    args = (wd["mu"], wd["sigma"], wd["counts"])
    with pytest.raises(ValueError):                        # offsets one entry short
        c.decode(s, offs[:-1], *args)
    with pytest.raises(ValueError):                        # offsets as int32
        c.decode(s, offs.to(torch.int32), *args)
    with pytest.raises(ValueError):                        # bitstream not bytes
        c.decode(s[: s.numel() // 4 * 4].view(torch.int32), offs, *args)
    out, o2 = c.alloc_output()
    with pytest.raises(ValueError):                        # encoder offsets too short
        c.encode_into(wd["kv"], wd["mu"], wd["sigma"], wd["counts"], out, o2[:1])
    ids = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    half = torch.empty(2 * lay.page_elems, dtype=torch.uint8, device="cuda")   # 1-byte codes for bf16
    with pytest.raises(ValueError):
        c.decode_chunks_into(s, offs, *args, ids, half)
    strided = torch.tensor([0, 9, 1, 9], dtype=torch.int32, device="cuda")[::2]
    pages = torch.empty((2, lay.page_elems), dtype=wd["mu"].dtype, device="cuda")
    with pytest.raises(ValueError):                        # non-contiguous ids
        c.decode_chunks_into(s, offs, *args, strided, pages)
    c.prepare_decode(wd["sigma"], wd["counts"])
    with pytest.raises(ValueError):                        # mu of the wrong size
        c.decode_chunks_prepared_into(s, offs, wd["mu"].view(-1)[:16], ids, pages)
    with pytest.raises(ValueError):                        # query arrays of unequal length
        cdf_eval(lay, wd["counts"], torch.zeros(3, dtype=torch.int32, device="cuda"),
                 torch.ones(2, dtype=torch.float32, device="cuda"), torch.zeros(3, dtype=torch.int32, device="cuda"))
    # and the valid call still works
    c.decode_chunks_prepared_into(s, offs, wd["mu"], ids, pages)
    c.check_status("pages")


# ------------------------------------------------------------------ errors

def test_status_errors():
    cfg = synth.CONFIGS["tiny"]
    wd, _ = _workload(cfg)
    lay = H.layout_of(cfg)
    c = Coder(lay)
    sig = wd["sigma"].clone()
    sig.view(-1)[7] = float("nan")
    with pytest.raises(SKVError) as e:
        c.encode(wd["kv"], wd["mu"], sig, wd["counts"])
    assert e.value.name == "BAD_SIGMA"
    mu = wd["mu"].clone()
    mu.view(-1)[123] = 0x7F80
    with pytest.raises(SKVError) as e:
        c.encode(wd["kv"], mu, wd["sigma"], wd["counts"])
    assert e.value.name == "NONFINITE_MU"
    with pytest.raises(SKVError) as e:
        c.encode(wd["kv"], wd["mu"], wd["sigma"], torch.zeros_like(wd["counts"]))
    assert e.value.name == "EMPTY_MARGINAL"
    out, offs = c.alloc_output()
    small = out[: 100000]
    c.encode_into(wd["kv"], wd["mu"], wd["sigma"], wd["counts"], small, offs)
    with pytest.raises(SKVError) as e:
        c.check_status("encode")
    assert e.value.name == "CAPACITY"
    assert int(offs[-1]) > 100000


def test_corruption_detected():
    cfg = synth.CONFIGS["tiny"]
    wd, _ = _workload(cfg)
    c = Coder(H.layout_of(cfg))
    s, offs = c.encode(wd["kv"], wd["mu"], wd["sigma"], wd["counts"])
    rng = np.random.default_rng(1)
    for _ in range(6):
        bad = s.clone()
        pos = int(rng.integers(8 * 64 + 64, int(offs[1]) - 64))
        bad[pos] ^= 1 << int(rng.integers(0, 8))
        with pytest.raises(SKVError) as e:
            c.decode(bad, offs, wd["mu"], wd["sigma"], wd["counts"])
        assert e.value.name == "CORRUPT"
    with pytest.raises(SKVError):
        c.decode(s[:-16], offs, wd["mu"], wd["sigma"], wd["counts"])
    bo = offs.clone()
    bo[1] += 16
    with pytest.raises(SKVError):
        c.decode(s, bo, wd["mu"], wd["sigma"], wd["counts"])
    bad = s.clone()
    bad[7] = 0xFF
    with pytest.raises(SKVError):
        c.decode(bad, offs, wd["mu"], wd["sigma"], wd["counts"])
    # the context is still usable after all of the above
    back = c.decode(s, offs, wd["mu"], wd["sigma"], wd["counts"])
    assert torch.equal(back, wd["kv"])


# -------------------------------------------------------------- full sizes

FULL = ["qwen3_0p6b", "qwen3_8b", "fp8_32b", "paged_14b"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(name):
    cfg = synth.CONFIGS[name]
    wd = synth.generate(cfg, device="cuda")
    lay = H.layout_of(cfg)
    c = Coder(lay)
    s, offs = c.encode(wd["kv"], wd["mu"], wd["sigma"], wd["counts"])
    back = torch.empty_like(wd["mu"])
    c.decode_into(s, offs, wd["mu"], wd["sigma"], wd["counts"], back)
    c.check_status("decode")
    assert torch.equal(back, wd["kv"])
    del back
    # 64 chunks byte-compared with the oracle: the first and last, and 62 drawn
    # (fixed seed per workload) from every layer, K and V alike
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    n = lay.n_chunks
    ks = sorted(set([0, n - 1] + rng.choice(n, 62, replace=False).tolist()))
    offs_h = offs.cpu().numpy()
    sub, part = H.slice_chunks(lay, wd, ks)
    so, oo = O.encode(H.o_layout(sub), part["kv"], part["mu"], part["sigma"], part["counts"])
    for i, k in enumerate(ks):
        got = s[int(offs_h[k]):int(offs_h[k + 1])].cpu().numpy()
        assert np.array_equal(got, so[int(oo[i]):int(oo[i + 1])]), (name, k)
    bits = 8.0 * float(offs_h[-1]) / lay.n_elems
    assert bits < (7.0 if lay.dtype == "bf16" else 4.0), bits


def test_concurrent_coders_on_two_streams():
    """Two Coders (own workspaces, own work counters) encoding and decoding
    different caches at once on two streams give the serial results: no state
    is shared between calls beyond what the caller passes."""
    a = synth.generate(synth.CONFIGS["qwen3_0p6b"].scaled(n_layers=2, n_tokens=1024), "cuda")
    b = synth.generate(synth.CONFIGS["fp8_32b"].scaled(n_layers=2, n_tokens=600), "cuda")
    la, lb = H.layout_of(synth.CONFIGS["qwen3_0p6b"].scaled(n_layers=2, n_tokens=1024)), \
        H.layout_of(synth.CONFIGS["fp8_32b"].scaled(n_layers=2, n_tokens=600))
    ca, cb = Coder(la), Coder(lb)
    sa_ref, oa_ref = ca.encode(a["kv"], a["mu"], a["sigma"], a["counts"])
    sb_ref, ob_ref = cb.encode(b["kv"], b["mu"], b["sigma"], b["counts"])
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outa, offa = ca.alloc_output()
    outb, offb = cb.alloc_output()
    torch.cuda.synchronize()
    for _ in range(3):
        ca.encode_into(a["kv"], a["mu"], a["sigma"], a["counts"], outa, offa, stream=s1)
        cb.encode_into(b["kv"], b["mu"], b["sigma"], b["counts"], outb, offb, stream=s2)
    torch.cuda.synchronize()
    ca.check_status("a", s1)
    cb.check_status("b", s2)
    assert torch.equal(offa, oa_ref) and torch.equal(offb, ob_ref)
    assert torch.equal(outa[: sa_ref.numel()], sa_ref) and torch.equal(outb[: sb_ref.numel()], sb_ref)
    ka, kb = torch.empty_like(a["kv"]), torch.empty_like(b["kv"])
    for _ in range(3):
        ca.decode_into(sa_ref, oa_ref, a["mu"], a["sigma"], a["counts"], ka, stream=s1)
        cb.decode_into(sb_ref, ob_ref, b["mu"], b["sigma"], b["counts"], kb, stream=s2)
    torch.cuda.synchronize()
    ca.check_status("a", s1)
    cb.check_status("b", s2)
    assert torch.equal(ka, a["kv"]) and torch.equal(kb, b["kv"])
