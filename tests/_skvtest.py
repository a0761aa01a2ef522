"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and the CPU oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

from lossless_kv_cache_scalar_gb300 import Coder, Layout, synth
from oracle import oracle as O


def o_layout(lay: Layout) -> O.Layout:
    w = lay.weights
    return O.Layout(O.BF16 if lay.dtype == "bf16" else O.E4M3, lay.n_layers, lay.n_kv, lay.n_heads,
                    lay.head_dim, lay.n_tokens, lay.tokens_per_chunk, lay.streams_per_chunk,
                    w[0], w[1], w[2])


def layout_of(cfg: synth.SynthConfig, **kw) -> Layout:
    return Layout(cfg.dtype, cfg.n_layers, cfg.n_kv, cfg.n_heads, cfg.head_dim, cfg.n_tokens, **kw)


def host(w: dict) -> dict:
    return synth.to_numpy(w)


def dev(w: dict, device="cuda") -> dict:
    return {k: v.to(device) for k, v in w.items()}


def gpu_encode(lay: Layout, wd: dict):
    c = Coder(lay, wd["kv"].device)
    s, offs = c.encode(wd["kv"], wd["mu"], wd["sigma"], wd["counts"])
    return s, offs, c


def oracle_encode(lay: Layout, wh: dict, chunk_ids=None):
    return O.encode(o_layout(lay), wh["kv"], wh["mu"], wh["sigma"], wh["counts"], chunk_ids=chunk_ids)


def assert_same_stream(lay: Layout, wd: dict, wh: dict):
    """GPU bitstream and offsets equal the oracle's byte for byte; GPU decode restores kv."""
    s, offs, c = gpu_encode(lay, wd)
    so, oo = oracle_encode(lay, wh)
    got_offs = offs.cpu().numpy().astype(np.uint64)
    assert np.array_equal(got_offs, oo), "offsets differ"
    got = s.cpu().numpy()
    if not np.array_equal(got, so):
        bad = np.flatnonzero(got != so)
        raise AssertionError(f"bitstream differs at {bad.size} bytes, first {bad[:8]}")
    back = c.decode(s, offs, wd["mu"], wd["sigma"], wd["counts"])
    assert torch.equal(back, wd["kv"]), "GPU decode does not restore the input"
    return s, offs, c


def slice_chunks(lay: Layout, wd: dict, ks):
    """The inputs of full-page chunks ks stacked as one layout of len(ks)
    one-page planes (host numpy): plane i is chunk ks[i], with its own sigma."""
    P = -(-lay.n_tokens // lay.tokens_per_chunk)
    kvs, mus, sigs = [], [], []
    for k in ks:
        plane, page = divmod(int(k), P)
        l, kv = divmod(plane, lay.n_kv)
        t0 = page * lay.tokens_per_chunk
        assert t0 + lay.tokens_per_chunk <= lay.n_tokens, "full pages only"
        kvs.append(wd["kv"][l, kv, t0:t0 + lay.tokens_per_chunk])
        mus.append(wd["mu"][l, kv, t0:t0 + lay.tokens_per_chunk])
        sigs.append(wd["sigma"][l, kv])
    sub = Layout(lay.dtype, len(ks), 1, lay.n_heads, lay.head_dim, lay.tokens_per_chunk, lay.tokens_per_chunk,
                 lay.streams_per_chunk, lay.weights)
    import torch
    part = {"kv": torch.stack(kvs)[:, None].contiguous(), "mu": torch.stack(mus)[:, None].contiguous(),
            "sigma": torch.stack(sigs)[:, None].contiguous(), "counts": wd["counts"]}
    return sub, host(part)


def slice_chunk(lay: Layout, wd: dict, k: int):
    """The inputs of chunk k alone, as a one-chunk layout (host numpy)."""
    P = -(-lay.n_tokens // lay.tokens_per_chunk)
    plane, page = divmod(k, P)
    l, kv = divmod(plane, lay.n_kv)
    t0 = page * lay.tokens_per_chunk
    t1 = min(lay.n_tokens, t0 + lay.tokens_per_chunk)
    sub = Layout(lay.dtype, 1, 1, lay.n_heads, lay.head_dim, t1 - t0, lay.tokens_per_chunk,
                 lay.streams_per_chunk, lay.weights)
    part = {"kv": wd["kv"][l, kv, t0:t1].contiguous(), "mu": wd["mu"][l, kv, t0:t1].contiguous(),
            "sigma": wd["sigma"][l, kv].contiguous(), "counts": wd["counts"]}
    return sub, host(part)
