"""The sharded coding path on one GPU (no process group): the cache's layers
split as bench.py splits them over N ranks, each part's codes counted by
skv_histogram on the GPU, the counts summed (what the all-reduce does), each
part encoded by a Coder of its own layers, and the parts stitched with the
exclusive scan of their byte totals: the result is byte for byte the one-GPU
encoding of the whole cache, and each part decodes back on its own.
"""
import pytest
import torch

import lossless_kv_cache_scalar_gb300 as skv
from lossless_kv_cache_scalar_gb300 import shard, synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,kw,world", [("qwen3_0p6b", dict(n_layers=5, n_tokens=600), 2),
                                           ("qwen3_0p6b", dict(n_layers=5, n_tokens=600), 3),
                                           ("fp8_32b", dict(n_layers=4, n_tokens=300), 4)])
def test_sharded_stitch_equals_one_gpu(name, kw, world):
    cfg = synth.CONFIGS[name].scaled(**kw)
    w = {k: v.cuda() for k, v in synth.generate(cfg).items()}
    full = skv.Layout(cfg.dtype, cfg.n_layers, cfg.n_kv, cfg.n_heads, cfg.head_dim, cfg.n_tokens)
    ref_bits, ref_offs = skv.Coder(full).encode(w["kv"], w["mu"], w["sigma"], w["counts"])
    # each rank's local histogram; their sum is what the all-reduce hands every rank
    parts = []
    for r in range(world):
        rng = shard.layer_ranges(cfg.n_layers, world)[r]
        sl = slice(rng.first, rng.first + rng.count)
        parts.append((rng, {k: w[k][sl] for k in ("kv", "mu", "sigma")}))
    counts = sum(skv.histogram(p["kv"], cfg.dtype) for _, p in parts)
    assert torch.equal(counts, w["counts"])
    streams, offsets = [], []
    for rng, p in parts:
        if rng.count == 0:
            continue
        lay = skv.Layout(cfg.dtype, rng.count, cfg.n_kv, cfg.n_heads, cfg.head_dim, cfg.n_tokens)
        coder = skv.Coder(lay)
        b, o = coder.encode(p["kv"], p["mu"], p["sigma"], counts)
        back = coder.decode(b, o, p["mu"], p["sigma"], counts)
        assert torch.equal(back, p["kv"])
        streams.append(b.cpu())
        offsets.append(o.cpu())
    s, o = shard.stitch(streams, offsets)
    assert torch.equal(o, ref_offs.cpu().to(torch.int64))
    assert torch.equal(s, ref_bits.cpu())
