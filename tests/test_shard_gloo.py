"""Sharded coding across ranks (world size 2, gloo on CPU).

Each rank codes its own contiguous layers; the p_hat histogram is all-reduced
first (it is global side information), and an exclusive scan of the per-rank
byte totals stitches the ranks' streams into the single-rank bitstream. The
per-rank coder here is the CPU oracle (no GPU in these tests); the stitching
and the collectives are the host logic the GPU path uses.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from lossless_kv_cache_scalar_gb300 import shard, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


CFG = synth.CONFIGS["qwen3_0p6b"].scaled(n_layers=3, n_tokens=300)


def _worker(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, ROOT)
    from oracle import oracle as O
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = synth.to_numpy(synth.generate(CFG))
    cache = {k: torch.from_numpy(w[k]) for k in ("kv", "mu", "sigma")}
    # the bench's sharding path, with the oracle's histogram as the rank's counter
    hist = lambda kv: torch.from_numpy(O.histogram(O.BF16, kv.numpy()).astype(np.int64))
    rng, part, counts = shard.rank_inputs(cache, rank, world, hist)
    kv, mu, sig = part["kv"].numpy(), part["mu"].numpy(), part["sigma"].numpy()
    counts = counts.numpy().astype(np.uint64)
    assert np.array_equal(counts, w["counts"])
    lay = O.Layout(O.BF16, rng.count, CFG.n_kv, CFG.n_heads, CFG.head_dim, CFG.n_tokens)
    s, offs = O.encode(lay, kv, mu, sig, counts, nthreads=2)
    base, total = shard.distributed_base(int(offs[-1]))
    np.save(os.path.join(out_dir, f"s{rank}.npy"), s)
    np.save(os.path.join(out_dir, f"o{rank}.npy"), offs.astype(np.int64))
    np.save(os.path.join(out_dir, f"b{rank}.npy"), np.array([base, total], np.int64))
    dist.barrier()
    dist.destroy_process_group()


def test_layer_ranges_cover_and_balance():
    for n, w in [(36, 8), (3, 2), (2, 4), (40, 1), (0, 3)]:
        r = shard.layer_ranges(n, w)
        assert [x.rank for x in r] == list(range(w))
        assert sum(x.count for x in r) == n
        assert all(r[i].first + r[i].count == r[i + 1].first for i in range(w - 1))
        assert max(x.count for x in r) - min(x.count for x in r) <= 1


def test_two_rank_sharded_encode_equals_single(tmp_path):
    from oracle import oracle as O
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    w = synth.to_numpy(synth.generate(CFG))
    lay = O.Layout(O.BF16, CFG.n_layers, CFG.n_kv, CFG.n_heads, CFG.head_dim, CFG.n_tokens)
    s_ref, o_ref = O.encode(lay, w["kv"], w["mu"], w["sigma"], w["counts"])
    streams = [torch.from_numpy(np.load(tmp_path / f"s{r}.npy")) for r in range(world)]
    offs = [torch.from_numpy(np.load(tmp_path / f"o{r}.npy")) for r in range(world)]
    s, o = shard.stitch(streams, offs)
    assert np.array_equal(s.numpy(), s_ref)
    assert np.array_equal(o.numpy(), o_ref.astype(np.int64))
    # each rank's all-gathered base is where its chunks start in the global stream
    for r in range(world):
        base, total = np.load(tmp_path / f"b{r}.npy")
        assert total == int(o_ref[-1])
        n_before = sum(x.count for x in shard.layer_ranges(CFG.n_layers, world)[:r]) * CFG.n_kv * 2
        assert base == int(o_ref[n_before])
