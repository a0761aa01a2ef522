"""Benchmark of the speculative KV coder on GB300.

One step = the whole hot path over one batch: encode the full synthetic KV
cache (set-up, model + rANS encode, offset scan, compaction) and decode it
back (set-up, CDF search + rANS decode). `value` is uncompressed KV bytes per
second over encode + decode, device-timed with CUDA events on the coder's
stream; the inputs (4.8 GB of KV and 4.8 GB of mu for the default workload)
are far larger than the 129 MB L2, so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl skv|reference]

--impl reference times the CPU oracle (oracle/), the only reference there is
for this method, on a bounded sample of the same workload.
Under torchrun (N > 1) the one cache is sharded by layer (strong scaling):
each rank codes its contiguous layers; the only exchanges are the all-reduce
of the code histogram (p_hat is global side information) before coding and
the all-gather of the ranks' byte totals that stitches their streams; rank 0
checks the stitched total against a one-GPU encoding of the whole cache.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

# The format's own arithmetic per scalar, by instruction class: the totals
# table of the SKV v1 format's section 9, read from the format text at the
# repository root and checked against the library's copy (skv_op_table). The arithmetic roofline
# is the scalars per second of the matching skv_peak_probe table probe.
OP_CLASSES = ["fp32", "fminmax", "iadd", "logic", "shift", "iminmax", "imad", "imad_hi", "imad_wide",
              "cvt", "mufu", "popc", "vote", "lds", "ldt", "sts"]
OP_TABLES = [("bf16", "encode"), ("bf16", "decode"), ("e4m3", "encode"), ("e4m3", "decode")]


def op_tables(check_lib: bool = True) -> dict:
    """{(dtype, op): {"counts": {class: n}, "instructions": n, "ops": weighted}} from SKV v1 format §9."""
    import re
    out = {}
    with open(os.path.join(ROOT, "FORMAT.md")) as fh:
        for line in fh:
            m = re.match(r"\| (bf16|e4m3) (encode|decode) \|(.*)\|\s*$", line)
            if not m:
                continue
            v = [int(x) for x in m.group(3).split("|")]
            if len(v) != len(OP_CLASSES) + 2:
                raise SystemExit(f"SKV v1 format §9: malformed row {line.strip()}")
            out[(m.group(1), m.group(2))] = {"counts": dict(zip(OP_CLASSES, v[:-2])), "instructions": v[-2],
                                             "ops": v[-1]}
    if sorted(out) != sorted(OP_TABLES):
        raise SystemExit("SKV v1 format §9: operation table rows missing")
    if check_lib:
        import ctypes as C
        from lossless_kv_cache_scalar_gb300 import _binding as B
        n = len(OP_CLASSES)
        for t, key in enumerate(OP_TABLES):
            counts, weights = (C.c_uint32 * n)(), (C.c_uint32 * n)()
            B.check("skv_op_table", B.lib().skv_op_table(t, counts, weights, n))
            if list(counts) != [out[key]["counts"][c] for c in OP_CLASSES]:
                raise SystemExit(f"skv_op_table({key}) differs from SKV v1 format §9")
            if sum(a * b for a, b in zip(counts, weights)) != out[key]["ops"]:
                raise SystemExit(f"skv_op_table({key}) weights differ from SKV v1 format §9")
    return out


SMS = 152               # GB300 streaming multiprocessors
LANES_PER_SM_CLK = 128  # 4 schedulers x 32 lanes issue per clock (the uniform issue peak, for comparison)


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            return json.load(fh)
    except OSError:
        return {}


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons. Started before the
    warm-up (so that it is sampling once the timed region begins); only the
    samples whose timestamps fall inside the timed region's host window
    (mark_start .. mark_end) are kept."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        fd, self.path = tempfile.mkstemp(prefix="skv_clocks_", suffix=".csv")
        self.fh = os.fdopen(fd, "w")
        self.proc = None
        self.t0 = self.t1 = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(gpu_index)], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
            self.fh.close()
            os.unlink(self.path)
        if self.proc is not None:
            import atexit
            atexit.register(self._end)

    def _end(self):
        if self.proc is not None and self.proc.poll() is None:
            self.proc.kill()

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        import datetime
        rows = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            for line in fh:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(p[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append((ts, float(p[2]), float(p[3]), {n for n, v in zip(names, p[6:10])
                                                                 if v.lower() == "active"}))
                except ValueError:
                    continue
        os.unlink(self.path)
        inside = [r for r in rows if self.t0 is not None and self.t1 is not None and self.t0 <= r[0] <= self.t1]
        window = "timed region"
        if not inside and rows:     # a region shorter than the sampling period: the sample nearest to it
            mid = 0.5 * (self.t0 + self.t1) if self.t0 is not None and self.t1 is not None else rows[-1][0]
            inside, window = [min(rows, key=lambda r: abs(r[0] - mid))], "sample nearest to the timed region"
        return {"sm_mhz": statistics.median(r[1] for r in inside) if inside else None,
                "sm_max_mhz": max(r[2] for r in inside) if inside else None,
                "samples": len(inside), "window": window,
                "reasons": sorted(set().union(*(r[3] for r in inside))) if inside else []}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def cpu_oracle_run(cfg, sample_chunks: int, nthreads: int, seconds_hint: float = 0.0):
    """Encode + decode `sample_chunks` chunks of the workload with the CPU oracle.

    Returns (uncompressed bytes processed, seconds, description)."""
    from lossless_kv_cache_scalar_gb300 import synth
    from oracle import oracle as O
    T = min(cfg.n_tokens, 256 * max(1, sample_chunks // 2))
    sub = cfg.scaled(n_layers=1, n_tokens=T)
    w = synth.to_numpy(synth.generate(sub))
    lay = O.Layout(O.BF16 if cfg.dtype == "bf16" else O.E4M3, 1, sub.n_kv, sub.n_heads, sub.head_dim, T)
    t0 = time.perf_counter()
    s, offs = O.encode(lay, w["kv"], w["mu"], w["sigma"], w["counts"], nthreads=nthreads)
    back = O.decode(lay, s, offs, w["mu"], w["sigma"], w["counts"], nthreads=nthreads)
    dt = time.perf_counter() - t0
    assert np.array_equal(back, w["kv"].reshape(-1))
    nbytes = lay.n_elems * sub.bytes_per_code
    desc = (f"{O.num_chunks(lay)} chunks ({lay.n_elems} scalars) of the {cfg.name} recipe, "
            f"1 layer x {sub.n_kv} x {T} tokens, encode+decode, oracle threads={nthreads}")
    return nbytes, dt, desc


def rate_sample(w, offsets, lay, layers: int = 4):
    """Coded bits over the ideal cross-entropy (the CPU oracle's real-valued
    mixture, libm) on a sample of the workload: the first 256-token page of K
    and V in `layers` evenly spaced layers, coded bits from the GPU stream's
    offsets. The rate bound of the method asks for at most 1.01."""
    from oracle import oracle as O
    L, T = w["kv"].shape[0], w["kv"].shape[2]
    tc = min(lay.tokens_per_chunk, T)
    pages = -(-T // lay.tokens_per_chunk)
    offs = offsets.cpu().numpy().astype(np.int64)
    counts = w["counts"].cpu().numpy().astype(np.uint64)
    coded = ideal = 0.0
    picked = sorted(set(int(i * L / layers) for i in range(layers)))
    for l in picked:
        sub = O.Layout(O.BF16 if lay.dtype == "bf16" else O.E4M3, 1, lay.n_kv, lay.n_heads, lay.head_dim, tc,
                       tokens_per_chunk=lay.tokens_per_chunk, streams_per_chunk=lay.streams_per_chunk,
                       w_n=lay.weights[0], w_w=lay.weights[1], w_h=lay.weights[2])
        kv = w["kv"][l:l + 1, :, :tc].cpu().numpy()
        mu = w["mu"][l:l + 1, :, :tc].cpu().numpy()
        sig = w["sigma"][l:l + 1].cpu().numpy()
        if lay.sigma_block_tokens:
            sig = sig[:, :, :1]
        ideal += O.ideal_bits(sub, kv, mu, sig.reshape(1, lay.n_kv, lay.n_heads, lay.head_dim), counts)
        for kvi in range(lay.n_kv):
            k = (l * lay.n_kv + kvi) * pages
            coded += 8.0 * (offs[k + 1] - offs[k])
    return {"bits_over_ideal": coded / ideal, "sample": f"page 0 of K and V in layers {picked}",
            "ideal": "sum of -log2 q over the sample, q the real-valued mixture over each code's interval"}


def cpu_table(single_chunks: int = 8, parallel_chunks: int = 64):
    """The CPU oracle on every workload recipe: encode + decode throughput
    (GB/s of uncompressed KV) single-threaded and chunk-parallel over all the
    host's cores, each on a bounded sample of the recipe (1 layer, K and V,
    the first tokens)."""
    from lossless_kv_cache_scalar_gb300 import synth
    from oracle import oracle as O
    rows = {}
    for name, cfg in synth.CONFIGS.items():
        row = {}
        for label, chunks, threads in (("single_thread", single_chunks, 1),
                                       ("parallel", parallel_chunks, O.threads())):
            nb, dt, desc = cpu_oracle_run(cfg, chunks, threads)
            row[label] = {"gbs": nb / dt / 1e9, "threads": threads, "seconds": dt, "sample": desc}
        rows[name] = row
    import platform
    print(json.dumps({"cpu_baseline_table": rows, "unit": "GB/s of uncompressed KV, encode + decode",
                      "host": platform.machine(), "cores": O.threads()}), flush=True)
    return 0


def run_reference(args, cfg):
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    from oracle import oracle as O
    nthreads = O.threads()
    total_b, total_t = 0, 0.0
    desc = ""
    for i in range(args.warmup + args.steps):
        b, t, desc = cpu_oracle_run(cfg, args.ref_chunks, nthreads)
        if i >= args.warmup:
            total_b += b
            total_t += t
    gbs = total_b / total_t / 1e9
    line = {"metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
            "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "u32/u64 int + f32",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": cfg.name, "shape": [cfg.n_layers, cfg.n_kv, cfg.n_tokens, cfg.n_heads,
                                                       cfg.head_dim],
                       "code_dtype": cfg.dtype, "scalars": cfg.n_elems, "sample": desc},
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": nthreads, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


METRIC = "KV encode+decode GB/s (uncompressed bytes) on GB300"


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default="qwen3_8b")
    ap.add_argument("--impl", default="skv", choices=["skv", "reference"])
    ap.add_argument("--ref-chunks", type=int, default=32, help="chunks per oracle step")
    ap.add_argument("--cpu-chunks", type=int, default=128,
                    help="chunks in the cpu_baseline sample (about 15 core-seconds of oracle work on 16 cores)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-layers", type=int, default=0,
                    help="layers per batch of the host pipelines (0: the library's default, four batches)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the cpu_baseline leg")
    ap.add_argument("--layers", type=int, default=None, help="override n_layers (profiling cases)")
    ap.add_argument("--streams", type=int, default=64, help="streams per chunk (32..256)")
    ap.add_argument("--tokens", type=int, default=None, help="override n_tokens (profiling cases)")
    ap.add_argument("--page-latency", type=int, default=200,
                    help="single-page random decodes timed after the run (0: skip)")
    ap.add_argument("--sigma-block", type=int, default=0,
                    help="tokens per sigma block (0: the workload's frozen per-channel sigma); "
                         "blocks are calibrated on the device from their own tokens")
    ap.add_argument("--offload", type=int, default=1,
                    help="time the offload decode from pinned host memory (0: skip)")
    ap.add_argument("--staging-mb", type=int, default=1024, help="offload staging buffer (two halves)")
    ap.add_argument("--requant", type=int, default=1,
                    help="time skv_requantize (8 -> 4 bits) on the workload's KV quantised to 8 bits (0: skip)")
    ap.add_argument("--alu-probe", type=int, default=1,
                    help="measure the integer / binary32 issue rates with skv_peak_probe (0: skip)")
    ap.add_argument("--model-inputs", type=int, default=1,
                    help="time skv_histogram and skv_calibrate_sigma on the workload (0: skip)")
    ap.add_argument("--traffic-json", default=os.path.join(ROOT, "profiles", "traffic.json"))
    ap.add_argument("--cpu-table", action="store_true",
                    help="only time the CPU oracle on every workload recipe (single-thread and chunk-parallel "
                         "samples) and print that table as one JSON line")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3) if args.impl == "skv" else args.warmup

    from lossless_kv_cache_scalar_gb300 import synth
    if args.cpu_table:
        return cpu_table()
    cfg = synth.CONFIGS[args.config]
    if args.layers or args.tokens:
        cfg = cfg.scaled(n_layers=args.layers, n_tokens=args.tokens)
    if args.impl == "reference":
        return run_reference(args, cfg)

    import lossless_kv_cache_scalar_gb300 as skv
    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    # One cache, sharded by layer (the path's own partition): every rank draws
    # the same cache, keeps its contiguous layers, counts their codes on the
    # GPU and all-reduces the histogram (p_hat is global); N = 1 is the whole
    # cache on one GPU.
    from lossless_kv_cache_scalar_gb300 import shard
    w_all = synth.generate(cfg, device=dev, with_mask=args.sigma_block > 0)
    rng, part, counts = shard.rank_inputs(w_all, rank, world, lambda kv: skv.histogram(kv, cfg.dtype))
    if world == 1 and not torch.equal(counts, w_all["counts"]):
        raise SystemExit("bench: skv_histogram differs from the workload's counts")
    w = dict(part, counts=counts)
    if "mask" in w_all:
        w["mask"] = w_all["mask"][rng.first: rng.first + rng.count]
    full_layers = cfg.n_layers
    cfg = cfg.scaled(n_layers=rng.count)
    del w_all
    torch.cuda.empty_cache()
    lay = skv.Layout(cfg.dtype, cfg.n_layers, cfg.n_kv, cfg.n_heads, cfg.head_dim, cfg.n_tokens,
                     streams_per_chunk=args.streams, sigma_block_tokens=args.sigma_block)
    if args.sigma_block:
        # position-aware sigma: each block's own RMS over its Gaussian-drawn elements
        mask = w.pop("mask").view(torch.uint8)
        w["sigma"] = skv.calibrate_sigma(lay, w["kv"], w["mu"], min(args.sigma_block, cfg.n_tokens),
                                         mask=mask)
        del mask
    sigma_side_bits = 32.0 * w["sigma"].numel() / lay.n_elems
    coder = skv.Coder(lay, dev)
    out, offsets = coder.alloc_output()
    back = torch.empty_like(w["mu"])
    stream = torch.cuda.Stream(device=dev)
    n_el = lay.n_elems
    raw_bytes = n_el * lay.bytes_per_code

    def step(s):
        coder.encode_into(w["kv"], w["mu"], w["sigma"], w["counts"], out, offsets, s)
        coder.decode_into(out, offsets, w["mu"], w["sigma"], w["counts"], back, s)

    sampler = ClockSampler(local) if rank == 0 else None
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step(stream)
    coder.check_status("warmup", stream)
    if not torch.equal(back, w["kv"]):
        raise SystemExit("bench: decode did not restore the input")
    total_bytes = int(offsets[-1].item())

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    barrier()
    if sampler:
        sampler.mark_start()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            ev[i][0].record(stream)
            coder.encode_into(w["kv"], w["mu"], w["sigma"], w["counts"], out, offsets, stream)
            ev[i][1].record(stream)
            coder.decode_into(out, offsets, w["mu"], w["sigma"], w["counts"], back, stream)
            ev[i][2].record(stream)
    barrier()
    if sampler:
        sampler.mark_end()
    clocks = sampler.stop() if sampler else {}
    coder.check_status("timed", stream)
    t_enc = sum(e[0].elapsed_time(e[1]) for e in ev) / 1e3
    t_dec = sum(e[1].elapsed_time(e[2]) for e in ev) / 1e3
    t_tot = t_enc + t_dec
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([t_tot, t_enc, t_dec], device=dev, dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        t_tot, t_enc, t_dec = t.tolist()
    # the whole cache's bytes (every rank's layers) over the slowest rank's time
    cache_bytes = raw_bytes * full_layers // max(cfg.n_layers, 1) if world > 1 else raw_bytes
    if world > 1:
        t = torch.tensor([raw_bytes], device=dev, dtype=torch.int64)
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        cache_bytes = int(t.item())
    value = cache_bytes * args.steps / t_tot / 1e9
    # this rank's byte base in the stitched stream and the cache's total
    base, stitched_total = shard.distributed_base(total_bytes, device=dev) if world > 1 else (0, total_bytes)
    enc_gbs = raw_bytes * args.steps / t_enc / 1e9
    dec_gbs = raw_bytes * args.steps / t_dec / 1e9

    # roofline of the dominant kernel (encode or decode call): the format's
    # operations per scalar (SKV v1 format §9) over the rate at which the
    # table probe runs that same operation mix on this GPU
    dom = "decode" if t_dec >= t_enc else "encode"
    t_dom = (t_dec if dom == "decode" else t_enc) / args.steps
    sm_mhz = clocks.get("sm_mhz") or _peaks().get("sm_max_mhz", 2070.0)
    uniform_tops = SMS * LANES_PER_SM_CLK * sm_mhz * 1e6 / 1e12
    tables = op_tables()
    traffic = inst_per_scalar = None
    try:
        with open(args.traffic_json) as fh:
            prof = json.load(fh)
        traffic = prof.get(f"{cfg.name}:{dom}")
        inst_per_scalar = {k: prof.get(f"{cfg.name}:{k}:thread_inst_per_scalar") for k in ("encode", "decode")}
    except (OSError, ValueError):
        traffic = None
    hbm_peak = _peaks().get("hbm_gbs", 6685.5)
    probes = alu_peaks(dev) if (args.alu_probe and rank == 0) else None

    def arith(op, t_total):
        """(achieved Tops, peak Tops, frac, frac against the uniform issue peak) for one direction."""
        tab = tables[(lay.dtype, op)]
        scal_s = n_el * args.steps / t_total
        achieved = tab["ops"] * scal_s / 1e12
        peak = tab["ops"] * probes["tables"][f"{lay.dtype} {op}"] / 1e12 if probes else None
        return achieved, peak, (achieved / peak if peak else None), achieved / uniform_tops

    a_enc, a_dec = arith("encode", t_enc), arith("decode", t_dec)
    achieved, peak_tops, frac, frac_uniform = a_dec if dom == "decode" else a_enc
    # per-GPU characterisations: rank 0 on its own layers
    lead = rank == 0
    page_lat = page_latency(coder, out, offsets, w, lay, args, dev) if (args.page_latency and lead) else None
    inputs = model_inputs_run(w, lay, args, dev, hbm_peak) if (args.model_inputs and lead) else None
    offload = offload_run(coder, out, offsets, w, lay, args, dev, total_bytes) if (args.offload and lead) else None
    requant = requant_run(w, lay, dev, hbm_peak) if (args.requant and lay.dtype == "bf16" and lead) else None
    bits = 8.0 * stitched_total / (cache_bytes / lay.bytes_per_code)

    # end to end through the public API with host buffers, every rank on its layers
    e2e = None
    if not args.no_e2e:
        barrier()
        e2e = e2e_run(coder, w, lay, args, dev, total_bytes)
        if world > 1:
            tmax = torch.tensor([e2e["seconds"]], device=dev, dtype=torch.float64)
            dist.all_reduce(tmax, op=dist.ReduceOp.MAX)
            sums = torch.tensor([lay.n_elems * lay.bytes_per_code, e2e["h2d_bytes_per_step"],
                                 e2e["d2h_bytes_per_step"]], device=dev, dtype=torch.int64)
            dist.all_reduce(sums, op=dist.ReduceOp.SUM)
            e2e["value"] = int(sums[0]) * e2e["steps"] / float(tmax[0]) / 1e9
            e2e["h2d_bytes_per_step"], e2e["d2h_bytes_per_step"] = int(sums[1]), int(sums[2])
            e2e["seconds"] = float(tmax[0])
    # N > 1: the stitched total equals the one-GPU encoding of the whole cache
    single_total = None
    if world > 1 and lead:
        wf = synth.generate(synth.CONFIGS[args.config].scaled(n_layers=args.layers, n_tokens=args.tokens)
                            if (args.layers or args.tokens) else synth.CONFIGS[args.config], device=dev)
        del coder, out, back
        torch.cuda.empty_cache()
        layf = skv.Layout(cfg.dtype, full_layers, cfg.n_kv, cfg.n_heads, cfg.head_dim, cfg.n_tokens,
                          streams_per_chunk=args.streams)
        cf = skv.Coder(layf, dev)
        sf, of = cf.encode(wf["kv"], wf["mu"], wf["sigma"], wf["counts"])
        single_total = int(of[-1].item())
        del wf, cf, sf, of
        if single_total != stitched_total:
            raise SystemExit(f"bench: stitched total {stitched_total} != one-GPU total {single_total}")
    line = None
    if rank == 0:
        cpu = None
        if args.no_cpu:
            cpu = {"value": None, "unit": "GB/s", "cores": None, "kind": "oracle", "sample": "skipped (--no-cpu)"}
        else:
          try:
            from oracle import oracle as O
            nb, dt, desc = cpu_oracle_run(cfg, args.cpu_chunks, O.threads())
            cpu = {"value": nb / dt / 1e9, "unit": "GB/s", "cores": O.threads(), "kind": "oracle",
                   "sample": desc}
          except Exception as e:  # the baseline must not hide the GPU number
            cpu = {"value": None, "unit": "GB/s", "cores": None, "kind": "oracle", "sample": f"failed: {e}"}
        try:
            rate = rate_sample(w, offsets, lay)
        except Exception as e:  # a check beside the number, not the number
            rate = {"bits_over_ideal": None, "sample": f"failed: {e}"}
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * t_tot / args.steps, "higher_is_better": True,
            "scaling": "strong", "vs_baseline": None, "dtype": "u32/u64 int + f32", "data": "synthetic",
            "config": {"workload": cfg.name, "shape": [full_layers, cfg.n_kv, cfg.n_tokens, cfg.n_heads,
                                                       cfg.head_dim],
                       "sharding": (f"layers split over {world} GPUs ({rng.count} on rank 0), p_hat counts "
                                    "all-reduced, byte bases all-gathered" if world > 1 else "one GPU, all layers"),
                       "stitched_bytes": stitched_total, "one_gpu_bytes": single_total if world > 1 else stitched_total,
                       "code_dtype": cfg.dtype, "scalars": cache_bytes // lay.bytes_per_code,
                       "tokens_per_chunk": lay.tokens_per_chunk,
                       "streams_per_chunk": lay.streams_per_chunk, "weights": list(lay.weights),
                       "sigma_block_tokens": lay.sigma_block_tokens,
                       "l2": "inputs 2 x %.1f GB >> 129 MB L2, no flush" % (raw_bytes / 1e9)},
            "encode_gbs": enc_gbs, "decode_gbs": dec_gbs, "bits_per_scalar": bits, "rate": rate,
            "compression_ratio": 8.0 * lay.bytes_per_code / bits,
            "sigma_side_bits_per_scalar": sigma_side_bits,
            "roofline": {"bound": "alu", "kernel": dom, "achieved": achieved, "peak": peak_tops,
                         "unit": "Tops/s", "frac": frac, "traffic": traffic,
                         "alg_ops_per_scalar": tables[(lay.dtype, dom)]["ops"],
                         "alg_instructions_per_scalar": tables[(lay.dtype, dom)]["instructions"],
                         "ncu_thread_inst_per_scalar": inst_per_scalar,
                         "peak_basis": ("measured: skv_peak_probe running the format's %s %s operation table "
                                        "(SKV v1 format §9) with full instruction-level parallelism"
                                        % (lay.dtype, dom)) if probes else "not measured (--alu-probe 0)",
                         "frac_of_uniform_issue": frac_uniform,
                         "uniform_issue_tops": uniform_tops,
                         "uniform_basis": f"{SMS} SMs x {LANES_PER_SM_CLK} lane-ops/clk x {sm_mhz:.0f} MHz (sampled)",
                         "hbm_bound_gbs": hbm_peak * lay.bytes_per_code / (2 * lay.bytes_per_code + bits / 8),
                         "probes": probes,
                         "hbm_peak_gbs": hbm_peak},
            "roofline_encode_frac": a_enc[2],
            "roofline_decode_frac": a_dec[2],
            "roofline_encode_frac_uniform": a_enc[3],
            "roofline_decode_frac_uniform": a_dec[3],
            "cpu_baseline": cpu,
            "page_decode_latency_us": page_lat,
            "model_inputs": inputs,
            "offload": offload,
            "requantize": requant,
            "e2e": e2e,
            "gpu_launches": 8 * args.steps,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


def page_latency(coder, out, offsets, w, lay, args, dev):
    """Random single-page decodes after a one-time skv_decode_prepare: per-call
    device time (CUDA events around each call, same stream), p50/p99 in us."""
    stream = torch.cuda.Stream(device=dev)
    rng = np.random.default_rng(7)
    ids = rng.integers(0, lay.n_chunks, args.page_latency)
    page = torch.empty(lay.page_elems, dtype=w["mu"].dtype, device=dev)
    idt = torch.tensor(ids, dtype=torch.int32, device=dev)
    with torch.cuda.stream(stream):
        coder.prepare_decode(w["sigma"], w["counts"], stream)
        for i in range(min(5, len(ids))):       # warm-up
            coder.decode_chunks_prepared_into(out, offsets, w["mu"], idt[i:i + 1], page, stream)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in ids]
        for i, (e0, e1) in enumerate(evs):
            e0.record(stream)
            coder.decode_chunks_prepared_into(out, offsets, w["mu"], idt[i:i + 1], page, stream)
            e1.record(stream)
    stream.synchronize()
    coder.check_status("page latency", stream)
    t = np.array([e0.elapsed_time(e1) * 1e3 for e0, e1 in evs])
    return {"p50": float(np.percentile(t, 50)), "p99": float(np.percentile(t, 99)),
            "pages": int(len(ids)), "page_scalars": lay.page_elems,
            "streams_per_chunk": lay.streams_per_chunk,
            "note": "one 256-token page per skv_decode_chunks_prepared call, tables prepared once"}


def model_inputs_run(w, lay, args, dev, hbm_peak, reps=5):
    """The two steps before the coder, on the bench workload: the code
    histogram over every scalar (checked against the workload's counts) and
    the sigma calibration over the first 1,024 tokens. Median device time of
    `reps` calls (CUDA events on the launching stream, 3 untimed calls first);
    the inputs (>> L2) are not reused between calls of the histogram."""
    import lossless_kv_cache_scalar_gb300 as skv
    stream = torch.cuda.Stream(device=dev)
    t_cal = min(1024, lay.n_tokens, lay.sigma_block_tokens or lay.n_tokens)
    counts = torch.empty_like(w["counts"])

    def timed(fn):
        ts = []
        with torch.cuda.stream(stream):
            for i in range(3 + reps):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                stream.synchronize()
                if i >= 3:
                    ts.append(e0.elapsed_time(e1))
        return float(np.median(ts))

    def hist():
        counts.zero_()
        skv.histogram(w["kv"], lay.dtype, counts=counts, stream=stream)

    t_h = timed(hist)
    if not torch.equal(counts, w["counts"]):
        raise SystemExit("bench: skv_histogram differs from the workload's counts")
    t_c = timed(lambda: skv.calibrate_sigma(lay, w["kv"], w["mu"], t_cal, stream=stream))
    hist_bytes = lay.n_elems * lay.bytes_per_code
    cal_elems = lay.n_layers * lay.n_kv * t_cal * lay.n_heads * lay.head_dim
    cal_bytes = cal_elems * 2 * lay.bytes_per_code
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    return {"histogram_ms": t_h, "histogram_gbs": hist_bytes / t_h / 1e6,
            "histogram_hbm_frac": hist_bytes / t_h / 1e6 / hbm_peak,
            "calibrate_ms": t_c, "calibrate_tokens": t_cal, "calibrate_gbs": cal_bytes / t_c / 1e6,
            "calibrate_f64_gops": 3 * cal_elems / t_c / 1e6,
            "calibrate_bound": "fp64 pipe (3 binary64 ops per element; %d SMs)" % sms,
            "note": "histogram over all scalars (counts checked equal to the workload's); "
                    "sigma from tokens < %d without a mask; median of %d calls" % (t_cal, reps)}


def offload_run(coder, out, offsets, w, lay, args, dev, total_bytes, reps=3):
    """Decode the whole cache from a pinned host copy of its bitstream
    (skv_decode_offload: batches copied on a second stream while the previous
    batch decodes), against the host link itself: a pinned host-to-device copy
    of the compressed bytes, and of the uncompressed KV (what offloading the
    raw cache would move). Median of `reps` runs, CUDA events; 2 untimed first."""
    stream = torch.cuda.Stream(device=dev)
    copy_stream = torch.cuda.Stream(device=dev)
    host = torch.empty(total_bytes, dtype=torch.uint8).pin_memory()
    host.copy_(out[:total_bytes])
    host_offs = offsets.cpu()
    staging = torch.empty(args.staging_mb << 20, dtype=torch.uint8, device=dev)
    back = torch.empty_like(w["kv"])
    raw_bytes = lay.n_elems * lay.bytes_per_code
    kv_host = torch.empty(raw_bytes, dtype=torch.uint8).pin_memory()
    kv_dev = torch.empty(raw_bytes, dtype=torch.uint8, device=dev)
    comp_dev = torch.empty(total_bytes, dtype=torch.uint8, device=dev)

    def timed(fn):
        ts = []
        for i in range(2 + reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            copy_stream.wait_stream(stream)
            fn()
            stream.wait_stream(copy_stream)
            e1.record(stream)
            stream.synchronize()
            if i >= 2:
                ts.append(e0.elapsed_time(e1) / 1e3)
        return float(np.median(ts))

    t_off = timed(lambda: coder.decode_offload_into(host, host_offs, offsets, w["mu"], w["sigma"],
                                                    w["counts"], back, staging, stream, copy_stream))
    coder.check_status("offload", stream)
    if not torch.equal(back, w["kv"]):
        raise SystemExit("bench: offload decode did not restore the input")

    def h2d(dst, src):
        with torch.cuda.stream(copy_stream):
            dst.copy_(src, non_blocking=True)

    t_comp = timed(lambda: h2d(comp_dev, host))
    t_raw = timed(lambda: h2d(kv_dev, kv_host))
    # the library's plan: halves of the staging buffer, batches of whole decoder waves
    half = (staging.numel() // 2) & ~15
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    wave = max(1, sms * 32 // (lay.streams_per_chunk // 32))
    per = max(1, half // max(1, total_bytes // lay.n_chunks) // wave) * wave
    n_batches = len(offload_plan_host(host_offs, half, per)) - 1
    dec_gbs = raw_bytes / t_off / 1e9
    link_comp = total_bytes / t_comp / 1e9
    link_raw = raw_bytes / t_raw / 1e9
    return {"decode_gbs": dec_gbs, "link_compressed_gbs": link_comp, "link_raw_gbs": link_raw,
            "kv_gbs_if_link_bound": link_comp * raw_bytes / total_bytes,
            "decode_over_link_kv_rate": dec_gbs / (link_comp * raw_bytes / total_bytes),
            "decode_over_raw_offload": dec_gbs / link_raw,
            "staging_mb": args.staging_mb, "batches": n_batches,
            "note": "GB/s of uncompressed KV for decode; link = pinned host-to-device copy of the "
                    "compressed stream / of the raw KV; median of %d" % reps}


def requant_run(w, lay, dev, hbm_peak, reps=5, group=128):
    """The PM-KVQ step beside the coder: KV values quantised to 8 bits (min/max
    per token and 128 channels; torch, input preparation only), then lowered
    to 4 bits by skv_requantize with each of the page's three rules. The values
    are the workload's predictor codes mu, which have the cache's shape and
    per-channel scales but none of its 2% uniform-random outlier codes (those
    span the whole bf16 range and defeat any 8-bit min/max grid).
    Device time of the ERS call (median of `reps`, CUDA events), and the RMS
    reconstruction error of each rule against the 8-bit values."""
    from lossless_kv_cache_scalar_gb300.api import requantize
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        v = w["mu"].view(torch.bfloat16).reshape(-1, group)
        lo = v.min(1).values.float()
        scale = ((v.max(1).values.float() - lo) / 255.0).clamp_min(1e-30)
        q = torch.empty(v.numel(), dtype=torch.uint8, device=dev)
        rows = 1 << 22
        for r0 in range(0, v.shape[0], rows):           # in slices, to bound the temporaries
            vr = v[r0:r0 + rows].float()
            q.view(-1, group)[r0:r0 + rows] = torch.round((vr - lo[r0:r0 + rows, None])
                                                          / scale[r0:r0 + rows, None]).clamp(0, 255).to(torch.uint8)
        ts = []
        for i in range(3 + reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            out, s_out = requantize(q, q.numel(), 4, scale, group, "ers", stream=stream)
            e1.record(stream)
            stream.synchronize()
            if i >= 3:
                ts.append(e0.elapsed_time(e1))
        t = float(np.median(ts))
        err = {}
        rs = min(v.shape[0], (1 << 26) // group)          # rows in the error sample
        x8 = lo[:rs, None] + scale[:rs, None] * q.view(-1, group)[:rs].float()
        for mode in ("ers", "drs", "mrs"):
            o4, s4 = requantize(q, q.numel(), 4, scale, group, mode, stream=stream)
            nib = torch.stack([o4[: rs * group // 2] & 15, o4[: rs * group // 2] >> 4], 1).reshape(rs, group).float()
            x4 = lo[:rs, None] + s4[:rs, None] * nib
            err[mode] = float(torch.sqrt(torch.mean((x4 - x8) ** 2)) / torch.sqrt(torch.mean(x8 ** 2)))
        stream.synchronize()
    nbytes = q.numel() + q.numel() // 2
    return {"bits": "8 -> 4", "mode": "ers", "ms": t, "gbs": nbytes / t / 1e6, "hbm_frac": nbytes / t / 1e6 / hbm_peak,
            "codes": q.numel(), "group": group,
            "relative_rms_error_vs_8bit": err,
            "values": "the workload's mu codes (bf16), 8-bit min/max per 128 channels",
            "note": "HBM-bound: reads the 8-bit codes, writes 4-bit codes; error over the first 2^26 codes"}


def alu_peaks(dev, target_ms=20.0):
    """skv_peak_probe: the rate of each instruction class of the SKV v1
    format's section 9 alone (Tops/s, 32-bit operations) and of each whole operation
    table (scalars/s), each the best of 3 launches sized to about target_ms."""
    import ctypes as C
    from lossless_kv_cache_scalar_gb300 import _binding as B
    stream = torch.cuda.Stream(device=dev)
    sink = torch.zeros(1, dtype=torch.int32, device=dev)

    def rate(kind):
        iters = 16
        ops = C.c_uint64()
        for _ in range(10):                      # grow until a launch takes target_ms
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            B.check("skv_peak_probe", B.lib().skv_peak_probe(kind, iters, C.c_void_p(sink.data_ptr()),
                                                             C.byref(ops), C.c_void_p(stream.cuda_stream)))
            e1.record(stream)
            stream.synchronize()
            ms = e0.elapsed_time(e1)
            if ms >= target_ms / 2 or iters >= (1 << 22):
                break
            iters = int(iters * max(2.0, target_ms / max(ms, 1e-3)))
        best = 0.0
        for _ in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            B.check("skv_peak_probe", B.lib().skv_peak_probe(kind, iters, C.c_void_p(sink.data_ptr()),
                                                             C.byref(ops), C.c_void_p(stream.cuda_stream)))
            e1.record(stream)
            stream.synchronize()
            best = max(best, ops.value / (e0.elapsed_time(e1) / 1e3))
        return best

    classes = {name: rate(k) / 1e12 for k, name in enumerate(OP_CLASSES)}
    tabs = {f"{d} {o}": rate(len(OP_CLASSES) + t) for t, (d, o) in enumerate(OP_TABLES)}
    return {"class_tops": classes, "tables": tabs, "tables_unit": "scalars/s"}


def offload_plan_host(host_offs, batch_bytes, max_chunks):
    from lossless_kv_cache_scalar_gb300.api import offload_plan
    return offload_plan(host_offs.numpy(), batch_bytes, max_chunks)


def e2e_run(coder, w, lay, args, dev, total_bytes):
    """The same round trip with the cache in host memory, through the public
    host-buffer API (skv_encode_host + skv_decode_host): every step copies the
    KV and mu from pinned host memory, encodes into a host bitstream, decodes
    it back into host memory; the library overlaps the copies with the kernels
    over batches of layers. Host wall clock; sigma and counts are copied to the
    device every step too."""
    import lossless_kv_cache_scalar_gb300 as skv
    hc = skv.HostCoder(lay, dev, layers_per_batch=args.e2e_layers or None)
    kv_h = w["kv"].cpu().pin_memory()
    mu_h = w["mu"].cpu().pin_memory()
    sig_h = w["sigma"].cpu().pin_memory()
    cnt_h = w["counts"].cpu().pin_memory()
    sig_d = torch.empty_like(w["sigma"])
    cnt_d = torch.empty_like(w["counts"])
    out_h = torch.empty(total_bytes + (1 << 20), dtype=torch.uint8).pin_memory()
    offs_h = torch.empty(lay.n_chunks + 1, dtype=torch.int64).pin_memory()
    back_h = torch.empty(kv_h.shape, dtype=kv_h.dtype).pin_memory()
    stream = torch.cuda.Stream(device=dev)
    steps = max(1, min(args.steps, 5))
    t_enc, t_dec = [], []
    with torch.cuda.stream(stream):
        for i in range(1 + steps):
            if i == 1:
                torch.cuda.synchronize(dev)
                t0 = time.perf_counter()
            ta = time.perf_counter()
            sig_d.copy_(sig_h, non_blocking=True)
            cnt_d.copy_(cnt_h, non_blocking=True)
            n = hc.encode_into(kv_h, mu_h, sig_d, cnt_d, out_h, offs_h, stream)
            tb = time.perf_counter()
            hc.decode_into(out_h, n, offs_h, mu_h, sig_d, cnt_d, back_h, stream)
            tc = time.perf_counter()
            if i >= 1:
                t_enc.append(tb - ta)
                t_dec.append(tc - tb)
        torch.cuda.synchronize(dev)
        dt = time.perf_counter() - t0
    hc.check_status("e2e")
    if n != total_bytes or not torch.equal(back_h, kv_h):
        raise SystemExit("bench e2e: round trip through host buffers failed")
    raw = lay.n_elems * lay.bytes_per_code
    h2d = 2 * raw + total_bytes + raw + 2 * 8 * (lay.n_chunks + 1) + sig_h.numel() * 4 + cnt_h.numel() * 8
    d2h = total_bytes + 8 * (lay.n_chunks + 1) + raw
    return {"value": raw * steps / dt / 1e9, "unit": "GB/s", "seconds": dt, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "layers_per_batch": hc.lpb,
            "encode_host_ms": 1e3 * float(np.median(t_enc)), "decode_host_ms": 1e3 * float(np.median(t_dec)),
            "step_ms": [round(1e3 * (a + b), 1) for a, b in zip(t_enc, t_dec)],
            "median_step_gbs": raw / float(np.median([a + b for a, b in zip(t_enc, t_dec)])) / 1e9,
            "timing": "host wall clock around skv_encode_host (host KV, mu -> host bitstream) and "
                      "skv_decode_host (host bitstream, mu -> host KV), copies overlapped with the kernels"}


if __name__ == "__main__":
    sys.exit(main())
