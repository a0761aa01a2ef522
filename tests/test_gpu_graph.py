"""The page decoder inside a CUDA graph: skv_decode_chunks_prepared is
captured once (its tables built beforehand by skv_decode_prepare) and
replayed with new page ids written into the captured id buffer, as a server
decoding a few pages per request would; every replay must give the pages a
direct call gives."""
import numpy as np
import pytest
import torch

from lossless_kv_cache_scalar_gb300 import Coder, Layout, synth

pytestmark = pytest.mark.gpu


def test_page_decode_replays_from_a_graph():
    cfg = synth.CONFIGS["qwen3_0p6b"].scaled(n_layers=2, n_tokens=512)
    w = synth.generate(cfg, "cuda")
    lay = Layout("bf16", 2, 2, 8, 128, 512, tokens_per_chunk=64, streams_per_chunk=64)
    c = Coder(lay, "cuda")
    bits, offs = c.encode(w["kv"], w["mu"], w["sigma"], w["counts"])
    c.prepare_decode(w["sigma"], w["counts"])
    ids = torch.zeros(3, dtype=torch.int32, device="cuda")
    pages = torch.zeros((3, lay.page_elems), dtype=torch.int16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        c.decode_chunks_prepared_into(bits, offs, w["mu"], ids, pages, stream=s)   # warm-up outside capture
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        c.decode_chunks_prepared_into(bits, offs, w["mu"], ids, pages, stream=s)
    rng = np.random.default_rng(3)
    for _ in range(5):
        want_ids = rng.integers(0, lay.n_chunks, 3).astype(np.int32)
        ids.copy_(torch.from_numpy(want_ids))
        g.replay()
        torch.cuda.synchronize()
        c.check_status("graph replay")
        direct = c.decode_chunks(bits, offs, w["mu"], w["sigma"], w["counts"],
                                 torch.from_numpy(want_ids).cuda())
        assert torch.equal(pages, direct)
