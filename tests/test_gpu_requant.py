"""GPU parity of skv_requantize (the PM-KVQ section's 2b -> b bit lowering:
Equivalent Right Shift, and the Direct / Modified Right Shift baselines)
against the CPU oracle: packed codes and new scales bit-equal, for every
width, whole and partial 32-byte units, several group sizes, and KV codes
quantised from a synthetic cache."""
import numpy as np
import pytest
import torch

from lossless_kv_cache_scalar_gb300 import SKVError, synth
from lossless_kv_cache_scalar_gb300.api import requantize
from oracle import oracle as O

pytestmark = pytest.mark.gpu
MODES = {"ers": O.RQ_ERS, "drs": O.RQ_DRS, "mrs": O.RQ_MRS}


@pytest.mark.parametrize("b", [1, 2, 4, 8])
@pytest.mark.parametrize("mode", ["ers", "drs", "mrs"])
def test_requantize_parity(b, mode):
    rng = np.random.default_rng(10 * b + MODES[mode])
    unit = 128 // b
    for n, group in [(unit, 1), (7 * unit + 3 * (8 // b), 64), (8 // b, 1000), (200 * unit + 8 // b, 17)]:
        packed = rng.integers(0, 256, n * 2 * b // 8, dtype=np.uint8)
        scale = (rng.random(-(-n // group)) * 3 + 0.01).astype(np.float32)
        out, s = requantize(torch.from_numpy(packed).cuda(), n, b, torch.from_numpy(scale).cuda(), group, mode)
        ref, rs = O.requantize(MODES[mode], b, packed, n, scale, group)
        assert np.array_equal(out.cpu().numpy(), ref), (n, group)
        assert np.array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))


def test_requantize_kv_codes():
    """8-bit codes of synthetic bf16 KV values (the workload's predictor codes,
    which hold no uniform-random outliers; per token-and-head min/max groups of
    128 channels) lowered to 4 bits: equal to the oracle's dequantise-requantise."""
    w = synth.generate(synth.CONFIGS["tiny"], "cuda")
    v = (w["mu"].view(torch.bfloat16).float()).reshape(-1, 128)
    lo, hi = v.min(1).values, v.max(1).values
    scale = ((hi - lo) / 255.0).clamp_min(1e-30)
    q = torch.round((v - lo[:, None]) / scale[:, None]).clamp(0, 255).to(torch.uint8).reshape(-1)
    out, s = requantize(q.contiguous(), q.numel(), 4, scale.float().contiguous(), 128, "ers")
    ref, rs = O.requantize(O.RQ_ERS, 4, q.cpu().numpy(), q.numel(), scale.cpu().numpy(), 128,
                           zero_in=lo.cpu().numpy())
    assert np.array_equal(out.cpu().numpy(), ref)
    assert np.array_equal(s.cpu().numpy(), rs)


def test_requantize_rejects_bad_args():
    x = torch.zeros(64, dtype=torch.uint8, device="cuda")
    sc = torch.ones(4, dtype=torch.float32, device="cuda")
    with pytest.raises(SKVError):
        requantize(x[1:33], 32, 4, sc, 8)          # not 16-byte aligned
    with pytest.raises(SKVError):
        requantize(x, 6, 2, sc, 8)                 # 6 x 2 bits is not whole bytes
    with pytest.raises(KeyError):
        requantize(x, 32, 4, sc, 8, "nearest")
