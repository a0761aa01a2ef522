"""Seeded synthetic KV-cache workloads.

This module only draws inputs: KV codes, predictor codes mu, per-channel
sigma and the code histogram. It holds none of the coder's arithmetic, and it
is the one module that both the CUDA path's tests/benchmark and the CPU
oracle's tests take their inputs from.

The pages measure on Qwen3 models over C4 text (the results table of the
Speculative KV Coding wiki; the measured-rates section of the 推测性KV编码
blog). Neither weights nor data are available, so these generators stand in
with the same tensor shapes and the structure the pages describe: a residual
KV_full - mu that is mostly small and Gaussian per channel, a wider Gaussian
tail, and rare outliers that only the empirical marginal explains (the
wiki's mixture section); a per-(kv, head, channel) sigma calibrated once on
the first tokens and frozen (wiki, predictor-choice section; blog, predictor
engineering section).

Recipe (all draws from one torch Generator seeded per config):
  s      ~ LogNormal(0, 1) per (layer, kv, head, channel); in K, `outlier_channels`
           seeded channels per (layer, head) get s x 20.
  mu     = round(s * N(0, 1)) to the code dtype.
  sigma  = 0.02 * s * LogNormal(0, 0.3) per channel (the generating scale).
  r      ~ 0.95 N(0, sigma^2) + 0.03 N(0, 9 sigma^2); KV_full = round(mu + r);
           with probability 0.02 instead KV_full = a uniformly drawn finite code.
  e4m3   : KV_true = s * N(0,1) + r in fp32, per-(layer, kv) scale
           max|KV_true| / 448, KV_full = e4m3(KV_true / scale) (saturating),
           mu = e4m3((KV_true + 0.5 sigma N(0,1)) / scale); outliers replace
           KV_full only; sigma is in code units.
  coding sigma: the generating sigma, or (calibrate=True) the RMS of
           value(KV_full) - value(mu) over the first `calib_tokens` tokens,
           Gaussian-drawn elements only, frozen for all tokens.
  counts : the histogram of KV_full over all codes (the empirical marginal).
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch

BF16_FINITE = 65536 - 256      # finite bf16 codes
E4M3_FINITE = 256 - 2          # finite e4m3 codes (0x7F and 0xFF are NaN)


@dataclass(frozen=True)
class SynthConfig:
    name: str
    dtype: str                  # "bf16" or "e4m3"
    n_layers: int
    n_tokens: int
    n_kv: int = 2
    n_heads: int = 8
    head_dim: int = 128
    outlier_channels: int = 0   # per (layer, K head), scale x20
    calibrate: bool = False
    calib_tokens: int = 1024
    seed: int = 1000

    @property
    def n_elems(self) -> int:
        return self.n_layers * self.n_kv * self.n_tokens * self.n_heads * self.head_dim

    @property
    def bytes_per_code(self) -> int:
        return 2 if self.dtype == "bf16" else 1

    def scaled(self, n_layers: int | None = None, n_tokens: int | None = None, **kw) -> "SynthConfig":
        return replace(self, n_layers=n_layers or self.n_layers,
                       n_tokens=self.n_tokens if n_tokens is None else n_tokens, **kw)


CONFIGS = {
    # 1 layer, K and V, 8 x 128 channels, 256 tokens: 524,288 bf16 scalars.
    "tiny": SynthConfig("tiny", "bf16", 1, 256, seed=1000),
    # Qwen3-0.6B-shaped: 28 layers x 1,024 tokens, outlier channels in K.
    "qwen3_0p6b": SynthConfig("qwen3_0p6b", "bf16", 28, 1024, outlier_channels=4, seed=1001),
    # Qwen3-8B-shaped: 36 layers x 32,768 tokens (2.42e9 scalars), sigma calibrated.
    "qwen3_8b": SynthConfig("qwen3_8b", "bf16", 36, 32768, outlier_channels=4,
                            calibrate=True, seed=1002),
    # FP8 KV, Qwen3-32B-shaped: 64 layers x 16,384 tokens of e4m3.
    "fp8_32b": SynthConfig("fp8_32b", "e4m3", 64, 16384, calibrate=True, seed=1003),
    # Long-context paged, Qwen3-14B-shaped: 40 layers x 131,072 tokens.
    "paged_14b": SynthConfig("paged_14b", "bf16", 40, 131072, outlier_channels=4,
                             calibrate=True, seed=1004),
}


def _uniform_finite_bf16(n: int, gen: torch.Generator, device) -> torch.Tensor:
    """Uniform draw over the finite bf16 codes, as int32 code values."""
    k = torch.randint(0, BF16_FINITE, (n,), generator=gen, device=device, dtype=torch.int32)
    # finite codes: sign s, exponent 0..254, mantissa 0..127 -> 2 * 255 * 128 codes
    sign = k // (255 * 128)
    rest = k % (255 * 128)
    return (sign << 15) | rest


def _uniform_finite_e4m3(n: int, gen: torch.Generator, device) -> torch.Tensor:
    k = torch.randint(0, E4M3_FINITE, (n,), generator=gen, device=device, dtype=torch.int32)
    sign = k // 127
    rest = k % 127
    return (sign << 7) | rest


def _bf16_codes(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.bfloat16).view(torch.int16).to(torch.int32) & 0xFFFF


def _bf16_values(codes: torch.Tensor) -> torch.Tensor:
    return (codes.to(torch.int32) << 16).view(torch.float32)


def _e4m3_codes(x: torch.Tensor) -> torch.Tensor:
    x = x.clamp(-448.0, 448.0)
    return x.to(torch.float8_e4m3fn).view(torch.uint8).to(torch.int32)


def _e4m3_values(codes: torch.Tensor) -> torch.Tensor:
    return codes.to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float32)


def _narrow(codes: torch.Tensor, bf: bool) -> torch.Tensor:
    """int32 code values -> the storage dtype (int16 bit pattern or uint8)."""
    if bf:
        return torch.where(codes >= 32768, codes - 65536, codes).to(torch.int16)
    return codes.to(torch.uint8)


def generate(cfg: SynthConfig, device: str | torch.device = "cpu", with_mask: bool = False):
    """Draw one workload. Returns a dict of tensors on `device`:

    kv, mu : int16 (bf16 codes) or uint8 (e4m3 codes), shape [L, n_kv, T, H, D]
    sigma  : float32 [L, n_kv, H, D]      coding sigma
    counts : int64 [N]                    histogram of kv over codes
    mask   : bool [L, n_kv, T, H, D]      (with_mask) element drawn from a Gaussian
    """
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(cfg.seed)
    L, K, T, H, D = cfg.n_layers, cfg.n_kv, cfg.n_tokens, cfg.n_heads, cfg.head_dim
    HD = H * D
    bf = cfg.dtype == "bf16"
    code_t = torch.int16 if bf else torch.uint8
    kv = torch.empty((L, K, T, H, D), dtype=code_t, device=device)
    mu = torch.empty_like(kv)
    sigma = torch.empty((L, K, H, D), dtype=torch.float32, device=device)
    counts = torch.zeros(65536 if bf else 256, dtype=torch.int64, device=device)
    mask_all = torch.empty((L, K, T, H, D), dtype=torch.bool, device=device) if with_mask else None

    for layer in range(L):
        for k in range(K):
            s = torch.exp(torch.randn(HD, generator=gen, device=device))
            if k == 0 and cfg.outlier_channels:
                for h in range(H):
                    ch = torch.randperm(D, generator=gen, device=device)[: cfg.outlier_channels]
                    s[h * D + ch] *= 20.0
            sig = 0.02 * s * torch.exp(0.3 * torch.randn(HD, generator=gen, device=device))
            n = T * HD
            z = torch.randn(n, generator=gen, device=device).view(T, HD)
            u = torch.rand(n, generator=gen, device=device).view(T, HD)
            rn = torch.randn(n, generator=gen, device=device).view(T, HD)
            wide = (u >= 0.95) & (u < 0.98)
            outl = u >= 0.98
            r = rn * sig * torch.where(wide, 3.0, 1.0)
            if bf:
                mu_c = _bf16_codes(s * z)
                kv_c = _bf16_codes(_bf16_values(mu_c) + r)
                rnd = _uniform_finite_bf16(n, gen, device).view(T, HD)
            else:
                true = s * z + r
                scale = true.abs().max() / 448.0
                pert = torch.randn(n, generator=gen, device=device).view(T, HD)
                kv_c = _e4m3_codes(true / scale)
                mu_c = _e4m3_codes((true + 0.5 * sig * pert) / scale)
                sig = sig / scale
                rnd = _uniform_finite_e4m3(n, gen, device).view(T, HD)
            kv_c = torch.where(outl, rnd, kv_c)
            if cfg.calibrate:
                tc = min(cfg.calib_tokens, T)
                vals = (_bf16_values if bf else _e4m3_values)
                res = (vals(kv_c[:tc]).double() - vals(mu_c[:tc]).double())
                keep = (~outl[:tc]).double()
                ms = (res * res * keep).sum(0) / keep.sum(0).clamp_min(1.0)
                sig = ms.sqrt().float()
            sig = torch.nan_to_num(sig, nan=1.0, posinf=3.0e38).clamp(min=2.0 ** -126)
            kv[layer, k] = _narrow(kv_c, bf).view(T, H, D)
            mu[layer, k] = _narrow(mu_c, bf).view(T, H, D)
            sigma[layer, k] = sig.view(H, D)
            counts += torch.bincount(kv_c.reshape(-1), minlength=counts.numel())
            if with_mask:
                mask_all[layer, k] = (~outl).view(T, H, D)
    out = {"kv": kv, "mu": mu, "sigma": sigma, "counts": counts}
    if with_mask:
        out["mask"] = mask_all
    return out


def histogram(codes: torch.Tensor, bf16: bool = True) -> torch.Tensor:
    """Histogram of a code tensor over all N codes (int64)."""
    c = codes.reshape(-1)
    c = (c.to(torch.int32) & 0xFFFF) if bf16 else c.to(torch.int32)
    return torch.bincount(c, minlength=65536 if bf16 else 256)


def to_numpy(w: dict):
    """Host numpy copies (codes as uint16/uint8, counts as uint64) for the oracle."""
    import numpy as np
    kv = w["kv"].cpu()
    bf = kv.dtype == torch.int16
    cd = np.uint16 if bf else np.uint8
    return {
        "kv": kv.numpy().view(cd),
        "mu": w["mu"].cpu().numpy().view(cd),
        "sigma": w["sigma"].cpu().numpy().astype(np.float32),
        "counts": w["counts"].cpu().numpy().astype(np.uint64),
    }
