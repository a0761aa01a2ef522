"""Golden fixtures: the pages' printed figures and a digest of the oracle's output.

tests/golden/pages_rates.json holds numbers printed by the pages (cited in the
file). They measure Qwen3 models on C4, which are not available, so they
cannot pin the coder's rate; they do pin the metric: bits per scalar is
compared against 16 bits for bf16 and 8 for e4m3, so 16/bits must reproduce
the printed compression ratios (the wiki's results table; the blog's FP8
paragraph).

tests/golden/oracle_tiny.json is written by tests/golden/make_golden.py from
the oracle alone and guards the format against silent drift.
"""
import hashlib
import json
import os

import pytest

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(HERE, name)) as fh:
        return json.load(fh)


def test_wiki_ratio_column_is_sixteen_over_bits():
    g = _load("pages_rates.json")
    for row in g["wiki_mixture_table"]:
        assert abs(16.0 / row["bits"] - row["ratio"]) < 0.006, row


def test_blog_fp8_extra_ratio_is_eight_over_bits():
    g = _load("pages_rates.json")["blog_fp8"]
    lo, hi = g["bits_range"]
    rlo, rhi = g["extra_ratio_range"]
    assert abs(8.0 / hi - rlo) < 0.015 and abs(8.0 / lo - rhi) < 0.015


def test_blog_single_gaussian_pairing_is_inconsistent():
    # The blog pairs 6.87 bits with 2.37x; 16/6.87 = 2.33, while 2.37x is
    # 16/6.74, the wiki's mixture figure. The build reports bits per scalar
    # and derives ratios as 16/bits, so it follows the wiki's column.
    g = _load("pages_rates.json")
    assert abs(16.0 / g["blog_single_gaussian"]["bits_0p6b"] - 2.37) > 0.03
    assert abs(16.0 / g["wiki_mixture_table"][0]["bits"] - 2.37) < 0.006


def test_mixture_weights_sum_to_one_hundred():
    w = _load("pages_rates.json")["mixture_weights_percent"]
    assert w["narrow"] + w["wide"] + w["marginal"] == 100 and w["wide_sigma_factor"] == 3


def test_oracle_tiny_digest():
    from oracle import oracle as O
    from lossless_kv_cache_scalar_gb300 import synth
    g = _load("oracle_tiny.json")
    w = synth.to_numpy(synth.generate(synth.CONFIGS["tiny"]))
    h_in = hashlib.sha256(w["kv"].tobytes() + w["mu"].tobytes() + w["sigma"].tobytes()).hexdigest()
    if h_in != g["input_sha256"]:
        pytest.skip("this torch build draws different random inputs")
    lay = O.Layout(O.BF16, 1, 2, 8, 128, 256)
    s, offs = O.encode(lay, w["kv"], w["mu"], w["sigma"], w["counts"])
    assert [int(x) for x in offs] == g["offsets"]
    assert hashlib.sha256(s.tobytes()).hexdigest() == g["bitstream_sha256"]
