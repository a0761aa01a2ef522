"""The operation count of the format (SKV v1 format §9) that defines the
arithmetic roofline: the totals table, the per-step tables it sums, the
library's copy (skv_op_table) and bench.py's reader agree. No GPU work.
"""
import ctypes as C
import os
import re
import sys

from lossless_kv_cache_scalar_gb300 import _binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

CLASSES = ["fp32", "fminmax", "iadd", "logic", "shift", "iminmax", "imad", "imad_hi", "imad_wide",
           "cvt", "mufu", "popc", "vote", "lds", "ldt", "sts"]
WEIGHT = {c: (2 if c == "imad_wide" else 1) for c in CLASSES}


def _section9():
    text = open(os.path.join(ROOT, "FORMAT.md")).read()
    return text[text.index("## 9. Operation count"):]


def _step_tables(sec):
    """The three per-step tables (one C(o), decode extras, encode extras) as class counters."""
    blocks = re.split(r"\*\*(One C\(o\)|Decode|Encode|Totals)", sec)
    out = {}
    for name, body in zip(blocks[1::2], blocks[2::2]):
        if name == "Totals":
            continue
        bf, e4 = {c: 0 for c in CLASSES}, {c: 0 for c in CLASSES}
        for line in body.splitlines():
            m = re.match(r"\| (.+) \| (.+) \|$", line)
            if not m or m.group(1) in ("step", "---"):
                continue
            # comma-separated "class n", each optionally followed by "(e4m3: class n)"
            for piece in m.group(2).split(","):
                pm = re.match(r"\s*([a-z_0-9]+) (\d+)(?: \(e4m3: ([a-z_0-9]+) (\d+)\))?\s*$", piece)
                assert pm, piece
                bf[pm.group(1)] += int(pm.group(2))
                if pm.group(3):
                    e4[pm.group(3)] += int(pm.group(4))
                else:
                    e4[pm.group(1)] += int(pm.group(2))
        out[name] = (bf, e4)
    return out


def _totals(sec):
    rows = {}
    for line in sec.splitlines():
        m = re.match(r"\| (bf16|e4m3) (encode|decode) \|(.*)\|\s*$", line)
        if m:
            v = [int(x) for x in m.group(3).split("|")]
            rows[(m.group(1), m.group(2))] = v
    return rows


def test_totals_rows_are_sums_and_weights():
    rows = _totals(_section9())
    assert sorted(rows) == [("bf16", "decode"), ("bf16", "encode"), ("e4m3", "decode"), ("e4m3", "encode")]
    for key, v in rows.items():
        counts = dict(zip(CLASSES, v[:16]))
        assert sum(counts.values()) == v[16], key
        assert sum(n * WEIGHT[c] for c, n in counts.items()) == v[17], key


def test_totals_follow_the_step_tables():
    sec = _section9()
    steps = _step_tables(sec)
    rows = _totals(sec)
    c_bf, _ = steps["One C(o)"]
    assert sum(c_bf.values()) == 33
    c_e4 = dict(c_bf)
    c_e4["ldt"] -= 1
    c_e4["lds"] += 2          # E(o) and P_hat(o) from two on-chip tables
    for op, name in (("decode", "Decode"), ("encode", "Encode")):
        bf, e4 = steps[name]
        for dt, extra, c in (("bf16", bf, c_bf), ("e4m3", e4, c_e4)):
            want = [2 * c[k] + extra[k] for k in CLASSES]
            assert rows[(dt, op)][:16] == want, (dt, op)


def test_library_copy_matches():
    rows = _totals(_section9())
    n = len(CLASSES)
    for t, key in enumerate([("bf16", "encode"), ("bf16", "decode"), ("e4m3", "encode"), ("e4m3", "decode")]):
        counts, weights = (C.c_uint32 * n)(), (C.c_uint32 * n)()
        assert B.lib().skv_op_table(t, counts, weights, n) == 0
        assert list(counts) == rows[key][:16]
        assert list(weights) == [WEIGHT[c] for c in CLASSES]
    counts, weights = (C.c_uint32 * n)(), (C.c_uint32 * n)()
    assert B.lib().skv_op_table(4, counts, weights, n) != 0
    assert B.lib().skv_op_table(0, counts, weights, n - 1) != 0


def test_bench_reader():
    import bench
    t = bench.op_tables()
    assert t[("bf16", "decode")]["instructions"] == 94 and t[("bf16", "decode")]["ops"] == 97
    assert t[("bf16", "encode")]["ops"] == 111
