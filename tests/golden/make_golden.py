"""Write tests/golden/oracle_tiny.json: a digest of the oracle's bitstream for
the `tiny` synthetic workload (the SKV v1 format). Calls only the oracle and the
seeded input generator; run it again only when the format itself changes,
and say in the commit which reading of the pages justified the change.
"""
import hashlib
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import oracle as O  # noqa: E402
from lossless_kv_cache_scalar_gb300 import synth  # noqa: E402


def digest():
    w = synth.to_numpy(synth.generate(synth.CONFIGS["tiny"]))
    lay = O.Layout(O.BF16, 1, 2, 8, 128, 256)
    s, offs = O.encode(lay, w["kv"], w["mu"], w["sigma"], w["counts"])
    return {
        "workload": "tiny (1 layer x 2 x 256 tokens x 8 heads x 128, bf16, seed 1000)",
        "input_sha256": hashlib.sha256(w["kv"].tobytes() + w["mu"].tobytes()
                                       + w["sigma"].tobytes()).hexdigest(),
        "bitstream_sha256": hashlib.sha256(s.tobytes()).hexdigest(),
        "offsets": [int(x) for x in offs],
        "bits_per_scalar": 8.0 * float(offs[-1]) / lay.n_elems,
    }


if __name__ == "__main__":
    with open(os.path.join(HERE, "oracle_tiny.json"), "w") as fh:
        json.dump(digest(), fh, indent=1)
        fh.write("\n")
