"""Writes tests/golden/tiny_oracle.json: the CPU oracle's k_cache bytes and comp32 for the tiny
workload (4 requests, windows ending at positions 127, 255, 383, 511). Calls only ``oracle``
and the seeded input generator; re-run it only when the oracle's arithmetic changes for a
reason the pages justify."""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from deepseek_v4_sparse_c128_gb300 import inputs  # noqa: E402


def main():
    p = inputs.make_problem("tiny")
    kc = p.k_cache.copy()
    comp = np.zeros((p.num_tokens, 512), np.float32)
    err = oracle.forward(p, k_cache=kc, comp_out=comp)
    assert err == 0
    out = {"workload": "tiny (seed 0)", "writer": "tests/golden/make_golden.py",
           "k_cache_hex": kc.tobytes().hex(), "comp32_hex": comp.tobytes().hex()}
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle.json"), "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
