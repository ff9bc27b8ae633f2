"""Writes the stored expected values under tests/golden/ from the fp64 oracle.

Only the oracle (and the seeded input generator) is called here; no value
comes from the CUDA path.  Run from the repository root:
    python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

from oracle.oracle import attention_of  # noqa: E402
from paged_kv_varlen_gb300 import workloads as wl  # noqa: E402


def tiny_decode():
    w = wl.workload(0)
    out = attention_of(w, nthreads=1)
    return {
        "description": "fp64 oracle output of the tiny fp32 decode workload (seed 1000): "
                       "2 requests, context 17 and 40, one query row each, H_q=4, H_kv=2, "
                       "D=64, block_size=16, 16-page pool, scale 1/8, no sinks",
        "source": "oracle.attention_of (paged attention written from the page "
                  "'What is Paged Attention' and the packed-query section)",
        "shape": list(out.shape),
        "q_checksum": float(np.asarray(w.q, np.float64).sum()),
        "block_tables": w.block_tables.tolist(),
        "out": [float(x) for x in out.ravel()],
    }


if __name__ == "__main__":
    path = os.path.join(HERE, "tiny_decode_f32.json")
    with open(path, "w") as f:
        json.dump(tiny_decode(), f, indent=0)
    print("wrote", path)
