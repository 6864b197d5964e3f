"""Write the stored oracle values of tests/golden/tiny_decode.txt.

The TinyServe pages print no worked numeric example, so every stored value
here is written by this script from the oracle alone (and the seeded input
generator); tests/test_oracle_pins.py recomputes them and compares, so a later
change of the oracle's arithmetic shows up as a diff of this file.

    python tests/golden/make_golden.py > tests/golden/tiny_decode.txt
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from query_aware_sparse_append_gb300 import workloads as W  # noqa: E402


def golden_lines():
    cfg = W.CONFIGS["tiny"]
    lens = W.seq_lens(cfg, 0)
    bud = W.budgets(cfg, lens)
    s = W.sequence(cfg, 0, int(lens[0]), 0)
    G, P = cfg.group, cfg.page_size
    out = ["# oracle decode of workload 'tiny', seed 0, sequence 0: per KV head the kept pages,",
           "# the eight largest page scores and the first four output values of query head h*G"]
    for h in range(cfg.num_kv_heads):
        K = W.widen(s.k[:, h], cfg.dtype)
        V = W.widen(s.v[:, h], cfg.dtype)
        q = W.widen(s.q[h * G:(h + 1) * G], cfg.dtype)
        lo, hi = oracle.page_bounds(K, P)
        sc, sel, o = oracle.decode_unit(q, K, V, lo, hi, int(lens[0]), P, int(bud[0]))
        top = np.sort(sc)[::-1][:8]
        out.append("head %d kept %s" % (h, " ".join(str(int(x)) for x in sel)))
        out.append("head %d top_scores %s" % (h, " ".join("%.12e" % x for x in top)))
        out.append("head %d out %s" % (h, " ".join("%.12e" % x for x in o[0, :4])))
    return out


if __name__ == "__main__":
    print("\n".join(golden_lines()))
