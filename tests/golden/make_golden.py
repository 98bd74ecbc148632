"""Writes the stored oracle snapshots under tests/golden/.

Calls only the oracle (and the seeded input generators for its inputs); no
value here ever comes from the CUDA path.  Run from the repository root:

    python tests/golden/make_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from invariant_rl_logprob_gb300 import synth  # noqa: E402


def tiny_snapshot():
    pool = synth.tiny_pool()
    lay = synth.packed(pool, [0, 1, 2, 3])
    logp, lse = oracle.linear_logp(synth.bf16_bits(lay.h), synth.bf16_bits(pool.W),
                                   lay.targets.numpy(), lay.cu_seqlens.numpy())
    return {
        "what": "fp64 oracle logp/lse of the tiny workload (4 packed sequences x 16 tokens, "
                "H=256, V=4096, h~N(0,1), W~N(0,0.02), targets uniform, seed 0)",
        "source": "oracle/ via tests/golden/make_golden.py (regression snapshot of the oracle, "
                  "not an independent pin)",
        "logp": [float(x) for x in logp],
        "lse": [float(x) for x in lse],
    }


if __name__ == "__main__":
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_linear_logp_oracle.json")
    with open(out, "w") as f:
        json.dump(tiny_snapshot(), f, indent=1)
    print("wrote", out)
