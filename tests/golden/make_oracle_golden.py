"""Write oracle_tiny_step.json: the oracle's loss and per-tensor gradient norms
for the tiny fp32 workload (seeded inputs from nc_synth).  Calls only oracle/.

    python tests/golden/make_oracle_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import nc_synth  # noqa: E402
import oracle  # noqa: E402


def compute():
    w = nc_synth.TINY
    ids, tg = nc_synth.make_tokens(w.shape.vocab, w.batch, w.seq, seed=0, dist=w.ids)
    P = nc_synth.make_weights(w.shape, seed=1, bf16=False)
    loss, grads = oracle.step(w.shape, P, ids, tg)
    return {"_written_by": "tests/golden/make_oracle_golden.py (oracle only)",
            "workload": w.name, "loss": loss,
            "grad_norms": {k: float(np.linalg.norm(v)) for k, v in sorted(grads.items())}}


if __name__ == "__main__":
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_tiny_step.json")
    with open(out, "w") as f:
        json.dump(compute(), f, indent=1, sort_keys=True)
    print("wrote", out)
