"""Writes tests/golden/tiny_oracle_snapshot.json: sampled fp64 oracle values on the tiny workload.

Calls only oracle/ (plus the seeded input generator, which holds none of the method's arithmetic).
The snapshot guards the oracle against accidental edits: a deliberate change to its arithmetic
regenerates this file, and the commit that does so names the passage of the page that justifies it.

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from lightning_attention_gb300 import workloads  # noqa: E402


def snapshot():
    w = workloads.tiny(0)
    s32 = oracle.slopes(w.H, w.layer_id, w.L).astype(np.float32).astype(np.float64)
    pool = w.materialize_pool().double().numpy()
    out, pool_after = oracle.extend(w.q.float().numpy(), w.k.float().numpy(), w.v.float().numpy(),
                                    s32, pool, w.state_idx.numpy(), w.cu_seqlens.numpy(),
                                    w.prefix_mask.numpy(), w.H, w.D, nthreads=1)
    rows = [0, 1, 36, 37, 60, 100]
    cols = [0, 5, 127, 128, 200, 255]
    out_s = [[r, c, float(out[r, c])] for r in rows for c in cols]
    st = []
    for b in range(w.B):
        slot = int(w.state_idx[b])
        for h in range(w.H):
            for (i, j) in [(0, 0), (3, 77), (127, 127), (64, 1)]:
                st.append([slot, h, i, j, float(pool_after[slot, h, i, j])])
    return {"workload": "tiny (seed 0)", "slopes_fp32": [float(x) for x in s32],
            "out_samples": out_s, "state_samples": st}


if __name__ == "__main__":
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle_snapshot.json")
    with open(path, "w") as f:
        json.dump(snapshot(), f, indent=1)
    print("wrote", path)
