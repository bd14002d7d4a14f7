"""Golden fixtures for the oracle (CPU only).

worked_example_d2.json is derived by hand from the page's recurrence (section
"独立参考实现：逐 token 递推公式" of "SGLang Lightning Attention 能力矩阵与 seg_la 线性注意力测试覆盖深度解析");
tiny_oracle_snapshot.json was written by tests/golden/make_golden.py, which calls only the oracle.
"""
import json
import math
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_hand_worked_example():
    with open(os.path.join(GOLDEN, "worked_example_d2.json")) as f:
        g = json.load(f)
    D = g["D"]
    q, k, v = (np.array(g[x], dtype=np.float64) for x in ("q", "k", "v"))
    out, pool = oracle.extend(q, k, v, [math.log(2.0)], np.zeros((1, 1, D, D)), [0], [0, 2], [0],
                              1, D)
    np.testing.assert_allclose(out * math.sqrt(2.0), np.array(g["out_times_sqrt2"]), rtol=1e-15,
                               atol=1e-15)
    np.testing.assert_allclose(pool[0, 0], np.array(g["final_state"]), rtol=1e-15, atol=1e-15)


def test_tiny_snapshot_reproduces():
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_golden",
                                                  os.path.join(GOLDEN, "make_golden.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    with open(os.path.join(GOLDEN, "tiny_oracle_snapshot.json")) as f:
        stored = json.load(f)
    fresh = mod.snapshot()
    assert stored["slopes_fp32"] == fresh["slopes_fp32"]
    np.testing.assert_allclose(np.array(fresh["out_samples"]), np.array(stored["out_samples"]),
                               rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(np.array(fresh["state_samples"]), np.array(stored["state_samples"]),
                               rtol=1e-12, atol=1e-14)
