"""Shared helpers for the parity tests: tolerances, comparisons, oracle-side input preparation.

The tolerance is the one the page "SGLang Lightning Attention 能力矩阵与 seg_la 线性注意力测试覆盖深度解析"
(section "独立参考实现") uses for bf16 I/O: atol = rtol = 3e-2, in assert_close form
|actual - expected| <= atol + rtol * |expected|, applied to outputs (bf16 against fp64) and to
states (fp32 against fp64).
"""
import numpy as np
import torch

import oracle

ATOL = 3e-2
RTOL = 3e-2


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


def oracle_slopes_fp32(H, layer_id, L) -> np.ndarray:
    """The oracle's fp64 slopes rounded once to fp32 (the reading: both sides use one fp32 slope)."""
    return oracle.slopes(H, layer_id, L).astype(np.float32).astype(np.float64)


def assert_close(actual, expected, what: str, atol=ATOL, rtol=RTOL):
    a = np.asarray(actual, dtype=np.float64)
    e = np.asarray(expected, dtype=np.float64)
    assert a.shape == e.shape, f"{what}: shape {a.shape} != {e.shape}"
    if a.size == 0:
        return
    assert np.isfinite(a).all(), f"{what}: non-finite values in the GPU result"
    err = np.abs(a - e)
    bad = err > atol + rtol * np.abs(e)
    if bad.any():
        idx = np.unravel_index(np.argmax(err - (atol + rtol * np.abs(e))), a.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {a.size} elements outside atol={atol} rtol={rtol}; "
            f"worst at {idx}: gpu={a[idx]!r} oracle={e[idx]!r}")


def max_err(actual, expected) -> float:
    a = np.asarray(actual, dtype=np.float64)
    e = np.asarray(expected, dtype=np.float64)
    return float(np.max(np.abs(a - e))) if a.size else 0.0
