"""fp64 CPU oracle for seg_la (segmented lightning attention).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline leg (and its ``--impl reference`` arm) import this package.  The product path never does,
and this package never imports the product package: the two sides share only the seeded input
generator, which holds none of the method's arithmetic.

The arithmetic lives in ``la_oracle.c`` (plain C, double precision), written from the page
"SGLang Lightning Attention 能力矩阵与 seg_la 线性注意力测试覆盖深度解析", section
"独立参考实现：逐 token 递推公式" (independent reference: per-token recurrence), and its section
"生产环境不支持" item 3 (chain verify and the commit of the accepted draft state).  This module only compiles that file with gcc and
marshals numpy float64 arrays into it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "la_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liblaoracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile la_oracle.c into a shared library next to it (plain gcc, -O2, no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-Wall", "-Wextra",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    dp = ctypes.POINTER(ctypes.c_double)
    ip = ctypes.POINTER(ctypes.c_int32)
    up = ctypes.POINTER(ctypes.c_uint8)
    ci = ctypes.c_int
    lib.la_oracle_slopes.argtypes = [ci, ci, ci, dp]
    lib.la_oracle_slopes.restype = None
    lib.la_oracle_extend.argtypes = [dp, dp, dp, dp, dp, ip, ip, up, dp, ci, ci, ci, ci]
    lib.la_oracle_extend.restype = ci
    lib.la_oracle_decode.argtypes = [dp, dp, dp, dp, dp, ip, dp, ci, ci, ci, ci]
    lib.la_oracle_decode.restype = ci
    lib.la_oracle_verify_chain.argtypes = [dp, dp, dp, dp, dp, ip, dp, dp, ci, ci, ci, ci, ci]
    lib.la_oracle_verify_chain.restype = ci
    lib.la_oracle_verify_tree.argtypes = [dp, dp, dp, dp, dp, ip, ip, dp, dp, ci, ci, ci, ci]
    lib.la_oracle_verify_tree.restype = ci
    lib.la_oracle_extend_tracked.argtypes = [dp, dp, dp, dp, dp, ip, ip, up, ip, ip, dp, ci, ci,
                                             ci, ci]
    lib.la_oracle_extend_tracked.restype = ci
    lib.la_oracle_commit_accepted.argtypes = [dp, ip, dp, ip, ci, ci, ci, ci]
    lib.la_oracle_commit_accepted.restype = ci
    lib.la_oracle_extend_gqa.argtypes = [dp, dp, dp, dp, dp, ip, ip, up, dp, ci, ci, ci, ci, ci]
    lib.la_oracle_extend_gqa.restype = ci
    lib.la_oracle_decode_gqa.argtypes = [dp, dp, dp, dp, dp, ip, dp, ci, ci, ci, ci, ci]
    lib.la_oracle_decode_gqa.restype = ci
    return lib


def load_library(path: str):
    """Bind an oracle shared library built from a (possibly edited) copy of la_oracle.c; the
    result can be passed as ``lib=`` to the functions below (used by the mutation tests)."""
    return _bind(ctypes.CDLL(path))


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def slopes(H: int, layer_id: int, L: int, lib=None) -> np.ndarray:
    """Per-head slopes in float64: ALiBi base 2^(-8(i+1)/H) times the per-layer factor."""
    out = np.zeros(H, dtype=np.float64)
    (lib or _load()).la_oracle_slopes(H, layer_id, L, _ptr(out, ctypes.c_double))
    return out


def extend(q, k, v, slopes_, pool, state_idx, cu_seqlens, prefix_mask, H: int, D: int,
           nthreads: int | None = None, lib=None):
    """Packed varlen extend.  q, k, v: [T, H*D]; pool: [S, H, D, D] (a float64 copy is updated
    and returned).  Returns (out [T, H*D], pool_after)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    T = q.shape[0]
    assert q.shape == (T, H * D) and k.shape == q.shape and v.shape == q.shape
    s = _f64(slopes_)
    pool_c = _f64(pool).copy()
    idx = _i32(state_idx)
    cu = _i32(cu_seqlens)
    pm = np.ascontiguousarray(np.asarray(prefix_mask, dtype=np.uint8))
    B = idx.shape[0]
    assert cu.shape == (B + 1,) and pm.shape == (B,)
    out = np.zeros((T, H * D), dtype=np.float64)
    (lib or _load()).la_oracle_extend(_ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double),
                             _ptr(v, ctypes.c_double), _ptr(s, ctypes.c_double),
                             _ptr(pool_c, ctypes.c_double), _ptr(idx, ctypes.c_int32),
                             _ptr(cu, ctypes.c_int32), _ptr(pm, ctypes.c_uint8),
                             _ptr(out, ctypes.c_double), B, H, D,
                             nthreads or default_threads())
    return out, pool_c


def extend_tracked(q, k, v, slopes_, pool, state_idx, cu_seqlens, prefix_mask, track_lens,
                   track_idx, H: int, D: int, nthreads: int | None = None, lib=None):
    """Packed varlen extend with state tracking: as extend(), and for every request b with
    track_lens[b] >= 0 the state after its first track_lens[b] tokens is also written to slot
    track_idx[b].  Returns (out, pool_after); raises ValueError on a track length outside
    [-1, length] or a track slot that is the request's own slot."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    T = q.shape[0]
    assert q.shape == (T, H * D) and k.shape == q.shape and v.shape == q.shape
    s = _f64(slopes_)
    pool_c = _f64(pool).copy()
    idx = _i32(state_idx)
    cu = _i32(cu_seqlens)
    pm = np.ascontiguousarray(np.asarray(prefix_mask, dtype=np.uint8))
    tl = _i32(track_lens)
    ti = _i32(track_idx)
    B = idx.shape[0]
    assert cu.shape == (B + 1,) and pm.shape == (B,) and tl.shape == (B,) and ti.shape == (B,)
    assert all(0 <= int(ti[b]) < pool_c.shape[0] for b in range(B) if tl[b] >= 0)
    out = np.zeros((T, H * D), dtype=np.float64)
    rc = (lib or _load()).la_oracle_extend_tracked(
        _ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double), _ptr(v, ctypes.c_double),
        _ptr(s, ctypes.c_double), _ptr(pool_c, ctypes.c_double), _ptr(idx, ctypes.c_int32),
        _ptr(cu, ctypes.c_int32), _ptr(pm, ctypes.c_uint8), _ptr(tl, ctypes.c_int32),
        _ptr(ti, ctypes.c_int32), _ptr(out, ctypes.c_double), B, H, D,
        nthreads or default_threads())
    if rc != 0:
        raise ValueError("track_lens must lie in [-1, request length] and track slots must not "
                         "be the request's own slot")
    return out, pool_c


def decode(q, k, v, slopes_, pool, state_idx, H: int, D: int, nthreads: int | None = None,
           lib=None):
    """One decode token per request.  q, k, v: [B, H*D].  Returns (out [B, H*D], pool_after)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    s = _f64(slopes_)
    pool_c = _f64(pool).copy()
    idx = _i32(state_idx)
    B = idx.shape[0]
    assert q.shape == (B, H * D)
    out = np.zeros((B, H * D), dtype=np.float64)
    (lib or _load()).la_oracle_decode(_ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double),
                             _ptr(v, ctypes.c_double), _ptr(s, ctypes.c_double),
                             _ptr(pool_c, ctypes.c_double), _ptr(idx, ctypes.c_int32),
                             _ptr(out, ctypes.c_double), B, H, D,
                             nthreads or default_threads())
    return out, pool_c


def verify_chain(q, k, v, slopes_, pool, state_idx, N: int, H: int, D: int,
                 nthreads: int | None = None, lib=None):
    """Chain verify of N draft tokens per request.  q, k, v: [B*N, H*D] (request-major).
    The pool is only read.  Returns (out [B*N, H*D], inter [B, N, H, D, D])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    s = _f64(slopes_)
    pool_c = _f64(pool)
    idx = _i32(state_idx)
    B = idx.shape[0]
    assert q.shape == (B * N, H * D)
    out = np.zeros((B * N, H * D), dtype=np.float64)
    inter = np.zeros((B, N, H, D, D), dtype=np.float64)
    (lib or _load()).la_oracle_verify_chain(_ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double),
                                   _ptr(v, ctypes.c_double), _ptr(s, ctypes.c_double),
                                   _ptr(pool_c, ctypes.c_double), _ptr(idx, ctypes.c_int32),
                                   _ptr(inter, ctypes.c_double), _ptr(out, ctypes.c_double),
                                   B, N, H, D, nthreads or default_threads())
    return out, inter


def verify_tree(q, k, v, slopes_, pool, state_idx, parents, N: int, H: int, D: int, lib=None):
    """Tree verify: token t of request b continues from the state after token parents[b, t] (-1:
    the pool state).  q, k, v: [B*N, H*D]; parents: [B, N] int32.  Returns (out, inter) like
    verify_chain; raises ValueError if a parent does not point backwards."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    s = _f64(slopes_)
    pool_c = _f64(pool)
    idx = _i32(state_idx)
    par = _i32(parents)
    B = idx.shape[0]
    assert q.shape == (B * N, H * D) and par.shape == (B, N)
    out = np.zeros((B * N, H * D), dtype=np.float64)
    inter = np.zeros((B, N, H, D, D), dtype=np.float64)
    rc = (lib or _load()).la_oracle_verify_tree(
        _ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double), _ptr(v, ctypes.c_double),
        _ptr(s, ctypes.c_double), _ptr(pool_c, ctypes.c_double), _ptr(idx, ctypes.c_int32),
        _ptr(par, ctypes.c_int32), _ptr(inter, ctypes.c_double), _ptr(out, ctypes.c_double),
        B, N, H, D)
    if rc != 0:
        raise ValueError("parents must satisfy -1 <= parents[b, t] < t")
    return out, inter


def commit_accepted(inter, accept_idx, pool, state_idx, lib=None) -> np.ndarray:
    """Accepted-state commit: returns a copy of ``pool`` in which slot state_idx[b] holds
    inter[b, accept_idx[b]] for every b with accept_idx[b] >= 0.  inter: [B, N, H, D, D];
    pool: [num_slots, H, D, D].  Raises ValueError if an index is outside [-1, N-1]."""
    inter_c = _f64(inter)
    acc = _i32(accept_idx)
    idx = _i32(state_idx)
    pool_c = _f64(pool).copy()
    B, N, H, D = inter_c.shape[0], inter_c.shape[1], inter_c.shape[2], inter_c.shape[3]
    assert acc.shape == (B,) and idx.shape == (B,) and pool_c.shape[1:] == (H, D, D)
    assert B == 0 or (idx.min() >= 0 and idx.max() < pool_c.shape[0])
    rc = (lib or _load()).la_oracle_commit_accepted(
        _ptr(inter_c, ctypes.c_double), _ptr(acc, ctypes.c_int32), _ptr(pool_c, ctypes.c_double),
        _ptr(idx, ctypes.c_int32), B, N, H, D)
    if rc != 0:
        raise ValueError("accept_idx must satisfy -1 <= accept_idx[b] < N")
    return pool_c


def extend_gqa(q, k, v, slopes_, pool, state_idx, cu_seqlens, prefix_mask, H: int, Hkv: int,
               D: int, nthreads: int | None = None, lib=None):
    """Packed varlen extend with grouped-query heads: q [T, H*D], k and v [T, Hkv*D], slopes
    [Hkv], pool [S, Hkv, D, D] (a float64 copy is updated and returned); query head h reads the
    state of kv head h // (H // Hkv).  Returns (out [T, H*D], pool_after)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    T = q.shape[0]
    assert q.shape == (T, H * D) and k.shape == (T, Hkv * D) and v.shape == k.shape
    s = _f64(slopes_)
    assert s.shape == (Hkv,)
    pool_c = _f64(pool).copy()
    assert pool_c.shape[1:] == (Hkv, D, D)
    idx = _i32(state_idx)
    cu = _i32(cu_seqlens)
    pm = np.ascontiguousarray(np.asarray(prefix_mask, dtype=np.uint8))
    B = idx.shape[0]
    assert cu.shape == (B + 1,) and pm.shape == (B,)
    out = np.zeros((T, H * D), dtype=np.float64)
    rc = (lib or _load()).la_oracle_extend_gqa(
        _ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double), _ptr(v, ctypes.c_double),
        _ptr(s, ctypes.c_double), _ptr(pool_c, ctypes.c_double), _ptr(idx, ctypes.c_int32),
        _ptr(cu, ctypes.c_int32), _ptr(pm, ctypes.c_uint8), _ptr(out, ctypes.c_double),
        B, H, Hkv, D, nthreads or default_threads())
    if rc != 0:
        raise ValueError("H must be a positive multiple of Hkv")
    return out, pool_c


def decode_gqa(q, k, v, slopes_, pool, state_idx, H: int, Hkv: int, D: int,
               nthreads: int | None = None, lib=None):
    """One decode token per request with grouped-query heads: q [B, H*D], k and v [B, Hkv*D],
    slopes [Hkv], pool [S, Hkv, D, D].  Returns (out [B, H*D], pool_after)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    s = _f64(slopes_)
    pool_c = _f64(pool).copy()
    idx = _i32(state_idx)
    B = idx.shape[0]
    assert q.shape == (B, H * D) and k.shape == (B, Hkv * D) and v.shape == k.shape
    out = np.zeros((B, H * D), dtype=np.float64)
    rc = (lib or _load()).la_oracle_decode_gqa(
        _ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double), _ptr(v, ctypes.c_double),
        _ptr(s, ctypes.c_double), _ptr(pool_c, ctypes.c_double), _ptr(idx, ctypes.c_int32),
        _ptr(out, ctypes.c_double), B, H, Hkv, D, nthreads or default_threads())
    if rc != 0:
        raise ValueError("H must be a positive multiple of Hkv")
    return out, pool_c
