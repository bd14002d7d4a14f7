"""ctypes binding of the seg_la C ABI (include/la.h).

Argument marshalling only: every step of the computation runs in the CUDA library.  Tensors are
checked for device, dtype, shape and contiguity, their ``data_ptr()`` and the current CUDA stream
are passed through, and a non-OK status raises ``LAError``.  PyTorch provides device memory and
streams; outputs the caller does not pass are allocated here with ``torch.empty``.

If the compiled library is missing or cannot be loaded, every call raises: there is no fallback.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading

import torch

from . import _build

_lock = threading.Lock()
_lib = None

STATUS = {0: "LA_OK", 1: "LA_ERR_INVALID", 2: "LA_ERR_UNSUPPORTED", 3: "LA_ERR_CUDA",
          4: "LA_ERR_TIMEOUT", 5: "LA_ERR_DEVICE_INPUT"}

EXPORTS = ("la_slopes", "la_extend", "la_extend_ex", "la_extend_workspace_size", "la_decode",
           "la_verify_chain", "la_verify_tree", "la_commit_accepted", "la_poll_error", "la_status_string",
           "la_set_wait_limit", "la_set_column_split", "la_set_persistent", "la_set_balanced", "la_extend_noalloc", "la_extend_gqa",
           "la_extend_gqa_workspace_size", "la_decode_gqa")


class LAError(RuntimeError):
    def __init__(self, func: str, status: int, message: str):
        super().__init__(f"{func} failed: {message}")
        self.status = status
        self.func = func


def library_path() -> str:
    return _build.LIB_PATH


def load():
    """Load the compiled library (building nothing); raise if it is absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"seg_la CUDA library not found at {path}; build it first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(path)
        vp, ip, fp = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(ctypes.c_float)
        lib.la_slopes.argtypes = [ip, ip, ip, fp]
        lib.la_slopes.restype = ip
        sz = ctypes.c_size_t
        lib.la_extend.argtypes = [vp, vp, vp, vp, vp, ip, vp, vp, vp, vp, ip, ip, ip, ip, ip, vp, sz,
                                  vp]
        lib.la_extend.restype = ip
        lib.la_extend_workspace_size.argtypes = [ip, ip, ip, ip, ip, ctypes.POINTER(sz)]
        lib.la_extend_workspace_size.restype = ip
        lib.la_decode.argtypes = [vp, vp, vp, vp, vp, ip, vp, vp, ip, ip, ip, vp]
        lib.la_decode.restype = ip
        lib.la_verify_chain.argtypes = [vp, vp, vp, vp, vp, ip, vp, vp, vp, ip, ip, ip, ip, vp]
        lib.la_verify_chain.restype = ip
        lib.la_verify_tree.argtypes = [vp, vp, vp, vp, vp, ip, vp, vp, vp, vp, ip, ip, ip, ip, vp]
        lib.la_verify_tree.restype = ip
        i64 = ctypes.c_int64
        lib.la_extend_ex.argtypes = [vp, vp, vp, vp, vp, ip, vp, vp, vp, vp, vp, vp, i64, i64, ip,
                                     ip, ip, ip, ip, vp, sz, vp]
        lib.la_extend_ex.restype = ip
        lib.la_commit_accepted.argtypes = [vp, vp, vp, ip, vp, ip, ip, ip, ip, vp]
        lib.la_commit_accepted.restype = ip
        lib.la_poll_error.argtypes = [vp]
        lib.la_poll_error.restype = ip
        lib.la_status_string.argtypes = [ip]
        lib.la_status_string.restype = ctypes.c_char_p
        lib.la_set_wait_limit.argtypes = [ctypes.c_uint64]
        lib.la_set_wait_limit.restype = None
        lib.la_set_column_split.argtypes = [ctypes.c_int]
        lib.la_set_column_split.restype = None
        lib.la_set_persistent.argtypes = [ctypes.c_int]
        lib.la_set_persistent.restype = None
        lib.la_set_balanced.argtypes = [ctypes.c_int]
        lib.la_set_balanced.restype = None
        lib.la_extend_gqa.argtypes = [vp, vp, vp, vp, vp, ip, vp, vp, vp, vp, ip, ip, ip, ip, ip,
                                      ip, vp, sz, vp]
        lib.la_extend_gqa.restype = ip
        lib.la_extend_gqa_workspace_size.argtypes = [ip, ip, ip, ip, ip, ip, ctypes.POINTER(sz)]
        lib.la_extend_gqa_workspace_size.restype = ip
        lib.la_decode_gqa.argtypes = [vp, vp, vp, vp, vp, ip, vp, vp, ip, ip, ip, ip, vp]
        lib.la_decode_gqa.restype = ip
        _lib = lib
        return lib


def _check(func: str, status: int):
    if status != 0:
        msg = load().la_status_string(status).decode()
        raise LAError(func, status, msg)


def _ptr(t: torch.Tensor | None):
    # the arguments are declared c_void_p, so ctypes takes the integer address as is
    return None if t is None else t.data_ptr()


# The current stream's raw handle without building a torch.cuda.Stream object per call (the
# public route below is the fallback); a decode call is short enough that the binding's own
# per-call cost shows up next to the kernel.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_handle(device: torch.device):
    if _raw_stream is not None:
        return _raw_stream(device.index)
    return torch.cuda.current_stream(device).cuda_stream


_NO_SWITCH = contextlib.nullcontext()


def _on(device: torch.device):
    """Make `device` current for the library call; no switch when it already is."""
    if torch.cuda.current_device() == device.index:
        return _NO_SWITCH
    return torch.cuda.device(device)


def _need(t: torch.Tensor, name: str, dtype, device, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _out_layout(out, dev, T: int, H: int, D: int):
    """(row stride, head stride) in elements of an extend output: a [T, H*D] or [T, H, D] bf16
    tensor whose innermost elements are contiguous (rows and heads may be strided)."""
    if not isinstance(out, torch.Tensor) or out.dtype != torch.bfloat16 or out.device != dev:
        raise TypeError(f"out must be a bf16 tensor on {dev}")
    if tuple(out.shape) == (T, H * D):
        if out.stride(1) != 1:
            raise ValueError("out rows must be contiguous")
        return (out.stride(0) if T > 1 else H * D), D
    if tuple(out.shape) == (T, H, D):
        if out.stride(2) != 1:
            raise ValueError("out heads must be contiguous")
        # a stride of a dimension of size 1 is arbitrary in torch: give it a valid value
        hs = out.stride(1) if H > 1 else D
        rs = out.stride(0) if T > 1 else ((H - 1) * hs + D + 7) // 8 * 8
        return rs, hs
    raise ValueError(f"out must have shape {(T, H * D)} or {(T, H, D)}, got {tuple(out.shape)}")


def slopes(H: int, layer_id: int, L: int) -> torch.Tensor:
    """Per-head slopes (fp32, on the host) from the library's slope rule."""
    out = (ctypes.c_float * H)() if H > 0 else (ctypes.c_float * 1)()
    _check("la_slopes", load().la_slopes(H, layer_id, L, out))
    return torch.tensor(list(out)[:H], dtype=torch.float32)


def set_wait_limit(microseconds: int) -> None:
    """Bound (in microseconds) on every device wait inside the extend kernels; 0 restores the
    default of two seconds (la_set_wait_limit)."""
    load().la_set_wait_limit(int(microseconds))


def set_column_split(enable: bool) -> None:
    """Scheduling switch of the extend calls (on by default): with SMs to spare, the longest
    requests run as two CTAs per head, one per 64-column half of the values."""
    load().la_set_column_split(1 if enable else 0)


def set_persistent(enable: bool) -> None:
    """Scheduling switch of the extend calls (on by default): a batch of more (request, head)
    pairs than SMs runs on a persistent grid of one CTA per SM; results are bit-identical."""
    load().la_set_persistent(1 if enable else 0)


def set_balanced(enable: bool) -> None:
    """Scheduling switch of the extend calls (on by default): a one-wave batch of uneven lengths
    runs as segments planned on the device, on one CTA per SM; results agree up to rounding."""
    load().la_set_balanced(1 if enable else 0)


def poll_error(device=None) -> None:
    """Synchronise the current stream and raise if a kernel recorded a device-side fault."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    _check("la_poll_error", load().la_poll_error(ctypes.c_void_p(_stream_handle(dev))))


_ws_cache: dict = {}


def extend_workspace_size(B: int, T: int, H: int, D: int, max_seqlen: int) -> int:
    """Bytes of scratch la_extend uses for this batch shape on the current device (0: none)."""
    n = ctypes.c_size_t(0)
    _check("la_extend_workspace_size",
           load().la_extend_workspace_size(B, T, H, D, max_seqlen, ctypes.byref(n)))
    return int(n.value)


def _cached_workspace(dev: torch.device, nbytes: int) -> torch.Tensor:
    # one growing scratch buffer per device, shared by calls on that device: calls that use it
    # on different streams concurrently must pass their own workspace instead
    t = _ws_cache.get(dev.index)
    if t is None or t.numel() < nbytes:
        t = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        _ws_cache[dev.index] = t
    return t


def extend(q, k, v, slopes_, state_pool, state_idx, cu_seqlens, prefix_mask, out=None,
           max_seqlen: int | None = None, workspace=None, track_lens=None, track_state_idx=None):
    """Packed varlen extend (la_extend).  q, k, v: bf16 [T, H*D]; state_pool fp32
    [S, H, D, D] updated in place; returns out (allocated as bf16 [T, H*D] when not given).

    out may be [T, H*D] or per-head [T, H, D], and a strided view (say a slice of a wider buffer,
    or a head-major [H, T, D] buffer transposed): any layout other than the packed one goes
    through la_extend_ex with its strides.

    workspace: None lets the binding supply the scratch la_extend_workspace_size asks for (a
    cached per-device buffer); False runs without scratch (no sequence split); a uint8 CUDA
    tensor is used as given.  Under CUDA-graph capture pass max_seqlen and a workspace tensor
    (or make one eager call of the same shape first), so that nothing is allocated.

    track_lens, track_state_idx: int32 [B] device tensors (both or neither) select
    la_extend_ex's state tracking: the state after the first track_lens[b] tokens of request b is also
    written to slot track_state_idx[b] (-1: no snapshot)."""
    dev = q.device
    T = q.shape[0]
    num_slots, H, D, D2 = state_pool.shape
    B = state_idx.shape[0]
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need(t, name, torch.bfloat16, dev, (T, H * D))
    _need(slopes_, "slopes", torch.float32, dev, (H,))
    _need(state_pool, "state_pool", torch.float32, dev)
    _need(state_idx, "state_idx", torch.int32, dev, (B,))
    _need(cu_seqlens, "cu_seqlens", torch.int32, dev, (B + 1,))
    _need(prefix_mask, "prefix_mask", torch.uint8, dev, (B,))
    if out is None:
        out = torch.empty_like(q)
    rs, hs = _out_layout(out, dev, T, H, D)
    if max_seqlen is None:
        max_seqlen = T
    if (track_lens is None) != (track_state_idx is None):
        raise ValueError("track_lens and track_state_idx go together")
    if track_lens is not None:
        _need(track_lens, "track_lens", torch.int32, dev, (B,))
        _need(track_state_idx, "track_state_idx", torch.int32, dev, (B,))
    with _on(dev):
        if workspace is None:
            nbytes = extend_workspace_size(B, T, H, D, int(max_seqlen))
            ws = _cached_workspace(dev, nbytes) if nbytes > 0 else None
        elif workspace is False:
            ws = None
        else:
            ws = workspace
            _need(ws, "workspace", torch.uint8, dev)
        ws_ptr = _ptr(ws)
        ws_bytes = ws.numel() if ws is not None else 0
        plain = track_lens is None and (rs, hs) == (H * D, D)
        if plain:
            st = load().la_extend(_ptr(q), _ptr(k), _ptr(v), _ptr(slopes_), _ptr(state_pool),
                                  num_slots, _ptr(state_idx), _ptr(cu_seqlens), _ptr(prefix_mask),
                                  _ptr(out), B, T, H, D, int(max_seqlen), ws_ptr, ws_bytes,
                                  _stream_handle(dev))
        else:
            st = load().la_extend_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(slopes_), _ptr(state_pool),
                                     num_slots, _ptr(state_idx), _ptr(cu_seqlens),
                                     _ptr(prefix_mask), _ptr(track_lens), _ptr(track_state_idx),
                                     _ptr(out), rs, hs, B, T, H, D, int(max_seqlen), ws_ptr,
                                     ws_bytes, _stream_handle(dev))
    _check("la_extend" if plain else "la_extend_ex", st)
    return out


def extend_noalloc(q, k, v, slopes_, state_pool, state_idx, cu_seqlens, prefix_mask, out=None,
                   max_seqlen: int | None = None):
    """la_extend_noalloc: la_extend for callers that cannot allocate device memory.  Same result
    as extend(); any scratch comes from the library's fixed 16 MiB device array instead of a
    caller buffer, so calls on one device must not overlap on the GPU.  (This wrapper allocates
    `out` only when the caller does not pass it.)"""
    lib = load()
    if not getattr(lib.la_extend_noalloc, "_la_bound", False):
        vp, ip = ctypes.c_void_p, ctypes.c_int
        lib.la_extend_noalloc.argtypes = [vp, vp, vp, vp, vp, ip, vp, vp, vp, vp, ip, ip, ip, ip,
                                          ip, vp]
        lib.la_extend_noalloc.restype = ip
        lib.la_extend_noalloc._la_bound = True
    dev = q.device
    T = q.shape[0]
    num_slots, H, D, _ = state_pool.shape
    B = state_idx.shape[0]
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need(t, name, torch.bfloat16, dev, (T, H * D))
    _need(slopes_, "slopes", torch.float32, dev, (H,))
    _need(state_pool, "state_pool", torch.float32, dev)
    _need(state_idx, "state_idx", torch.int32, dev, (B,))
    _need(cu_seqlens, "cu_seqlens", torch.int32, dev, (B + 1,))
    _need(prefix_mask, "prefix_mask", torch.uint8, dev, (B,))
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, dev, (T, H * D))
    if max_seqlen is None:
        max_seqlen = T
    with _on(dev):
        st = lib.la_extend_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(slopes_), _ptr(state_pool),
                                   num_slots, _ptr(state_idx), _ptr(cu_seqlens), _ptr(prefix_mask),
                                   _ptr(out), B, T, H, D, int(max_seqlen), _stream_handle(dev))
    _check("la_extend_noalloc", st)
    return out


def decode(q, k, v, slopes_, state_pool, state_idx, out=None):
    """One-token decode (la_decode).  q, k, v: bf16 [B, H*D]; pool updated in place."""
    dev = q.device
    num_slots, H, D, _ = state_pool.shape
    B = state_idx.shape[0]
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need(t, name, torch.bfloat16, dev, (B, H * D))
    _need(slopes_, "slopes", torch.float32, dev, (H,))
    _need(state_pool, "state_pool", torch.float32, dev)
    _need(state_idx, "state_idx", torch.int32, dev, (B,))
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, dev, (B, H * D))
    with _on(dev):
        st = load().la_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(slopes_), _ptr(state_pool), num_slots,
                              _ptr(state_idx), _ptr(out), B, H, D, _stream_handle(dev))
    _check("la_decode", st)
    return out


def verify_chain(q, k, v, slopes_, state_pool, state_idx, N: int, inter_states=None, out=None):
    """Chain verify (la_verify_chain).  q, k, v: bf16 [B*N, H*D]; returns (out, inter_states)
    with inter_states fp32 [B, N, H, D, D]; the pool is not modified."""
    dev = q.device
    num_slots, H, D, _ = state_pool.shape
    B = state_idx.shape[0]
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need(t, name, torch.bfloat16, dev, (B * N, H * D))
    _need(slopes_, "slopes", torch.float32, dev, (H,))
    _need(state_pool, "state_pool", torch.float32, dev)
    _need(state_idx, "state_idx", torch.int32, dev, (B,))
    if inter_states is None:
        inter_states = torch.empty((B, N, H, D, D), dtype=torch.float32, device=dev)
    _need(inter_states, "inter_states", torch.float32, dev, (B, N, H, D, D))
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, dev, (B * N, H * D))
    with _on(dev):
        st = load().la_verify_chain(_ptr(q), _ptr(k), _ptr(v), _ptr(slopes_), _ptr(state_pool),
                                    num_slots, _ptr(state_idx), _ptr(inter_states), _ptr(out), B,
                                    N, H, D, _stream_handle(dev))
    _check("la_verify_chain", st)
    return out, inter_states


def verify_tree(q, k, v, slopes_, state_pool, state_idx, parents, N: int, inter_states=None,
                out=None):
    """Tree verify (la_verify_tree).  parents: int32 [B, N] with entries in [-1, t-1] (-1: the
    pool state).  q, k, v: bf16 [B*N, H*D]; returns (out, inter_states); the pool is not modified."""
    dev = q.device
    num_slots, H, D, _ = state_pool.shape
    B = state_idx.shape[0]
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need(t, name, torch.bfloat16, dev, (B * N, H * D))
    _need(slopes_, "slopes", torch.float32, dev, (H,))
    _need(state_pool, "state_pool", torch.float32, dev)
    _need(state_idx, "state_idx", torch.int32, dev, (B,))
    _need(parents, "parents", torch.int32, dev, (B, N))
    if inter_states is None:
        inter_states = torch.empty((B, N, H, D, D), dtype=torch.float32, device=dev)
    _need(inter_states, "inter_states", torch.float32, dev, (B, N, H, D, D))
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, dev, (B * N, H * D))
    with _on(dev):
        st = load().la_verify_tree(_ptr(q), _ptr(k), _ptr(v), _ptr(slopes_), _ptr(state_pool),
                                   num_slots, _ptr(state_idx), _ptr(parents), _ptr(inter_states),
                                   _ptr(out), B, N, H, D, _stream_handle(dev))
    _check("la_verify_tree", st)
    return out, inter_states


def commit_accepted(inter_states, accept_idx, state_pool, state_idx):
    """la_commit_accepted: pool[state_idx[b]] = inter_states[b, accept_idx[b]] where accept_idx[b]
    >= 0 (-1 leaves the slot as is)."""
    dev = state_pool.device
    num_slots, H, D, _ = state_pool.shape
    B, N = inter_states.shape[0], inter_states.shape[1]
    _need(inter_states, "inter_states", torch.float32, dev, (B, N, H, D, D))
    _need(accept_idx, "accept_idx", torch.int32, dev, (B,))
    _need(state_pool, "state_pool", torch.float32, dev)
    _need(state_idx, "state_idx", torch.int32, dev, (B,))
    with _on(dev):
        st = load().la_commit_accepted(_ptr(inter_states), _ptr(accept_idx), _ptr(state_pool),
                                       num_slots, _ptr(state_idx), B, N, H, D, _stream_handle(dev))
    _check("la_commit_accepted", st)


def extend_gqa_workspace_size(B: int, T: int, H: int, Hkv: int, D: int, max_seqlen: int) -> int:
    """Bytes of scratch la_extend_gqa uses for this batch shape on the current device."""
    n = ctypes.c_size_t(0)
    _check("la_extend_gqa_workspace_size",
           load().la_extend_gqa_workspace_size(B, T, H, Hkv, D, max_seqlen, ctypes.byref(n)))
    return int(n.value)


def extend_gqa(q, k, v, slopes_, state_pool, state_idx, cu_seqlens, prefix_mask, out=None,
               max_seqlen: int | None = None, workspace=None):
    """Grouped-query extend (la_extend_gqa): q bf16 [T, H*D]; k, v bf16 [T, Hkv*D]; slopes fp32
    [Hkv]; state_pool fp32 [S, Hkv, D, D] updated in place; returns out bf16 [T, H*D].  H comes
    from q, Hkv from the pool.  workspace: None lets the binding supply the scratch (a cached
    per-device buffer); otherwise a uint8 CUDA tensor of at least extend_gqa_workspace_size()."""
    dev = q.device
    T = q.shape[0]
    num_slots, Hkv, D, _ = state_pool.shape
    H = q.shape[1] // D
    B = state_idx.shape[0]
    _need(q, "q", torch.bfloat16, dev, (T, H * D))
    for name, t in (("k", k), ("v", v)):
        _need(t, name, torch.bfloat16, dev, (T, Hkv * D))
    _need(slopes_, "slopes", torch.float32, dev, (Hkv,))
    _need(state_pool, "state_pool", torch.float32, dev)
    _need(state_idx, "state_idx", torch.int32, dev, (B,))
    _need(cu_seqlens, "cu_seqlens", torch.int32, dev, (B + 1,))
    _need(prefix_mask, "prefix_mask", torch.uint8, dev, (B,))
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, dev, (T, H * D))
    if max_seqlen is None:
        max_seqlen = T
    with _on(dev):
        if workspace is None:
            nbytes = extend_gqa_workspace_size(B, T, H, Hkv, D, int(max_seqlen))
            ws = _cached_workspace(dev, nbytes) if nbytes > 0 else None
        else:
            ws = workspace
            _need(ws, "workspace", torch.uint8, dev)
        st = load().la_extend_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(slopes_), _ptr(state_pool),
                                  num_slots, _ptr(state_idx), _ptr(cu_seqlens), _ptr(prefix_mask),
                                  _ptr(out), B, T, H, Hkv, D, int(max_seqlen), _ptr(ws),
                                  ws.numel() if ws is not None else 0, _stream_handle(dev))
    _check("la_extend_gqa", st)
    return out


def decode_gqa(q, k, v, slopes_, state_pool, state_idx, out=None):
    """Grouped-query decode (la_decode_gqa): q bf16 [B, H*D]; k, v bf16 [B, Hkv*D]; slopes fp32
    [Hkv]; state_pool fp32 [S, Hkv, D, D] updated in place; returns out bf16 [B, H*D]."""
    dev = q.device
    num_slots, Hkv, D, _ = state_pool.shape
    B = state_idx.shape[0]
    H = q.shape[1] // D
    _need(q, "q", torch.bfloat16, dev, (B, H * D))
    for name, t in (("k", k), ("v", v)):
        _need(t, name, torch.bfloat16, dev, (B, Hkv * D))
    _need(slopes_, "slopes", torch.float32, dev, (Hkv,))
    _need(state_pool, "state_pool", torch.float32, dev)
    _need(state_idx, "state_idx", torch.int32, dev, (B,))
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, dev, (B, H * D))
    with _on(dev):
        st = load().la_decode_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(slopes_), _ptr(state_pool),
                                  num_slots, _ptr(state_idx), _ptr(out), B, H, Hkv, D,
                                  _stream_handle(dev))
    _check("la_decode_gqa", st)
    return out
