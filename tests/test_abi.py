"""CPU-side checks of the C ABI: the library loads, exports every symbol include/la.h declares,
and its host-only paths (slopes, argument checks, status strings) behave without a GPU."""
import ctypes
import os
import re

import numpy as np
import pytest

import lightning_attention_gb300 as la
from lightning_attention_gb300 import _build, binding
from la_testutil import oracle_slopes_fp32

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(la_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return binding.load()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("la_extend", "la_decode", "la_verify_chain", "la_slopes", "la_poll_error",
                     "la_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    # the binding knows every entry point the header declares, and no other
    assert set(declared_functions()) == set(binding.EXPORTS)


def test_slopes_match_oracle_rule(lib):
    for (H, l, L) in [(2, 0, 1), (16, 3, 8), (16, 0, 4), (32, 5, 12), (64, 10, 20), (8, 7, 8),
                      (12, 1, 3)]:
        got = la.slopes(H, l, L).double().numpy()
        ref = oracle_slopes_fp32(H, l, L)
        # both sides round one fp64 value to fp32; allow one fp32 ulp for libm differences
        np.testing.assert_allclose(got, ref, rtol=2 ** -23, atol=0)


def test_slopes_reject_bad_arguments(lib):
    buf = (ctypes.c_float * 4)()
    for args in [(0, 0, 1), (4, 1, 1), (4, -1, 2), (4, 0, 0)]:
        assert lib.la_slopes(*args, buf) == 1
    assert lib.la_slopes(4, 0, 1, None) == 1


def test_host_argument_checks_need_no_gpu(lib):
    n = None
    # unsupported head_dim is refused before anything touches the device
    assert lib.la_extend(n, n, n, n, n, 1, n, n, n, n, 1, 1, 1, 64, 1, n, 0, n) == 2
    assert lib.la_decode(n, n, n, n, n, 1, n, n, 1, 1, 64, n) == 2
    assert lib.la_verify_chain(n, n, n, n, n, 1, n, n, n, 1, 1, 1, 64, n) == 2
    # negative sizes / bad counts
    assert lib.la_extend(n, n, n, n, n, 1, n, n, n, n, -1, 0, 1, 128, 0, n, 0, n) == 1
    assert lib.la_extend(n, n, n, n, n, 0, n, n, n, n, 1, 1, 1, 128, 1, n, 0, n) == 1
    assert lib.la_decode(n, n, n, n, n, 1, n, n, 1, 0, 128, n) == 1
    assert lib.la_verify_chain(n, n, n, n, n, 1, n, n, n, 1, 0, 1, 128, n) == 1
    # null pointers with work to do
    assert lib.la_extend(n, n, n, n, n, 1, n, n, n, n, 1, 1, 1, 128, 1, n, 0, n) == 1
    assert lib.la_decode(n, n, n, n, n, 1, n, n, 1, 1, 128, n) == 1
    assert lib.la_verify_chain(n, n, n, n, n, 1, n, n, n, 1, 2, 1, 128, n) == 1
    import ctypes as ct
    nb = ct.c_size_t(7)
    assert lib.la_extend_workspace_size(1, 1, 1, 64, 1, ct.byref(nb)) == 2
    assert lib.la_extend_workspace_size(-1, 1, 1, 128, 1, ct.byref(nb)) == 1
    assert lib.la_extend_workspace_size(1, 1, 1, 128, 1, None) == 1
    assert lib.la_extend_workspace_size(0, 0, 1, 128, 0, ct.byref(nb)) == 0 and nb.value == 0
    # empty batch is a no-op
    assert lib.la_extend(n, n, n, n, n, 1, n, n, n, n, 0, 0, 1, 128, 0, n, 0, n) == 0
    assert lib.la_decode(n, n, n, n, n, 1, n, n, 0, 1, 128, n) == 0
    assert lib.la_verify_chain(n, n, n, n, n, 1, n, n, n, 0, 1, 1, 128, n) == 0
    # extend with options: the two track arrays go together; output strides must be multiples
    # of 8 that keep heads and rows apart; otherwise la_extend's checks
    ext = (n, n, n, n, n, 1, n, n, n)
    assert lib.la_extend_ex(*ext, n, n, n, 0, 0, 1, 1, 1, 64, 1, n, 0, n) == 2
    assert lib.la_extend_ex(*ext, n, n, n, 0, 0, 0, 0, 1, 128, 0, n, 0, n) == 0
    one = ct.c_void_p(16)
    assert lib.la_extend_ex(*ext, one, n, n, 0, 0, 0, 0, 1, 128, 0, n, 0, n) == 1
    assert lib.la_extend_ex(*ext, n, one, n, 0, 0, 0, 0, 1, 128, 0, n, 0, n) == 1
    assert lib.la_extend_ex(*ext, n, n, n, 260, 0, 0, 0, 2, 128, 0, n, 0, n) == 1  # not x8
    assert lib.la_extend_ex(*ext, n, n, n, 128, 128, 0, 4, 2, 128, 0, n, 0, n) == 1  # overlap
    assert lib.la_extend_ex(*ext, n, n, n, -8, 0, 0, 0, 2, 128, 0, n, 0, n) == 1
    assert lib.la_extend_ex(*ext, n, n, n, 128, 512, 0, 4, 2, 128, 0, n, 0, n) == 0  # head-major
    assert lib.la_extend_ex(*ext, n, n, n, 384, 128, 0, 4, 2, 128, 0, n, 0, n) == 0  # wide rows
    # accepted-state commit: same rules
    assert lib.la_commit_accepted(n, n, n, 1, n, 1, 1, 1, 64, n) == 2
    assert lib.la_commit_accepted(n, n, n, 1, n, 1, 0, 1, 128, n) == 1
    assert lib.la_commit_accepted(n, n, n, 0, n, 1, 1, 1, 128, n) == 1
    assert lib.la_commit_accepted(n, n, n, 1, n, 1, 1, 1, 128, n) == 1
    assert lib.la_commit_accepted(n, n, n, 1, n, 0, 1, 1, 128, n) == 0


def test_misaligned_pointers_are_refused_before_any_launch(lib):
    """Every pointer the kernels move with 16-byte accesses must be 16-byte aligned, and the int32
    and fp32 arrays 4-byte aligned: a misaligned one returns LA_ERR_INVALID on the host, so it can
    never become a misaligned-address fault on the device.  (Each call below has one misaligned
    pointer and is refused before any CUDA call, so it runs the same with or without a GPU.)"""
    ct = ctypes
    ok, bad16, bad4 = ct.c_void_p(4096), ct.c_void_p(4096 + 8), ct.c_void_p(4096 + 2)

    def decode(q=ok, k=ok, v=ok, s=ok, pool=ok, idx=ok, out=ok):
        return lib.la_decode(q, k, v, s, pool, 4, idx, out, 1, 1, 128, None)

    for kw in ({"q": bad16}, {"k": bad16}, {"v": bad16}, {"pool": bad16}, {"out": bad16},
               {"s": bad4}, {"idx": bad4}):
        assert decode(**kw) == 1, kw

    def chain(q=ok, k=ok, v=ok, s=ok, pool=ok, idx=ok, inter=ok, out=ok):
        return lib.la_verify_chain(q, k, v, s, pool, 4, idx, inter, out, 1, 2, 1, 128, None)

    for kw in ({"q": bad16}, {"k": bad16}, {"v": bad16}, {"pool": bad16}, {"inter": bad16},
               {"out": bad16}, {"s": bad4}, {"idx": bad4}):
        assert chain(**kw) == 1, kw

    def tree(q=ok, k=ok, v=ok, s=ok, pool=ok, idx=ok, par=ok, inter=ok, out=ok):
        return lib.la_verify_tree(q, k, v, s, pool, 4, idx, par, inter, out, 1, 2, 1, 128, None)

    for kw in ({"q": bad16}, {"k": bad16}, {"v": bad16}, {"pool": bad16}, {"inter": bad16},
               {"out": bad16}, {"s": bad4}, {"idx": bad4}, {"par": bad4}):
        assert tree(**kw) == 1, kw

    def extend(q=ok, k=ok, v=ok, s=ok, pool=ok, idx=ok, cu=ok, pm=ok, out=ok):
        return lib.la_extend(q, k, v, s, pool, 4, idx, cu, pm, out, 1, 8, 1, 128, 8, None, 0, None)

    for kw in ({"q": bad16}, {"k": bad16}, {"v": bad16}, {"pool": bad16}, {"out": bad16},
               {"s": bad4}, {"idx": bad4}, {"cu": bad4}):
        assert extend(**kw) == 1, kw

    def commit(inter=ok, acc=ok, pool=ok, idx=ok):
        return lib.la_commit_accepted(inter, acc, pool, 4, idx, 1, 2, 1, 128, None)

    for kw in ({"inter": bad16}, {"pool": bad16}, {"acc": bad4}, {"idx": bad4}):
        assert commit(**kw) == 1, kw


def test_status_strings(lib):
    for code, name in binding.STATUS.items():
        assert lib.la_status_string(code).decode().startswith(name)
    assert lib.la_status_string(99).decode() == "LA_ERR_UNKNOWN"
