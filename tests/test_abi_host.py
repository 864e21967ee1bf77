"""The C-ABI library builds, loads and exports every entry point the header declares;
argument checking happens on the host before any device work (no GPU needed)."""
import ctypes as C
import os
import re

import pytest

import prefill_gemv_q8_gb300 as pgq
from prefill_gemv_q8_gb300 import build as pbuild
from util import cuda_ok

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pgq.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b(pgq_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def L():
    pbuild.build()
    return pgq.lib()


def test_header_declares_entry_points():
    names = declared_functions()
    for must in ("pgq_gemv_f16", "pgq_gemv_q8", "pgq_add_rmsnorm", "pgq_relu2"):
        assert must in names


def test_every_declared_symbol_is_exported(L):
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, f"declared but not exported: {missing}"


def test_binding_covers_header():
    assert set(declared_functions()) <= set(pgq._SIGS), set(declared_functions()) - set(pgq._SIGS)


def test_status_strings(L):
    for s in range(8):
        assert pgq.status_string(s)
    assert L.pgq_abi_version() == 1


# Every call below fails an argument check, so nothing reaches a device even on a
# machine with a GPU.
FAKE = 0x10000000


def test_null_pointers_rejected(L):
    assert L.pgq_add_rmsnorm(None, None, None, 1e-6, 1, 64, None, None, None) == pgq.EINVAL
    assert b"non-null" in L.pgq_last_error()
    assert L.pgq_gemv_q8(None, None, 4, 64, None, 1, None, 1e-6, None, 0, None, None) == pgq.EINVAL
    assert L.pgq_relu2(None, 16, None) == pgq.EINVAL
    assert L.pgq_relu2(None, 0, None) == pgq.OK


def test_shapes_rejected(L):
    p = C.c_void_p(FAKE)
    # B out of range
    assert L.pgq_gemv_f16(p, 8, 64, p, 9, None, 1e-6, p, 0, None, None) == pgq.EINVAL
    assert L.pgq_gemv_f16(p, 8, 64, p, 0, None, 1e-6, p, 0, None, None) == pgq.EINVAL
    # cols not a multiple of 32
    assert L.pgq_gemv_f16(p, 8, 48, p, 1, None, 1e-6, p, 0, None, None) == pgq.EINVAL
    # input too large to stage
    assert L.pgq_gemv_f16(p, 8, 32768, p, 2, None, 1e-6, C.c_void_p(FAKE * 2), 0, None, None) == pgq.EUNSUPPORTED
    # bad epilogue / add without residual
    assert L.pgq_gemv_f16(p, 8, 64, p, 1, None, 1e-6, C.c_void_p(FAKE * 2), 7, None, None) == pgq.EINVAL
    assert L.pgq_gemv_f16(p, 8, 64, p, 1, None, 1e-6, C.c_void_p(FAKE * 2), 2, None, None) == pgq.EINVAL
    # norm width
    assert L.pgq_add_rmsnorm(p, None, p, 1e-6, 1, 6, C.c_void_p(FAKE * 2), None, None) == pgq.EINVAL
    assert L.pgq_add_rmsnorm(p, None, p, 1e-6, 0, 64, C.c_void_p(FAKE * 2), None, None) == pgq.EINVAL


def test_alignment_rejected(L):
    p = C.c_void_p(FAKE)
    q = C.c_void_p(FAKE * 2)
    odd = C.c_void_p(FAKE + 4)
    assert L.pgq_gemv_f16(odd, 8, 64, p, 1, None, 1e-6, q, 0, None, None) == pgq.EALIGN
    assert L.pgq_add_rmsnorm(odd, None, p, 1e-6, 1, 64, q, None, None) == pgq.EALIGN
    assert L.pgq_gemv_q8(C.c_void_p(FAKE + 4), p, 4, 64, q, 1, None, 1e-6, C.c_void_p(FAKE * 3), 0, None,
                         None) == pgq.EALIGN


def test_overlap_rejected(L):
    p = C.c_void_p(FAKE)
    # y == h for the norm
    assert L.pgq_add_rmsnorm(p, None, C.c_void_p(FAKE * 2), 1e-6, 2, 64, p, None, None) == pgq.EINVAL
    # y overlapping x for a projection
    assert L.pgq_gemv_f16(C.c_void_p(FAKE * 2), 8, 64, p, 1, None, 1e-6, C.c_void_p(FAKE + 16), 0, None,
                          None) == pgq.EINVAL


def test_workspace_rejected(L):
    p = C.c_void_p(FAKE)
    ids = C.c_void_p(FAKE * 3)
    st = L.pgq_gemv_f16_argmax(C.c_void_p(FAKE * 2), 64, 64, p, 1, None, 1e-6, None, ids, None, 0, None)
    # no device here gives ENODEV before the workspace check; with a device, EWORKSPACE
    assert st in (pgq.EWORKSPACE, pgq.ENODEV)


@pytest.mark.skipif(cuda_ok(), reason="checks the no-device path; a GPU is present")
def test_no_device_no_fallback(L):
    """Without a GPU a well-formed call must fail with ENODEV, not compute on the CPU."""
    p, q = C.c_void_p(FAKE), C.c_void_p(FAKE * 2)
    assert L.pgq_add_rmsnorm(p, None, q, 1e-6, 1, 64, C.c_void_p(FAKE * 3), None, None) == pgq.ENODEV
    assert L.pgq_gemv_f16(q, 8, 64, p, 1, None, 1e-6, C.c_void_p(FAKE * 3), 0, None, None) == pgq.ENODEV
    assert L.pgq_device_check() == pgq.ENODEV
