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


# The entry points of the decode layer, the prefill pass and the MoE stages reject bad
# arguments before they look for a device.  Run where there is no GPU only, so that a
# call that got past its checks could never reach one with these made-up addresses.
no_gpu = pytest.mark.skipif(cuda_ok(), reason="made-up device addresses: only where no GPU exists")


def _p(k):
    return C.c_void_p(FAKE * k)


@no_gpu
def test_prefill_q8_arguments_rejected(L):
    X, ws = _p(1), _p(2)
    job = pgq.Q8Job(_p(3).value, _p(4).value, 256, 0, _p(5).value, pgq.EPI_NONE, None)
    jobs = (pgq.Q8Job * 5)(*([job] * 5))
    call = lambda **kw: L.pgq_prefill_q8(kw.get("jobs", jobs), kw.get("njobs", 1), kw.get("X", X), kw.get("cols", 512),
                                         kw.get("B", 16), kw.get("ws", ws), 1 << 30, None)
    assert call(jobs=None) == pgq.EINVAL
    assert call(njobs=0) == pgq.EINVAL
    assert call(njobs=5) == pgq.EINVAL            # at most 4 matrices reading one X
    assert call(B=0) == pgq.EINVAL
    assert call(B=65) == pgq.EINVAL
    assert call(cols=480) == pgq.EUNSUPPORTED      # cols % 128
    assert call(X=C.c_void_p(FAKE + 4)) == pgq.EALIGN
    assert call(ws=C.c_void_p(FAKE * 2 + 128)) == pgq.EWORKSPACE
    bad = (pgq.Q8Job * 1)(pgq.Q8Job(_p(3).value, _p(4).value, 0, 0, _p(5).value, pgq.EPI_NONE, None))
    assert call(jobs=bad) == pgq.EINVAL            # rows 0
    bad = (pgq.Q8Job * 1)(pgq.Q8Job(_p(3).value, _p(4).value, 256, 0, _p(5).value, pgq.EPI_ADD, None))
    assert call(jobs=bad) == pgq.EINVAL            # add without a residual
    bad = (pgq.Q8Job * 1)(pgq.Q8Job(_p(3).value, _p(4).value, 256, 0, X.value + 64, pgq.EPI_NONE, None))
    assert call(jobs=bad) == pgq.EINVAL            # output overlaps X
    assert L.pgq_prefill_q8_workspace_bytes((C.c_int * 1)(256), 1, 512, 65) == 0


@no_gpu
def test_prefill_pass_arguments_rejected(L):
    def layer(h, kv, i):
        m = pgq.Q8Matrix(_p(3).value, _p(4).value)
        return pgq.Q8Layer(m, m, m, m, m, m, h, kv, i)
    two = (pgq.Q8Layer * 2)(layer(512, 128, 1024), layer(512, 128, 1024))
    h, g1, g2, ws = _p(1), _p(5), _p(6), _p(7)
    call = lambda **kw: L.pgq_q8_prefill_pass(kw.get("layers", two), kw.get("L", 2), kw.get("h", h), kw.get("B", 8),
                                              g1, g2, 1e-6, kw.get("ws", ws), 1 << 30, None)
    assert call(L=0) == pgq.EINVAL
    assert call(B=65) == pgq.EINVAL
    assert call(h=C.c_void_p(FAKE + 8)) == pgq.EALIGN
    assert call(layers=(pgq.Q8Layer * 2)(layer(512, 128, 1024), layer(512, 128, 2048))) == pgq.EINVAL
    assert call(layers=(pgq.Q8Layer * 2)(layer(576, 128, 1024), layer(576, 128, 1024))) == pgq.EUNSUPPORTED
    assert call(ws=C.c_void_p(FAKE * 7 + 64)) == pgq.EWORKSPACE
    offs = (C.c_size_t * 7)()
    assert L.pgq_q8_prefill_pass_layout(512, 128, 1024, 0, offs) == pgq.EINVAL
    assert L.pgq_q8_prefill_pass_workspace_bytes(512, 128, 1024, 65) == 0
    assert L.pgq_q8_prefill_pass_layout(512, 128, 1024, 8, offs) == pgq.OK
    assert list(offs) == sorted(offs) and all(o % 256 == 0 for o in offs)


@no_gpu
def test_decode_layer_and_multi_arguments_rejected(L):
    m = pgq.Q8Matrix(_p(3).value, _p(4).value)
    lay = pgq.Q8Layer(m, m, m, m, m, m, 512, 128, 1024)
    outs = [_p(10 + i) for i in range(6)]
    assert L.pgq_q8_decode_layer_ex(C.byref(lay), _p(1), _p(2), _p(5), 1e-6, *outs, 2, None) == pgq.EINVAL  # flags
    assert L.pgq_q8_decode_layer(None, _p(1), _p(2), _p(5), 1e-6, *outs, None) == pgq.EINVAL
    job = pgq.Q8Job(_p(3).value, _p(4).value, 64, 0, _p(5).value, pgq.EPI_NONE, None)
    jobs = (pgq.Q8Job * 9)(*([job] * 9))
    ins = (pgq.Input * 5)(*([pgq.Input(_p(1).value, None)] * 5))
    assert L.pgq_gemv_q8_multi(jobs, 9, ins, 1, 512, 1, 1e-6, None) == pgq.EINVAL          # > 8 jobs
    assert L.pgq_gemv_q8_multi(jobs, 1, ins, 5, 512, 1, 1e-6, None) == pgq.EINVAL          # > 4 inputs
    assert L.pgq_gemv_q8_multi(jobs, 1, ins, 4, 16384, 1, 1e-6, None) == pgq.EUNSUPPORTED  # staged values
    bad = (pgq.Q8Job * 1)(pgq.Q8Job(_p(3).value, _p(4).value, 64, 3, _p(5).value, pgq.EPI_NONE, None))
    assert L.pgq_gemv_q8_multi(bad, 1, ins, 1, 512, 1, 1e-6, None) == pgq.EINVAL          # input index


@no_gpu
def test_moe_arguments_rejected(L):
    a, b, c = _p(1), _p(2), _p(3)
    assert L.pgq_moe_router(a, 0, 64, b, 4, c, None) == pgq.EINVAL
    assert L.pgq_moe_router(a, 8, 66, b, 4, c, None) == pgq.EINVAL                  # cols % 4
    assert L.pgq_moe_router(a, 8, 64, C.c_void_p(FAKE * 2 + 4), 4, c, None) == pgq.EALIGN
    assert L.pgq_moe_router(a, 8, 64, b, 4, C.c_void_p(FAKE * 2 + 64), None) == pgq.EINVAL  # logits overlap n
    assert L.pgq_moe_route_topk(a, 4, 257, 6, 0, b, c, None) == pgq.EINVAL          # E > 256
    assert L.pgq_moe_route_topk(a, 4, 8, 9, 0, b, c, None) == pgq.EINVAL            # k > E
    assert L.pgq_moe_route_topk(a, 4, 64, 33, 0, b, c, None) == pgq.EINVAL          # k > 32
    assert L.pgq_moe_group_gather(a, 64, 6, 6000, b, c, _p(4), None, 0, 1, None, None) == pgq.EUNSUPPORTED
    assert L.pgq_moe_group_gather(a, 4, 2, 8, b, c, _p(4), None, 0, 1, _p(5), None) == pgq.EINVAL  # gather, no x
    assert L.pgq_moe_experts_q8(a, b, 8, 64, 6176, c, _p(4), _p(5), 8, _p(6), 1, _p(7), 0, None) == pgq.EUNSUPPORTED
    assert L.pgq_moe_experts_q8(a, b, 8, 64, 512, c, _p(4), _p(5), 8, _p(6), 1, _p(7), pgq.EPI_ADD,
                                None) == pgq.EINVAL
    assert L.pgq_moe_combine_rmsnorm(a, None, b, c, 2, _p(4), 1e-6, 2, 66, _p(5), None, None) == pgq.EINVAL  # n % 4
    assert L.pgq_moe_combine_rmsnorm(a, None, b, c, 2, _p(4), 1e-6, 2, 64, C.c_void_p(FAKE + 256), None,
                                     None) == pgq.EINVAL                                # y overlaps h
    lay = pgq.MoeLayer(_p(1).value, _p(2).value, _p(3).value, _p(4).value, _p(5).value, 8, 9, 256, 128, 0)
    assert L.pgq_moe_layer_workspace_bytes(C.byref(lay), 16) == 0                   # k > E
    lay.k = 2
    need = L.pgq_moe_layer_workspace_bytes(C.byref(lay), 16)
    assert need > 0
    assert L.pgq_moe_prefill_layer(C.byref(lay), _p(6), 16, _p(7), _p(8), 1e-6, _p(9), _p(10), need - 256,
                                   None) == pgq.EWORKSPACE
    assert L.pgq_moe_prefill_layer(C.byref(lay), _p(6), 65, _p(7), _p(8), 1e-6, _p(9), _p(10), need,
                                   None) == pgq.EINVAL


def test_norm_ex_and_sandwich_arguments_rejected(L):
    f = C.c_void_p(FAKE)
    g = C.c_void_p(FAKE + (1 << 20))
    # unknown flags, non-finite scale, bad n, misalignment, overlap
    assert L.pgq_add_rmsnorm_ex(f, None, g, 1e-6, 0.0, 2, 1, 64, C.c_void_p(FAKE + (2 << 20)), None, None) == pgq.EINVAL
    assert L.pgq_add_rmsnorm_ex(f, None, g, 1e-6, float("inf"), 0, 1, 64, C.c_void_p(FAKE + (2 << 20)), None,
                                None) == pgq.EINVAL
    assert L.pgq_add_rmsnorm_ex(f, None, g, 1e-6, 1.0, 0, 1, 66, C.c_void_p(FAKE + (2 << 20)), None, None) == pgq.EINVAL
    assert L.pgq_add_rmsnorm_ex(C.c_void_p(FAKE + 4), None, g, 1e-6, 1.0, 0, 1, 64, C.c_void_p(FAKE + (2 << 20)), None,
                                None) == pgq.EALIGN
    assert L.pgq_add_rmsnorm_ex(f, None, g, 1e-6, 1.0, 0, 1, 64, f, None, None) == pgq.EINVAL
    x, h, o = C.c_void_p(FAKE), C.c_void_p(FAKE + (1 << 20)), C.c_void_p(FAKE + (2 << 20))
    w = C.c_void_p(FAKE + (3 << 20))
    assert L.pgq_sandwich_rmsnorm(x, w, h, w, 1e-6, 0.0, 4, 1, 64, o, None, None, None, None) == pgq.EINVAL
    assert L.pgq_sandwich_rmsnorm(x, w, h, w, 1e-6, 0.0, 0, 1, 16388, o, None, None, None, None) == pgq.EINVAL
    assert L.pgq_sandwich_rmsnorm(x, w, h, w, 1e-6, float("nan"), 0, 1, 64, o, None, None, None, None) == pgq.EINVAL
    assert L.pgq_sandwich_rmsnorm(x, w, x, w, 1e-6, 0.0, 0, 1, 64, o, None, None, None, None) == pgq.EINVAL
    assert L.pgq_sandwich_rmsnorm(x, w, h, w, 1e-6, 0.0, 0, 1, 64, o, h, None, None, None) == pgq.EINVAL
    assert L.pgq_sandwich_rmsnorm(x, w, h, w, 1e-6, 0.0, 0, 1, 64, C.c_void_p(FAKE + (2 << 20) + 8), None, None, None,
                                  None) == pgq.EALIGN
    assert L.pgq_sandwich_rmsnorm(None, w, h, w, 1e-6, 0.0, 0, 1, 64, o, None, None, None, None) == pgq.EINVAL


def test_wait_limit_and_stall_arguments(L):
    assert L.pgq_set_wait_limit_ns(10) == pgq.EINVAL
    assert L.pgq_set_wait_limit_ns(10 ** 12) == pgq.EINVAL
    assert L.pgq_set_wait_limit_ns(5000) == pgq.OK
    assert L.pgq_wait_limit_ns() == 5000
    assert L.pgq_set_wait_limit_ns(0) == pgq.OK
    assert L.pgq_wait_limit_ns() == 2_000_000_000
    assert L.pgq_debug_stall(3) == pgq.EINVAL
    assert L.pgq_debug_stall(0) == pgq.OK


def test_q82f_arguments_rejected(L):
    p = lambda k: C.c_void_p(FAKE + k * (1 << 24))  # noqa: E731
    # cols not a multiple of 128, null pointers, misaligned column field, bad B
    assert L.pgq_gemv_q82f(p(1), p(2), p(3), 64, 80, p(4), 1, None, 1e-6, p(5), 0, None, None) == pgq.EINVAL
    assert L.pgq_gemv_q82f(p(1), None, p(3), 64, 128, p(4), 1, None, 1e-6, p(5), 0, None, None) == pgq.EINVAL
    assert L.pgq_gemv_q82f(p(1), p(2), C.c_void_p(FAKE + 3 * (1 << 24) + 8), 64, 128, p(4), 1, None, 1e-6, p(5), 0,
                           None, None) == pgq.EALIGN
    assert L.pgq_gemv_q82f(p(1), p(2), p(3), 64, 128, p(4), 9, None, 1e-6, p(5), 0, None, None) == pgq.EINVAL
    m = pgq.Q82Matrix(p(1).value, p(2).value, p(3).value)
    lay = pgq.Q82Layer(m, m, m, m, m, m, 512, 128, 1024)
    outs = [p(10 + i) for i in range(6)]
    assert L.pgq_q82f_decode_layer(C.byref(lay), p(6), p(7), p(8), 1e-6, *outs, 4, None) == pgq.EINVAL
    assert L.pgq_q82f_decode_layer(None, p(6), p(7), p(8), 1e-6, *outs, 0, None) == pgq.EINVAL


@no_gpu
def test_q82f_prefill_arguments_rejected(L):
    X, ws = _p(1), _p(2)
    job = pgq.Q82Job(_p(3).value, _p(4).value, _p(6).value, 256, _p(5).value, pgq.EPI_NONE, None)
    jobs = (pgq.Q82Job * 1)(job)
    call = lambda **kw: L.pgq_prefill_q82f(kw.get("jobs", jobs), kw.get("njobs", 1), kw.get("X", X),  # noqa: E731
                                           kw.get("cols", 512), kw.get("B", 16), ws, 1 << 30, None)
    assert call(jobs=None) == pgq.EINVAL
    assert call(B=65) == pgq.EINVAL
    assert call(cols=480) == pgq.EUNSUPPORTED
    assert call(X=C.c_void_p(FAKE + 4)) == pgq.EALIGN
    bad = (pgq.Q82Job * 1)(pgq.Q82Job(_p(3).value, None, _p(6).value, 256, _p(5).value, pgq.EPI_NONE, None))
    assert call(jobs=bad) == pgq.EINVAL            # no row scales
    bad = (pgq.Q82Job * 1)(pgq.Q82Job(_p(3).value, _p(4).value + 8, _p(6).value, 256, _p(5).value, pgq.EPI_NONE,
                                      None))
    assert call(jobs=bad) == pgq.EALIGN            # row scales 16-byte aligned
    bad = (pgq.Q82Job * 1)(pgq.Q82Job(_p(3).value, _p(4).value, _p(6).value, 256, _p(5).value, pgq.EPI_ADD, None))
    assert call(jobs=bad) == pgq.EINVAL            # add without a residual
    m = pgq.Q82Matrix(_p(3).value, _p(4).value, _p(6).value)
    lay = (pgq.Q82Layer * 2)(pgq.Q82Layer(m, m, m, m, m, m, 512, 128, 1024),
                             pgq.Q82Layer(m, m, m, m, m, m, 512, 128, 1024))
    h, g1, g2 = _p(7), _p(8), _p(9)
    pcall = lambda **kw: L.pgq_q82f_prefill_pass(kw.get("layers", lay), kw.get("L", 2), h, 8, g1, g2,  # noqa: E731
                                                 1e-6, kw.get("ws", ws), 1 << 30, None)
    assert pcall(L=0) == pgq.EINVAL
    assert pcall(layers=None) == pgq.EINVAL
    nocf = pgq.Q82Matrix(_p(3).value, _p(4).value, None)
    assert pcall(layers=(pgq.Q82Layer * 1)(pgq.Q82Layer(m, m, m, m, m, nocf, 512, 128, 1024)), L=1) == pgq.EINVAL
    odd = pgq.Q82Matrix(_p(3).value, _p(4).value + 2, _p(6).value)
    assert pcall(layers=(pgq.Q82Layer * 1)(pgq.Q82Layer(m, odd, m, m, m, m, 512, 128, 1024)), L=1) == pgq.EALIGN


@no_gpu
def test_moe_q82f_arguments_rejected(L):
    q = lambda k: _p(k).value  # noqa: E731
    lay = pgq.MoeQ82Layer(q(1), q(2), q(3), q(4), q(5), q(6), q(7), 128, 6, 2688, 1856, 0)
    h, g1, g2, y, ws = _p(8), _p(9), _p(10), _p(11), _p(12)
    call = lambda s_, B=64: L.pgq_moe_q82f_prefill_layer(C.byref(s_), h, B, g1, g2, 1e-6, y, ws,  # noqa: E731
                                                         1 << 34, None)
    big = pgq.MoeQ82Layer(q(1), q(2), q(3), q(4), q(5), q(6), q(7), 300, 6, 2688, 1856, 0)
    assert call(big) == pgq.EUNSUPPORTED           # more experts than the tensor-core bank takes
    odd = pgq.MoeQ82Layer(q(1), q(2), q(3), q(4), q(5), q(6), q(7), 128, 6, 2688 + 16, 1856, 0)
    assert call(odd) == pgq.EUNSUPPORTED           # hidden not a multiple of 32
    nocf = pgq.MoeQ82Layer(q(1), q(2), q(3), None, q(5), q(6), q(7), 128, 6, 2688, 1856, 0)
    assert call(nocf) == pgq.EINVAL
    assert call(lay, B=65) == pgq.EINVAL
    mis = pgq.MoeQ82Layer(q(1), q(2), q(3) + 8, q(4), q(5), q(6), q(7), 128, 6, 2688, 1856, 0)
    assert call(mis) == pgq.EALIGN
    assert L.pgq_moe_q82f_layer_workspace_bytes(C.byref(nocf), 64) == 0
    assert L.pgq_moe_q82f_layer_workspace_bytes(C.byref(lay), 64) > 0
