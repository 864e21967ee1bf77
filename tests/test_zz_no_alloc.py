"""The allocation-free vocab-head entry point (pgq_gemv_f16_argmax_static).

Some callers cannot allocate device memory at the moment they need the vocab head:
a plugin living inside a host framework that owns every byte of device memory
through its own pools, or a decode loop that cannot take the device-wide
synchronisation an allocation may bring.  For them the library keeps the argmax
scratch in a fixed device array.  This test calls that entry point through the C
ABI several times in a row (one position, which takes the CUDA-core kernel, and 3
and 8 positions, which take the tensor-core kernel) and checks each result against
the ordinary entry point, which takes caller-allocated scratch, and against the
oracle.  It lives in its own file, collected last.
"""
import ctypes as C

import numpy as np
import pytest

import oracle
import synth
from util import TOL, check_proj, dev, host, cuda_ok

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA device")]
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def built():
    from prefill_gemv_q8_gb300 import build
    build.build()


def test_static_scratch_matches_caller_scratch_twice():
    import prefill_gemv_q8_gb300 as pgq
    L = pgq.lib()
    rows, cols = 6000, 4096
    for call, B in enumerate((1, 3, 8, 1)):
        W = synth.f16_matrix(rows, cols, 960, call)
        W[4321] = W[17]                                    # an exact tie: row 17 must win
        x = synth.normal((B, cols), 1.0, 961, call)
        x[0] = W[17].astype(np.float32) * 8
        g = synth.gamma(cols, 962)
        Wd, xd, gd = dev(W), dev(x), dev(g)
        stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)

        ids_s = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        lg_s = torch.empty(B, rows, dtype=torch.float32, device="cuda")
        st = L.pgq_gemv_f16_argmax_static(C.c_void_p(Wd.data_ptr()), rows, cols, C.c_void_p(xd.data_ptr()), B,
                                          C.c_void_p(gd.data_ptr()), 1e-6, C.c_void_p(lg_s.data_ptr()),
                                          C.c_void_p(ids_s.data_ptr()), stream)
        assert st == pgq.OK, L.pgq_last_error()

        ids_w, lg_w = pgq.gemv_f16_argmax(Wd, xd, gamma=gd)       # caller-allocated scratch
        torch.cuda.synchronize()
        ref = oracle.vocab_head(x, g, 1e-6, W)
        check_proj(host(lg_s), host(lg_w), ref["e"], tol=TOL, what="static vs caller scratch logits")
        check_proj(host(lg_s), ref["logits"], ref["e"], tol=TOL, what="static scratch logits vs oracle")
        assert host(ids_s).tolist() == host(ids_w).tolist()
        assert host(ids_s).tolist() == oracle.argmax(host(lg_s)).tolist()
        assert int(host(ids_s)[0]) == 17


def test_static_scratch_rejects_bad_batch():
    import prefill_gemv_q8_gb300 as pgq
    L = pgq.lib()
    p = C.c_void_p(0x10000000)
    assert L.pgq_gemv_f16_argmax_static(p, 64, 64, p, 9, None, 1e-6, None, p, None) == pgq.EINVAL
