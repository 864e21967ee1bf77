"""The q8_2f weight format (gemma_batch.rs `Q82_MM_WGSL` / `q8_2f_mm_r2`: int8 body,
binary16 row scale, binary16 column field) through the decode kernel, against the
oracle at |Δ| ≤ 1e-3·Σ|w||x| per element."""
import numpy as np
import pytest

import oracle
import synth
from util import check_proj, check_relu2, dev, host, cuda_ok

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA device")]
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def built():
    from prefill_gemv_q8_gb300 import build
    build.build()


import prefill_gemv_q8_gb300 as pgq  # noqa: E402

CASES = [(1, 128, 1), (37, 1152, 2), (513, 4096, 1), (300, 2688 + 128, 3), (64, 14336, 1), (1024, 4096, 8),
         (129, 1920, 4), (5, 96, 1), (33, 1856, 3), (17, 2688, 8)]


@pytest.mark.parametrize("rows,cols,B", CASES)
@pytest.mark.parametrize("prenorm", [False, True])
def test_gemv_q82f(rows, cols, B, prenorm):
    codes, rs, cf = synth.q82f_matrix(rows, cols, 970, rows + cols + B)
    x = synth.normal((B, cols), 1.0, 971, rows + B)
    g = synth.gamma(cols, 972) if prenorm else None
    y = pgq.gemv_q82f(dev(codes), dev(rs), dev(cf), dev(x), gamma=dev(g) if prenorm else None)
    xin = oracle.rmsnorm(x, g, 1e-6)[0] if prenorm else x
    ref, e = oracle.gemv_q82f(codes, rs, cf, xin)
    check_proj(host(y), ref, e, what=f"q8_2f {rows}x{cols} B={B}")


def test_gemv_q82f_epilogues_and_identity():
    rows, cols = 257, 4096
    codes, rs, cf = synth.q82f_matrix(rows, cols, 973, 1)
    x = synth.normal((2, cols), 1.0, 973, 2)
    res = synth.normal((2, rows), 5.0, 973, 3)
    ref, e = oracle.gemv_q82f(codes, rs, cf, x)
    u = pgq.gemv_q82f(dev(codes), dev(rs), dev(cf), dev(x), epilogue="relu2")
    check_relu2(host(u), ref, e)
    y = dev(res)
    pgq.gemv_q82f(dev(codes), dev(rs), dev(cf), dev(x), epilogue="add", residual=y, y=y)
    check_proj(host(y), res.astype(np.float64) + ref, e, extra=np.abs(res) * 2.0 ** -23, what="q8_2f add")
    # identity body, unit scales: x back bit for bit at several positions, and within
    # the tolerance at one position
    n = 4096
    eye = dev(np.eye(n, dtype=np.int8))
    ones = dev(np.ones(n, np.float16))
    xi = synth.normal((3, n), 1.0, 974, 3)
    assert np.array_equal(host(pgq.gemv_q82f(eye, ones, ones, dev(xi))), xi)
    x1 = synth.normal((1, n), 1.0, 974, 1)
    check_proj(host(pgq.gemv_q82f(eye, ones, ones, dev(x1))), x1.astype(np.float64), np.abs(x1), what="identity B=1")


def test_q82f_decode_layer_full_size():
    """The q8 decode layer's shapes (hidden 4096, kv 1024, inter 14336) in q8_2f, every
    element of every projection against the oracle (down fed the kernel's own u)."""
    c = synth.Q8_LAYER
    H, KV, I, wl = c["hidden"], c["kv"], c["inter"], c["workload"]
    mats = synth.q82f_layer(wl, 0, H, KV, I)
    x = synth.normal((H,), 1.0, wl, synth.T_X)
    xo = synth.normal((H,), 1.0, wl, synth.T_XO)
    g = synth.gamma(H, wl)
    dm = {s: tuple(dev(a) for a in m) for s, m in mats.items()}
    for stable in (False, True):
        out = pgq.q82f_decode_layer(dm, dev(x), dev(xo), dev(g), 1e-6, weights_stable=stable)
        torch.cuda.synchronize()
        n, _ = oracle.rmsnorm(x, g, 1e-6)
        for s, inp in (("q", n), ("k", n), ("v", n), ("o", xo)):
            ref, e = oracle.gemv_q82f(*mats[s], inp)
            check_proj(host(out[s])[None, :], ref, e, what=f"q8_2f layer {s}")
        up, e = oracle.gemv_q82f(*mats["up"], n)
        check_relu2(host(out["u"])[None, :], up, e, what="q8_2f layer u")
        dn, e = oracle.gemv_q82f(*mats["down"], host(out["u"]))
        check_proj(host(out["down"])[None, :], dn, e, what="q8_2f layer down")
    assert pgq.last_device_status() == pgq.OK
