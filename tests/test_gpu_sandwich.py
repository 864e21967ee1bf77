"""The fused sandwich residual (gemma_batch.rs `g4_sandwich`): one launch that must
give the same bits as the chain of two add + RMSNorm launches it replaces, and match
the oracle (inverse RMS within 1e-4 relative, outputs by first-order propagation)."""
import numpy as np
import pytest

import oracle
import synth
from util import NORM_TOL, check_rel, dev, host, cuda_ok

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA device")]
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def built():
    from prefill_gemv_q8_gb300 import build
    build.build()


import prefill_gemv_q8_gb300 as pgq  # noqa: E402

CASES = [  # B, n, scale, gemma
    (1, 4096, 0.0, False), (64, 2688, 0.5, True), (3, 16384, 1.25, False), (2, 4, 0.0, True),
    (7, 5120, 0.0625, True), (64, 4096, 0.0, False)]


def _inputs(B, n, seed):
    r = np.random.default_rng(seed)
    x = (r.standard_normal((B, n)) * r.uniform(0.1, 30, (B, 1))).astype(np.float32)
    h = r.standard_normal((B, n)).astype(np.float32)
    w1 = synth.gamma(n, seed, 1) - 0.5    # around 0 (the Gemma form adds 1) or around 1
    w2 = synth.gamma(n, seed, 2) - 0.5
    return x, h, w1.astype(np.float32), w2.astype(np.float32)


@pytest.mark.parametrize("B,n,scale,gemma", CASES)
def test_sandwich_equals_two_norm_chain(B, n, scale, gemma):
    x, h, w1, w2 = _inputs(B, n, B * 7 + n)
    xd, w1d, w2d = dev(x), dev(w1), dev(w2)
    f = lambda: torch.empty(B, dtype=torch.float32, device="cuda")  # noqa: E731
    # fused
    hf = dev(h)
    mid_f = torch.empty_like(hf)
    i1f, i2f = f(), f()
    out_f = pgq.sandwich_rmsnorm(xd, w1d, hf, w2d, 1e-6, scale=scale, gemma=gemma, mid=mid_f, inv1=i1f, inv2=i2f)
    # the chain of two launches
    hc = dev(h)
    x_copy = xd.clone()
    i1c, i2c = f(), f()
    mid_c = pgq.add_rmsnorm_ex(x_copy, w1d, 1e-6, gemma=gemma, inv=i1c)
    out_c = pgq.add_rmsnorm_ex(hc, w2d, 1e-6, add=mid_c, scale=scale, gemma=gemma, inv=i2c)
    torch.cuda.synchronize()
    assert torch.equal(x_copy, xd)                   # the first norm does not write its input
    for a, b, nm in ((mid_f, mid_c, "mid"), (hf, hc, "h"), (out_f, out_c, "out"), (i1f, i1c, "inv1"),
                     (i2f, i2c, "inv2")):
        assert torch.equal(a, b), f"{nm} differs between the fused and the chained form"
    # against the oracle
    ref = oracle.sandwich(x, w1, h, w2, 1e-6, scale=scale, gemma=gemma)
    check_rel(host(i1f), ref["inv1"], NORM_TOL, "inv1")
    check_rel(host(mid_f), ref["mid"], NORM_TOL + 1e-6, "mid", abs_=1e-30)
    # h' = (h + mid)·s: mid's relative error carried by |mid|, plus f32 rounding of h'
    sc = scale if scale else 1.0
    lim = (NORM_TOL + 1e-6) * np.abs(ref["mid"]) * abs(sc) + 2.0 ** -22 * np.abs(ref["h"]) + 1e-30
    assert np.all(np.abs(host(hf) - ref["h"]) <= lim), "h"
    # out = w2'·h'·inv2 taken from the kernel's own h' (stage-wise), inv2 within 1e-4
    _, y_ref, inv2_ref = oracle.add_rmsnorm_ex(host(hf), None, w2, 1e-6, None, gemma)
    check_rel(host(i2f), inv2_ref, NORM_TOL, "inv2")
    check_rel(host(out_f), y_ref, NORM_TOL + 1e-6, "out", abs_=1e-30)


def test_add_rmsnorm_ex_without_options_is_add_rmsnorm():
    B, n = 5, 4096
    x, h, _, w2 = _inputs(B, n, 3)
    ha, hb = dev(h), dev(h)
    ia = torch.empty(B, dtype=torch.float32, device="cuda")
    ib = torch.empty_like(ia)
    ya = pgq.add_rmsnorm(ha, dev(w2), 1e-6, add=dev(x), inv=ia)
    yb = pgq.add_rmsnorm_ex(hb, dev(w2), 1e-6, add=dev(x), inv=ib)
    assert torch.equal(ha, hb) and torch.equal(ya, yb) and torch.equal(ia, ib)
