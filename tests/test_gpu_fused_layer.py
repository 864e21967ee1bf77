"""The decode layer and the tiny MLP block in one launch (persistent, with a
device-side dependency between the first projections and the second): the same
outputs as the two-launch forms bit for bit (the same per-row arithmetic), every
element against the oracle, several calls in a row on one sync word (which each call
leaves zeroed), and a shape where part of the grid has no second-half work."""
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


def _layer_case(H, KV, I, wl):
    mats = synth.q8_layer(wl, 0, H, KV, I)
    x = synth.normal((H,), 1.0, wl, synth.T_X)
    xo = synth.normal((H,), 1.0, wl, synth.T_XO)
    g = synth.gamma(H, wl)
    return mats, x, xo, g


@pytest.mark.parametrize("H,KV,I", [(4096, 1024, 14336), (512, 128, 1024), (1024, 256, 2816)])
def test_q8_layer_fused_equals_two_launches_and_oracle(H, KV, I):
    mats, x, xo, g = _layer_case(H, KV, I, 980 + H // 512)
    dm = {s: (dev(c), dev(p)) for s, (c, p) in mats.items()}
    xd, xod, gd = dev(x), dev(xo), dev(g)
    sync = pgq.layer_sync()
    ref2 = pgq.q8_decode_layer(dm, xd, xod, gd, 1e-6)
    for call, stable in enumerate((False, True, True)):
        out = pgq.q8_decode_layer_fused(dm, xd, xod, gd, 1e-6, sync=sync, weights_stable=stable)
        torch.cuda.synchronize()
        for s in ("q", "k", "v", "o", "u", "down"):
            assert torch.equal(out[s], ref2[s]), f"call {call}: {s} differs from the two-launch form"
        assert int(sync.abs().sum()) == 0, "the sync word is left zeroed"
    assert pgq.last_device_status() == pgq.OK
    n, _ = oracle.rmsnorm(x, g, 1e-6)
    for s, inp in (("q", n), ("k", n), ("v", n), ("o", xo)):
        y, e = oracle.gemv_q8(*mats[s], inp)
        check_proj(host(out[s])[None, :], y, e, what=f"fused layer {s}")
    up, e = oracle.gemv_q8(*mats["up"], n)
    check_relu2(host(out["u"])[None, :], up, e, what="fused layer u")
    dn, e = oracle.gemv_q8(*mats["down"], host(out["u"]))
    check_proj(host(out["down"])[None, :], dn, e, what="fused layer down")


def test_tiny_mlp_fused_full_size():
    c = synth.TINY_MLP
    H, I, wl = c["hidden"], c["inter"], c["workload"]
    h = synth.normal((H,), 1.0, wl, synth.T_X)
    Wu = synth.f16_matrix(I, H, wl, synth.T_WUP)
    Wd = synth.f16_matrix(H, I, wl, synth.T_WDOWN)
    g = synth.gamma(H, wl)
    hd, Wud, Wdd, gd = dev(h), dev(Wu), dev(Wd), dev(g)
    sync = pgq.layer_sync()
    y2, u2 = pgq.mlp_f16_decode(hd, Wud, Wdd, gd, 1e-6)
    for _ in range(3):
        y, u = pgq.mlp_f16_decode_fused(hd, Wud, Wdd, gd, 1e-6, sync=sync)
        torch.cuda.synchronize()
        assert torch.equal(y, y2) and torch.equal(u, u2)
        assert int(sync.abs().sum()) == 0
    ref = oracle.tiny_mlp(h, Wu, Wd, g, 1e-6)
    check_relu2(host(u)[None, :], ref["up"], ref["e_up"], what="fused mlp u")
    dn, e = oracle.gemv_f16(Wd, host(u))          # stage-wise: down fed the kernel's own u
    check_proj(host(y)[None, :], h.astype(np.float64)[None, :] + dn, e, extra=np.abs(h)[None, :] * 2.0 ** -23,
               what="fused mlp y")


def test_fused_rejects_bad_sync():
    c = synth.TINY_MLP
    H, I = c["hidden"], c["inter"]
    h = torch.zeros(H, device="cuda")
    W = torch.zeros(I, H, dtype=torch.float16, device="cuda")
    Wd = torch.zeros(H, I, dtype=torch.float16, device="cuda")
    g = torch.ones(H, device="cuda")
    u = torch.empty(I, device="cuda")
    y = torch.empty(H, device="cuda")
    L = pgq.lib()
    bad = torch.zeros(8, dtype=torch.int32, device="cuda")
    assert L.pgq_mlp_f16_decode_fused(pgq._ptr(h), pgq._ptr(W), pgq._ptr(Wd), H, I, pgq._ptr(g), 1e-6, pgq._ptr(u),
                                      pgq._ptr(y), None, pgq._stream()) == pgq.EINVAL
    import ctypes as C
    assert L.pgq_mlp_f16_decode_fused(pgq._ptr(h), pgq._ptr(W), pgq._ptr(Wd), H, I, pgq._ptr(g), 1e-6, pgq._ptr(u),
                                      pgq._ptr(y), C.c_void_p(bad.data_ptr() + 4), pgq._stream()) == pgq.EINVAL
