"""The timeout path of the bounded device-side waits, made to run on purpose.

A wait that runs past the wait limit must end the call cleanly and be reported
through pgq_last_device_status as PGQ_ETIMEOUT; the next call, with the default
limit, must give correct results again.  The expired wait is made with the test
hook pgq_debug_stall (a wait for an event that never comes: inputs that are never
copied, one tile more than the projection has), never with a fault: every kernel wait
is bounded, so the call ends after a few wait limits."""
import numpy as np
import pytest

import oracle
import synth
from util import check_proj, dev, host, cuda_ok

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA device")]
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def built():
    from prefill_gemv_q8_gb300 import build
    build.build()


import prefill_gemv_q8_gb300 as pgq  # noqa: E402

SHORT_NS = 2_000_000   # 2 ms: far below the default, far above a normal wait here


class stalled:
    """The hook on and a short limit inside the block; both restored on the way out."""

    def __enter__(self):
        pgq.set_wait_limit_ns(SHORT_NS)
        pgq.debug_stall(True)

    def __exit__(self, *a):
        pgq.debug_stall(False)
        pgq.set_wait_limit_ns(0)
        return False


def test_wait_limit_setting():
    assert pgq.wait_limit_ns() == 2_000_000_000
    pgq.set_wait_limit_ns(5000)
    assert pgq.wait_limit_ns() == 5000
    pgq.set_wait_limit_ns(0)
    assert pgq.wait_limit_ns() == 2_000_000_000
    assert pgq.lib().pgq_set_wait_limit_ns(10) == pgq.EINVAL
    assert pgq.lib().pgq_debug_stall(2) == pgq.EINVAL
    assert pgq.last_device_status() == pgq.OK


def test_decode_timeout_is_reported_then_parity():
    rows, cols = 1024, 4096
    codes, params = synth.q8_matrix(rows, cols, 990, 1)
    x = synth.normal((1, cols), 1.0, 990, 2)
    g = synth.gamma(cols, 990)
    c, p, xd, gd = dev(codes), dev(params), dev(x), dev(g)
    assert pgq.last_device_status() == pgq.OK
    with stalled():
        pgq.gemv_q8(c, p, xd, gamma=gd)
        assert pgq.last_device_status() == pgq.ETIMEOUT
    assert pgq.last_device_status() == pgq.OK          # reading cleared the record
    y = pgq.gemv_q8(c, p, xd, gamma=gd)
    assert pgq.last_device_status() == pgq.OK
    ref, e = oracle.gemv_q8(codes, params, oracle.rmsnorm(x, g, 1e-6)[0])
    check_proj(host(y), ref, e, what="q8 after a timeout")


def test_prefill_pass_timeout_is_reported_then_parity():
    H, KV, I, B = 512, 128, 1024, 16
    mats = synth.q8_layer(991, 0, H, KV, I)
    dm = {s: (dev(c), dev(p)) for s, (c, p) in mats.items()}
    h0 = synth.normal((B, H), 1.0, 991, synth.T_X)
    g1 = synth.uniform((1, H), 0.5, 1.5, 991, synth.T_GAMMA)
    g2 = synth.uniform((1, H), 0.5, 1.5, 991, synth.T_GAMMA2)
    ws = pgq.prefill_pass_workspace(H, KV, I, B)
    with stalled():
        pgq.prefill_pass([dm], dev(h0), dev(g1), dev(g2), 1e-6, workspace=ws)
        assert pgq.prefill_status(ws) == pgq.ETIMEOUT
        assert pgq.last_device_status(ws) == pgq.ETIMEOUT
    h = dev(h0)
    pgq.prefill_pass([dm], h, dev(g1), dev(g2), 1e-6, workspace=ws)
    assert pgq.last_device_status(ws) == pgq.OK
    # the layer's output against the oracle (each stage fed its own reference)
    ref = oracle.prefill_layer(h0, mats, g1[0], g2[0], 1e-6)
    taps = pgq.prefill_pass_taps(ws, H, KV, I, B)
    t = {k: host(v) for k, v in taps.items()}
    y, e = oracle.gemv_q8(*mats["down"], t["u"])
    check_proj(host(h), t["h1"].astype(np.float64) + y, e, extra=np.abs(t["h1"]) * 2.0 ** -23, what="h2")
    y, e = oracle.gemv_q8(*mats["q"], t["n1"])
    check_proj(t["q"], y, e, what="q")
    assert np.isfinite(ref["h2"]).all()
