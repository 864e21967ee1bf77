"""The batched prefill pass (add+RMSNorm, q/k/v, o with the residual add, add+RMSNorm,
up with relu², down with the residual add, per layer) checked stage by stage against
the oracle, each stage fed the kernel's own previous stage."""
import numpy as np
import pytest

import oracle
import synth
from util import NORM_TOL, check_proj, check_relu2, check_rel, dev, host, cuda_ok

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA device")]
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def built():
    from prefill_gemv_q8_gb300 import build
    build.build()


import prefill_gemv_q8_gb300 as pgq  # noqa: E402


def check_layer(mats, h0, g1, g2, taps, h2, rows_sample=None):
    """Stage-wise: every stage's oracle gets the kernel's previous stage output."""
    t = {k: host(v) for k, v in taps.items()}
    n1_ref, _ = oracle.rmsnorm(h0, g1, 1e-6)
    check_rel(t["n1"], n1_ref, NORM_TOL + 1e-6, "n1", abs_=1e-30)
    sel = slice(None) if rows_sample is None else rows_sample
    for s in ("q", "k", "v"):
        c, p = mats[s]
        r = rows_sample if rows_sample is not None and s == "q" else slice(None)
        y, e = oracle.gemv_q8(c[r], p[r], t["n1"])
        check_proj(t[s][:, r], y, e, what=s)
    y, e = oracle.gemv_q8(mats["o"][0][sel], mats["o"][1][sel], t["q"])
    check_proj(t["h1"][:, sel], h0[:, sel].astype(np.float64) + y, e, extra=np.abs(h0[:, sel]) * 2.0 ** -23,
               what="h1")
    n2_ref, _ = oracle.rmsnorm(t["h1"], g2, 1e-6)
    check_rel(t["n2"], n2_ref, NORM_TOL + 1e-6, "n2", abs_=1e-30)
    up, e = oracle.gemv_q8(*mats["up"], t["n2"]) if rows_sample is None else \
        oracle.gemv_q8(mats["up"][0][sel], mats["up"][1][sel], t["n2"])
    check_relu2(t["u"][:, sel], up, e, what="u")
    dn, e = oracle.gemv_q8(mats["down"][0][sel], mats["down"][1][sel], t["u"])
    check_proj(h2[:, sel], t["h1"][:, sel].astype(np.float64) + dn, e, extra=np.abs(t["h1"][:, sel]) * 2.0 ** -23,
               what="h2")


def _one_layer(H, KV, I, B, wl, backend):
    d = "cuda" if backend == "torch" else None
    mats = synth.q8_layer(wl, 0, H, KV, I, backend, d)
    h0 = synth.normal((B, H), 1.0, wl, synth.T_X, backend, d)
    g1 = synth.uniform((1, H), 0.5, 1.5, wl, synth.T_GAMMA, backend, d)
    g2 = synth.uniform((1, H), 0.5, 1.5, wl, synth.T_GAMMA2, backend, d)
    return mats, h0, g1, g2


@pytest.mark.parametrize("H,KV,I,B", [(512, 128, 1024, 16), (1024, 256, 2048, 64), (512, 128, 1536, 5)])
def test_pass_one_layer_small(H, KV, I, B):
    mats, h0, g1, g2 = _one_layer(H, KV, I, B, 940 + B, "numpy")
    dm = {s: (dev(c), dev(p)) for s, (c, p) in mats.items()}
    h = dev(h0)
    ws = pgq.prefill_pass([dm], h, dev(g1), dev(g2), 1e-6)
    taps = pgq.prefill_pass_taps(ws, H, KV, I, B)
    check_layer(mats, h0, g1[0], g2[0], taps, host(h))


def test_pass_full_layer_sampled():
    """One layer at the full size (hidden 4096, kv 1024, inter 14336, B = 64): the
    launch shapes the benchmark times; q/o/up/down checked on a row sample."""
    c = synth.PREFILL
    mats_d, h0, g1, g2 = _one_layer(c["hidden"], c["kv"], c["inter"], c["B"], c["workload"], "torch")
    h = h0.clone()
    ws = pgq.prefill_pass([mats_d], h, g1, g2, 1e-6)
    taps = pgq.prefill_pass_taps(ws, c["hidden"], c["kv"], c["inter"], c["B"])
    rng = np.random.default_rng(0)
    rows = np.sort(rng.choice(c["hidden"], 256, replace=False))
    mats = {s: (host(cc), host(pp)) for s, (cc, pp) in mats_d.items()}
    check_layer(mats, host(h0), host(g1)[0], host(g2)[0], taps, host(h), rows_sample=rows)


def test_pass_many_layers_equals_layer_by_layer():
    """L layers in one call give bit-identical results to L calls of one layer."""
    H, KV, I, B, L = 512, 128, 1024, 32, 3
    layers = [{s: (dev(cc), dev(pp)) for s, (cc, pp) in synth.q8_layer(950, l, H, KV, I).items()}
              for l in range(L)]
    h0 = dev(synth.normal((B, H), 1.0, 950, synth.T_X))
    g1 = dev(synth.uniform((L, H), 0.5, 1.5, 950, synth.T_GAMMA))
    g2 = dev(synth.uniform((L, H), 0.5, 1.5, 950, synth.T_GAMMA2))
    ha = h0.clone()
    pgq.prefill_pass(layers, ha, g1, g2, 1e-6)
    hb = h0.clone()
    for l in range(L):
        pgq.prefill_pass([layers[l]], hb, g1[l:l + 1].contiguous(), g2[l:l + 1].contiguous(), 1e-6)
    assert torch.equal(ha, hb)
    assert torch.isfinite(ha).all()
