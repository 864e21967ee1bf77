"""The q8_2f format (gemma_batch.rs `Q82_MM_WGSL` / `q8_2f_mm_r2`: int8 body, binary16
row scale, binary16 column field) on the tensor-core prefill path: single projections
with every epilogue, and the prefill pass checked stage by stage against the oracle
(each stage fed the kernel's own previous stage), at |Δ| ≤ 1e-3·Σ|w||x| per element."""
import numpy as np
import pytest

import oracle
import synth
from util import NORM_TOL, check_proj, check_rel, check_relu2, dev, host, cuda_ok

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA device")]
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def built():
    from prefill_gemv_q8_gb300 import build
    build.build()


import prefill_gemv_q8_gb300 as pgq  # noqa: E402


@pytest.mark.parametrize("rows,cols,B", [(256, 512, 16), (300, 384, 5), (1024, 1024, 64), (132, 2688, 33),
                                         (4096, 128, 1)])
def test_prefill_q82f_projection(rows, cols, B):
    codes, rs, cf = synth.q82f_matrix(rows, cols, 1200, rows + B)
    x = synth.normal((B, cols), 1.0, 1201, cols + B)
    ref, e = oracle.gemv_q82f(codes, rs, cf, x)
    y = torch.empty(B, rows, dtype=torch.float32, device="cuda")
    pgq.prefill_q82f([dict(codes=dev(codes), row_scale=dev(rs), col_field=dev(cf), y=y)], dev(x))
    check_proj(host(y), ref, e, what=f"q8_2f prefill {rows}x{cols} B={B}")


@pytest.mark.parametrize("rows", [257, 301])   # 301: rows not a multiple of 4 (element-wise epilogue)
def test_prefill_q82f_epilogues(rows):
    cols, B = 640, 24
    codes, rs, cf = synth.q82f_matrix(rows, cols, 1202, rows)
    x = synth.normal((B, cols), 1.0, 1203, 1)
    res = synth.normal((B, rows), 5.0, 1203, 2)
    ref, e = oracle.gemv_q82f(codes, rs, cf, x)
    W = dict(codes=dev(codes), row_scale=dev(rs), col_field=dev(cf))
    u = torch.empty(B, rows, dtype=torch.float32, device="cuda")
    y = dev(res)
    pgq.prefill_q82f([dict(W, y=u, epilogue="relu2"), dict(W, y=y, epilogue="add", residual=y)], dev(x))
    check_relu2(host(u), ref, e, what="q8_2f prefill relu²")
    check_proj(host(y), res.astype(np.float64) + ref, e, extra=np.abs(res) * 2.0 ** -23, what="q8_2f prefill add")


def test_prefill_q82f_identity_and_field():
    """Identity body with unit row scales and a column field of powers of two: every
    product is exact in binary16, so y = x·cf up to the input's binary16 rounding."""
    n, B = 512, 16
    eye = np.eye(n, dtype=np.int8)
    rs = np.ones(n, np.float16)
    cf = (2.0 ** (np.arange(n) % 5 - 2)).astype(np.float16)
    x = synth.normal((B, n), 1.0, 1204, 1)
    y = torch.empty(B, n, dtype=torch.float32, device="cuda")
    pgq.prefill_q82f([dict(codes=dev(eye), row_scale=dev(rs), col_field=dev(cf), y=y)], dev(x))
    ref, e = oracle.gemv_q82f(eye, rs, cf, x)
    check_proj(host(y), ref, e, what="identity × field")
    np.testing.assert_allclose(host(y), x * cf.astype(np.float32)[None, :], rtol=2.0 ** -11, atol=0)


def check_layer_q82f(mats, h0, g1, g2, t, h2, rows=None):
    """Stage-wise check of one q8_2f pass layer from the workspace taps ``t``."""
    sel = slice(None) if rows is None else rows
    proj = lambda s, x: oracle.gemv_q82f(mats[s][0][sel], mats[s][1][sel], mats[s][2], x)  # noqa: E731
    n1_ref, _ = oracle.rmsnorm(h0, g1, 1e-6)
    check_rel(t["n1"], n1_ref, NORM_TOL + 1e-6, "n1", abs_=1e-30)
    for s in ("q", "k", "v"):
        if s == "q" or rows is None:
            y, e = proj(s, t["n1"]) if s == "q" else oracle.gemv_q82f(*mats[s], t["n1"])
            check_proj(t[s][:, sel] if s == "q" else t[s], y, e, what=s)
    y, e = proj("o", t["q"])
    check_proj(t["h1"][:, sel], h0[:, sel].astype(np.float64) + y, e, extra=np.abs(h0[:, sel]) * 2.0 ** -23, what="h1")
    n2_ref, _ = oracle.rmsnorm(t["h1"], g2, 1e-6)
    check_rel(t["n2"], n2_ref, NORM_TOL + 1e-6, "n2", abs_=1e-30)
    up, e = proj("up", t["n2"])
    check_relu2(t["u"][:, sel], up, e, what="u")
    dn, e = proj("down", t["u"])
    check_proj(h2[:, sel], t["h1"][:, sel].astype(np.float64) + dn, e, extra=np.abs(t["h1"][:, sel]) * 2.0 ** -23,
               what="h2")


@pytest.mark.parametrize("H,KV,I,B", [(512, 128, 1024, 16), (1024, 256, 2048, 64)])
def test_q82f_pass_one_layer(H, KV, I, B):
    mats = synth.q82f_layer(1210 + B, 0, H, KV, I)
    h0 = synth.normal((B, H), 1.0, 1210 + B, synth.T_X)
    g1 = synth.uniform((1, H), 0.5, 1.5, 1210 + B, synth.T_GAMMA)
    g2 = synth.uniform((1, H), 0.5, 1.5, 1210 + B, synth.T_GAMMA2)
    dm = {s: tuple(dev(a) for a in m) for s, m in mats.items()}
    h = dev(h0)
    ws = pgq.q82f_prefill_pass([dm], h, dev(g1), dev(g2), 1e-6)
    assert pgq.last_device_status(ws) == pgq.OK
    t = {k: host(v) for k, v in pgq.prefill_pass_taps(ws, H, KV, I, B).items()}
    check_layer_q82f(mats, h0, g1[0], g2[0], t, host(h))


def test_q82f_pass_across_launches_equals_layer_by_layer():
    """L = 10 layers (two launches of the pass kernel) give bit-identical results to
    ten calls of one layer."""
    H, KV, I, B, L = 512, 128, 1024, 32, 10
    layers = [{s: tuple(dev(a) for a in m) for s, m in synth.q82f_layer(1220, l, H, KV, I).items()} for l in range(L)]
    h0 = dev(synth.normal((B, H), 1.0, 1220, synth.T_X))
    g1 = dev(synth.uniform((L, H), 0.5, 1.5, 1220, synth.T_GAMMA))
    g2 = dev(synth.uniform((L, H), 0.5, 1.5, 1220, synth.T_GAMMA2))
    ha = h0.clone()
    pgq.q82f_prefill_pass(layers, ha, g1, g2, 1e-6)
    hb = h0.clone()
    for l in range(L):
        pgq.q82f_prefill_pass([layers[l]], hb, g1[l:l + 1].contiguous(), g2[l:l + 1].contiguous(), 1e-6)
    assert torch.equal(ha, hb)
    assert torch.isfinite(ha).all()


def test_q82f_pass_full_layer_sampled():
    """One layer at the full size (hidden 4096, kv 1024, inter 14336, B = 64), checked
    stage-wise on a sample of 256 rows of q, o, up and down."""
    c = synth.PREFILL
    H, KV, I, B, wl = c["hidden"], c["kv"], c["inter"], c["B"], c["workload"]
    md = synth.q82f_layer(wl, 0, H, KV, I, "torch", "cuda")
    h0 = synth.normal((B, H), 1.0, wl, synth.T_X, "torch", "cuda")
    g1 = synth.uniform((1, H), 0.5, 1.5, wl, synth.T_GAMMA, "torch", "cuda")
    g2 = synth.uniform((1, H), 0.5, 1.5, wl, synth.T_GAMMA2, "torch", "cuda")
    h = h0.clone()
    ws = pgq.q82f_prefill_pass([md], h, g1, g2, 1e-6)
    t = {k: host(v) for k, v in pgq.prefill_pass_taps(ws, H, KV, I, B).items()}
    rows = np.sort(np.random.default_rng(1).choice(H, 256, replace=False))
    mats = {s: tuple(host(a) for a in m) for s, m in md.items()}
    check_layer_q82f(mats, host(h0), host(g1)[0], host(g2)[0], t, host(h), rows=rows)
