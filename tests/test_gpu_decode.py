"""Parity of the decode kernels (add+RMSNorm, relu², argmax, f16 and q8 GEMV, the
tiny MLP block and the q8 decode layer) with the f64 oracle on seeded inputs."""
import numpy as np
import pytest

import oracle
import synth
from util import TOL, NORM_TOL, check_proj, check_relu2, check_rel, dev, host, cuda_ok

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA device")]

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def built():
    from prefill_gemv_q8_gb300 import build
    build.build()


import prefill_gemv_q8_gb300 as pgq  # noqa: E402


def loaded_libraries():
    return open("/proc/self/maps").read()


def test_native_library_is_loaded():
    assert pgq.lib().pgq_device_check() == pgq.OK, pgq.lib().pgq_last_error()
    assert "libpgq.so" in loaded_libraries()


# ------------------------------------------------------------------ a1 add + RMSNorm
@pytest.mark.parametrize("B,n,with_add", [(1, 512, False), (3, 4096, True), (64, 4096, True),
                                          (5, 2688, False), (2, 4, True), (7, 14336, True)])
def test_add_rmsnorm(B, n, with_add):
    r = np.random.default_rng(B * 1000 + n)
    h = (r.standard_normal((B, n)) * r.uniform(0.01, 100, (B, 1))).astype(np.float32)
    a = r.standard_normal((B, n)).astype(np.float32) if with_add else None
    g = synth.gamma(n, 0)
    h_d = dev(h)
    inv_d = torch.empty(B, dtype=torch.float32, device="cuda")
    y_d = pgq.add_rmsnorm(h_d, dev(g), 1e-6, add=dev(a) if with_add else None, inv=inv_d)
    h_ref, y_ref, inv_ref = oracle.add_rmsnorm(h, a, g, 1e-6)
    check_rel(host(h_d), h_ref, 1e-6, "h + add", abs_=1e-30)
    check_rel(host(inv_d), inv_ref, NORM_TOL, "inv")
    # y = γ·h·inv: inv within 1e-4 relative, plus f32 rounding of the products
    check_rel(host(y_d), y_ref, NORM_TOL + 1e-6, "y", abs_=1e-30)


# ------------------------------------------------------------------ a5 relu²
@pytest.mark.parametrize("n", [1, 3, 4, 1000, 14336 * 64 + 3])
def test_relu2(n):
    v = np.random.default_rng(n).standard_normal(n).astype(np.float32) * 10
    v[::7] = -0.0
    d = dev(v)
    pgq.relu2(d)
    want = oracle.relu2(v).astype(np.float32)      # relu² of an f32 value, rounded once
    assert np.array_equal(host(d), want)


# ------------------------------------------------------------------ argmax
def test_argmax_rules():
    r = np.random.default_rng(5)
    l = r.standard_normal((8, 5000)).astype(np.float32)
    l[1, [17, 300, 4000]] = 50.0                      # exact ties → 17
    l[2, :] = np.nan
    l[2, 999] = 1.0                                    # NaN never chosen
    l[3, :] = np.nan                                   # nothing valid → 0
    l[4, :] = -np.inf
    l[5, :] = -3.0e38                                  # nothing above the floor → 0
    l[6, 4999] = 1e30                                  # last element
    l[7, :] = 0.0
    l[7, 2] = -0.0                                     # −0 == +0 tie → lowest index 0
    ids = host(pgq.argmax(dev(l)))
    assert ids.tolist() == oracle.argmax(l).tolist()
    assert ids[1] == 17 and ids[2] == 999 and ids[3] == 0 and ids[5] == 0 and ids[6] == 4999 and ids[7] == 0


# ------------------------------------------------------------------ q8 GEMV
Q8_CASES = [  # rows, cols, B
    (1, 32, 1), (5, 64, 3), (37, 288, 2), (513, 4096, 1), (300, 2688, 8), (129, 1856, 4),
    (64, 512, 5), (1024, 4096, 7), (8, 14336, 1), (333, 2048, 6)]


def _q8(rows, cols, seed):
    return synth.q8_matrix(rows, cols, 900, seed)


@pytest.mark.parametrize("rows,cols,B", Q8_CASES)
@pytest.mark.parametrize("prenorm", [False, True])
def test_gemv_q8(rows, cols, B, prenorm):
    codes, params = _q8(rows, cols, rows * 7 + cols + B)
    x = synth.normal((B, cols), 1.0, 901, rows + B)
    g = synth.gamma(cols, 902) if prenorm else None
    y = pgq.gemv_q8(dev(codes), dev(params), dev(x), gamma=dev(g) if prenorm else None, eps=1e-6)
    xin = oracle.rmsnorm(x, g, 1e-6)[0] if prenorm else x
    ref, e = oracle.gemv_q8(codes, params, xin)
    check_proj(host(y), ref, e, what=f"q8 {rows}x{cols} B={B}")


@pytest.mark.parametrize("epi", ["relu2", "add"])
def test_gemv_q8_epilogues(epi):
    rows, cols, B = 257, 4096, 2
    codes, params = _q8(rows, cols, 11)
    x = synth.normal((B, cols), 1.0, 903, 1)
    res = synth.normal((B, rows), 5.0, 903, 2)
    ref, e = oracle.gemv_q8(codes, params, x)
    if epi == "relu2":
        u = pgq.gemv_q8(dev(codes), dev(params), dev(x), epilogue="relu2")
        check_relu2(host(u), ref, e)
    else:
        y = dev(res)
        pgq.gemv_q8(dev(codes), dev(params), dev(x), epilogue="add", residual=y, y=y)   # in place
        check_proj(host(y), res.astype(np.float64) + ref, e, extra=np.abs(res) * 2.0 ** -23, what="q8 add")


def test_gemv_q8_identity_exact():
    """Identity weights (scale 1, offset 0, code 1 on the diagonal) return x bit for bit."""
    n = 4096
    codes = np.eye(n, dtype=np.int8)
    params = np.zeros((n, n // 32, 2), np.float16)
    params[..., 0] = 1.0
    x = synth.normal((3, n), 1.0, 904, 1)
    y = host(pgq.gemv_q8(dev(codes), dev(params), dev(x)))
    assert np.array_equal(y, x)


def test_gemv_q8_identity_one_position():
    """Identity weights at one position (the register-resident kernel): within
    1e-3·Σ|w||x| = 1e-3·|x_i| of x for every element, however small x_i is."""
    n = 4096
    codes = np.eye(n, dtype=np.int8)
    params = np.zeros((n, n // 32, 2), np.float16)
    params[..., 0] = 1.0
    x = synth.normal((1, n), 1.0, 904, 2)
    y = host(pgq.gemv_q8(dev(codes), dev(params), dev(x)))
    check_proj(y, x.astype(np.float64), np.abs(x), what="q8 identity B=1")


def test_gemv_q8_equal_rows_equal_bits_and_deterministic():
    codes, params = _q8(64, 4096, 12)
    codes[40] = codes[3]
    params[40] = params[3]
    x = dev(synth.normal((1, 4096), 1.0, 905, 1))
    c, p = dev(codes), dev(params)
    y1 = host(pgq.gemv_q8(c, p, x))
    y2 = host(pgq.gemv_q8(c, p, x))
    assert np.array_equal(y1, y2)
    assert y1[0, 40] == y1[0, 3]


def test_gemv_q8_multi_mixed_inputs():
    cols, B = 1024, 2
    mats = [_q8(r, cols, 20 + r) for r in (96, 33, 256)]
    x0 = synth.normal((B, cols), 1.0, 906, 1)
    x1 = synth.normal((B, cols), 1.0, 906, 2)
    g = synth.gamma(cols, 906)
    outs = [torch.empty(B, m[0].shape[0], device="cuda") for m in mats]
    jobs = [dict(codes=dev(m[0]), params=dev(m[1]), y=o, input=i, epilogue=e)
            for m, o, i, e in zip(mats, outs, (0, 1, 0), ("none", "none", "relu2"))]
    pgq.gemv_q8_multi(jobs, [(dev(x0), dev(g)), (dev(x1), None)], eps=1e-6)
    n0 = oracle.rmsnorm(x0, g, 1e-6)[0]
    r0, e0 = oracle.gemv_q8(*mats[0], n0)
    r1, e1 = oracle.gemv_q8(*mats[1], x1)
    r2, e2 = oracle.gemv_q8(*mats[2], n0)
    check_proj(host(outs[0]), r0, e0)
    check_proj(host(outs[1]), r1, e1)
    check_relu2(host(outs[2]), r2, e2)


# ------------------------------------------------------------------ f16 GEMV
F16_CASES = [(1, 32, 1), (2048, 512, 1), (512, 2048, 1), (77, 4096, 8), (1000, 4096, 3), (31, 6144, 2)]


@pytest.mark.parametrize("rows,cols,B", F16_CASES)
@pytest.mark.parametrize("prenorm", [False, True])
def test_gemv_f16(rows, cols, B, prenorm):
    W = synth.f16_matrix(rows, cols, 910, rows + cols)
    x = synth.normal((B, cols), 1.0, 911, B)
    g = synth.gamma(cols, 912) if prenorm else None
    y = pgq.gemv_f16(dev(W), dev(x), gamma=dev(g) if prenorm else None)
    xin = oracle.rmsnorm(x, g, 1e-6)[0] if prenorm else x
    ref, e = oracle.gemv_f16(W, xin)
    check_proj(host(y), ref, e, what=f"f16 {rows}x{cols} B={B}")


@pytest.mark.parametrize("B", [1, 2, 3, 8])
def test_vocab_head_argmax(B):
    rows, cols = 20000, 4096
    W = synth.f16_matrix(rows, cols, 913, B)
    # plant exact ties: copies of some rows further down
    W[15000] = W[123]
    W[19999] = W[7]
    x = synth.normal((B, cols), 1.0, 914, B)
    x[0] = W[123].astype(np.float32) * 10       # position 0 prefers row 123 (and its copy 15000)
    g = synth.gamma(cols, 915)
    ids, logits = pgq.gemv_f16_argmax(dev(W), dev(x), gamma=dev(g))
    ids, lg = host(ids), host(logits)
    ref = oracle.vocab_head(x, g, 1e-6, W)
    check_proj(lg, ref["logits"], ref["e"], what="vocab logits")
    # (i) bit-exact against the oracle's argmax of the kernel's own f32 logits
    assert ids.tolist() == oracle.argmax(lg).tolist()
    assert lg[0, 123] == lg[0, 15000] and ids[0] == 123
    # (ii) against the f64 logits, unless the f64 gap is inside the tolerance
    for b in range(B):
        rl = ref["logits"][b]
        top = np.sort(rl)[-2:]
        if top[1] - top[0] >= 2 * TOL * ref["e"][b].max():
            assert ids[b] == ref["ids"][b]
        else:
            assert rl[ids[b]] >= rl.max() - 2 * TOL * ref["e"][b, ids[b]]


def test_vocab_head_without_logits_matches():
    rows, cols = 3001, 4096
    W = synth.f16_matrix(rows, cols, 916, 1)
    x = synth.normal((4, cols), 1.0, 917, 1)
    Wd, xd = dev(W), dev(x)
    ids_a, lg = pgq.gemv_f16_argmax(Wd, xd)
    ids_b, none = pgq.gemv_f16_argmax(Wd, xd, logits=False)
    assert none is None and host(ids_a).tolist() == host(ids_b).tolist()
    assert host(ids_a).tolist() == oracle.argmax(host(lg)).tolist()


# ------------------------------------------------------------------ workloads
def test_tiny_mlp_full_size():
    """Tiny decode MLP block at its full size (hidden 512, inter 2048, seed 0)."""
    c = synth.TINY_MLP
    H, I, wl = c["hidden"], c["inter"], c["workload"]
    h = synth.normal((H,), 1.0, wl, synth.T_X)
    Wu = synth.f16_matrix(I, H, wl, synth.T_WUP)
    Wd = synth.f16_matrix(H, I, wl, synth.T_WDOWN)
    g = synth.gamma(H, wl)
    y, u = pgq.mlp_f16_decode(dev(h), dev(Wu), dev(Wd), dev(g), 1e-6)
    ref = oracle.tiny_mlp(h, Wu, Wd, g, 1e-6)
    check_relu2(host(u), ref["up"][0], ref["e_up"][0])
    # stage-wise: down checked on the kernel's own u
    dn, e_dn = oracle.gemv_f16(Wd, host(u))
    check_proj(host(y), h.astype(np.float64) + dn[0], e_dn[0], extra=np.abs(h) * 2.0 ** -23, what="mlp y")


def _layer(hidden, kv, inter, wl=1, backend="numpy"):
    return synth.q8_layer(wl, 0, hidden, kv, inter, backend, "cuda" if backend == "torch" else None)


def _check_layer(out, mats, x, x_o, g):
    u = host(out["u"])
    ref = oracle.q8_decode_layer(x, x_o, g, 1e-6, mats, u_in=u)
    for s in ("q", "k", "v", "o"):
        check_proj(host(out[s]), ref[s][0], ref["e_" + s][0], what=s)
    check_relu2(u, ref["up"][0], ref["e_up"][0], what="u")
    check_proj(host(out["down"]), ref["down"][0], ref["e_down"][0], what="down")


def test_q8_decode_layer_small():
    hidden, kv, inter = 512, 128, 1792
    mats = _layer(hidden, kv, inter, wl=920)
    x = synth.normal((hidden,), 1.0, 920, synth.T_X)
    x_o = synth.normal((hidden,), 1.0, 920, synth.T_XO)
    g = synth.gamma(hidden, 920)
    dm = {s: (dev(c), dev(p)) for s, (c, p) in mats.items()}
    out = pgq.q8_decode_layer(dm, dev(x), dev(x_o), dev(g), 1e-6)
    _check_layer(out, mats, x, x_o, g)


def test_q8_decode_layer_full_size():
    """The full q8 decode layer (hidden 4096, kv 1024, inter 14336) in the launch
    configuration the benchmark times; every output element checked."""
    c = synth.Q8_LAYER
    dm = _layer(c["hidden"], c["kv"], c["inter"], wl=c["workload"], backend="torch")
    x = synth.normal((c["hidden"],), 1.0, c["workload"], synth.T_X, "torch", "cuda")
    x_o = synth.normal((c["hidden"],), 1.0, c["workload"], synth.T_XO, "torch", "cuda")
    g = synth.gamma(c["hidden"], c["workload"], backend="torch", device="cuda")
    out = pgq.q8_decode_layer(dm, x, x_o, g, 1e-6)
    mats = {s: (host(cc), host(pp)) for s, (cc, pp) in dm.items()}
    _check_layer(out, mats, host(x), host(x_o), host(g))


def _chain(dms, x0, x_o, g):
    """Layer calls back to back with weights_stable, no host synchronisation between
    them: call i+1 reads x = call i's down output (written by the launch just before)."""
    outs, xs = [], [x0]
    for dm in dms:
        outs.append(pgq.q8_decode_layer(dm, xs[-1], x_o, g, 1e-6, weights_stable=True))
        xs.append(outs[-1]["down"])
    return outs, xs


def test_q8_decode_layers_chained_weights_stable():
    """Three layers with distinct weights chained through their down outputs: each
    step checked against the oracle on the input the kernels actually read."""
    hidden, kv, inter = 512, 128, 1792
    mats = [_layer(hidden, kv, inter, wl=930 + i) for i in range(3)]
    x = synth.normal((hidden,), 1.0, 930, synth.T_X)
    x_o = synth.normal((hidden,), 1.0, 930, synth.T_XO)
    g = synth.gamma(hidden, 930)
    dms = [{s: (dev(c), dev(p)) for s, (c, p) in m.items()} for m in mats]
    outs, xs = _chain(dms, dev(x), dev(x_o), dev(g))
    for out, m, xi in zip(outs, mats, xs):
        _check_layer(out, m, host(xi), x_o, g)


def test_q8_decode_layers_chained_full_size():
    """Two chained full-size layers (hidden 4096, kv 1024, inter 14336) with
    weights_stable, as the benchmark runs them."""
    c = synth.Q8_LAYER
    dm = _layer(c["hidden"], c["kv"], c["inter"], wl=c["workload"], backend="torch")
    x = synth.normal((c["hidden"],), 1.0, c["workload"], synth.T_X, "torch", "cuda")
    x_o = synth.normal((c["hidden"],), 1.0, c["workload"], synth.T_XO, "torch", "cuda")
    g = synth.gamma(c["hidden"], c["workload"], backend="torch", device="cuda")
    outs, xs = _chain([dm, dm], x, x_o, g)
    mats = {s: (host(cc), host(pp)) for s, (cc, pp) in dm.items()}
    for out, xi in zip(outs, xs):
        _check_layer(out, mats, host(xi), host(x_o), host(g))
