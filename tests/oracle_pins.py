"""Pins of the oracle against facts that do not come from the oracle itself.

Each ``pin_*`` raises AssertionError when the oracle disagrees with a closed form,
an invariant, a brute-force evaluation written independently below (pure Python
loops with a hand-written binary16 decoder), or a value the source pages print
(``tests/golden/pages_constants.json``).  ``test_oracle_pins.py`` runs them as they
are; ``test_oracle_mutations.py`` plants plausible mistakes in the oracle and checks
that at least one pin fails for each.
"""
from __future__ import annotations

import json
import math
import os
import struct

import numpy as np

import oracle.ref as R

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_constants.json")


# ------------------------------------------------------------ independent helpers
def half_bits_to_float(bits: int) -> float:
    """IEEE-754 binary16 decoding from the definition (1 sign, 5 exponent, 10
    fraction bits, bias 15), independent of numpy's conversion."""
    sign = -1.0 if bits & 0x8000 else 1.0
    exp = (bits >> 10) & 0x1F
    frac = bits & 0x3FF
    if exp == 0:
        return sign * frac * 2.0 ** -24
    if exp == 31:
        return sign * math.inf if frac == 0 else math.nan
    return sign * (1.0 + frac / 1024.0) * 2.0 ** (exp - 15)


def f16_list(a):
    bits = np.asarray(a, np.float16).view(np.uint16).reshape(-1)
    return [half_bits_to_float(int(b)) for b in bits]


def brute_q8(codes, params, x):
    """y[r] = Σ_c (scale·q + offset)·x[c], pure Python, f16 decoded by hand."""
    rows, cols = codes.shape
    nb = cols // 32
    p = f16_list(params)
    xs = [float(v) for v in np.asarray(x, np.float32)]
    out = []
    for r in range(rows):
        acc = 0.0
        for c in range(cols):
            s = p[(r * nb + c // 32) * 2]
            o = p[(r * nb + c // 32) * 2 + 1]
            acc += (s * int(codes[r, c]) + o) * xs[c]
        out.append(acc)
    return out


def brute_f16(W, x):
    rows, cols = W.shape
    w = f16_list(W)
    xs = [float(v) for v in np.asarray(x, np.float32)]
    return [sum(w[r * cols + c] * xs[c] for c in range(cols)) for r in range(rows)]


def _rng(seed):
    return np.random.default_rng(seed)


def _q8(rows, cols, seed):
    r = _rng(seed)
    codes = np.clip(np.rint(r.standard_normal((rows, cols)) * 40), -127, 127).astype(np.int8)
    params = np.empty((rows, cols // 32, 2), np.float16)
    params[..., 0] = r.uniform(1e-3, 4e-3, (rows, cols // 32))
    params[..., 1] = r.standard_normal((rows, cols // 32)) * 1e-3
    return codes, params


def close(a, b, rel=1e-12, abs_=0.0):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert a.shape == b.shape, (a.shape, b.shape)
    err = np.abs(a - b)
    lim = rel * np.maximum(np.abs(a), np.abs(b)) + abs_
    assert np.all(err <= lim), f"max err {err.max()} (limit {lim.max()})"


# ------------------------------------------------------------ projections
def pin_q8_identity():
    n = 96
    codes = np.eye(n, dtype=np.int8)
    params = np.zeros((n, n // 32, 2), np.float16)
    params[..., 0] = 1.0
    x = _rng(1).standard_normal((3, n)).astype(np.float32)
    y, _ = R.gemv_q8(codes, params, x)
    assert np.array_equal(y, x.astype(np.float64)), "identity q8 must return x exactly"


def pin_f16_identity():
    n = 64
    x = _rng(2).standard_normal((2, n)).astype(np.float32)
    y, _ = R.gemv_f16(np.eye(n, dtype=np.float16), x)
    assert np.array_equal(y, x.astype(np.float64))


def pin_q8_onehot_rectangular():
    """Row r holds one code at column π(r): y[r] = s·q·x[π(r)] (offset 0).  The
    matrix is 64×96, so a transposed operand or a swapped axis cannot pass."""
    rows, cols = 64, 96
    r = _rng(3)
    perm = r.permutation(cols)[:rows]
    codes = np.zeros((rows, cols), np.int8)
    qv = r.integers(-127, 128, rows)
    codes[np.arange(rows), perm] = qv
    params = np.zeros((rows, cols // 32, 2), np.float16)
    params[..., 0] = r.uniform(1e-3, 4e-3, (rows, cols // 32))
    x = r.standard_normal((2, cols)).astype(np.float32)
    y, e = R.gemv_q8(codes, params, x)
    s = params[np.arange(rows), perm // 32, 0].astype(np.float64)
    want = s[None, :] * qv[None, :] * x[:, perm].astype(np.float64)
    close(y, want, rel=0)
    close(e, np.abs(want), rel=0)


def pin_q8_zero_x():
    codes, params = _q8(32, 64, 4)
    y, e = R.gemv_q8(codes, params, np.zeros((1, 64), np.float32))
    assert np.all(y == 0) and np.all(e == 0)


def pin_q8_ones_closed_form():
    """x = 1: y[r] = Σ_blk (scale·Σ_{c∈blk} q + 32·offset)."""
    codes, params = _q8(40, 128, 5)
    y, _ = R.gemv_q8(codes, params, np.ones((1, 128), np.float32))
    p = params.astype(np.float64)
    want = [sum(p[r, b, 0] * int(codes[r, 32 * b:32 * b + 32].astype(np.int64).sum()) + 32 * p[r, b, 1]
                for b in range(4)) for r in range(40)]
    close(y[0], want, rel=1e-12)


def pin_q8_offset_only():
    """Codes 0: y[r] = Σ_blk offset·Σ_{c∈blk} x[c] (the offset is additive)."""
    rows, cols = 8, 96
    codes = np.zeros((rows, cols), np.int8)
    params = np.zeros((rows, cols // 32, 2), np.float16)
    params[..., 0] = 3e-3
    params[..., 1] = np.arange(rows * 3).reshape(rows, 3) * 0.125 - 1.0
    x = _rng(6).standard_normal(cols).astype(np.float32)
    y, _ = R.gemv_q8(codes, params, x)
    xs = x.astype(np.float64).reshape(3, 32).sum(axis=1)
    want = params[..., 1].astype(np.float64) @ xs
    close(y[0], want, rel=1e-12)


def pin_q8_bruteforce_tiny():
    for rows, cols, seed in ((32, 32, 7), (33, 64, 8), (5, 96, 9)):
        codes, params = _q8(rows, cols, seed)
        x = _rng(seed + 100).standard_normal(cols).astype(np.float32)
        y, e = R.gemv_q8(codes, params, x)
        close(y[0], brute_q8(codes, params, x), rel=1e-11, abs_=1e-12)
        w_abs = [[abs(v) for v in row] for row in R.dequant_q8(codes, params)]
        e_bf = [sum(w_abs[r][c] * abs(float(x[c])) for c in range(cols)) for r in range(rows)]
        close(e[0], e_bf, rel=1e-11)


def pin_f16_bruteforce_tiny():
    for rows, cols, seed in ((7, 32, 10), (64, 96, 11)):
        W = (_rng(seed).standard_normal((rows, cols)) / np.sqrt(cols)).astype(np.float16)
        x = _rng(seed + 1).standard_normal(cols).astype(np.float32)
        y, _ = R.gemv_f16(W, x)
        close(y[0], brute_f16(W, x), rel=1e-11, abs_=1e-12)


def pin_projection_linearity():
    codes, params = _q8(48, 160, 12)
    r = _rng(13)
    x1, x2 = r.standard_normal(160), r.standard_normal(160)
    a = 2.5
    y1, _ = R.gemv_q8(codes, params, x1)
    y2, _ = R.gemv_q8(codes, params, x2)
    y3, _ = R.gemv_q8(codes, params, a * x1 + x2)
    close(y3, a * y1 + y2, rel=1e-9, abs_=1e-12)


def pin_batch_rows_independent():
    """Row b of a batch depends only on x[b]; permuting positions permutes outputs."""
    codes, params = _q8(24, 64, 14)
    X = _rng(15).standard_normal((5, 64))
    Y, _ = R.gemv_q8(codes, params, X)
    P = [3, 0, 4, 1, 2]
    Yp, _ = R.gemv_q8(codes, params, X[P])
    assert np.array_equal(Yp, Y[P])
    for b in range(5):
        yb, _ = R.gemv_q8(codes, params, X[b])
        close(yb[0], Y[b], rel=1e-13, abs_=1e-15)


def pin_quantize_roundtrip_bound():
    """quantize → dequantize error ≤ scale/2 per element, plus any clamp excess."""
    W = _rng(16).standard_normal((16, 256)) * 0.1
    codes, params = R.quantize_q8(W)
    Wd = R.dequant_q8(codes, params)
    s = np.repeat(params[..., 0].astype(np.float64), 32, axis=1)
    o = np.repeat(params[..., 1].astype(np.float64), 32, axis=1)
    excess = np.maximum(0.0, np.abs(W - o) - 127.5 * s)
    assert np.all(np.abs(W - Wd) <= s / 2 + excess + 1e-15)
    assert np.all(np.abs(codes.astype(int)) <= 127)


# ------------------------------------------------------------ norm, activation
def pin_rmsnorm_invariant():
    """mean_i (y_i/γ_i)² = ms/(ms + eps) with ms = mean(h²)."""
    r = _rng(17)
    h = r.standard_normal((4, 300)) * np.array([[1e-3], [1.0], [30.0], [1e3]])
    g = r.uniform(0.5, 1.5, 300)
    eps = 1e-6
    y, inv = R.rmsnorm(h, g, eps)
    ms = np.mean(h * h, axis=1)
    close(np.mean((y / g) ** 2, axis=1), ms / (ms + eps), rel=1e-12)
    close(inv, 1 / np.sqrt(ms + eps), rel=1e-14)


def pin_rmsnorm_constant():
    """h = c, γ = 1: y = c/√(c² + eps) (eps inside the root, as the pages write)."""
    for c in (1e-3, 0.5, -2.0, 7.0):
        y, _ = R.rmsnorm(np.full((1, 64), c), np.ones(64), 1e-6)
        close(y, np.full((1, 64), c / math.sqrt(c * c + 1e-6)), rel=1e-14)


def pin_add_rmsnorm_residual():
    r = _rng(18)
    h, a = r.standard_normal((3, 50)), r.standard_normal((3, 50))
    g = r.uniform(0.5, 1.5, 50)
    hn, y, inv = R.add_rmsnorm(h, a, g, 1e-6)
    assert np.array_equal(hn, h + a)
    y2, _ = R.rmsnorm(h + a, g, 1e-6)
    assert np.array_equal(y, y2)
    hn0, _, _ = R.add_rmsnorm(h, None, g, 1e-6)
    assert np.array_equal(hn0, h)


def pin_relu2_closed_form():
    v = np.array([-3.0, -0.0, 0.0, 0.5, 2.0, -1e-30, 1e10])
    assert np.array_equal(R.relu2(v), np.array([0, 0, 0, 0.25, 4.0, 0, 1e20]))


# ------------------------------------------------------------ MoE
def pin_softmax():
    r = _rng(19)
    l = r.standard_normal((6, 128)) * 3
    p = R.softmax(l)
    close(p.sum(axis=1), np.ones(6), rel=1e-12)
    e = np.exp(l - l.max(axis=1, keepdims=True))
    close(p[:, :5], (e / e.sum(axis=1, keepdims=True))[:, :5], rel=1e-12)
    # shift invariance and a huge logit must not overflow
    close(R.softmax(l + 1000.0), p, rel=1e-9)
    big = R.softmax(np.array([[1000.0, 0.0]]))
    assert np.isfinite(big).all() and big[0, 0] > 0.999
    # two logits: p0 = 1/(1+e^(l1-l0))
    close(R.softmax(np.array([[0.3, -0.2]]))[0, 0], 1 / (1 + math.exp(-0.5)), rel=1e-14)


def pin_topk_bruteforce():
    r = _rng(20)
    s = np.round(r.standard_normal((10, 20)), 1)          # many exact ties
    sel = R.topk(s, 6)
    for b in range(10):
        want = sorted(range(20), key=lambda i: (-s[b, i], i))[:6]
        assert list(sel[b]) == want


def pin_route_weights():
    r = _rng(21)
    l = r.standard_normal((4, 16))
    sel, w = R.route(l, 3)
    p = R.softmax(l)
    for b in range(4):
        assert list(sel[b]) == sorted(range(16), key=lambda i: (-p[b, i], i))[:3]
        close(w[b], p[b, sel[b]], rel=0)
    _, wn = R.route(l, 3, renorm=True)
    close(wn.sum(axis=1), np.ones(4), rel=1e-14)


def pin_group_bruteforce():
    r = _rng(22)
    B, k, E = 13, 4, 9
    sel = np.array([r.choice(E, k, replace=False) for _ in range(B)], np.int32)
    counts, offsets, entries = R.group(sel, E)
    assert counts.sum() == B * k and offsets[0] == 0 and offsets[-1] == B * k
    assert np.array_equal(np.diff(offsets), counts)
    assert sorted(entries.tolist()) == list(range(B * k))
    for e in range(E):
        want = [j for j in range(B * k) if sel.reshape(-1)[j] == e]
        assert entries[offsets[e]:offsets[e + 1]].tolist() == want


def pin_combine_closed_form():
    B, k, n = 3, 2, 5
    eo = np.arange(B * k * n, dtype=np.float64).reshape(B * k, n)
    w = np.array([[1.0, 10.0], [100.0, 0.0], [0.5, -1.0]])
    m = R.combine(eo, w, k)
    want = np.stack([1 * eo[0] + 10 * eo[1], 100 * eo[2] + 0 * eo[3], 0.5 * eo[4] - 1 * eo[5]])
    assert np.array_equal(m, want)
    o = np.ones((B, n))
    assert np.array_equal(R.combine(eo, w, k, o), want + 1)


def pin_argmax_rules():
    l = np.array([[1.0, 5.0, 5.0, -2.0],
                  [np.nan, 0.5, np.nan, 0.5],
                  [np.nan, np.nan, np.nan, np.nan],
                  [-np.inf, -3.0e38, -3.1e38, -np.inf],
                  [-0.0, 0.0, -1.0, -0.0],
                  [-4.0, -1.0, -1.0, -9.0]])
    assert R.argmax(l).tolist() == [1, 1, 0, 0, 0, 1]


# ------------------------------------------------------------ the pages' constants
def pin_pages_constants():
    g = json.load(open(GOLDEN))
    assert R.PASS_MAX == g["pass_max"]["value"]
    assert R.ARGMAX_FLOOR == g["argmax_floor"]["value"]
    a = g["argmax_tie"]
    assert int(R.argmax(np.array([a["example_logits"]]))[0]) == a["expected_index"]
    t = g["route_tie"]
    assert R.topk(np.array([t["example_scores"]]), t["k"])[0].tolist() == t["expected_sel"]
    gr = g["group_order"]
    counts, offsets, entries = R.group(np.array(gr["example_sel"]), gr["experts"])
    assert counts.tolist() == gr["expected_counts"]
    assert entries.tolist() == gr["expected_entries"]


# ------------------------------------------------------------ workloads
def pin_tiny_mlp_composition():
    """Identity up (as f16 I), down = I: y = h + relu²(rms(h)·γ)."""
    n = 32
    h = _rng(23).standard_normal(n).astype(np.float32)
    g = np.linspace(0.5, 1.5, n)
    out = R.tiny_mlp(h, np.eye(n, dtype=np.float16), np.eye(n, dtype=np.float16), g, 1e-6)
    nrm, _ = R.rmsnorm(h, g, 1e-6)
    close(out["y"], h[None].astype(np.float64) + R.relu2(nrm), rel=1e-14)


def pin_prefill_layer_composition():
    """With q, o, up, down the identity (scale 1, code 1 on the diagonal) the layer
    reduces to h1 = h + rms(h)·γ1, h2 = h1 + relu²(rms(h1)·γ2)."""
    n = 64
    eye = np.eye(n, dtype=np.int8)
    par = np.zeros((n, n // 32, 2), np.float16)
    par[..., 0] = 1.0
    mats = {s: (eye, par) for s in ("q", "k", "v", "o", "up", "down")}
    r = _rng(24)
    h = r.standard_normal((3, n))
    g1, g2 = r.uniform(0.5, 1.5, n), r.uniform(0.5, 1.5, n)
    out = R.prefill_layer(h, mats, g1, g2, 1e-6)
    n1, _ = R.rmsnorm(h, g1, 1e-6)
    h1 = h + n1
    n2, _ = R.rmsnorm(h1, g2, 1e-6)
    close(out["h1"], h1, rel=1e-14)
    close(out["h2"], h1 + R.relu2(n2), rel=1e-14)


def _scaled_slots(n, scales):
    """Slot matrices that are the identity times a power of two (code 1 on the
    diagonal, offset 0): exact in binary16, and distinct per slot, so a slot fed
    the wrong input or the wrong matrix changes the result."""
    eye = np.eye(n, dtype=np.int8)
    mats = {}
    for s, sc in scales.items():
        par = np.zeros((n, n // 32, 2), np.float16)
        par[..., 0] = sc
        mats[s] = (eye, par)
    return mats


def _rms_closed(h, g, eps):
    """RMSNorm from its definition, row by row: h / sqrt(mean(h²) + eps) · γ."""
    h = np.atleast_2d(np.asarray(h, np.float64))
    return np.stack([row / math.sqrt(float(np.mean(row * row)) + eps) * np.asarray(g, np.float64) for row in h])


def _relu2_closed(v):
    v = np.asarray(v, np.float64)
    return np.where(v > 0, v * v, 0.0)


# ------------------------------------------------------------ q8_2f (row scale × column field)
def _q82f(rows, cols, seed):
    r = _rng(seed)
    codes = np.clip(np.rint(r.standard_normal((rows, cols)) * 40), -127, 127).astype(np.int8)
    rs = r.uniform(1e-3, 4e-3, rows).astype(np.float16)
    cf = r.uniform(0.5, 2.0, cols).astype(np.float16)
    return codes, rs, cf


def brute_q82f(codes, rs, cf, x):
    """y[r] = Σ_c rs[r]·q[r][c]·cf[c]·x[c], pure Python, binary16 decoded by hand."""
    rows, cols = codes.shape
    rsv, cfv = f16_list(rs), f16_list(cf)
    xs = [float(v) for v in np.asarray(x, np.float32)]
    return [sum(rsv[r] * int(codes[r, c]) * cfv[c] * xs[c] for c in range(cols)) for r in range(rows)]


def pin_q82f_identity():
    """Identity body, unit row scales and column field: y == x exactly."""
    n = 64
    x = _rng(40).standard_normal((3, n)).astype(np.float32)
    y, _ = R.gemv_q82f(np.eye(n, dtype=np.int8), np.ones(n, np.float16), np.ones(n, np.float16), x)
    assert np.array_equal(y, x.astype(np.float64))


def pin_q82f_onehot_rectangular():
    """One code per row at column π(r), on a 48×80 matrix: y[r] = rs[r]·q·cf[π(r)]·x[π(r)],
    so a row scale read per column (or a column field read per row) cannot pass."""
    rows, cols = 48, 80
    r = _rng(41)
    perm = r.permutation(cols)[:rows]
    codes = np.zeros((rows, cols), np.int8)
    qv = r.integers(-127, 128, rows)
    codes[np.arange(rows), perm] = qv
    rs = r.uniform(1e-3, 4e-3, rows).astype(np.float16)
    cf = r.uniform(0.5, 2.0, cols).astype(np.float16)
    x = r.standard_normal((2, cols)).astype(np.float32)
    y, e = R.gemv_q82f(codes, rs, cf, x)
    want = (rs.astype(np.float64)[None, :] * qv[None, :] * cf.astype(np.float64)[perm][None, :]
            * x[:, perm].astype(np.float64))
    close(y, want, rel=1e-15)
    close(e, np.abs(want), rel=1e-15)


def pin_q82f_ones_closed_form():
    """x = 1: y[r] = rs[r]·Σ_c q[r][c]·cf[c]."""
    codes, rs, cf = _q82f(24, 96, 42)
    y, _ = R.gemv_q82f(codes, rs, cf, np.ones((1, 96), np.float32))
    want = [float(rs[r]) * sum(int(codes[r, c]) * float(cf[c]) for c in range(96)) for r in range(24)]
    close(y[0], want, rel=1e-12)


def pin_q82f_brute_force():
    for rows, cols, seed in ((5, 32, 43), (7, 64, 44), (3, 96, 45)):
        codes, rs, cf = _q82f(rows, cols, seed)
        x = _rng(seed + 100).standard_normal((2, cols)).astype(np.float32)
        y, _ = R.gemv_q82f(codes, rs, cf, x)
        for b in range(2):
            close(y[b], brute_q82f(codes, rs, cf, x[b]), rel=1e-12, abs_=1e-300)


def pin_q82f_folds_like_the_page():
    """The page's arithmetic order: the column field folded into the activations,
    the row scale applied to the finished integer-weighted sum."""
    codes, rs, cf = _q82f(16, 64, 46)
    x = _rng(47).standard_normal((3, 64))
    y, _ = R.gemv_q82f(codes, rs, cf, x)
    folded = x * cf.astype(np.float64)[None, :]
    want = (folded @ codes.astype(np.float64).T) * rs.astype(np.float64)[None, :]
    close(y, want, rel=1e-12)


# ------------------------------------------------------------ sandwich residual
def pin_add_rmsnorm_ex_closed_forms():
    """h = 0, d = c (constant): h' = s·c, y = s·c/√((s·c)² + eps)·w, with w = 1 + γ
    under the gemma switch; no scale when scale is 0 or None."""
    n, c, s, eps = 16, 0.75, 2.5, 1e-6
    g = _rng(48).uniform(0.5, 1.5, n)
    h0 = np.zeros((1, n))
    d = np.full((1, n), c)
    hn, y, inv = R.add_rmsnorm_ex(h0, d, g, eps, scale=s, gemma=True)
    close(hn, np.full((1, n), s * c), rel=1e-15)
    close(inv, [1.0 / math.sqrt((s * c) ** 2 + eps)], rel=1e-15)
    close(y, (s * c / math.sqrt((s * c) ** 2 + eps)) * (1.0 + g)[None, :], rel=1e-14)
    for none in (None, 0.0):
        hn, y, _ = R.add_rmsnorm_ex(h0, d, g, eps, scale=none)
        close(hn, d, rel=0)
        close(y, (c / math.sqrt(c * c + eps)) * g[None, :], rel=1e-14)


def pin_sandwich_constant_inputs():
    """x = a and h = b constant, w1 = 1, w2 = γ: mid = a/√(a² + eps),
    h' = (b + mid)·s, n = h'/√(h'² + eps)·γ."""
    n, a, b, s, eps = 32, -1.25, 0.5, 0.75, 1e-6
    g = _rng(49).uniform(0.5, 1.5, n)
    out = R.sandwich(np.full((2, n), a), np.ones(n), np.full((2, n), b), g, eps, scale=s)
    mid = a / math.sqrt(a * a + eps)
    hp = (b + mid) * s
    close(out["mid"], np.full((2, n), mid), rel=1e-15)
    close(out["h"], np.full((2, n), hp), rel=1e-15)
    close(out["n"], np.tile(hp / math.sqrt(hp * hp + eps) * g, (2, 1)), rel=1e-14)


def pin_sandwich_invariants_and_order():
    """mean((n/w2)²) = ms/(ms + eps) with ms = mean(h'²); h' − h·s = mid·s (the add
    comes before the scale); gemma with zero weights equals unit weights."""
    n, eps, s = 40, 1e-6, 1.5
    r = _rng(50)
    x, h = r.standard_normal((3, n)) * 3, r.standard_normal((3, n))
    w1, w2 = r.uniform(0.5, 1.5, n), r.uniform(0.5, 1.5, n)
    out = R.sandwich(x, w1, h, w2, eps, scale=s)
    ms = np.mean(out["h"] ** 2, axis=1)
    close(np.mean((out["n"] / w2[None, :]) ** 2, axis=1), ms / (ms + eps), rel=1e-13)
    ms1 = np.mean(x * x, axis=1)
    close(np.mean((out["mid"] / w1[None, :]) ** 2, axis=1), ms1 / (ms1 + eps), rel=1e-13)
    close(out["h"] - h * s, out["mid"] * s, rel=1e-12, abs_=1e-15)
    a = R.sandwich(x, np.zeros(n), h, np.zeros(n), eps, gemma=True)
    b = R.sandwich(x, np.ones(n), h, np.ones(n), eps)
    for k in ("mid", "h", "n"):
        close(a[k], b[k], rel=0)


def pin_sandwich_brute_force():
    """Pure-Python statement of the two norms on a tiny row."""
    x = [0.5, -2.0, 1.0, 3.0]
    h = [1.0, 0.25, -0.5, 2.0]
    w1 = [1.5, 0.5, 1.0, 0.75]
    w2 = [0.5, 1.25, 1.0, 2.0]
    eps, s = 1e-6, 0.5
    inv1 = 1.0 / math.sqrt(sum(v * v for v in x) / 4 + eps)
    mid = [x[i] * inv1 * (1.0 + w1[i]) for i in range(4)]
    hp = [(h[i] + mid[i]) * s for i in range(4)]
    inv2 = 1.0 / math.sqrt(sum(v * v for v in hp) / 4 + eps)
    nn = [hp[i] * inv2 * (1.0 + w2[i]) for i in range(4)]
    out = R.sandwich(np.array([x]), np.array(w1), np.array([h]), np.array(w2), eps, scale=s, gemma=True)
    close(out["mid"][0], mid, rel=1e-15)
    close(out["h"][0], hp, rel=1e-15)
    close(out["n"][0], nn, rel=1e-14)
    close(out["inv1"], [inv1], rel=1e-15)
    close(out["inv2"], [inv2], rel=1e-15)


SLOT_SCALES = {"q": 2.0, "k": 4.0, "v": 0.5, "o": 8.0, "up": 0.25, "down": 16.0}


def pin_q8_decode_layer_slots():
    """Decode layer wiring: q, k, v and up read n = rms(x)·γ, o reads its own input
    x_o, down reads relu²(up); each slot's scale shows which matrix it used."""
    n = 64
    mats = _scaled_slots(n, SLOT_SCALES)
    r = _rng(27)
    x, x_o, g = r.standard_normal(n), r.standard_normal(n), r.uniform(0.5, 1.5, n)
    out = R.q8_decode_layer(x, x_o, g, 1e-6, mats)
    nrm = _rms_closed(x, g, 1e-6)
    for s in ("q", "k", "v", "up"):
        close(out[s], SLOT_SCALES[s] * nrm, rel=1e-13)
    close(out["o"], SLOT_SCALES["o"] * np.atleast_2d(x_o), rel=1e-13)
    close(out["down"], SLOT_SCALES["down"] * _relu2_closed(SLOT_SCALES["up"] * nrm), rel=1e-13)


def pin_prefill_layer_slots():
    """Prefill layer wiring with distinct slot scales: h1 = h + s_o·(s_q·n1),
    n2 = rms(h1)·γ2, h2 = h1 + s_down·relu²(s_up·n2), and k, v = s_k·n1, s_v·n1."""
    n = 64
    mats = _scaled_slots(n, SLOT_SCALES)
    r = _rng(28)
    h = r.standard_normal((3, n))
    g1, g2 = r.uniform(0.5, 1.5, n), r.uniform(0.5, 1.5, n)
    out = R.prefill_layer(h, mats, g1, g2, 1e-6)
    n1 = _rms_closed(h, g1, 1e-6)
    for s in ("q", "k", "v"):
        close(out[s], SLOT_SCALES[s] * n1, rel=1e-13)
    h1 = h + SLOT_SCALES["o"] * (SLOT_SCALES["q"] * n1)
    close(out["h1"], h1, rel=1e-13)
    n2 = _rms_closed(h1, g2, 1e-6)
    close(out["h2"], h1 + SLOT_SCALES["down"] * _relu2_closed(SLOT_SCALES["up"] * n2), rel=1e-12)


def pin_moe_layer_composition():
    """Experts whose up and down are the identity scaled by (e+1): the MoE output for
    a position is Σ_s w_s·relu²((e_s+1)·n) (up scale e+1, down scale 1), and the
    layer's output is the second norm of the updated residual, y = rms(h + m)·γ2,
    with γ1 ≠ γ2 so that a norm taking the wrong weight (or none) is seen."""
    n, E, k, B = 32, 5, 2, 4
    eye = np.eye(n, dtype=np.int8)
    experts = []
    for e in range(E):
        pu = np.zeros((n, 1, 2), np.float16)
        pu[..., 0] = e + 1
        pd = np.zeros((n, 1, 2), np.float16)
        pd[..., 0] = 1.0
        experts.append((eye, pu, eye, pd))
    r = _rng(25)
    h = r.standard_normal((B, n))
    g1, g2 = r.uniform(0.5, 1.5, n), r.uniform(0.5, 1.5, n)
    router = r.standard_normal((E, n))
    out = R.moe_layer(h, g1, g2, 1e-6, router, experts, k)
    nrm = _rms_closed(h, g1, 1e-6)
    close(out["n"], nrm, rel=1e-13)
    logits = nrm @ router.T
    sel, w = R.route(logits, k)
    m = np.zeros_like(h)
    for b in range(B):
        for s in range(k):
            m[b] += w[b, s] * _relu2_closed((sel[b, s] + 1) * nrm[b])
    close(out["m"], m, rel=1e-12, abs_=1e-15)
    close(out["h"], h + m, rel=1e-13)
    hn = h + m
    close(out["y"], _rms_closed(hn, g2, 1e-6), rel=1e-12)
    close(out["inv2"], 1.0 / np.sqrt(np.mean(hn * hn, axis=1) + 1e-6), rel=1e-13)


def pin_moe_layer_q82f_closed_form():
    """q8_2f experts (nemotron_prefill.rs's q8_2f bank payload): expert e's up matrix is
    a permutation P (row r reads column π(r) = (3r + 1) mod n) with row scales
    (e+1)·a_r and a column field b_c, its down matrix the identity with unit scales, so
    up_e(x)_r = (e+1)·a_r·b_π(r)·x_π(r) and m[b] = Σ_s w_s·relu²(up_e(n[b])).  Row scales
    and column fields differ in pattern and the permutation is not symmetric, so a
    transposed or swapped factor, or the down bank's scales used for up, is seen."""
    n, E, k, B = 32, 4, 2, 5
    pi = (3 * np.arange(n) + 1) % n
    perm = np.zeros((n, n), np.int8)
    perm[np.arange(n), pi] = 1
    a = 2.0 ** (np.arange(n) % 3 - 1)
    bfield = 1.0 + (np.arange(n) % 4) / 4.0
    eye = np.eye(n, dtype=np.int8)
    ones = np.ones(n, np.float16)
    experts = [(perm, ((e + 1) * a).astype(np.float16), bfield.astype(np.float16), eye, ones, ones) for e in range(E)]
    r = _rng(27)
    h = r.standard_normal((B, n))
    g1, g2 = r.uniform(0.5, 1.5, n), r.uniform(0.5, 1.5, n)
    router = r.standard_normal((E, n))
    out = R.moe_layer(h, g1, g2, 1e-6, router, experts, k)
    nrm = _rms_closed(h, g1, 1e-6)
    sel, w = R.route(nrm @ router.T, k)
    m = np.zeros_like(h)
    for b in range(B):
        for s in range(k):
            up = (sel[b, s] + 1) * a * bfield[pi] * nrm[b][pi]
            close(out["up"][b * k + s], up, rel=1e-13, abs_=1e-15)
            m[b] += w[b, s] * _relu2_closed(up)
    close(out["m"], m, rel=1e-12, abs_=1e-15)
    close(out["y"], _rms_closed(h + m, g2, 1e-6), rel=1e-12)


def pin_vocab_head_ties():
    """Duplicated rows give exact ties, which go to the lowest row."""
    r = _rng(26)
    W = (r.standard_normal((10, 64)) / 8).astype(np.float16)
    x = r.standard_normal((2, 64)).astype(np.float32)
    g = np.ones(64)
    out = R.vocab_head(x, g, 1e-6, W)
    best = out["ids"]
    W2 = np.concatenate([W[best[0]:best[0] + 1], W])   # the winner of position 0 at row 0 and row best+1
    out2 = R.vocab_head(x, g, 1e-6, W2)
    assert out2["logits"][0, 0] == out2["logits"][0, best[0] + 1]
    assert out2["ids"][0] == 0


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_") and callable(v)]
