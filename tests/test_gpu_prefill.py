"""Parity of the tensor-core prefill projection (B <= 64 positions, q8 weights read
once per pass) with the f64 oracle."""
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


def run(mats, X, epis=None, residuals=None, ws=None):
    B = X.shape[0]
    jobs, outs = [], []
    for i, (c, p) in enumerate(mats):
        y = torch.empty(B, c.shape[0], dtype=torch.float32, device="cuda") if residuals is None or \
            residuals[i] is None else residuals[i]
        jobs.append(dict(codes=dev(c), params=dev(p), y=y, epilogue=(epis or ["none"] * len(mats))[i],
                         residual=None if residuals is None else residuals[i]))
        outs.append(y)
    ws = pgq.prefill_q8(jobs, dev(X), workspace=ws)
    assert pgq.prefill_status(ws) == pgq.OK
    return [host(o) for o in outs], ws


CASES = [  # rows, cols, B
    (128, 128, 1), (128, 128, 16), (256, 512, 16), (300, 1024, 64), (64, 4096, 7), (1000, 4096, 33),
    (1024, 4096, 64), (4096, 4096, 64), (4096, 14336, 64), (14336, 4096, 64), (513, 2688, 50)]


@pytest.mark.parametrize("rows,cols,B", CASES)
def test_prefill_q8(rows, cols, B):
    c, p = synth.q8_matrix(rows, cols, 930, rows + cols)
    X = synth.normal((B, cols), 1.0, 931, B)
    (y,), _ = run([(c, p)], X)
    ref, e = oracle.gemv_q8(c, p, X)
    check_proj(y, ref, e, what=f"prefill {rows}x{cols} B={B}")


def test_prefill_identity_layout():
    """Identity weights: every position's row comes back (within binary16 rounding of
    x), which pins the operand layouts (a transposed or permuted K would not)."""
    n, B = 256, 16
    codes = np.eye(n, dtype=np.int8)
    params = np.zeros((n, n // 32, 2), np.float16)
    params[..., 0] = 1.0
    X = (np.arange(B * n, dtype=np.float32).reshape(B, n) % 97) - 48.0   # exact in binary16
    (y,), _ = run([(codes, params)], X)
    assert np.array_equal(y, X)


def test_prefill_multi_and_epilogues():
    cols, B = 4096, 64
    mats = [synth.q8_matrix(r, cols, 932, r) for r in (4096, 1024, 1024)]
    X = synth.normal((B, cols), 1.0, 933, 1)
    res = synth.normal((B, 1024), 3.0, 933, 2)
    r_d = dev(res)
    outs, _ = run(mats, X, epis=["none", "relu2", "add"], residuals=[None, None, r_d])
    r0, e0 = oracle.gemv_q8(*mats[0], X)
    r1, e1 = oracle.gemv_q8(*mats[1], X)
    r2, e2 = oracle.gemv_q8(*mats[2], X)
    check_proj(outs[0], r0, e0)
    check_relu2(outs[1], r1, e1)
    check_proj(outs[2], res + r2, e2, extra=np.abs(res) * 2.0 ** -23)


def test_prefill_large_activations_and_zero_rows():
    """relu²-sized inputs (hundreds to thousands) and an all-zero position stay exact
    in range thanks to the per-position power-of-two scale."""
    rows, cols, B = 512, 4096, 24
    c, p = synth.q8_matrix(rows, cols, 934, 1)
    X = synth.normal((B, cols), 1.0, 934, 2)
    X = (X * X * 500).astype(np.float32)
    X[5] = 0.0
    X[7] *= 1e-20
    (y,), _ = run([(c, p)], X)
    ref, e = oracle.gemv_q8(c, p, X)
    check_proj(y, ref, e)
    assert np.all(y[5] == 0)


def test_prefill_deterministic():
    rows, cols, B = 2048, 4096, 64
    c, p = synth.q8_matrix(rows, cols, 935, 1)
    X = synth.normal((B, cols), 1.0, 935, 2)
    (y1,), ws = run([(c, p)], X)
    (y2,), _ = run([(c, p)], X, ws=ws)
    assert np.array_equal(y1, y2)


def test_prefill_matches_decode_rows():
    """A prompt through the prefill pass and position by position through the decode
    GEMV give the same products (nemotron_prefill.rs: the arithmetic is the decode
    frame's) — within the tolerance of both."""
    rows, cols, B = 700, 4096, 8
    c, p = synth.q8_matrix(rows, cols, 936, 1)
    X = synth.normal((B, cols), 1.0, 936, 2)
    (y,), _ = run([(c, p)], X)
    yd = host(pgq.gemv_q8(dev(c), dev(p), dev(X)))
    ref, e = oracle.gemv_q8(c, p, X)
    check_proj(y, yd, 2 * e)


@pytest.mark.parametrize("rows,epi", [(1024, "add"), (1024, "relu2"), (513, "none")])
def test_prefill_split_fixup_halves_agree(rows, epi):
    """Tiles that three or more blocks share are finished by two blocks, one per half of
    the positions, each adding the tile's partial sums in the same block order: with the
    two halves of the input swapped, the outputs come back swapped, bit for bit (a
    helper that added its sources in another order would round differently)."""
    cols, B = 4096, 64
    c, p = synth.q8_matrix(rows, cols, 937, rows)
    X = synth.normal((B, cols), 1.0, 937, 2)
    swap = lambda a: np.concatenate([a[32:], a[:32]])
    res = synth.normal((B, rows), 3.0, 937, 3) if epi == "add" else None
    r1 = [dev(res)] if res is not None else None
    r2 = [dev(swap(res))] if res is not None else None
    (y1,), _ = run([(c, p)], X, epis=[epi], residuals=r1)
    (y2,), _ = run([(c, p)], swap(X), epis=[epi], residuals=r2)
    assert np.array_equal(y1, swap(y2))
    ref, e = oracle.gemv_q8(c, p, X)
    if epi == "add":
        check_proj(y1, res + ref, e, extra=np.abs(res) * 2.0 ** -23)
    elif epi == "relu2":
        check_relu2(y1, ref, e)
    else:
        check_proj(y1, ref, e)
