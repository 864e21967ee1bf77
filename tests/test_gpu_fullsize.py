"""Parity at the launch shapes the benchmark times.

* The vocab head at its full size (262144 × 4096 binary16, 2 GiB: the last row ends
  exactly at the 2^31-byte mark) for one position (CUDA-core kernel) and eight
  (tensor-core kernel): every logit against the oracle, the ids under both argmax
  checks, and an exact tie planted among the last rows, which the earlier row wins.
* The prefill pass across its launch boundary: more than PASS_LMAX layers take several
  persistent launches (PASS_LMAX layers each), each starting from the previous launch's
  h and the next layer's norm weights; results must be bit-identical to one layer
  per call, and the last layer must match the oracle stage by stage.
* One full-size launch of PASS_LMAX layers (hidden 4096, kv 1024, inter 14336, 64
  positions): the last layer stage by stage on a row sample.
"""
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


import prefill_gemv_q8_gb300 as pgq  # noqa: E402
from test_gpu_prefill_pass import check_layer  # noqa: E402


# ------------------------------------------------------------------ vocab head
@pytest.mark.parametrize("B", [1, 8])
def test_vocab_head_full_size(B):
    c = synth.VOCAB
    V, H, wl = c["vocab"], c["hidden"], c["workload"]
    W = synth.f16_matrix(V, H, wl, synth.T_W, "torch", "cuda")
    early, late = 1234, V - 300                       # the copy sits in the last 1024 rows
    W[late] = W[early]
    x = synth.normal((B, H), 1.0, wl, synth.T_X + B, "torch", "cuda")
    x[0] = W[early].float() * 8.0                     # position 0 prefers the early row (and its copy)
    g = synth.gamma(H, wl, backend="torch", device="cuda")
    ids, logits = pgq.gemv_f16_argmax(W, x, gamma=g)
    torch.cuda.synchronize()
    ids, lg = host(ids), host(logits)
    xh, gh = host(x), host(g)
    n, _ = oracle.rmsnorm(xh, gh, 1e-6)
    # the oracle over row chunks (host memory bounded)
    ref = np.empty((B, V))
    err = np.empty((B, V))
    step = 16384
    for r0 in range(0, V, step):
        Wc = host(W[r0:r0 + step])
        y, e = oracle.gemv_f16(Wc, n)
        ref[:, r0:r0 + step], err[:, r0:r0 + step] = y, e
    check_proj(lg, ref, err, what=f"vocab logits B={B}")
    # (i) bit-exact against the oracle's argmax of the kernel's own f32 logits
    assert ids.tolist() == oracle.argmax(lg).tolist()
    assert lg[0, early] == lg[0, late] and ids[0] == early
    # (ii) against the f64 logits, unless the f64 gap is inside the tolerance
    ref_ids = oracle.argmax(ref)
    for b in range(B):
        rl = ref[b]
        top = np.partition(rl, -2)[-2:]
        if abs(top[1] - top[0]) >= 2 * TOL * err[b].max():
            assert ids[b] == ref_ids[b]
        else:
            assert rl[ids[b]] >= rl.max() - 2 * TOL * err[b, ids[b]]


# ------------------------------------------------------------------ prefill pass across launches
def _layers(wl, L, H, KV, I):
    return [{s: (dev(cc), dev(pp)) for s, (cc, pp) in synth.q8_layer(wl, l, H, KV, I).items()} for l in range(L)]


@pytest.mark.parametrize("L,B", [(10, 64), (17, 32)])
def test_pass_across_launches_equals_layer_by_layer(L, B):
    H, KV, I = 512, 128, 1024
    wl = 960 + L
    layers = _layers(wl, L, H, KV, I)
    h0 = dev(synth.normal((B, H), 1.0, wl, synth.T_X))
    g1 = dev(synth.uniform((L, H), 0.5, 1.5, wl, synth.T_GAMMA))
    g2 = dev(synth.uniform((L, H), 0.5, 1.5, wl, synth.T_GAMMA2))
    ha = h0.clone()
    ws = pgq.prefill_pass(layers, ha, g1, g2, 1e-6)
    assert pgq.last_device_status(ws) == pgq.OK
    hb = h0.clone()
    h_before_last = None
    for l in range(L):
        if l == L - 1:
            h_before_last = hb.clone()
        pgq.prefill_pass([layers[l]], hb, g1[l:l + 1].contiguous(), g2[l:l + 1].contiguous(), 1e-6)
    assert torch.equal(ha, hb)
    # the last layer, stage by stage, from the multi-launch call's own taps
    taps = pgq.prefill_pass_taps(ws, H, KV, I, B)
    mats = {s: (host(cc), host(pp)) for s, (cc, pp) in layers[-1].items()}
    check_layer(mats, host(h_before_last), host(g1)[L - 1], host(g2)[L - 1], taps, host(ha))


def test_pass_full_size_one_launch():
    """PASS_LMAX layers at the benchmark's shapes in one persistent launch: the last
    layer checked stage by stage on a row sample, the h it started from taken from a
    call over the layers before it."""
    c = synth.PREFILL
    H, KV, I, B, wl = c["hidden"], c["kv"], c["inter"], c["B"], c["workload"]
    L = pgq.PASS_LMAX
    layers = [synth.q8_layer(wl, l, H, KV, I, "torch", "cuda") for l in range(L)]
    h0 = synth.normal((B, H), 1.0, wl, synth.T_X, "torch", "cuda")
    g1 = synth.uniform((L, H), 0.5, 1.5, wl, synth.T_GAMMA, "torch", "cuda")
    g2 = synth.uniform((L, H), 0.5, 1.5, wl, synth.T_GAMMA2, "torch", "cuda")
    hp = h0.clone()
    pgq.prefill_pass(layers[:L - 1], hp, g1[:L - 1].contiguous(), g2[:L - 1].contiguous(), 1e-6)
    h = h0.clone()
    ws = pgq.prefill_pass(layers, h, g1, g2, 1e-6)
    assert pgq.last_device_status(ws) == pgq.OK
    # one launch of L layers equals a launch of L - 1 layers and a one-layer call
    hl = hp.clone()
    pgq.prefill_pass(layers[L - 1:], hl, g1[L - 1:].contiguous(), g2[L - 1:].contiguous(), 1e-6)
    assert torch.equal(h, hl)
    taps = pgq.prefill_pass_taps(ws, H, KV, I, B)
    rng = np.random.default_rng(8)
    rows = np.sort(rng.choice(H, 192, replace=False))
    mats = {s: (host(cc), host(pp)) for s, (cc, pp) in layers[-1].items()}
    check_layer(mats, host(hp), host(g1)[L - 1], host(g2)[L - 1], taps, host(h), rows_sample=rows)
