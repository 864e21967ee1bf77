"""Parity of the MoE pieces (router, softmax top-k, grouping, grouped expert
projections, weighted combine + RMSNorm) and of the whole MoE layer with the oracle.
Integer outputs (selection, counts, offsets, entries, gathered rows) are bit-exact."""
import numpy as np
import pytest

import oracle
import synth
from util import NORM_TOL, TOL, check_proj, check_relu2, check_rel, dev, host, cuda_ok

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA device")]
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def built():
    from prefill_gemv_q8_gb300 import build
    build.build()


import prefill_gemv_q8_gb300 as pgq  # noqa: E402


@pytest.mark.parametrize("E,cols,B", [(16, 256, 5), (128, 2688, 64), (7, 3072, 3)])
def test_router(E, cols, B):
    R = synth.normal((E, cols), 1.0 / np.sqrt(cols), 970, E)
    n = synth.normal((B, cols), 1.0, 971, B)
    lg = host(pgq.moe_router(dev(R), dev(n)))
    ref, e = oracle.project(R, n)
    check_proj(lg, ref, e, what="router")


@pytest.mark.parametrize("renorm", [False, True])
def test_route_topk(renorm):
    B, E, k = 64, 128, 6
    r = np.random.default_rng(3)
    lg = r.standard_normal((B, E)).astype(np.float32)
    lg[0, [5, 9, 100]] = 4.0            # exact ties: 5, 9, 100 in that order
    lg[1, :] = 0.0                      # all tied: 0..5
    lg[2, 7] = np.nan                   # never preferred
    lg[3, :] = np.round(lg[3, :], 1)    # many ties
    sel, w = pgq.moe_route_topk(dev(lg), k, renorm)
    sel, w = host(sel), host(w)
    lg_clean = np.where(np.isnan(lg), -np.inf, lg)
    ref_sel, ref_w = oracle.route(lg_clean, k, renorm)
    assert np.array_equal(sel, ref_sel)
    assert sel[0, :3].tolist() == [5, 9, 100] and sel[1].tolist() == list(range(6))
    check_rel(w, ref_w, 1e-5, "routing weights")


def test_group_gather():
    B, k, E, n = 64, 6, 128, 40
    r = np.random.default_rng(4)
    sel = np.array([r.choice(E, k, replace=False) for _ in range(B)], np.int32)
    sel[10] = sel[11]                   # two positions choosing the same experts
    x = r.standard_normal((B, n)).astype(np.float32)
    counts, offsets, entries, xg = pgq.moe_group_gather(dev(sel), E, x=dev(x), xdiv=k)
    rc, ro, re = oracle.group(sel, E)
    assert np.array_equal(host(counts), rc)
    assert np.array_equal(host(offsets), ro)
    assert np.array_equal(host(entries), re)
    assert np.array_equal(host(xg), x[re // k])


def test_group_skips_invalid_ids():
    sel = np.array([[1, -1], [7, 1], [0, 3]], np.int32)     # -1 and 7 are outside [0, 4)
    counts, offsets, entries, _ = pgq.moe_group_gather(dev(sel), 4)
    assert host(counts).tolist() == [1, 2, 0, 1]
    assert host(offsets).tolist() == [0, 1, 3, 3, 4]
    assert host(entries).tolist() == [4, 0, 3, 5, -1, -1]


def _bank_case(E, rows, cols, B, k, seed):
    codes, params = synth.q8_bank(E, rows, cols, seed, "up")
    r = np.random.default_rng(seed)
    sel = np.array([r.choice(E, k, replace=False) for _ in range(B)], np.int32)
    return codes, params, sel


@pytest.mark.parametrize("E,rows,cols,B,k", [(8, 96, 256, 16, 3), (4, 70, 2688, 13, 4), (3, 1856, 512, 40, 2)])
def test_experts_up_and_down(E, rows, cols, B, k):
    codes, params, sel = _bank_case(E, rows, cols, B, k, 972 + E)
    x = synth.normal((B, cols), 1.0, 973, B)
    counts, offsets, entries, _ = pgq.moe_group_gather(dev(sel), E)
    u = torch.empty(B * k, rows, device="cuda")
    pgq.moe_experts_q8(dev(codes), dev(params), counts, offsets, entries, dev(x), k, u, "relu2")
    u = host(u)
    for j in range(B * k):
        e = sel.reshape(-1)[j]
        y, ey = oracle.gemv_q8(codes[e], params[e], x[j // k])
        check_relu2(u[j], y[0], ey[0], what=f"up entry {j}")
    # down: input row of entry j is entry j's own row (xdiv = 1)
    dcodes, dparams = synth.q8_bank(E, cols, rows if rows % 32 == 0 else 96, 974, "down")
    if rows % 32 == 0:
        eo = torch.empty(B * k, cols, device="cuda")
        pgq.moe_experts_q8(dev(dcodes), dev(dparams), counts, offsets, entries, dev(u), 1, eo, "none")
        eo = host(eo)
        for j in range(0, B * k, 3):
            e = sel.reshape(-1)[j]
            y, ey = oracle.gemv_q8(dcodes[e], dparams[e], u[j])
            check_proj(eo[j], y[0], ey[0], what=f"down entry {j}")


def test_expert_with_many_entries():
    """Every position picks expert 0 (64 entries for one expert: 8 chunks)."""
    E, rows, cols, B, k = 4, 64, 256, 64, 2
    codes, params = synth.q8_bank(E, rows, cols, 975, "up")
    sel = np.zeros((B, k), np.int32)
    sel[:, 1] = np.arange(B) % 3 + 1
    x = synth.normal((B, cols), 1.0, 976, 1)
    counts, offsets, entries, _ = pgq.moe_group_gather(dev(sel), E)
    y = torch.empty(B * k, rows, device="cuda")
    pgq.moe_experts_q8(dev(codes), dev(params), counts, offsets, entries, dev(x), k, y, "none")
    y = host(y)
    for j in range(B * k):
        ref, e = oracle.gemv_q8(codes[sel.reshape(-1)[j]], params[sel.reshape(-1)[j]], x[j // k])
        check_proj(y[j], ref[0], e[0], what=f"entry {j}")


def test_combine_rmsnorm():
    B, k, n = 9, 3, 2688
    r = np.random.default_rng(5)
    h = r.standard_normal((B, n)).astype(np.float32)
    eo = (r.standard_normal((B * k, n)) * 10).astype(np.float32)
    w = r.uniform(0, 0.4, (B, k)).astype(np.float32)
    g = synth.gamma(n, 977)
    hd = dev(h)
    inv = torch.empty(B, device="cuda")
    y = pgq.moe_combine_rmsnorm(hd, dev(eo), dev(w), dev(g), 1e-6, inv=inv)
    m = oracle.combine(eo, w, k)
    # f32 sum of k products and one add: a few ulp of the magnitudes involved
    scale = np.abs(h) + np.abs(w[:, :, None] * eo.reshape(B, k, n)).sum(axis=1)
    check_proj(host(hd), h + m, scale, tol=4 * 2.0 ** -23, what="h")
    y_ref, inv_ref = oracle.rmsnorm(host(hd), g, 1e-6)
    check_rel(host(inv), inv_ref, NORM_TOL, "inv")
    check_rel(host(y), y_ref, NORM_TOL + 1e-6, "y", abs_=1e-30)


def _layer_check(W_np, router, h0, g1, g2, k, taps, h_after, y, entries_sample=None, renorm=False):
    """Stage-wise check of a MoE layer from its workspace taps."""
    t = {kk: host(v) for kk, v in taps.items()}
    E = router.shape[0]
    n_ref, _ = oracle.rmsnorm(h0, g1, 1e-6)
    check_rel(t["n"], n_ref, NORM_TOL + 1e-6, "n", abs_=1e-30)
    lg, e_lg = oracle.project(router, t["n"])
    check_proj(t["logits"], lg, e_lg, what="logits")
    # selection from the kernel's own f32 logits: bit-exact (R12-i)
    sel_ref, w_ref = oracle.route(t["logits"], k, renorm)
    assert np.array_equal(t["sel"], sel_ref)
    check_rel(t["w"], w_ref, 1e-5, "w")
    c, o, en = oracle.group(t["sel"], E)
    assert np.array_equal(t["counts"], c) and np.array_equal(t["offsets"], o) and np.array_equal(t["entries"], en)
    up, down = W_np   # (codes, params) banks, or (codes, row_scale, col_field) for q8_2f

    def proj(bank, e, x):
        return oracle.gemv_q82f(bank[0][e], bank[1][e], bank[2][e], x) if len(bank) == 3 else \
            oracle.gemv_q8(bank[0][e], bank[1][e], x)
    B = h0.shape[0]
    js = range(B * k) if entries_sample is None else entries_sample
    for j in js:
        e = t["sel"].reshape(-1)[j]
        yu, eu = proj(up, e, t["n"][j // k])
        check_relu2(t["u"][j], yu[0], eu[0], what=f"u[{j}]")
        yd, ed = proj(down, e, t["u"][j])
        check_proj(t["eo"][j], yd[0], ed[0], what=f"eo[{j}]")
    m = oracle.combine(t["eo"], t["w"], k)
    scale = np.abs(h0) + np.abs(t["w"][:, :, None] * t["eo"].reshape(B, k, -1)).sum(axis=1)
    check_proj(host(h_after), h0.astype(np.float64) + m, scale, tol=4 * 2.0 ** -23, what="h")
    y_ref, _ = oracle.rmsnorm(host(h_after), g2, 1e-6)
    check_rel(host(y), y_ref, NORM_TOL + 1e-6, "y", abs_=1e-30)


@pytest.mark.parametrize("E,H,I,B,k", [(16, 256, 128, 24, 4), (8, 288, 96, 24, 3), (6, 160, 224, 40, 2)])
def test_moe_layer_small(E, H, I, B, k):
    """(The second and third shapes have an odd number of (scale, offset) pairs per row
    in both banks (9 and 3; 5 and 7): rows that start on 4-byte boundaries and a ragged
    last k-step whose missing pairs are zero-filled.)"""
    router, up, down = synth.moe_layer(978, E, H, I)
    h0 = synth.normal((B, H), 1.0, 978, synth.T_X)
    g1, g2 = synth.gamma(H, 978), synth.gamma(H, 978, synth.T_GAMMA2)
    Wd = pgq.MoeWeights(dev(router), dev(up[0]), dev(up[1]), dev(down[0]), dev(down[1]), k)
    h = dev(h0)
    ws = torch.full((pgq.moe_layer_workspace(Wd, B).numel(),), 0x55, dtype=torch.uint8, device="cuda")
    y, ws = pgq.moe_prefill_layer(Wd, h, dev(g1), dev(g2), 1e-6, workspace=ws)
    # the workspace's status words (the banks' area comes first) start from garbage
    # and are set by the call itself
    assert pgq.last_device_status(ws) == pgq.OK
    taps = pgq.moe_layer_taps(Wd, ws, B)
    _layer_check((up, down), router, h0, g1, g2, k, taps, h, y)


@pytest.mark.parametrize("E,B,k,renorm", [(256, 64, 8, True), (40, 7, 32, False), (1, 3, 1, True),
                                         (1, 64, 1, False), (2, 64, 1, False), (4, 64, 2, True)])
def test_moe_layer_routing_extremes(E, B, k, renorm):
    """The routing in the router launch at its limits: 256 experts and 8 full position
    groups; a partial position group with k = 32 (2048-entry ceiling: 224 entries);
    a single expert.  Then crowded experts (64 entries for one expert; about 32; about
    32 of 128 entries), which cut the grouped banks' input ring into 3, 4 or 6 stages
    of 4, 3 or 2 boxes.  Selection and lists bit-exact, weights renormalised or not."""
    H, I = 128, 64
    router, up, down = synth.moe_layer(979, E, H, I)
    h0 = synth.normal((B, H), 1.0, 979, synth.T_X)
    g1, g2 = synth.gamma(H, 979), synth.gamma(H, 979, synth.T_GAMMA2)
    Wd = pgq.MoeWeights(dev(router), dev(up[0]), dev(up[1]), dev(down[0]), dev(down[1]), k, renorm)
    h = dev(h0)
    ws = torch.full((pgq.moe_layer_workspace(Wd, B).numel(),), 0x55, dtype=torch.uint8, device="cuda")
    for _ in range(2):   # the second call starts from the tickets the first one left
        h = dev(h0)
        y, ws = pgq.moe_prefill_layer(Wd, h, dev(g1), dev(g2), 1e-6, workspace=ws)
        assert pgq.last_device_status(ws) == pgq.OK
        taps = pgq.moe_layer_taps(Wd, ws, B)
        js = range(0, B * k, max(1, B * k // 48))
        _layer_check((up, down), router, h0, g1, g2, k, taps, h, y, entries_sample=js, renorm=renorm)


def test_moe_layer_full_size_sampled():
    """The MoE prefill layer at its full size (B = 64, hidden 2688, 128 experts of
    1856 x 2688, top-6), as the benchmark runs it; every integer output checked,
    float outputs on 36 sampled entries and every position."""
    c = synth.MOE
    E, H, I, B, k, wl = c["experts"], c["hidden"], c["inter"], c["B"], c["topk"], c["workload"]
    router, up, down = synth.moe_layer(wl, E, H, I, "torch", "cuda")
    h0 = synth.normal((B, H), 1.0, wl, synth.T_X, "torch", "cuda")
    g1 = synth.gamma(H, wl, backend="torch", device="cuda")
    g2 = synth.gamma(H, wl, synth.T_GAMMA2, "torch", "cuda")
    W = pgq.MoeWeights(router, up[0], up[1], down[0], down[1], k)
    h = h0.clone()
    y, ws = pgq.moe_prefill_layer(W, h, g1, g2, 1e-6)
    assert pgq.last_device_status(ws) == pgq.OK
    taps = pgq.moe_layer_taps(W, ws, B)
    sample = sorted(np.random.default_rng(0).choice(B * k, 36, replace=False).tolist())
    sel = host(taps["sel"]).reshape(-1)
    need = sorted(set(int(sel[j]) for j in sample))
    # host copies of only the experts the sampled entries use
    up_np = (np.zeros((E, I, H), np.int8), np.zeros((E, I, H // 32, 2), np.float16))
    dn_np = (np.zeros((E, H, I), np.int8), np.zeros((E, H, I // 32, 2), np.float16))
    for e in need:
        up_np[0][e], up_np[1][e] = host(up[0][e]), host(up[1][e])
        dn_np[0][e], dn_np[1][e] = host(down[0][e]), host(down[1][e])
    _layer_check((up_np, dn_np), host(router), host(h0), host(g1), host(g2), k, taps, h, y, entries_sample=sample)


@pytest.mark.parametrize("E,H,I,B,k", [(16, 256, 128, 24, 4), (8, 384, 96, 64, 2)])
def test_moe_q82f_layer_small(E, H, I, B, k):
    """The MoE layer with q8_2f experts (nemotron_prefill.rs's q8_2f bank payload);
    inter = 96 makes the down bank's last k-step ragged."""
    router, up, down = synth.moe_q82f_layer(1230 + E, E, H, I)
    h0 = synth.normal((B, H), 1.0, 1230 + E, synth.T_X)
    g1, g2 = synth.gamma(H, 1230 + E), synth.gamma(H, 1230 + E, synth.T_GAMMA2)
    W = pgq.MoeQ82Weights(dev(router), tuple(dev(a) for a in up), tuple(dev(a) for a in down), k)
    h = dev(h0)
    ws = torch.full((pgq.moe_layer_workspace(W, B).numel(),), 0x55, dtype=torch.uint8, device="cuda")
    y, ws = pgq.moe_prefill_layer(W, h, dev(g1), dev(g2), 1e-6, workspace=ws)
    assert pgq.last_device_status(ws) == pgq.OK
    taps = pgq.moe_layer_taps(W, ws, B)
    _layer_check((up, down), router, h0, g1, g2, k, taps, h, y)
    # the oracle's whole layer agrees with the kernel's final output
    ref = oracle.moe_layer(h0, g1, g2, 1e-6, router,
                           [(up[0][e], up[1][e], up[2][e], down[0][e], down[1][e], down[2][e]) for e in range(E)], k)
    assert np.array_equal(host(taps["sel"]), ref["sel"])


def test_moe_q82f_layer_full_size_sampled():
    """The q8_2f MoE layer at the full size (B = 64, hidden 2688, 128 experts of
    1856 x 2688, top-6); float outputs checked on 36 sampled entries."""
    c = synth.MOE
    E, H, I, B, k, wl = c["experts"], c["hidden"], c["inter"], c["B"], c["topk"], c["workload"]
    router, up, down = synth.moe_q82f_layer(wl, E, H, I, "torch", "cuda")
    h0 = synth.normal((B, H), 1.0, wl, synth.T_X, "torch", "cuda")
    g1 = synth.gamma(H, wl, backend="torch", device="cuda")
    g2 = synth.gamma(H, wl, synth.T_GAMMA2, "torch", "cuda")
    W = pgq.MoeQ82Weights(router, up, down, k)
    h = h0.clone()
    y, ws = pgq.moe_prefill_layer(W, h, g1, g2, 1e-6)
    assert pgq.last_device_status(ws) == pgq.OK
    taps = pgq.moe_layer_taps(W, ws, B)
    sample = sorted(np.random.default_rng(2).choice(B * k, 36, replace=False).tolist())
    sel = host(taps["sel"]).reshape(-1)
    need = sorted(set(int(sel[j]) for j in sample))
    up_np = (np.zeros((E, I, H), np.int8), np.zeros((E, I), np.float16), np.zeros((E, H), np.float16))
    dn_np = (np.zeros((E, H, I), np.int8), np.zeros((E, H), np.float16), np.zeros((E, I), np.float16))
    for e in need:
        for i in range(3):
            up_np[i][e], dn_np[i][e] = host(up[i][e]), host(down[i][e])
    _layer_check((up_np, dn_np), host(router), host(h0), host(g1), host(g2), k, taps, h, y, entries_sample=sample)
