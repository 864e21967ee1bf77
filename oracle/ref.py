"""f64 oracle of the projection path (see the package docstring)."""
from __future__ import annotations

import numpy as np

QBLOCK = 32                 # q8 format: one (scale, offset) pair per 32 columns of a row
ARGMAX_FLOOR = -3.0e38      # nemotron_prefill.rs `pb_argmax`: the running max starts here
PASS_MAX = 64               # nemotron_prefill.rs `PB_MAX`: positions per prefill pass

__all__ = [
    "QBLOCK", "ARGMAX_FLOOR", "PASS_MAX",
    "as_f64", "dequant_q8", "project", "gemv_f16", "gemv_q8", "dequant_q82f", "gemv_q82f",
    "rmsnorm", "add_rmsnorm", "add_rmsnorm_ex", "sandwich", "relu2", "softmax", "topk", "route", "group",
    "combine", "argmax", "quantize_q8",
    "tiny_mlp", "q8_decode_layer", "prefill_layer", "moe_layer", "vocab_head",
]


def as_f64(a) -> np.ndarray:
    """Exact widening of f32 / binary16 / integer arrays to f64."""
    return np.asarray(a).astype(np.float64)


# ----------------------------------------------------------------- weights
def dequant_q8(codes, params) -> np.ndarray:
    """q8 block format → f64 weights.

    w[r][c] = scale[r][c // 32] · q[r][c] + offset[r][c // 32], with (scale, offset)
    the binary16 pair ``params[r][c // 32]``.  The offset is additive in weight
    units (the plain reading of "scale and offset"; the q8_2f format of
    gemma_batch.rs `Q82_MM_WGSL`, row scale × column field, is a different format).
    """
    codes = np.asarray(codes)
    rows, cols = codes.shape
    assert cols % QBLOCK == 0
    p = as_f64(params).reshape(rows, cols // QBLOCK, 2)
    q = as_f64(codes).reshape(rows, cols // QBLOCK, QBLOCK)
    w = q * p[:, :, 0:1] + p[:, :, 1:2]
    return w.reshape(rows, cols)


def project(W, X):
    """y[b][r] = Σ_c W[r][c]·x[b][c] — the projection of gemma_batch.rs
    `encode_q82_mm` ("y[nb][rows] = x[nb][cols]·Wᵀ") — and its error scale
    e[b][r] = Σ_c |W[r][c]|·|x[b][c]|.  X is [B][cols] (or [cols]); returns
    (Y [B][rows], E [B][rows])."""
    W = as_f64(W)
    X = np.atleast_2d(as_f64(X))
    return X @ W.T, np.abs(X) @ np.abs(W).T


def gemv_f16(W16, X):
    """Projection through a binary16 matrix (embryo_wide.wgsl header: f16 matrices
    read by the row kernels)."""
    return project(as_f64(W16), X)


def gemv_q8(codes, params, X):
    """Projection through a q8 block-format matrix."""
    return project(dequant_q8(codes, params), X)


def dequant_q82f(codes, row_scale, col_field) -> np.ndarray:
    """q8_2f format → f64 weights (gemma_batch.rs `Q82_MM_WGSL`: an int8 body
    [rows][cols], one binary16 scale per row and one binary16 factor per column, the
    "column field"):  w[r][c] = row_scale[r] · q[r][c] · col_field[c].  The page's
    kernel folds the column field into the staged activations and multiplies the
    finished row sum by the row scale; this is the same product written per weight."""
    q = as_f64(codes)
    rows, cols = q.shape
    rs = as_f64(row_scale).reshape(rows)
    cf = as_f64(col_field).reshape(cols)
    return rs[:, None] * q * cf[None, :]


def gemv_q82f(codes, row_scale, col_field, X):
    """Projection through a q8_2f matrix (gemma_batch.rs `q8_2f_mm_r2`)."""
    return project(dequant_q82f(codes, row_scale, col_field), X)


# ----------------------------------------------------------------- norms, activation
def rmsnorm(h, gamma, eps):
    """nemotron_prefill.rs `pb_add_rms` / gemma_batch.rs `g4_add_norm_b`:
    inv = 1/√(mean_i h_i² + eps), y = γ·(h·inv), per row.  Returns (y, inv)."""
    h = np.atleast_2d(as_f64(h))
    ms = np.mean(h * h, axis=1)
    inv = 1.0 / np.sqrt(ms + float(eps))
    return h * inv[:, None] * as_f64(gamma)[None, :], inv


def add_rmsnorm(h, add, gamma, eps):
    """`pb_add_rms` with add=1: h ← h + add (``add`` may be None: plain norm),
    then y = rms(h)·γ.  Returns (h_new, y, inv)."""
    h = np.atleast_2d(as_f64(h))
    if add is not None:
        h = h + np.atleast_2d(as_f64(add))
    y, inv = rmsnorm(h, gamma, eps)
    return h, y, inv


def add_rmsnorm_ex(h, add, gamma, eps, scale=None, gemma=False):
    """gemma_batch.rs `g4_add_norm_b`: h ← (h + d)·scale (no scale when ``scale`` is
    None or 0: the page's "scale bits 0"), then y = h·inv·w with w = 1 + γ when
    ``gemma`` (the page's `gemma` switch) else γ.  Returns (h_new, y, inv)."""
    h = np.atleast_2d(as_f64(h))
    if add is not None:
        h = h + np.atleast_2d(as_f64(add))
    if scale:
        h = h * float(scale)
    w = as_f64(gamma)
    if gemma:
        w = 1.0 + w
    y, inv = rmsnorm(h, w, eps)
    return h, y, inv


def sandwich(x, w1, h, w2, eps, scale=None, gemma=False):
    """gemma_batch.rs `g4_sandwich` (Gemma's sandwich residual in one dispatch), in
    the page's order: mid = rms(x)·w1 (the mixer or FFN output norm), then
    h ← (h + mid)·scale and n = rms(h)·w2 (`g4_add_norm_b`); with ``gemma`` both norm
    weights are used as 1 + w.  Returns dict(mid, h, n, inv1, inv2)."""
    w1 = as_f64(w1)
    if gemma:
        w1 = 1.0 + w1
    mid, inv1 = rmsnorm(x, w1, eps)
    h_new, n, inv2 = add_rmsnorm_ex(h, mid, w2, eps, scale, gemma)
    return dict(mid=mid, h=h_new, n=n, inv1=inv1, inv2=inv2)


def relu2(v):
    """`pb_relu2`: v ← max(v, 0)²."""
    r = np.maximum(as_f64(v), 0.0)
    return r * r


# ----------------------------------------------------------------- MoE
def softmax(logits):
    """p_e = exp(l_e) / Σ exp(l), per row (shifted by the row max)."""
    l = np.atleast_2d(as_f64(logits))
    z = np.exp(l - l.max(axis=1, keepdims=True))
    return z / z.sum(axis=1, keepdims=True)


def topk(scores, k):
    """The k largest scores of each row, larger first; an exact tie goes to the
    lower expert id (nemotron_prefill.rs `pb_route`: lowest lane among equal
    maxima, strict `>` across warps).  Returns int32 [B][k]."""
    s = np.atleast_2d(as_f64(scores))
    B, E = s.shape
    ids = np.arange(E)
    out = np.empty((B, k), np.int32)
    for b in range(B):
        order = np.lexsort((ids, -s[b]))     # primary: −score, secondary: id
        out[b] = order[:k]
    return out


def route(logits, k, renorm=False):
    """Softmax router with top-k choice.  The weight of a chosen expert is its
    softmax probability; with ``renorm`` the k weights are divided by their sum
    (the `norm` switch of `pb_route`).  Returns (sel int32 [B][k], w f64 [B][k])."""
    p = softmax(logits)
    sel = topk(p, k)
    w = np.take_along_axis(p, sel.astype(np.int64), axis=1)
    if renorm:
        w = w / w.sum(axis=1, keepdims=True)
    return sel, w


def group(sel, E):
    """Per-expert grouping of the pass's selections (nemotron_prefill.rs
    `pb_lists`): for expert e, the entries j = b·k + s with sel[b][s] = e in
    ascending j.  Returned in CSR form: counts int32 [E], exclusive offsets int32
    [E+1], entries int32 [B·k] (expert-major)."""
    flat = np.asarray(sel, np.int64).reshape(-1)
    counts = np.zeros(E, np.int32)
    lists = [[] for _ in range(E)]
    for j, e in enumerate(flat):
        lists[e].append(j)
        counts[e] += 1
    offsets = np.zeros(E + 1, np.int32)
    offsets[1:] = np.cumsum(counts)
    entries = np.array([j for e in range(E) for j in lists[e]], np.int32)
    return counts, offsets, entries


def combine(eo, w, k, o=None):
    """Weighted MoE sum (`pb_add_rms`, add=2): m[b] = o[b] + Σ_s w[b][s]·eo[b·k+s],
    slots in ascending order; ``o`` may be None (no shared-expert term)."""
    eo = as_f64(eo)
    w = np.atleast_2d(as_f64(w))
    B = w.shape[0]
    m = np.zeros((B, eo.shape[1])) if o is None else np.atleast_2d(as_f64(o)).copy()
    for s in range(k):
        m += w[:, s:s + 1] * eo[np.arange(B) * k + s]
    return m


def argmax(logits):
    """Per-row argmax with the rules of nemotron_prefill.rs `pb_argmax`: the running
    best starts at −3e38 with index 0 and only a strictly greater value replaces it,
    so the lowest index wins a tie, NaN is never chosen, and a row with nothing
    above −3e38 gives 0.  Returns int32 [B]."""
    l = np.atleast_2d(as_f64(logits))
    out = np.zeros(l.shape[0], np.int32)
    for b in range(l.shape[0]):
        row = l[b]
        ok = row > ARGMAX_FLOOR                 # False for NaN too
        if ok.any():
            m = row[ok].max()
            out[b] = int(np.flatnonzero(ok & (row == m))[0])
    return out


# ----------------------------------------------------------------- test utility
def quantize_q8(W):
    """Test utility, not part of the path (the pages define no quantizer): per
    32-block, offset o = (max+min)/2 and scale s = (max−min)/254, both rounded to
    binary16, then q = clamp(round-half-even((w − o)/s), −127, 127).  Returns
    (codes int8, params binary16 [rows][cols/32][2])."""
    W = as_f64(W)
    rows, cols = W.shape
    blk = W.reshape(rows, cols // QBLOCK, QBLOCK)
    mx, mn = blk.max(axis=2), blk.min(axis=2)
    o16 = ((mx + mn) / 2).astype(np.float16)
    s16 = ((mx - mn) / 254).astype(np.float16)
    s = as_f64(s16)
    s_safe = np.where(s > 0, s, 1.0)
    q = np.rint((blk - as_f64(o16)[:, :, None]) / s_safe[:, :, None])
    q = np.where(s[:, :, None] > 0, q, 0.0)
    codes = np.clip(q, -127, 127).astype(np.int8).reshape(rows, cols)
    params = np.stack([s16, o16], axis=2)
    return codes, params


# ----------------------------------------------------------------- workloads
def tiny_mlp(h, W_up, W_down, gamma, eps):
    """Tiny decode MLP block: y = h + W_down·relu²(W_up·(rms(h)·γ)).  Returns the
    stages and the error scale of each projection."""
    n, inv = rmsnorm(h, gamma, eps)
    up, e_up = gemv_f16(W_up, n)
    u = relu2(up)
    dn, e_dn = gemv_f16(W_down, u)
    y = np.atleast_2d(as_f64(h)) + dn
    return dict(n=n, inv=inv, up=up, e_up=e_up, u=u, down=dn, e_down=e_dn, y=y)


def q8_decode_layer(x, x_o, gamma, eps, mats, u_in=None):
    """q8 decode layer, one position: n = rms(x)·γ feeds q, k, v and up; o reads its
    own input x_o (the attention output, not part of this path); down reads
    u = relu²(up) (or ``u_in`` when checking stage-wise).  ``mats`` maps slot →
    (codes, params)."""
    n, inv = rmsnorm(x, gamma, eps)
    out = dict(n=n, inv=inv)
    for s in ("q", "k", "v", "up"):
        out[s], out["e_" + s] = gemv_q8(*mats[s], n)
    out["o"], out["e_o"] = gemv_q8(*mats["o"], x_o)
    out["u"] = relu2(out["up"])
    out["down"], out["e_down"] = gemv_q8(*mats["down"], out["u"] if u_in is None else u_in)
    return out


def prefill_layer(h, mats, gamma1, gamma2, eps, stage_in=None):
    """One layer of the batched prefill pass over B positions:
    n1 = rms(h)·γ1; [q, k, v] = W·n1; the attention output is stood in for by q;
    h1 = h + W_o·q; n2 = rms(h1)·γ2; u = relu²(W_up·n2); h2 = h1 + W_down·u.
    ``stage_in`` (optional) replaces each stage's input by a given array (keys
    'q', 'h1', 'u') so that every stage can be checked on its own."""
    si = stage_in or {}
    h = np.atleast_2d(as_f64(h))
    n1, inv1 = rmsnorm(h, gamma1, eps)
    out = dict(n1=n1, inv1=inv1)
    for s in ("q", "k", "v"):
        out[s], out["e_" + s] = gemv_q8(*mats[s], n1)
    q_in = si.get("q", out["q"])
    out["o"], out["e_o"] = gemv_q8(*mats["o"], q_in)
    h1 = h + out["o"]
    out["h1"] = h1
    h1_in = np.atleast_2d(as_f64(si.get("h1", h1)))
    n2, inv2 = rmsnorm(h1_in, gamma2, eps)
    out["n2"], out["inv2"] = n2, inv2
    out["up"], out["e_up"] = gemv_q8(*mats["up"], n2)
    out["u"] = relu2(out["up"])
    u_in = si.get("u", out["u"])
    out["down"], out["e_down"] = gemv_q8(*mats["down"], u_in)
    out["h2"] = h1_in + out["down"]
    return out


def moe_layer(h, gamma1, gamma2, eps, router, experts, k, renorm=False, stage_in=None):
    """MoE prefill layer over B positions:
    n = rms(h)·γ1; logits = R·n; (sel, w) = softmax top-k; grouping per expert;
    for each entry j: u_j = relu²(up_e(n[j // k])), eo_j = down_e(u_j);
    m[b] = Σ_s w[b][s]·eo[b·k+s]; h' = h + m; y = rms(h')·γ2.
    ``experts[e]`` = (up_codes, up_params, down_codes, down_params) in the block format,
    or (up_codes, up_row_scale, up_col_field, down_codes, down_row_scale, down_col_field)
    in the q8_2f format (nemotron_prefill.rs's q8_2f bank payload of `pb_q8_bank`).
    ``stage_in`` may give 'sel', 'w', 'u', 'eo' to check stages on their own."""
    si = stage_in or {}
    h = np.atleast_2d(as_f64(h))
    B = h.shape[0]
    E = len(experts)
    n, inv = rmsnorm(h, gamma1, eps)
    logits, e_logits = project(as_f64(router), n)
    sel, w = route(logits, k, renorm)
    sel_in = np.asarray(si.get("sel", sel))
    w_in = as_f64(si.get("w", w))
    counts, offsets, entries = group(sel_in, E)
    rows_up = experts[0][0].shape[0]
    hid = h.shape[1]
    up = np.zeros((B * k, rows_up))
    e_up = np.zeros((B * k, rows_up))
    eo = np.zeros((B * k, hid))
    e_eo = np.zeros((B * k, hid))
    u_given = si.get("u")
    for e in range(E):
        js = entries[offsets[e]:offsets[e + 1]]
        if len(js) == 0:
            continue
        if len(experts[e]) == 6:
            uc, urs, ucf, dc, drs, dcf = experts[e]
            up_proj = lambda x: gemv_q82f(uc, urs, ucf, x)    # noqa: E731
            down_proj = lambda x: gemv_q82f(dc, drs, dcf, x)  # noqa: E731
        else:
            uc, up_p, dc, dp = experts[e]
            up_proj = lambda x: gemv_q8(uc, up_p, x)          # noqa: E731
            down_proj = lambda x: gemv_q8(dc, dp, x)          # noqa: E731
        y, ey = up_proj(n[js // k])
        up[js], e_up[js] = y, ey
        u_e = relu2(y) if u_given is None else as_f64(u_given)[js]
        y2, ey2 = down_proj(u_e)
        eo[js], e_eo[js] = y2, ey2
    u = relu2(up)
    eo_in = as_f64(si.get("eo", eo))
    m = combine(eo_in, w_in, k)
    h_new = h + m
    y, inv2 = rmsnorm(h_new, gamma2, eps)
    return dict(n=n, inv=inv, logits=logits, e_logits=e_logits, sel=sel, w=w,
                counts=counts, offsets=offsets, entries=entries,
                up=up, e_up=e_up, u=u, eo=eo, e_eo=e_eo, m=m, h=h_new, y=y, inv2=inv2)


def vocab_head(x, gamma, eps, W16):
    """Vocab head: n = rms(x)·γ, logits = W·n, ids = argmax (ties → lowest)."""
    n, inv = rmsnorm(x, gamma, eps)
    logits, e = gemv_f16(W16, n)
    return dict(n=n, inv=inv, logits=logits, e=e, ids=argmax(logits))
