"""Plant plausible mistakes in the oracle (on the CPU, by monkeypatching) and check
that at least one pin catches each: the pins are strong enough to trust."""
import numpy as np
import pytest

import oracle.ref as R
from oracle_pins import PINS

_orig = {k: getattr(R, k) for k in ("dequant_q8", "project", "rmsnorm", "relu2", "softmax",
                                    "topk", "route", "group", "combine", "argmax", "dequant_q82f",
                                    "add_rmsnorm_ex", "sandwich")}


def _dequant_no_offset(codes, params):
    rows, cols = np.asarray(codes).shape
    p = R.as_f64(params).reshape(rows, cols // 32, 2)
    q = R.as_f64(codes).reshape(rows, cols // 32, 32)
    return (q * p[:, :, 0:1]).reshape(rows, cols)


def _dequant_zero_point(codes, params):
    rows, cols = np.asarray(codes).shape
    p = R.as_f64(params).reshape(rows, cols // 32, 2)
    q = R.as_f64(codes).reshape(rows, cols // 32, 32)
    return ((q - p[:, :, 1:2]) * p[:, :, 0:1]).reshape(rows, cols)


def _dequant_block_index_mod(codes, params):
    # uses block c % nb instead of c // 32
    rows, cols = np.asarray(codes).shape
    nb = cols // 32
    p = R.as_f64(params).reshape(rows, nb, 2)
    idx = np.arange(cols) % nb
    return R.as_f64(codes) * p[:, idx, 0] + p[:, idx, 1]


def _dequant_block_16(codes, params):
    # blocks of 16 columns
    rows, cols = np.asarray(codes).shape
    nb = cols // 32
    p = R.as_f64(params).reshape(rows, nb, 2)
    idx = np.minimum(np.arange(cols) // 16, nb - 1)
    return R.as_f64(codes) * p[:, idx, 0] + p[:, idx, 1]


def _project_transposed(W, X):
    W = R.as_f64(W)
    X = np.atleast_2d(R.as_f64(X))
    if W.shape[0] == W.shape[1]:
        return X @ W, np.abs(X) @ np.abs(W)
    return _orig["project"](W, X)


def _project_abs_wrong(W, X):
    y, e = _orig["project"](W, X)
    return y, np.abs(y)


def _rms_eps_outside(h, gamma, eps):
    h = np.atleast_2d(R.as_f64(h))
    inv = 1.0 / (np.sqrt(np.mean(h * h, axis=1)) + eps)
    return h * inv[:, None] * R.as_f64(gamma)[None, :], inv


def _rms_sum_not_mean(h, gamma, eps):
    h = np.atleast_2d(R.as_f64(h))
    inv = 1.0 / np.sqrt(np.sum(h * h, axis=1) + eps)
    return h * inv[:, None] * R.as_f64(gamma)[None, :], inv


def _rms_no_gamma(h, gamma, eps):
    y, inv = _orig["rmsnorm"](h, np.ones_like(R.as_f64(gamma)), eps)
    return y, inv


def _relu_not_squared(v):
    return np.maximum(R.as_f64(v), 0.0)


def _square_no_relu(v):
    return R.as_f64(v) ** 2


def _softmax_unshifted(l):
    l = np.atleast_2d(R.as_f64(l))
    with np.errstate(over="ignore", invalid="ignore"):
        z = np.exp(l)
        return z / z.sum(axis=1, keepdims=True)


def _topk_ties_high(scores, k):
    s = np.atleast_2d(R.as_f64(scores))
    ids = np.arange(s.shape[1])
    return np.array([np.lexsort((-ids, -row))[:k] for row in s], np.int32)


def _route_always_renorm(logits, k, renorm=False):
    return _orig["route"](logits, k, True)


def _group_descending(sel, E):
    c, o, e = _orig["group"](sel, E)
    e = e.copy()
    for i in range(E):
        e[o[i]:o[i + 1]] = e[o[i]:o[i + 1]][::-1]
    return c, o, e


def _combine_slot_reversed(eo, w, k, o=None):
    return _orig["combine"](eo, np.atleast_2d(R.as_f64(w))[:, ::-1], k, o)


def _argmax_last(l):
    l = np.atleast_2d(R.as_f64(l))
    out = []
    for row in l:
        ok = row > R.ARGMAX_FLOOR
        out.append(int(np.flatnonzero(ok & (row == row[ok].max()))[-1]) if ok.any() else 0)
    return np.array(out, np.int32)


def _argmax_numpy(l):
    return np.argmax(np.atleast_2d(R.as_f64(l)), axis=1).astype(np.int32)


_layer = {k: getattr(R, k) for k in ("q8_decode_layer", "prefill_layer", "moe_layer")}


def _decode_o_reads_n(x, x_o, gamma, eps, mats, u_in=None):
    n, _ = _orig["rmsnorm"](x, gamma, eps)
    return _layer["q8_decode_layer"](x, n, gamma, eps, mats, u_in)


def _decode_down_reads_up(x, x_o, gamma, eps, mats, u_in=None):
    first = _layer["q8_decode_layer"](x, x_o, gamma, eps, mats)
    return _layer["q8_decode_layer"](x, x_o, gamma, eps, mats, u_in=first["up"])


def _decode_k_v_swapped(x, x_o, gamma, eps, mats, u_in=None):
    m = dict(mats)
    m["k"], m["v"] = mats["v"], mats["k"]
    return _layer["q8_decode_layer"](x, x_o, gamma, eps, m, u_in)


def _prefill_o_reads_n1(h, mats, gamma1, gamma2, eps, stage_in=None):
    n1, _ = _orig["rmsnorm"](np.atleast_2d(np.asarray(h, np.float64)), gamma1, eps)
    return _layer["prefill_layer"](h, mats, gamma1, gamma2, eps, stage_in={"q": n1})


def _prefill_second_norm_reads_h(h, mats, gamma1, gamma2, eps, stage_in=None):
    return _layer["prefill_layer"](h, mats, gamma1, gamma2, eps, stage_in={"h1": h})


def _prefill_h2_from_h(h, mats, gamma1, gamma2, eps, stage_in=None):
    out = _layer["prefill_layer"](h, mats, gamma1, gamma2, eps, stage_in)
    out["h2"] = np.atleast_2d(np.asarray(h, np.float64)) + out["down"]
    return out


def _moe_residual_from_n(h, gamma1, gamma2, eps, router, experts, k, renorm=False, stage_in=None):
    out = _layer["moe_layer"](h, gamma1, gamma2, eps, router, experts, k, renorm, stage_in)
    out["h"] = out["n"] + out["m"]
    return out


def _moe_second_norm_gamma1(h, gamma1, gamma2, eps, router, experts, k, renorm=False, stage_in=None):
    return _layer["moe_layer"](h, gamma1, gamma1, eps, router, experts, k, renorm, stage_in)


def _moe_second_norm_no_gamma(h, gamma1, gamma2, eps, router, experts, k, renorm=False, stage_in=None):
    out = _layer["moe_layer"](h, gamma1, gamma2, eps, router, experts, k, renorm, stage_in)
    out["y"] = out["y"] / np.asarray(gamma2, np.float64)[None, :]
    return out


def _q82f_scales_swapped(codes, row_scale, col_field):
    # the row scale read per column and the column field per row (square blocks only)
    q = R.as_f64(codes)
    rows, cols = q.shape
    rs = R.as_f64(row_scale).reshape(-1)
    cf = R.as_f64(col_field).reshape(-1)
    return cf[:rows, None] * q * rs[None, :cols] if rows <= cols else cf[:, None] * q * rs[None, :cols]


def _q82f_no_col_field(codes, row_scale, col_field):
    return _orig["dequant_q82f"](codes, row_scale, np.ones_like(R.as_f64(col_field)))


def _q82f_col_field_shifted(codes, row_scale, col_field):
    cf = np.roll(R.as_f64(col_field).reshape(-1), 1)
    return _orig["dequant_q82f"](codes, row_scale, cf)


def _add_norm_ex_scale_before_add(h, add, gamma, eps, scale=None, gemma=False):
    h = np.atleast_2d(R.as_f64(h))
    if scale:
        h = h * float(scale)
    if add is not None:
        h = h + np.atleast_2d(R.as_f64(add))
    w = R.as_f64(gamma) + (1.0 if gemma else 0.0)
    y, inv = R.rmsnorm(h, w, eps)
    return h, y, inv


def _add_norm_ex_gemma_ignored(h, add, gamma, eps, scale=None, gemma=False):
    return _orig["add_rmsnorm_ex"](h, add, gamma, eps, scale, False)


def _sandwich_first_norm_w2(x, w1, h, w2, eps, scale=None, gemma=False):
    return _orig["sandwich"](x, w2, h, w2, eps, scale, gemma)


def _sandwich_adds_raw_x(x, w1, h, w2, eps, scale=None, gemma=False):
    out = _orig["sandwich"](x, w1, h, w2, eps, scale, gemma)
    hn, n, inv2 = _orig["add_rmsnorm_ex"](h, x, w2, eps, scale, gemma)
    out.update(h=hn, n=n, inv2=inv2)
    return out


MUTATIONS = {
    "dequant drops the offset": ("dequant_q8", _dequant_no_offset),
    "offset read as a zero-point": ("dequant_q8", _dequant_zero_point),
    "block index c % nb": ("dequant_q8", _dequant_block_index_mod),
    "16-column blocks": ("dequant_q8", _dequant_block_16),
    "transposed weight operand": ("project", _project_transposed),
    "error scale |W x| instead of |W||x|": ("project", _project_abs_wrong),
    "eps outside the root": ("rmsnorm", _rms_eps_outside),
    "sum instead of mean": ("rmsnorm", _rms_sum_not_mean),
    "gamma dropped": ("rmsnorm", _rms_no_gamma),
    "relu not squared": ("relu2", _relu_not_squared),
    "square without relu": ("relu2", _square_no_relu),
    "softmax without max shift": ("softmax", _softmax_unshifted),
    "top-k tie to the higher id": ("topk", _topk_ties_high),
    "router always renormalises": ("route", _route_always_renorm),
    "groups in descending order": ("group", _group_descending),
    "combine with slots reversed": ("combine", _combine_slot_reversed),
    "argmax tie to the last index": ("argmax", _argmax_last),
    "argmax picks NaN / ignores the floor": ("argmax", _argmax_numpy),
    "decode: o reads n instead of its own input": ("q8_decode_layer", _decode_o_reads_n),
    "decode: down reads up instead of relu²(up)": ("q8_decode_layer", _decode_down_reads_up),
    "decode: k and v matrices swapped": ("q8_decode_layer", _decode_k_v_swapped),
    "prefill: o reads n1 instead of q": ("prefill_layer", _prefill_o_reads_n1),
    "prefill: second norm reads h instead of h1": ("prefill_layer", _prefill_second_norm_reads_h),
    "prefill: h2 adds the down output to h": ("prefill_layer", _prefill_h2_from_h),
    "moe: residual added to the normalised input": ("moe_layer", _moe_residual_from_n),
    "moe: second norm weighted by gamma1": ("moe_layer", _moe_second_norm_gamma1),
    "moe: second norm without gamma": ("moe_layer", _moe_second_norm_no_gamma),
    "q8_2f: row scale and column field swapped": ("dequant_q82f", _q82f_scales_swapped),
    "q8_2f: column field dropped": ("dequant_q82f", _q82f_no_col_field),
    "q8_2f: column field off by one column": ("dequant_q82f", _q82f_col_field_shifted),
    "add_rmsnorm_ex: scale applied before the add": ("add_rmsnorm_ex", _add_norm_ex_scale_before_add),
    "add_rmsnorm_ex: gemma switch ignored": ("add_rmsnorm_ex", _add_norm_ex_gemma_ignored),
    "sandwich: first norm weighted by w2": ("sandwich", _sandwich_first_norm_w2),
    "sandwich: residual adds the raw x": ("sandwich", _sandwich_adds_raw_x),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(R, attr, fn)
    failed = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin()
        except (AssertionError, ValueError, IndexError, FloatingPointError):
            failed.append(pin.__name__)
    assert failed, f"no pin catches the mutation: {name}"
