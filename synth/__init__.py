"""Seeded synthetic inputs shared by the oracle side and the CUDA side of the tests
and by the benchmark.

This module draws random numbers and casts them to the storage types of the
weight formats (int8 codes, binary16 scales/offsets, binary16 matrices, f32
activations).  It holds none of the method's arithmetic: no dequantization, no
products, no norms.  Every tensor is addressed by a ``(workload, tensor)`` seed
pair so that any tensor can be regenerated on its own.

Two backends give the same *recipe* (distribution, shape, dtype, layout) but not
the same values:

* ``"numpy"`` — ``numpy.random.default_rng(SeedSequence([workload, tensor]))``,
  on the host.  Used for every case the oracle evaluates in full.
* ``"torch"`` — a ``torch.Generator`` on the given device seeded from the same
  pair.  Used for the full-size workloads (gigabytes of weights), which a host
  generator would take minutes to draw; the oracle then reads the sampled rows it
  needs back from the device copy of these *inputs*.

Recipe (distributions as the workload descriptions state them; ``N(0, v)`` with a
``1/in_dim`` argument is a variance, the usual initialisation convention, while the
literal ``N(0,40)`` of the codes and ``N(0,1e-3)`` of the offsets are standard
deviations — codes clipped to the int8 range only make sense at a spread of 40):

* q8 block format: int8 codes ``[rows][cols]`` = round-half-even(N(0, 40²)) clipped
  to [-127, 127]; params binary16 ``[rows][cols/32][2]`` = (scale ~ U(1e-3, 4e-3),
  offset ~ N(0, (1e-3)²)).
* f16 matrices ``[rows][cols]`` ~ N(0, 1/cols) rounded to binary16.
* activations f32 ~ N(0, 1); RMSNorm weights gamma f32 ~ U(0.5, 1.5); eps = 1e-6.
"""
from __future__ import annotations

import numpy as np

QBLOCK = 32          # columns per (scale, offset) block of the q8 format
CODE_STD = 40.0
CODE_CLIP = 127
SCALE_LO, SCALE_HI = 1e-3, 4e-3
OFFSET_STD = 1e-3
CF_LO, CF_HI = 0.5, 1.5   # q8_2f column field (the pages give no distribution)
EPS = 1e-6

# tensor ids inside one workload seed space
T_X, T_XO, T_GAMMA, T_GAMMA2, T_ROUTER, T_WUP, T_WDOWN, T_W = 1, 2, 3, 4, 5, 6, 7, 8
# q8 matrices of a decode layer: tensor id = 100 + 10*layer + slot
Q8_SLOTS = ("q", "k", "v", "o", "up", "down")


def q8_tensor_id(layer: int, slot: str) -> int:
    return 100 + 10 * layer + Q8_SLOTS.index(slot)


def expert_tensor_id(expert: int, which: str) -> int:
    return 100_000 + 2 * expert + (0 if which == "up" else 1)


def _np_rng(workload: int, tensor: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(workload), int(tensor)]))


def _torch_gen(workload: int, tensor: int, device):
    import torch
    g = torch.Generator(device=device)
    # a fixed mixing of the pair into one 63-bit seed
    g.manual_seed((int(workload) * 1_000_003 + int(tensor) * 7_919 + 12_345) & ((1 << 63) - 1))
    return g


# ---------------------------------------------------------------- primitives
def normal(shape, std, workload, tensor, backend="numpy", device=None, dtype="f32"):
    """N(0, std²) values of ``shape``; dtype 'f32' or 'f16'."""
    if backend == "numpy":
        v = _np_rng(workload, tensor).standard_normal(shape) * std
        return v.astype(np.float32 if dtype == "f32" else np.float16)
    import torch
    g = _torch_gen(workload, tensor, device)
    v = torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std
    return v if dtype == "f32" else v.to(torch.float16)


def uniform(shape, lo, hi, workload, tensor, backend="numpy", device=None):
    if backend == "numpy":
        return _np_rng(workload, tensor).uniform(lo, hi, shape).astype(np.float32)
    import torch
    g = _torch_gen(workload, tensor, device)
    return torch.rand(shape, generator=g, device=device, dtype=torch.float32) * (hi - lo) + lo


def q8_matrix(rows, cols, workload, tensor, backend="numpy", device=None):
    """(codes int8 [rows][cols], params binary16 [rows][cols/32][2] = (scale, offset))."""
    assert cols % QBLOCK == 0
    nb = cols // QBLOCK
    if backend == "numpy":
        r = _np_rng(workload, tensor)
        codes = np.clip(np.rint(r.standard_normal((rows, cols)) * CODE_STD), -CODE_CLIP, CODE_CLIP)
        codes = codes.astype(np.int8)
        params = np.empty((rows, nb, 2), np.float16)
        params[..., 0] = r.uniform(SCALE_LO, SCALE_HI, (rows, nb)).astype(np.float16)
        params[..., 1] = (r.standard_normal((rows, nb)) * OFFSET_STD).astype(np.float16)
        return codes, params
    import torch
    g = _torch_gen(workload, tensor, device)
    codes = torch.empty((rows, cols), dtype=torch.int8, device=device)
    step = max(1, (1 << 26) // cols)            # bound the f32 temporary to 256 MB
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        t = torch.randn((r1 - r0, cols), generator=g, device=device) * CODE_STD
        codes[r0:r1] = torch.round(t).clamp_(-CODE_CLIP, CODE_CLIP).to(torch.int8)
    params = torch.empty((rows, nb, 2), dtype=torch.float16, device=device)
    params[..., 0] = (torch.rand((rows, nb), generator=g, device=device)
                      * (SCALE_HI - SCALE_LO) + SCALE_LO).to(torch.float16)
    params[..., 1] = (torch.randn((rows, nb), generator=g, device=device) * OFFSET_STD).to(torch.float16)
    return codes, params


def q82f_matrix(rows, cols, workload, tensor, backend="numpy", device=None):
    """q8_2f matrix: (codes int8 [rows][cols] as q8_matrix draws them, row_scale
    binary16 [rows] ~ U(SCALE_LO, SCALE_HI), col_field binary16 [cols] ~ U(CF_LO, CF_HI))."""
    if backend == "numpy":
        r = _np_rng(workload, tensor)
        codes = np.clip(np.rint(r.standard_normal((rows, cols)) * CODE_STD), -CODE_CLIP, CODE_CLIP)
        codes = codes.astype(np.int8)
        rs = r.uniform(SCALE_LO, SCALE_HI, rows).astype(np.float16)
        cf = r.uniform(CF_LO, CF_HI, cols).astype(np.float16)
        return codes, rs, cf
    import torch
    g = _torch_gen(workload, tensor, device)
    codes = torch.empty((rows, cols), dtype=torch.int8, device=device)
    step = max(1, (1 << 26) // cols)
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        t = torch.randn((r1 - r0, cols), generator=g, device=device) * CODE_STD
        codes[r0:r1] = torch.round(t).clamp_(-CODE_CLIP, CODE_CLIP).to(torch.int8)
    rs = (torch.rand(rows, generator=g, device=device) * (SCALE_HI - SCALE_LO) + SCALE_LO).to(torch.float16)
    cf = (torch.rand(cols, generator=g, device=device) * (CF_HI - CF_LO) + CF_LO).to(torch.float16)
    return codes, rs, cf


def q82f_layer(workload, layer, hidden, kv, inter, backend="numpy", device=None):
    """The six projections of a decode layer in the q8_2f format: {slot: (codes, rs, cf)}."""
    return {s: q82f_matrix(r, c, workload, q8_tensor_id(layer, s) + 500, backend, device)
            for s, (r, c) in q8_layer_shapes(hidden, kv, inter).items()}


def f16_matrix(rows, cols, workload, tensor, backend="numpy", device=None):
    """binary16 [rows][cols] ~ N(0, 1/cols)."""
    if backend == "numpy":
        return normal((rows, cols), 1.0 / np.sqrt(cols), workload, tensor, "numpy", dtype="f16")
    import torch
    g = _torch_gen(workload, tensor, device)
    out = torch.empty((rows, cols), dtype=torch.float16, device=device)
    step = max(1, (1 << 26) // cols)
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        out[r0:r1] = (torch.randn((r1 - r0, cols), generator=g, device=device)
                      / float(np.sqrt(cols))).to(torch.float16)
    return out


def gamma(n, workload, tensor=T_GAMMA, backend="numpy", device=None):
    return uniform((n,), 0.5, 1.5, workload, tensor, backend, device)


# ---------------------------------------------------------------- workloads
# Full sizes of the five workloads; tests shrink them through the keyword args.
TINY_MLP = dict(workload=0, hidden=512, inter=2048)
Q8_LAYER = dict(workload=1, hidden=4096, kv=1024, inter=14336)
PREFILL = dict(workload=2, B=64, layers=32, hidden=4096, kv=1024, inter=14336)
MOE = dict(workload=3, B=64, hidden=2688, inter=1856, experts=128, topk=6)
VOCAB = dict(workload=4, vocab=262144, hidden=4096)


def q8_layer_shapes(hidden, kv, inter):
    return {"q": (hidden, hidden), "k": (kv, hidden), "v": (kv, hidden),
            "o": (hidden, hidden), "up": (inter, hidden), "down": (hidden, inter)}


def q8_layer(workload, layer, hidden, kv, inter, backend="numpy", device=None):
    """The six q8 projections of one decode layer: {slot: (codes, params)}."""
    return {s: q8_matrix(r, c, workload, q8_tensor_id(layer, s), backend, device)
            for s, (r, c) in q8_layer_shapes(hidden, kv, inter).items()}


def q8_bank(E, rows, cols, workload, which, backend="numpy", device=None):
    """Contiguous bank of E q8 matrices (codes [E][rows][cols], params
    [E][rows][cols/32][2]); expert e drawn from seed (workload, expert_tensor_id(e, which))."""
    if backend == "numpy":
        cs, ps = zip(*[q8_matrix(rows, cols, workload, expert_tensor_id(e, which)) for e in range(E)])
        return np.stack(cs), np.stack(ps)
    import torch
    codes = torch.empty((E, rows, cols), dtype=torch.int8, device=device)
    params = torch.empty((E, rows, cols // QBLOCK, 2), dtype=torch.float16, device=device)
    for e in range(E):
        c, p = q8_matrix(rows, cols, workload, expert_tensor_id(e, which), "torch", device)
        codes[e].copy_(c)
        params[e].copy_(p)
    return codes, params


def q82f_bank(E, rows, cols, workload, which, backend="numpy", device=None):
    """Contiguous bank of E q8_2f matrices (codes [E][rows][cols], row scales [E][rows],
    column fields [E][cols]); expert e drawn as q82f_matrix from seed (workload,
    expert_tensor_id(e, which) + 500)."""
    if backend == "numpy":
        cs, rs, cf = zip(*[q82f_matrix(rows, cols, workload, expert_tensor_id(e, which) + 500) for e in range(E)])
        return np.stack(cs), np.stack(rs), np.stack(cf)
    import torch
    codes = torch.empty((E, rows, cols), dtype=torch.int8, device=device)
    rs = torch.empty((E, rows), dtype=torch.float16, device=device)
    cf = torch.empty((E, cols), dtype=torch.float16, device=device)
    for e in range(E):
        c, r, f = q82f_matrix(rows, cols, workload, expert_tensor_id(e, which) + 500, "torch", device)
        codes[e].copy_(c)
        rs[e].copy_(r)
        cf[e].copy_(f)
    return codes, rs, cf


def moe_q82f_layer(workload, E, hidden, inter, backend="numpy", device=None):
    """Router (as moe_layer) and the up / down expert banks in the q8_2f format."""
    router = normal((E, hidden), 1.0 / np.sqrt(hidden), workload, T_ROUTER, backend, device)
    up = q82f_bank(E, inter, hidden, workload, "up", backend, device)
    down = q82f_bank(E, hidden, inter, workload, "down", backend, device)
    return router, up, down


def moe_layer(workload, E, hidden, inter, backend="numpy", device=None):
    """Router f32 [E][hidden] ~ N(0, 1/hidden) and the up / down expert banks."""
    router = normal((E, hidden), 1.0 / np.sqrt(hidden), workload, T_ROUTER, backend, device)
    up = q8_bank(E, inter, hidden, workload, "up", backend, device)
    down = q8_bank(E, hidden, inter, workload, "down", backend, device)
    return router, up, down
