"""Host logic of bench.py that needs no GPU: the DRAM traffic figure of a launch comes
from a committed ncu capture only while the kernel's sources are the ones captured,
and the committed figures are plausible for the launches they describe."""
import importlib.util
import json
import os

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_host_mod", os.path.join(ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    return b


def test_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    b = _bench()
    csrc = tmp_path / "prefill_gemv_q8_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "k.cu").write_text("__global__ void k() {}\n")
    (csrc / "h.cuh").write_text("// header\n")
    monkeypatch.setattr(b, "ROOT", str(tmp_path))
    files = ["k.cu", "h.cuh"]
    # no capture file: no figure
    assert b.ncu_traffic("launch", files) is None
    entry = {"source_sha": b.source_sha(files), "dram_bytes_per_launch": 123456}
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(json.dumps({"launch": entry}))
    assert b.ncu_traffic("launch", files) == 123456
    assert b.ncu_traffic("other", files) is None
    # any change to any of the kernel's files, or to their order, voids the figure
    (csrc / "h.cuh").write_text("// header, edited\n")
    assert b.ncu_traffic("launch", files) is None
    (csrc / "h.cuh").write_text("// header\n")
    assert b.ncu_traffic("launch", files) == 123456
    assert b.ncu_traffic("launch", files[::-1]) is None


def test_committed_traffic_is_plausible():
    """Each committed figure (DRAM read + write bytes of one launch) is at least the
    launch's algorithmic weight bytes and at most 10 % above them: every weight byte is
    read, and little else (inputs, outputs, partials) is moved."""
    import prefill_gemv_q8_gb300 as pgq

    d = json.load(open(os.path.join(ROOT, "profiles", "ncu_traffic.json")))
    c = synth.Q8_LAYER
    shp = synth.q8_layer_shapes(c["hidden"], c["kv"], c["inter"])
    q8 = lambda names: sum(r * k for n, (r, k) in shp.items() if n in names) * 9 // 8
    launch1 = q8({"q", "k", "v", "o", "up"})                # norm + q,k,v,o,up of the decode layer
    p = synth.PREFILL
    shp_p = synth.q8_layer_shapes(p["hidden"], p["kv"], p["inter"])
    per_layer = sum(r * k for r, k in shp_p.values()) * 9 // 8
    pass_launch = per_layer * pgq.PASS_LMAX                 # one persistent launch of the pass
    for key, alg in (("gemv_q8_layer_multi", launch1), ("prefill_pass_launch", pass_launch)):
        v = d[key]["dram_bytes_per_launch"]
        assert alg <= v <= 1.10 * alg, (key, v, alg)
        assert len(d[key]["source_sha"]) == 16
