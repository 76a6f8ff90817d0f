"""The benchmark's layer roofline on CPU: the layer's algorithmic bytes, its intensity and the
roof that binds it (the lower of the bf16 peak and intensity x HBM rate).

The bytes are checked against an inventory of the tensors each step reads or writes once,
listed by shape; the roof is checked on both sides of the ridge."""
import sys

import pytest

from tests.conftest import ROOT

PK = {"hbm_gbs": 6693.8, "bf16_tflops": 1928.8, "bf16_tflops_sustained": 1741.1}


def _bench():
    sys.path.insert(0, ROOT)
    import bench
    return bench


def _inventory(spec, kept):
    """(elements, bytes per element) of every tensor one forward moves once."""
    T, d, N, K, dr, ds = spec.T, spec.d_model, spec.N, spec.K, spec.d_expert, spec.d_shared
    e = spec.elem_bytes
    items = [
        (T * d, e), (N * d, e), (T * K, 4), (T * K, 4),             # router: x, W_r; top-K idx, w
        (T * K, 4), (T * K, 4), (T * K, 4), (T * d, e), (kept * d, e),  # permutation
        (kept * d, e), (N * dr * d, e), (N * dr * d, e), (N * d * dr, e),  # gate/up, down reads
        (kept * dr, e), (kept * dr, e), (kept * d, e),              # h written and read, f written
        (kept * d, e), (T * d, 4), (T * K, 4), (T * K, 4),          # combine: f, y; tables
    ]
    if ds > 0:
        items += [(T * d, e), (ds * d, e), (ds * d, e), (d * ds, e), (T * ds, e), (T * ds, e),
                  (T * d, e), (T * d, e)]                          # shared; g written and read
    return items


@pytest.mark.parametrize("name", ["olmo", "dsv3", "mixtral", "qwen2", "tiny"])
def test_layer_bytes_match_the_tensor_inventory(name):
    from workloads import CONFIGS
    b = _bench()
    spec = CONFIGS[name]
    kept = spec.T * spec.K - 7
    assert b.layer_algorithmic_bytes(spec, kept) == sum(n * s for n, s in _inventory(spec, kept))


def test_layer_roof_is_hbm_below_the_ridge_and_tensor_above():
    from workloads import CONFIGS
    b = _bench()
    dsv3, olmo = CONFIGS["dsv3"], CONFIGS["olmo"]
    r = b.layer_roofline(dsv3, dsv3.T * dsv3.K, 5.7, PK)
    assert r["intensity_flop_per_byte"] < r["ridge_flop_per_byte"]
    assert r["bound"] == "hbm"
    assert r["roof_tflops"] == pytest.approx(r["intensity_flop_per_byte"] * PK["hbm_gbs"] / 1e3)
    assert r["frac"] == pytest.approx(r["achieved_tflops"] / r["roof_tflops"])
    assert r["achieved_tflops"] == pytest.approx(dsv3.expert_flops(dsv3.T * dsv3.K) / 5.7e-3 / 1e12)
    r = b.layer_roofline(olmo, olmo.T * olmo.K, 1.0, PK)
    assert r["bound"] == "tensor" and r["roof_tflops"] == PK["bf16_tflops"]
    assert r["frac"] == pytest.approx(olmo.expert_flops(olmo.T * olmo.K) / 1e-3 / 1e12 / PK["bf16_tflops"])


def test_stage_traffic_is_reported_only_for_the_captured_sources(monkeypatch):
    """The ncu traffic figure comes with the hash of the kernel sources it was captured on:
    the bench reports it while the sources hash to that value and null otherwise (a changed
    kernel has not been measured), and null for a workload without a capture."""
    import hashlib
    import os
    bench = _bench()
    h = hashlib.sha256()
    for f in bench.TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    current = h.hexdigest()[:16]
    monkeypatch.setattr(bench, "STAGE_TRAFFIC", {
        "same": {"sources_sha256": current, "bytes": 123},
        "changed": {"sources_sha256": "0" * 16 if current != "0" * 16 else "1" * 16, "bytes": 456}})
    assert bench.stage_traffic("same") == 123
    assert bench.stage_traffic("changed") is None
    assert bench.stage_traffic("no capture") is None
