"""Host-side arithmetic of bench.py (no GPU): the roofline fields and the
DRAM-traffic records, which must read as unknown (None) once a kernel's
source no longer matches the capture they came from."""
import hashlib
import json
import os

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_roofline_fields():
    r = bench.roofline(611_844_096, 0.36, 6689.5, traffic=592_056_064)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == 6689.5
    assert r["achieved"] == pytest.approx(611_844_096 / 0.36e-3 / 1e9, rel=1e-4)
    assert r["frac"] == pytest.approx(r["achieved"] / 6689.5, abs=1e-4)
    assert r["traffic"] == 592_056_064 and r["algorithmic_bytes"] == 611_844_096


def test_algorithmic_bytes_per_token():
    # q, k, v, out bf16 + g fp32 for 96 heads x 128 channels, beta fp32 per head
    assert bench.BYTES_PER_TOKEN == 96 * 128 * (4 * 2 + 4) + 96 * 4 == 147_840
    assert bench.STATE_BYTES == 96 * 128 * 128 * 4


def test_traffic_records_point_at_sources_and_scale_with_units(monkeypatch, tmp_path):
    records = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    assert records
    for name, e in records.items():
        assert os.path.exists(os.path.join(ROOT, e["source"])), name
        assert e["dram_bytes"] > 0 and e["units"] > 0 and len(e["sha256"]) == 64
    # a record whose source matches scales linearly; one that does not reads None
    src = tmp_path / "k.cu"
    src.write_text("kernel source\n")
    good = {"source": str(src), "sha256": hashlib.sha256(b"kernel source\n").hexdigest(),
            "dram_bytes": 1000, "units": 10}
    stale = dict(good, sha256="0" * 64)
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"a": good, "b": stale}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_for("a", 25) == 2500
    assert bench.traffic_for("b", 25) is None
    assert bench.traffic_for("missing", 25) is None
    src.write_text("kernel source, edited\n")
    assert bench.traffic_for("a", 25) is None


def test_leg_summaries_close_the_line():
    """Every leg's value and roofline fraction sit in the last 1.5 KB of the
    printed line, after the verbose records."""
    rf = lambda f: {"bound": "hbm", "achieved": 1.0, "peak": 2.0, "unit": "GB/s", "frac": f,
                    "traffic": None, "algorithmic_bytes": 1}
    verbose = {"workload": "x" * 400, "roofline": rf(0.5), "note": "y" * 400}
    dec = dict(verbose, value=2097.9, unit="steps/s", ms_per_step=0.4767, roofline=rf(1.03))
    lng = dict(verbose, value=1.0e7, unit="tokens/s", ms_per_step=26.0, roofline=rf(0.22),
               two_kernels={"prologue": {"ms": 3.0}, "prefill": {"ms": 22.1}})
    ext = {name: dict(verbose, value=1.0, unit="u", ms_per_step=1.0, roofline=rf(0.9))
           for name in ("decode_conv", "verify", "output_gate", "packed_documents",
                        "segmented_h8", "segmented_h96")}
    ext["clocks"] = {"sm_mhz": 2070.0}
    legs = bench.legs_summary(dec, lng, ext)
    assert legs["decode"] == {"value": 2097.9, "unit": "steps/s", "ms_per_step": 0.4767, "frac": 1.03}
    assert legs["long_context"]["prefill_alone_ms"] == 22.1
    assert legs["packed_documents"]["frac"] == 0.9
    assert set(legs["extras"]) == {"decode_conv", "verify", "output_gate", "segmented_h8", "segmented_h96"}
    line = {"metric": "m", "value": 1.0, "detail": {"decode": dec, "long_context": lng, "extras": ext},
            "legs": legs}
    tail = json.dumps(line)[-1500:]
    assert '"decode": {"value": 2097.9' in tail and '"frac": 1.03' in tail
    assert '"long_context": {"value": 10000000.0' in tail
