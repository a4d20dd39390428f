"""Host logic of bench.py's measured DRAM traffic: a per-unit figure from an ncu capture is
reported only while the kernel source still has the hash it was captured on."""
import hashlib
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    sys.path.insert(0, ROOT)
    import bench
    return bench


def test_traffic_scales_with_units_while_the_source_matches(tmp_path, monkeypatch):
    bench = _bench()
    src = tmp_path / "kernel.cu"
    src.write_bytes(b"// a kernel\n")
    digest = hashlib.sha256(src.read_bytes()).hexdigest()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setitem(bench.TRAFFIC, "probe", ("kernel.cu", digest, 1500.0))
    assert bench.traffic_bytes("probe", 4) == 6000.0
    assert bench.traffic_bytes("probe", 0) == 0.0


def test_traffic_is_null_once_the_source_changes_or_is_missing(tmp_path, monkeypatch):
    bench = _bench()
    src = tmp_path / "kernel.cu"
    src.write_bytes(b"// a kernel\n")
    digest = hashlib.sha256(src.read_bytes()).hexdigest()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setitem(bench.TRAFFIC, "probe", ("kernel.cu", digest, 1500.0))
    src.write_bytes(b"// a kernel, edited\n")
    assert bench.traffic_bytes("probe", 4) is None
    monkeypatch.setitem(bench.TRAFFIC, "gone", ("no_such_kernel.cu", digest, 1500.0))
    assert bench.traffic_bytes("gone", 4) is None


def test_every_entry_names_a_kernel_source_of_the_package():
    bench = _bench()
    for kind, (path, digest, per_unit) in bench.TRAFFIC.items():
        assert path.startswith("gated_delta_rule_kda_gb300/csrc/") and path.endswith(".cu"), kind
        assert os.path.exists(os.path.join(ROOT, path)), kind
        assert len(digest) == 64 and per_unit > 0, kind
