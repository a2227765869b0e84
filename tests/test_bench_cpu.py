"""Host-side pieces of bench.py that need no GPU."""
import hashlib
import json

import bench


def test_traffic_is_keyed_by_the_kernel_sources(tmp_path, monkeypatch):
    """The DRAM traffic recorded by a capture is reported only while the
    captured kernel sources are unchanged (key: sha256 of the files' bytes in
    order); after any edit the bench reports no traffic."""
    a, b = tmp_path / "plan.cu", tmp_path / "scan.cu"
    a.write_bytes(b"// plan\n")
    b.write_bytes(b"// scan\n")
    key = hashlib.sha256(a.read_bytes() + b.read_bytes()).hexdigest()
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic.json").write_text(json.dumps({key: {"bytes_per_launch": 123.0}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_for([str(a), str(b)]) == 123.0
    assert bench.traffic_for([str(b), str(a)]) is None     # order is part of the key
    b.write_bytes(b"// scan, edited\n")
    assert bench.traffic_for([str(a), str(b)]) is None

