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



def test_reference_arm_line_on_cpu():
    """`bench.py --impl reference` times the oracle on the host (no GPU) and
    prints one JSON line whose metric, unit and config keys are those of the
    CUDA line, with the contract's cpu_baseline and zero-copy e2e."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                          "--workload", "tiny", "--steps", "1", "--warmup", "3",
                          "--cpu-budget", "0.2"], capture_output=True, text=True, timeout=600,
                         cwd=root)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == "tokens/s"
    assert line["higher_is_better"] is True and line["value"] > 0
    cfg = line["config"]
    assert cfg["workload"] == "tiny" and cfg["variant"] == "forward"
    assert cfg["parallelism"] == "single"
    assert "fits or nearly fits in L2" in cfg["l2"]
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    assert cb["nproc"] >= 1 and cb["cpu_model"]
    e2e = line["e2e"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert e2e["value"] == line["value"]
