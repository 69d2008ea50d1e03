"""Host-side checks of bench.py: the reference arm's JSON line (it runs the
oracle on the host cores, no GPU) and the rule that a committed ncu summary
gives roofline.traffic only while it matches the kernel source it was taken
on, and only for the workload it covers."""
import hashlib
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def test_reference_arm_prints_the_contract_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                          "--warmup", "1"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["steps"] == 1 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["higher_is_better"] is True and d["value"] > 0
    assert "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"]
    assert cb["value"] == d["value"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def _summary(path, key, sha, traffic):
    with open(path, "w") as f:
        f.write("# summary\n\n%s: %s\ntraffic_bytes_per_launch: %d\n" % (key, sha, traffic))


def test_traffic_follows_the_kernel_source(tmp_path, monkeypatch):
    import bench
    src = tmp_path / "kernel.cu"
    src.write_text("// one kernel\n")
    prof = tmp_path / "profiles"
    prof.mkdir()
    sha = hashlib.sha256(src.read_bytes()).hexdigest()
    _summary(prof / "k.md", "score_source_sha256", sha, 123456)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "PROFILES", {2: ("k.md", str(src), "score_source_sha256")})
    assert bench.profiled_traffic(2) == 123456
    assert bench.profiled_traffic(5) is None          # no summary for that workload
    src.write_text("// one kernel, changed\n")
    assert bench.profiled_traffic(2) is None          # taken on another source
    (prof / "k.md").unlink()
    assert bench.profiled_traffic(2) is None


@pytest.mark.parametrize("idx", [1, 2, 3, 4, 5, "attn", "quantize_q", "write_index_k"])
def test_committed_summaries_name_their_source_and_traffic(idx):
    import bench
    name, src, key = bench.PROFILES[idx]
    txt = open(os.path.join(ROOT, "profiles", name)).read()
    assert key + ":" in txt and "traffic_bytes_per_launch:" in txt
    assert "--clock-control none" in txt and os.path.exists(src)
