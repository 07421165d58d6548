"""The benchmark's reference arm (the fp64 oracle on host cores) prints one
JSON line with the keys of the benchmark contract. CPU only."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "1", "--ref-budget", "2"], capture_output=True, text=True, timeout=600,
                       cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["impl"] == "reference" and line["value"] > 0 and line["steps"] == 2 and line["warmup"] == 1
    assert line["higher_is_better"] is True and line["dtype"] == "f64" and "workload" in line["config"]
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == line["value"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_kernel_hash_ignores_comments(tmp_path, monkeypatch):
    """The DRAM counters in profiles/traffic.json stay valid across comment
    edits of the kernel sources, and not across code edits."""
    import shutil
    sys.path.insert(0, ROOT)
    import bench
    csrc = tmp_path / "up_proj_gemm_gb300" / "csrc"
    shutil.copytree(os.path.join(ROOT, "up_proj_gemm_gb300", "csrc"), csrc)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0, hb = bench.kernel_hashes("fwd"), bench.kernel_hashes("dgrad")
    f = csrc / "fwd.cu"
    src = f.read_text()
    f.write_text("// a new comment line\n/* and a block\n   comment */\n" + src.replace("\n", "\n\n", 3))
    assert bench.kernel_hashes("fwd") == h0
    f.write_text(src.replace("constexpr int kBM = 128;", "constexpr int kBM = 64;"))
    assert bench.kernel_hashes("fwd") != h0
    assert bench.kernel_hashes("dgrad") == hb  # the backward's counters do not depend on fwd.cu
