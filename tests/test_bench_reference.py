"""bench.py's reference arm (the float64 oracle on the host cores) prints one
JSON line with the keys the benchmark contract asks for (CPU only)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "1", "--ref-budget", "0.3"], capture_output=True, text=True, timeout=600,
                       cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "dtype", "data", "config", "cpu_baseline", "e2e", "gpu_launches"):
        assert k in d, k
    assert d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 1 and d["higher_is_better"] is True
    assert d["gpu_launches"] == 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
    assert "workload" in d["config"]


def test_kernel_digest_ignores_comments_only():
    """The digest that vouches for the committed DRAM counters changes with
    the code, not with its comments or layout."""
    sys.path.insert(0, ROOT)
    import bench
    base = 'int f(int x) { // twice\n  return 2 * x; /* doubled */ }\nconst char *s = "a // b /* c */";\n'
    assert bench._code_only(base) == bench._code_only(base.replace("// twice", "// two times"))
    assert bench._code_only(base) == bench._code_only(base.replace("/* doubled */", "").replace("  ", "    "))
    assert bench._code_only(base) != bench._code_only(base.replace("2 * x", "3 * x"))
    assert '"a // b /* c */"' in bench._code_only(base)  # literals are code
    assert bench._code_only("char c = '\"'; int y; // z") == "char c = '\"'; int y;"
    assert len(bench.kernel_digest()) == 16
