"""The benchmark's JSON line, checked on the CPU through its reference arm (the
oracle timed on the host): one line with the contract's keys and types."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "1"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 1
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["vs_baseline"] is None and d["data"] == "synthetic"
    assert "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_breakdown_rows_are_calls_the_library_takes():
    # every breakdown row names a format and shape the library's own host-side
    # queries accept for the path the row's tag selects (no GPU): the
    # quantized-activation rows get a workspace size, the path-B rows (the MX
    # formats with a workspace) too, and every format is one of the library's
    sys.path.insert(0, ROOT)
    import bench
    import block_scaled_quantized_spec_gb300 as q
    from block_scaled_quantized_spec_gb300 import build
    build.build()
    q.load()
    for row in bench.BREAKDOWN:
        fmt, m, n, k = row[:4]
        tag = row[4] if len(row) > 4 else "auto"
        assert fmt in q.FORMATS, row
        assert m >= 1 and n >= 1 and k % 32 == 0, row
        if tag == "A8":
            assert q.qmm_a8_workspace_bytes(fmt, m, k) > 0, row
        elif tag == "A4":
            assert q.qmm_a4_workspace_bytes(fmt, m, k) > 0, row
        elif tag == "A":
            assert m > 16 and fmt not in q.SUB_BYTE, row
        else:
            assert tag == "auto", row
    for fmt, m, n, k, e in bench.GATHER + bench.GROUPED:
        assert q.qmm_grouped_workspace_bytes(fmt, m, k, e) > 0
