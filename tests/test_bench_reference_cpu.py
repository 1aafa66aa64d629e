"""The reference arm of bench.py (the CPU oracle, timed on the host cores) prints one
JSON line with the contract's fields; it needs no GPU."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                          "--steps", "2", "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["metric"].startswith("decoded tokens/s") and d["value"] > 0 and d["steps"] == 2
    assert d["config"]["workload"] == "tiny"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_kernel_roofline_takes_the_side_that_needs_more_time():
    sys.path.insert(0, ROOT)
    import bench

    # host bytes dominate: 0.95 GB at 211 GB/s (4.5 ms) vs 5.26 GB at 6812.7 GB/s (0.77 ms)
    r = bench.kernel_roofline(5.26e9, 0.95e9, 4.766, 6812.7, 211.1)
    assert r["bound"] == "host-link" and r["peak"] == 211.1
    assert abs(r["frac"] - 0.95e9 / 4.766e-3 / 211.1e9) < 1e-12
    assert abs(r["frac_hbm"] - 5.26e9 / 4.766e-3 / 6812.7e9) < 1e-12
    # a pool of 2-bit codes and no persistent copies: HBM bytes dominate
    r = bench.kernel_roofline(6.0e9, 0.02e9, 2.0, 6812.7, 211.1)
    assert r["bound"] == "hbm" and r["achieved"] == r["hbm_gbs"] and r["frac"] == r["frac_hbm"]
