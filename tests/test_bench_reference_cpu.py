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


def test_step_roofline_sums_each_steps_bound():
    sys.path.insert(0, ROOT)
    import bench

    # one link-bound step (2.111 GB over 211.1 GB/s = 10 ms) and one HBM-bound step
    # (6.8127 GB at 6812.7 GB/s = 1 ms): the ideal run takes 11 ms, 5.5 ms a step; the
    # aggregate form takes max(2.121 GB / 211.1, 6.8227 GB / 6812.7) = 10.05 ms, 5.02 a step
    sb = [(2.111e9, 0.01e9), (0.01e9, 6.8127e9)]
    r = bench.step_roofline(sb, 6.8227e9, 2.121e9, 6.0, 6812.7, 211.1)
    assert abs(r["ideal_ms"] - 5.5) < 1e-9 and abs(r["frac"] - 5.5 / 6.0) < 1e-9
    assert abs(r["aggregate_ideal_ms"] - 0.5 * 2.121e9 / 211.1e9 * 1e3) < 1e-9
    assert r["aggregate_ideal_ms"] < r["ideal_ms"]
    assert r["link_bound_steps"] == 1
    assert r["hbm_bytes_per_step"] == 6.8227e9 / 2 and r["host_bytes_per_step"] == 2.121e9 / 2
    # steps that are all bound on the same side: the two forms agree
    sb = [(1e9, 1e9), (2e9, 1e9), (3e9, 1e9)]
    r = bench.step_roofline(sb, 3e9, 6e9, 20.0, 6812.7, 211.1)
    assert abs(r["ideal_ms"] - r["aggregate_ideal_ms"]) < 1e-12 and r["link_bound_steps"] == 3


def test_profile_traffic_only_for_the_captured_kernel(tmp_path, monkeypatch):
    sys.path.insert(0, ROOT)
    import hashlib

    import bench

    src = tmp_path / "host_offloaded_kv_gb300" / "csrc"
    src.mkdir(parents=True)
    (src / "clo_fused.cu").write_text("// kernel A\n")
    prof = tmp_path / "profiles"
    prof.mkdir()
    digest = hashlib.sha256(b"// kernel A\n").hexdigest()
    (prof / "k_step_fused_w.md").write_text(f"# capture\nsource_sha256: {digest}\ntraffic_bytes_per_launch: 123456\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_from_profiles("k_step_fused", "w") == 123456.0
    assert bench.traffic_from_profiles("k_step_fused", "w_int4") is None  # no capture of that mode
    (src / "clo_fused.cu").write_text("// kernel B\n")  # the kernel changed since the capture
    assert bench.traffic_from_profiles("k_step_fused", "w") is None


def test_committed_profiles_describe_the_committed_kernel():
    # the ncu summaries that give bench.py its traffic figures were taken of this kernel
    sys.path.insert(0, ROOT)
    import bench

    for name in ("llama32k", "llama32k_int4", "llama32k_int2", "qwen512k"):
        assert bench.traffic_from_profiles("k_step_fused", name) is not None, name
