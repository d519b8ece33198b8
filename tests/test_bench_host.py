"""Host logic of the benchmark that needs no GPU: the per-kernel DRAM traffic
read from a committed ncu summary only while the kernel's sources match the
capture, the source hash over a marked section of a file, the clock sampler's
parsing of nvidia-smi samples (median SM clock, throttle reasons) and the
fallback peaks, and the reference arm's JSON line (it runs on the host cores)."""
import os

import bench


def test_traffic_only_while_the_kernel_sources_match(monkeypatch):
    path = os.path.join(bench.ROOT, "profiles", "decode_layer_kernel_decode_b1.txt")
    committed = None
    with open(path) as f:
        for line in f:
            if line.startswith("bench.traffic_bytes_per_launch:"):
                committed = float(line.split(":", 1)[1])
    assert committed and committed > 3e7
    assert bench.read_traffic("decode_layer_kernel_decode_b1.txt", "bench.traffic_bytes_per_launch") == committed
    monkeypatch.setattr(bench, "src_hash", lambda paths: "0" * 16)
    assert bench.read_traffic("decode_layer_kernel_decode_b1.txt", "bench.traffic_bytes_per_launch") is None
    assert bench.read_traffic("no_such_summary.txt", "bench.traffic_bytes_per_launch") is None


def test_section_hash_follows_only_the_marked_section(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    f = tmp_path / "k.cu"
    spec = [("k.cu", "// begin", "// end")]

    def write(before, inside, after):
        f.write_text(f"{before}\n// begin\n{inside}\n// end\n{after}\n")

    write("a", "kernel v1", "z")
    h1 = bench.src_hash(spec)
    write("b", "kernel v1", "y")  # outside the section
    assert bench.src_hash(spec) == h1
    write("a", "kernel v2", "z")  # inside the section
    assert bench.src_hash(spec) != h1


class _Proc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _sampler_with(tmp_path, rows):
    s = bench.ClockSampler(0)
    s.path = str(tmp_path / "clocks.csv")
    s.f = open(s.path, "w")
    for r in rows:
        s.f.write(", ".join(r) + "\n")
    s.f.flush()
    s.proc = _Proc()
    return s


def test_clock_sampler_median_and_reasons(tmp_path):
    ok = ["0", "2070", "2070", "900.0", "0x0", "Not Active", "Not Active", "Not Active", "Not Active"]
    capped = ["0", "1980", "2070", "1400.0", "0x4", "Not Active", "Not Active", "Not Active", "Active"]
    slow = ["0", "1500", "2070", "800.0", "0x8", "Active", "Not Active", "Not Active", "Not Active"]
    out = _sampler_with(tmp_path, [ok, ok, capped]).stop()
    assert out["sm_mhz"] == 2070.0 and out["sm_max_mhz"] == 2070.0 and out["samples"] == 3
    assert out["reasons"] == ["sw_power_cap"]
    out = _sampler_with(tmp_path, [ok, slow, slow]).stop()
    assert out["sm_mhz"] == 1500.0 and out["reasons"] == ["hw_slowdown"]


def test_clock_sampler_without_nvidia_smi():
    s = bench.ClockSampler(0)
    assert s.stop()["reasons"] == ["nvidia-smi unavailable"]


def test_peaks_fall_back_without_the_measured_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, src = bench.load_peaks()
    assert src == "fallback" and peaks["hbm_gbs"] > 0
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"hbm_gbs": 1234.0, "bf16_tflops": 1.0}')
    peaks, src = bench.load_peaks()
    assert src == "measured" and peaks["hbm_gbs"] == 1234.0


def test_reference_arm_prints_one_contract_line():
    # the reference arm is the oracle on the host cores: it runs here too
    import json
    import subprocess
    import sys

    env = dict(os.environ)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        env.pop(k, None)
    out = subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "3"], capture_output=True, text=True, timeout=600, env=env,
                         cwd=bench.ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    r = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in r, key
    assert r["impl"] == "reference" and r["steps"] == 1 and r["warmup"] == 3 and r["n_gpus"] == 1
    assert r["value"] > 0 and r["higher_is_better"] is True and r["unit"] == "tokens/s"
    assert r["config"]["workload"].startswith("decode_b1_resident")
    cb = r["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == r["value"] and cb["cores"] >= 1 and cb["sample"]
    assert r["e2e"] == {"value": r["value"], "unit": r["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
