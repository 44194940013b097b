"""The benchmark's reference arm: the CPU oracle timed on a token sample of
the benchmark's workload.  Its JSON line carries the keys of the
benchmark's own line with the same metric, unit and config; ranks other
than 0 of a multi-process launch exit 0 without work."""
import json
import os
import subprocess
import sys

import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(env_extra=None, *args):
    env = dict(os.environ)
    env.update(env_extra or {})
    return subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
         "--steps", "2", "--warmup", "1", "--ref-sample-tokens", "16",
         "--ref-sample-w-rows", "32", *args],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_reference_arm_line():
    r = _run()
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data",
                "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert (d["n_gpus"], d["steps"], d["warmup"]) == (1, 2, 1)
    assert d["unit"] == "us/layer" and d["higher_is_better"] is False
    assert d["value"] > 0 and abs(d["ms_per_step"] * 1e3 - d["value"]) <= 1e-9 * d["value"]
    assert d["vs_baseline"] is None and d["data"] == "synthetic"
    wl = workloads.WORKLOADS[3]          # the largest layer is the default
    assert d["config"]["workload"] == wl.name
    assert (d["config"]["T"], d["config"]["Cin"], d["config"]["Cout"]) == (wl.T, wl.Cin, wl.Cout)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert cb["unit"] == d["unit"] and cb["extrapolated"] is True
    assert f"first 16 of {wl.T} tokens" in cb["sample"]
    assert f"32 of {wl.Cout} rows" in cb["sample"]
    assert cb["host"]["nproc"] >= 1 and cb["host"]["machine"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"],
                        "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_exit_without_work():
    r = _run({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}, "--gpus", "2")
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def _bench():
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_under_test",
                                                  os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_cpu_baseline_leg_on_a_small_sample():
    """The oracle timing leg of the benchmark's own line, on the small
    workload: a positive per-layer figure scaled from the token sample."""
    bench = _bench()
    wl = workloads.WORKLOADS[0]
    inp = workloads.make_inputs(wl)
    cb = bench.cpu_baseline(wl, inp, 32)
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["unit"] == "us/layer"
    assert cb["value"] > 0 and cb["measured_s"] > 0
    assert cb["value"] >= cb["measured_s"] * 1e6 * 0.999      # scaled up to all T
    assert f"first 32 of {wl.T} tokens" in cb["sample"]
    assert cb["host"]["nproc"] >= 1


def test_host_cpu_names_an_arm_part(tmp_path):
    bench = _bench()
    f = tmp_path / "cpuinfo"
    f.write_text("processor\t: 0\nBogoMIPS\t: 2000.00\nCPU implementer\t: 0x41\n"
                 "CPU architecture: 8\nCPU part\t: 0xd4f\n\nprocessor\t: 1\n"
                 "CPU implementer\t: 0x41\nCPU part\t: 0xd4f\n")
    assert bench.host_cpu(str(f))["model"] == "implementer 0x41 part 0xd4f"
    f.write_text("processor\t: 0\nmodel name\t: Some CPU @ 3.0GHz\n")
    assert bench.host_cpu(str(f))["model"] == "Some CPU @ 3.0GHz"
    assert bench.host_cpu(str(tmp_path / "missing"))["model"] is None
