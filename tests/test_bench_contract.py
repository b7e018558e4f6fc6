"""The benchmark's JSON-line contract, checked on CPU: the reference arm (the
fp64 oracle) prints one well-formed line on rank 0 and nothing elsewhere, and
the library arm fails loudly, printing no line, when no GPU is present."""
import json
import os
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ARGS = ["bench.py", "--impl", "reference", "--workload", "tiny_ce_z_fp32", "--steps", "2",
        "--warmup", "3"]


def _run(args, **env):
    e = dict(os.environ, **{k: str(v) for k, v in env.items()})
    return subprocess.run([sys.executable, *args], cwd=ROOT, env=e, capture_output=True,
                          text=True, timeout=300)


def test_reference_arm_prints_one_contract_line():
    r = _run(ARGS)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key, typ in (("metric", str), ("value", float), ("unit", str), ("n_gpus", int),
                     ("steps", int), ("warmup", int), ("ms_per_step", float),
                     ("higher_is_better", bool), ("scaling", str), ("dtype", str),
                     ("data", str), ("config", dict), ("cpu_baseline", dict), ("e2e", dict)):
        assert isinstance(d[key], typ), key
    assert d["impl"] == "reference"
    assert d["vs_baseline"] is None
    assert d["steps"] == 2 and d["warmup"] >= 3 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["config"]["workload"] == "tiny_ce_z_fp32"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_runs_on_rank_zero_only():
    r1 = _run(ARGS + ["--gpus", "2"], RANK=1, WORLD_SIZE=2, LOCAL_RANK=1)
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    r0 = _run(ARGS + ["--gpus", "2"], RANK=0, WORLD_SIZE=2, LOCAL_RANK=0)
    assert r0.returncode == 0, r0.stderr[-2000:]
    d = json.loads(r0.stdout.strip())
    assert d["n_gpus"] == 2 and d["impl"] == "reference"


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU failure")
def test_library_arm_fails_loudly_without_a_gpu():
    r = _run(["bench.py", "--workload", "tiny_ce_z_fp32", "--steps", "1", "--warmup", "3"])
    assert r.returncode != 0
    assert r.stdout.strip() == ""


def _fake_smi(tmp_path, body):
    d = tmp_path / "bin"
    d.mkdir()
    f = d / "nvidia-smi"
    f.write_text("#!/bin/bash\n" + body)
    f.chmod(0o755)
    return str(d)


def test_clock_sampler_counts_only_samples_inside_the_timed_region(tmp_path, monkeypatch):
    """The sampler waits for nvidia-smi's first line before the region starts,
    so that line (taken before the region) is not counted; throttle reasons
    seen inside the region are reported."""
    import time
    sys.path.insert(0, ROOT)
    import bench
    d = _fake_smi(tmp_path, (
        "sleep 0.2\n"
        "echo '0, 1200, 2070, 500.0, 0x0, Active, Not Active, Not Active, Not Active'\n"
        "sleep 0.1\n"
        "echo '0, 2070, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active'\n"
        "sleep 10\n"))
    monkeypatch.setenv("PATH", d + os.pathsep + os.environ["PATH"])
    with bench.ClockSampler(0) as c:
        time.sleep(0.4)
    s = c.summary()
    assert s["samples"] == 1 and s["sm_mhz"] == 2070.0 and s["reasons"] == ["sw_power_cap"]


def test_clock_sampler_without_nvidia_smi_reports_nothing(tmp_path, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    empty = tmp_path / "empty"
    empty.mkdir()
    monkeypatch.setenv("PATH", str(empty))
    with bench.ClockSampler(0) as c:
        pass
    assert c.summary() is None
