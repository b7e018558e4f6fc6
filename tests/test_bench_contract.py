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
