"""bench.py's output contract, checked on CPU: the reference arm (the oracle) prints
one JSON line with the keys the driver reads, and the native arm refuses to run
without a GPU instead of falling back to the CPU."""
import json
import os
import subprocess
import sys

import pytest

from tests.conftest import ROOT

KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
        "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "impl"}


def _run(*args):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                          cwd=ROOT, env=env, timeout=600)


@pytest.mark.parametrize("extra", [["--sessions", "1"], ["--workload", "pool"]])
def test_reference_arm_prints_one_json_line(extra):
    r = _run("--impl", "reference", "--steps", "2", "--warmup", "1", *extra)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert KEYS <= set(line), KEYS - set(line)
    assert line["impl"] == "reference" and line["n_gpus"] == 1 and line["steps"] == 2 and line["warmup"] == 1
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert "workload" in line["config"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0


def test_native_arm_needs_a_gpu():
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    r = _run("--steps", "1", "--warmup", "1")
    assert r.returncode != 0
    assert "GPU" in (r.stderr + r.stdout)


def test_reference_arm_loads_only_the_oracle():
    """The reference arm builds its inputs with the seeded generator and runs the oracle: the
    CUDA library's package is never imported and its shared object never loaded."""
    code = ("import sys; sys.argv = ['bench.py', '--impl', 'reference', '--steps', '1', '--warmup', '0', "
            "'--sessions', '1', '--workload', 'd2t']; import bench; bench.main(); "
            "maps = open('/proc/self/maps').read(); "
            "assert 'serving_sampler_gb300' not in sys.modules; assert 'libspecverify' not in maps; "
            "assert 'liboracle' in maps; print('ONLY_ORACLE')")
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, cwd=ROOT, env=env, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    assert "ONLY_ORACLE" in r.stdout
