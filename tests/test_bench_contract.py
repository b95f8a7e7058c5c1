"""bench.py's JSON line on the CPU: the reference arm (the oracle timed on the
host cores) prints one line with the keys the benchmark contract names, the
same workload config as the CUDA arm, at least 3 warm-up steps, and nothing on
ranks other than 0."""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _reference_line(warmup: int) -> dict:
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny-fp32", "--steps", "2",
                        "--warmup", str(warmup)], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.strip()]
    assert len(lines) == 1
    return json.loads(lines[0])


def test_reference_arm_honours_the_warmup_it_is_given():
    assert _reference_line(5)["warmup"] == 5


def test_cpu_baseline_reports_all_cores_and_one_thread():
    import bench
    from medusa_head_tree_heads_b300 import synth
    s = synth.SHAPES["tiny-fp32"]
    inp = synth.make_inputs(s, synth.load_plans()[s.name])
    cb = bench.time_oracle(s, inp, budget_s=0.0)
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0 and cb["cpu_model"]
    st = cb["single_thread"]
    assert st["cores"] == 1 and st["value"] > 0 and st["unit"] == "steps/s"


def test_one_thread_blas_without_threadpoolctl(monkeypatch):
    """Hosts without threadpoolctl still hold numpy's bundled OpenBLAS to one
    thread (through its own setter) and restore the thread count after."""
    import builtins

    import bench
    real_import = builtins.__import__

    def no_threadpoolctl(name, *args, **kw):
        if name == "threadpoolctl":
            raise ImportError("hidden for this test")
        return real_import(name, *args, **kw)

    monkeypatch.setattr(builtins, "__import__", no_threadpoolctl)
    import ctypes
    import glob
    import os

    import numpy as np
    libs = glob.glob(os.path.join(os.path.dirname(np.__file__), "..", "numpy.libs", "*openblas*.so*"))
    get = None
    for path in libs:
        lib = ctypes.CDLL(path)
        get = getattr(lib, "scipy_openblas_get_num_threads64_", None)
        if get is not None:
            get.restype = ctypes.c_int
            break
    before = get() if get is not None else None
    with bench.blas_one_thread() as how:
        if get is not None:
            assert how == "openblas" and get() == 1
    if get is not None:
        assert get() == before


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny-fp32", "--steps", "2",
                        "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    import bench
    from medusa_head_tree_heads_b300 import synth
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "steps/s"
    assert d["higher_is_better"] is True and d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 3
    assert d["value"] > 0 and abs(d["ms_per_step"] - 1e3 / d["value"]) < 1e-6 * d["ms_per_step"]
    assert d["data"] == "synthetic" and d["vs_baseline"] is None
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert cb["cpu_model"]
    assert d["e2e"] == {"value": d["value"], "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    s = synth.SHAPES["tiny-fp32"]
    want = bench.workload_config(s, "oracle on the host cores")
    assert d["config"] == want


def test_reference_arm_is_silent_off_rank_0(capsys):
    import bench
    args = argparse.Namespace(workload="tiny-fp32", steps=1, warmup=3, gpus=2)
    bench.run_reference(args, world=2, rank=1)
    assert capsys.readouterr().out == ""
