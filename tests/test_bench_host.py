"""Host-side consistency of bench.py's tables (no GPU): every workload the
bench can time has a source-digest entry and a seeded input recipe, and every
recorded DRAM-traffic line names a known workload, a 16-hex-digit digest, a
positive byte count and a profile summary that exists."""
import inspect
import os
import re

import pytest

import bench
from dense_gemm_row_gb300 import workloads as w

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("name", sorted(bench.WORKLOADS))
def test_every_workload_is_complete(name):
    desc, kind, bound, launches = bench.WORKLOADS[name]
    assert kind in ("bf16", "f16", "f32", "s8")
    assert bound in ("tensor", "alu")
    assert launches >= 1
    assert name in bench.KERNEL_SOURCES
    for f in bench.KERNEL_SOURCES[name]:
        assert os.path.exists(os.path.join(ROOT, "dense_gemm_row_gb300", "csrc", f)), f
    assert re.fullmatch(r"[0-9a-f]{16}", bench.source_digest(name))
    # a recipe of its own in workloads.config (building the inputs here would
    # take too long at 8192^3)
    assert f'name == "{name}"' in inspect.getsource(w.config), name


def test_traffic_records_are_well_formed():
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    seen = set()
    for line in open(path).read().splitlines():
        if not line.strip() or line.startswith("#"):
            continue
        name, digest, nbytes, profile = line.split()
        assert name in bench.WORKLOADS, name
        assert name not in seen, f"{name} recorded twice"
        seen.add(name)
        assert re.fullmatch(r"[0-9a-f]{16}", digest)
        assert int(nbytes) > 0
        assert os.path.exists(os.path.join(ROOT, profile)), profile


def test_reference_arm_prints_the_contract_line(monkeypatch, capsys):
    """`bench.py --impl reference` times the CPU oracle and prints one JSON line
    with the same metric as the GPU arm, marked impl=reference, with a
    cpu_baseline describing the run and an e2e of zero copied bytes; ranks
    other than 0 print nothing. Run here on a small seeded problem standing in
    for the workload's inputs."""
    import argparse
    import json

    import torch

    small = w.problem(64, 48, 40, torch.bfloat16, "normal", 5)
    monkeypatch.setattr(w, "config", lambda name: small)
    args = argparse.Namespace(workload="bf16_8192", steps=2, warmup=1)
    assert bench.run_reference(args, 1, 1) == 0
    assert capsys.readouterr().out == ""
    assert bench.run_reference(args, 1, 0) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC
    assert line["unit"] == "TFLOP/s" and line["higher_is_better"] is True
    assert line["steps"] == 2 and line["warmup"] == 1 and line["n_gpus"] == 1
    assert line["value"] > 0 and line["ms_per_step"] > 0
    assert line["dtype"] == "f64" and line["data"] == "synthetic"
    assert line["config"]["workload"] == bench.WORKLOADS["bf16_8192"][0]
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] == line["value"]
    assert "rows 0..63 of A (64 of 64)" in cpu["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
