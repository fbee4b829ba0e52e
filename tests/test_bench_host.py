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
