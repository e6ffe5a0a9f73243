"""The committed ncu summaries that bench.py reads its DRAM traffic from:
every summary with a machine-readable header names a known kernel and a
workload bench.py runs, carries a 64-hex source hash and a numeric byte
count, and is found again by bench.py's own lookup when its hash is current."""
import os
import re

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PDIR = os.path.join(ROOT, "profiles")
KEYS = ("kernel", "workload", "source_sha256", "dram_bytes_per_launch")


def headers():
    out = []
    for fn in sorted(os.listdir(PDIR)):
        if not fn.endswith((".txt", ".md")):
            continue
        fields = {}
        with open(os.path.join(PDIR, fn), encoding="utf-8") as f:
            for line in f:
                if ":" in line and line.strip().startswith(KEYS):
                    k, v = line.split(":", 1)
                    fields.setdefault(k.strip(), []).append(v.strip())
        if fields:
            out.append((fn, fields))
    return out


def test_profiles_present():
    assert os.path.isdir(PDIR)
    assert len(headers()) >= 4


@pytest.mark.parametrize("fn,fields", headers(), ids=[h[0] for h in headers()])
def test_profile_header_well_formed(fn, fields):
    for k in KEYS:
        assert k in fields, f"{fn}: no '{k}:' line"
        assert len(fields[k]) == 1, f"{fn}: '{k}:' appears {len(fields[k])} times"
    kernel, workload = fields["kernel"][0], fields["workload"][0]
    assert kernel in bench.KERNEL_SOURCES, fn
    assert workload in bench.WORKLOADS, fn
    assert re.fullmatch(r"[0-9a-f]{64}", fields["source_sha256"][0]), fn
    assert float(fields["dram_bytes_per_launch"][0]) > 0, fn
    if fields["source_sha256"][0] == bench.source_sha(bench.KERNEL_SOURCES[kernel]):
        assert bench.profiled_traffic(kernel, workload) == float(fields["dram_bytes_per_launch"][0])
