"""The committed ncu summaries: each names its kernel, records the hash of the
kernel's sources it was captured on (which must be the current sources, else
the benchmark reports no DRAM traffic for it) and the command that made it;
on the streaming workloads its DRAM bytes per launch are close to the
algorithmic bytes it states."""

import glob
import os
import re

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUMMARIES = sorted(p for p in glob.glob(os.path.join(ROOT, "profiles", "*.md"))
                   if re.search(r"source_hash:", open(p).read()))
KERNELS = {"pa_tile_kernel": "pa_tile", "pa_mtp_kernel": "pa_mtp", "pa_reduce_kernel": "pa_reduce",
           "pa_logits_kernel": "pa_logits"}


def kernel_of(text):
    head = text.splitlines()[0]
    for name, key in KERNELS.items():
        if name in head:
            return key
    raise AssertionError(f"no known kernel in {head!r}")


def test_every_kernel_family_has_a_summary():
    found = {kernel_of(open(p).read()) for p in SUMMARIES}
    assert found == set(KERNELS.values())


@pytest.mark.parametrize("path", SUMMARIES, ids=[os.path.basename(p) for p in SUMMARIES])
def test_summary_is_current(path):
    text = open(path).read()
    key = kernel_of(text)
    h = re.search(r"source_hash:\s*([0-9a-f]+)", text).group(1)
    assert h == bench.kernel_source_hash(key), f"{os.path.basename(path)} was captured on other {key} sources"
    assert re.search(r"^ncu .*--clock-control none", text, re.M), "the capture command is recorded"
    traffic = int(re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text).group(1))
    assert traffic > 0
    name = os.path.basename(path)
    if name.startswith(("pa_tile_dense", "pa_tile_d256", "pa_mtp_")):
        # streaming workloads larger than L2: each KV byte comes from DRAM about once
        # (sparse gathers and the reducer re-read data that L2 holds)
        ratios = [float(r) for r in re.findall(r"traffic / algorithmic = ([0-9.]+)", text)]
        assert ratios and all(0.95 < r < 1.15 for r in ratios), (name, ratios)
