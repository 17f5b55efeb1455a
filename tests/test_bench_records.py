"""The bench's DRAM traffic records match the kernel sources they were taken on.

bench.py reports a record's bytes only while the sources still hash to the
recorded value (otherwise the line carries traffic = null).  These checks run
without a GPU and flag a kernel change committed without a fresh capture, and
a record whose workload or bytes cannot be right.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
import seeded_inputs as si  # noqa: E402


@pytest.mark.parametrize("rec", bench.TRAFFIC, ids=lambda r: f"{r[0]}:{r[1]}:{'c' if r[2] else 'nc'}")
def test_traffic_record_is_current(rec):
    kernel, workload, causal, files, sha, nbytes = rec
    assert sha is not None and nbytes is not None, "record without a capture"
    assert bench.source_sha(files) == sha, (
        f"{kernel} on {workload}: the sources changed since the DRAM capture; "
        "recapture it (one-pass ncu of the bench command) and update the record")
    assert bench.traffic_for(kernel, workload, causal) == nbytes


def test_traffic_records_are_unique_and_plausible():
    keys = [(k, w, c) for k, w, c, *_ in bench.TRAFFIC]
    assert len(keys) == len(set(keys))
    for kernel, workload, causal, files, sha, nbytes in bench.TRAFFIC:
        for rel in files:
            assert os.path.isfile(os.path.join(ROOT, rel)), rel
        # a prefill moves Q, K, V in and O out about once: between half (a
        # workload that fits in L2 starts partly resident) and four times
        # those bytes, or the record is mis-typed
        w = si.WORKLOADS[workload]
        if kernel.startswith("prefill"):
            once = 4 * w["B"] * w["H"] * w["S"] * w["D"] * 2
            assert 0.5 * once <= nbytes <= 4 * once, (workload, nbytes, once)
