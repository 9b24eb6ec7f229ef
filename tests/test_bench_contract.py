"""Host-side pieces of bench.py's JSON line that need no GPU: the DRAM-traffic
record lookup (valid only for the kernel source it was measured on) and the
CPU description of the oracle baseline."""

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from causal_gqa_prefill_gb300 import workloads as W  # noqa: E402


def _records():
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    out = {}
    with open(path) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            num, sha, val = line.split("\t")
            out[int(num)] = (sha, float(val))
    return out


def test_traffic_records_are_well_formed():
    recs = _records()
    assert recs, "no traffic records"
    for num, (sha, val) in recs.items():
        assert num in W.WORKLOADS
        assert len(sha) == 16 and all(c in "0123456789abcdef" for c in sha)
        # at least the algorithmic bytes' order of magnitude: a record far below the
        # bytes the kernel must move would be a measurement of the wrong launch
        w = W.WORKLOADS[num]
        assert val > 0.2 * w.io_bytes(), (num, val, w.io_bytes())


def test_traffic_lookup_follows_the_source_hash(monkeypatch):
    recs = _records()
    num, (sha, val) = next(iter(recs.items()))
    w = W.WORKLOADS[num]
    monkeypatch.setattr(bench, "kernel_source_hash", lambda w_: sha)
    assert bench.recorded_traffic(w) == val
    # a changed kernel source invalidates the record
    monkeypatch.setattr(bench, "kernel_source_hash", lambda w_: "0" * 16)
    assert bench.recorded_traffic(w) is None


def test_kernel_source_per_workload_family():
    assert bench.kernel_source(W.WORKLOADS[3]).endswith("attn_prefill.cu")
    assert bench.kernel_source(W.WORKLOADS[10]).endswith("attn_decode.cu")
    assert bench.kernel_source(W.WORKLOADS[12]).endswith("attn_backward.cu")
    for n in (3, 10, 12):
        assert os.path.exists(bench.kernel_source(W.WORKLOADS[n]))


def test_cpu_model_is_described():
    m = bench.cpu_model()
    assert isinstance(m, str) and m.strip()
