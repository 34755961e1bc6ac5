"""Host-side accounting of bench.py: the exact count of visible (query, key) pairs that
the valid-work figures divide by, against brute force."""
import itertools
import os
import sys

import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402
from sequence_head_attention_seq_b300 import workloads  # noqa: E402


def _brute(s, b, h, causal, lens):
    return h * sum(1 for bb, i, j in itertools.product(range(b), range(s), range(s))
                   if (not causal or j <= i) and j < lens[bb])


@pytest.mark.parametrize("s,b,h,causal,lens", [
    (7, 1, 2, True, None), (7, 2, 3, False, None), (9, 3, 1, True, [4, 9, 0]),
    (9, 2, 2, False, [1, 8]), (6, 2, 1, True, [12, -3]),
])
def test_valid_pairs_brute_force(s, b, h, causal, lens):
    w = workloads.Workload("t", 1, b=b, h=h, d=64, s=s, N=1, causal=causal, scale=1.0)
    kl = None if lens is None else torch.tensor(lens)
    want = _brute(s, b, h, causal, [max(0, min(n, s)) for n in (lens or [s] * b)])
    assert bench.valid_pairs(w, kl) == want


def test_valid_pairs_dense_causal_closed_form():
    w = workloads.WORKLOADS["llama70b"]
    assert bench.valid_pairs(w) == w.b * w.h * w.s * (w.s + 1) // 2


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` (the fp64 oracle on the host cores) prints one JSON line
    with the keys the benchmark contract names; it needs no GPU."""
    import json
    import subprocess
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload",
                          "tiny", "--steps", "1", "--warmup", "3"], cwd=root,
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0 and line["steps"] == 1
    assert line["config"]["workload"] == "tiny"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    assert "first 128 positions" in cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"],
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_cpu_relayout_rate_on_a_small_workload():
    """The host regrouping rate in `cpu_baseline` (the oracle's copy loop over one tensor)
    runs on CPU tensors and reports bytes read + written per second."""
    w = workloads.Workload("t", 3, b=2, h=4, d=64, s=256, N=2, causal=True, scale=1.0)
    ins = workloads.make_inputs(w, device="cpu", with_dout=False)
    r = bench.cpu_relayout(w, ins)
    assert r["unit"] == "GB/s" and r["value"] > 0 and r["cores"] == 1
    assert "seq2head" in r["sample"]
    one = workloads.Workload("t1", 4, b=1, h=2, d=64, s=128, N=1, causal=True, scale=1.0)
    assert bench.cpu_relayout(one, workloads.make_inputs(one, with_dout=False)) is None


def test_oracle_whole_on_a_small_workload():
    """The whole-workload oracle timing that the small workloads' entries carry: the
    shards are put back in sequence order and every head, row and key is computed."""
    w = workloads.Workload("t", 5, b=2, h=2, d=64, s=128, N=2, causal=False, scale=1.0,
                           key_len_range=(64, 128))
    r = bench.oracle_whole(w, workloads.make_inputs(w, device="cpu"))
    assert r["kind"] == "oracle" and r["value"] > 0 and r["cores"] >= 1
    assert "all 4 heads" in r["sample"]
