"""CPU checks of the benchmark's byte models and its reference arm (the FP64
oracle timed on the host cores), for every workload."""
import json
import subprocess
import sys
import os
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_single_byte_model():
    b = bench.algorithmic_bytes(S=10, N=32768, D=4096, R=4096, out_norm=True, P=152)
    v = 10 * 32768 * 4096 * 2
    row = 32768 * 4096 * 2
    stats = 3 * 32768 * 10 * 4 + 32768 * 4
    assert b["fwd"] == v + row + stats
    assert b["bwd"] == 2 * v + row + stats + 2 * 152 * (4096 + 4096) * 4
    assert b["total"] == b["fwd"] + b["bwd"]
    # a saved FP32 pre-norm mixture is written by the forward and read by the backward
    c = bench.algorithmic_bytes(S=10, N=32768, D=4096, R=4096, out_norm=True, P=152, o_pre=True)
    assert c["fwd"] - b["fwd"] == c["bwd"] - b["bwd"] == 32768 * 4096 * 4
    assert bench.algorithmic_bytes(S=2, N=8, D=64, R=64, out_norm=False, P=1, o_pre=True) == \
        bench.algorithmic_bytes(S=2, N=8, D=64, R=64, out_norm=False, P=1)


def test_sliced_step_reads_twice():
    w = bench.SlicedRead(tokens=8)
    assert [x.key_offset for x in w.wls] == [0, 3072]
    one = bench.algorithmic_bytes(9, 8, 4096, 1024, False, 1)
    assert w.bytes_for(1)["total"] == 2 * one["total"]
    assert w.wls[0].values is w.wls[1].values   # the same sources, read twice


def test_multi_byte_model():
    b = bench.multi_algorithmic_bytes(S=10, N=32768, D=4096, R=1024, M=2, P=152)
    v = 10 * 32768 * 4096 * 2
    out = 2 * 32768 * 4096 * 2
    stats = (2 * 2 * 10 + 10) * 32768 * 4
    assert b["fwd"] == v + out + stats
    assert b["bwd"] == 2 * v + out + stats + 2 * 152 * 2 * 1024 * 4


@pytest.mark.parametrize("workload", ["long", "short", "sliced", "deep", "multi", "multi16", "selected", "block"])
def test_reference_arm_prints_one_json_line(workload):
    t0 = time.time()
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", workload, "--steps", "2", "--warmup", "3", "--ref-tokens", "16"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    wall = time.time() - t0
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "impl", "cpu_baseline", "e2e", "config"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    # ms_per_step is what a timed step measured: the steps fit in the run's wall time
    assert d["steps"] * d["ms_per_step"] * 1e-3 < wall
    assert d["config"]["sample_tokens"] == 16


def test_sixteen_query_workload():
    w = bench.Multi16Read(tokens=8)
    assert (w.wl.S, w.wl.D, w.wl.R, w.wl.M) == (10, 1024, 1024, 16)
    assert w.bytes_for(76) == bench.multi_algorithmic_bytes(10, 8, 1024, 1024, 16, 76)
    assert "multi16" in bench.WORKLOADS and bench.FULL_TOKENS["multi16"] == 32768


def test_extension_byte_models():
    s = bench.selected_algorithmic_bytes(S=10, N=100, D=64, R=16, K=2, E=8, P=4)
    m = bench.multi_algorithmic_bytes(S=10, N=100, D=64, R=16, M=2, P=0)
    assert s["fwd"] == m["fwd"] + 100 * 2 * 8
    assert s["bwd"] == m["bwd"] + 100 * 2 * 8 + 2 * 4 * 8 * 16 * 4
    b = bench.block_algorithmic_bytes(S=9, N=10, D=64, R=16, P=3)
    row = 10 * 64 * 2
    # reads: S-1 completed + the previous partial + delta; writes: the new partial + y
    assert b["fwd"] == (8 + 2) * row + 2 * row + 3 * 10 * 9 * 4
    assert b["bwd"] == 2 * 9 * row + 2 * row + 3 * 10 * 9 * 4 + 2 * 3 * 16 * 4
