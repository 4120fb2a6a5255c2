"""Host-side pieces of bench.py, on the CPU: the algorithmic work model behind the
roofline figures, the L2 flush rule, the traffic record lookup, the split planner's
mirror, and the reference arm's JSON line (the oracle timed on the host)."""
import hashlib
import json
import os
import subprocess
import sys
import types

import bench
from gated_delta_rule_24_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_algorithmic_work_workload3():
    """16 x 4096 tokens, 16 q/k heads, 32 v heads, bf16 states, fp32 gates: 1.661 GB and
    0.344 TFLOP per call, the figures the roofline fractions divide by."""
    p = W.make_workload(3, seqs=1)  # one sequence: scale by 16 below
    b1, f1 = bench.algorithmic_work(p)
    T, D = 4096, 128
    qk = 2 * T * 16 * D * 2
    v_out = 2 * T * 32 * D * 2
    gates = 2 * T * 32 * 4
    states = 2 * 32 * D * D * 2
    assert b1 == qk + v_out + gates + states
    # every term is per token or per (sequence, head): 16 sequences are 16 times one
    assert 16 * b1 == 1660944384
    assert 16 * f1 == 343597383680


def test_flush_rule():
    assert bench.needs_flush(W.make_workload(1)) and bench.needs_flush(W.make_workload(2))
    assert bench.needs_flush(W.make_workload(3, seqs=1))  # 104 MB: below twice the L2
    assert not bench.needs_flush(W.make_workload(3, seqs=3))  # 312 MB


def test_recorded_traffic_follows_the_source_hash():
    text = open(os.path.join(ROOT, "profiles", "traffic.md")).read()
    rows = [[c.strip() for c in line.strip().strip("|").split("|")] for line in text.splitlines()
            if line.startswith("| gdn_")]
    assert rows
    for kernel, workload, digest, nbytes, _ in rows:
        src = "decode.cu" if "decode" in kernel else "prefill.cu"
        got = bench.recorded_traffic(kernel, workload, src)
        current = hashlib.sha256(open(os.path.join(ROOT, "gated_delta_rule_24_gb300", "csrc", src), "rb")
                                 .read()).hexdigest()[:16]
        assert got == (float(nbytes) if digest == current else None)
        assert bench.recorded_traffic(kernel, workload + "_other", src) is None


def test_planned_splits_follow_the_library_plan(force_split):
    w3 = types.SimpleNamespace(N=16, H=32, T=16 * 4096, batch_invariant=False)
    w4 = types.SimpleNamespace(N=2, H=32, T=2 * 65536, batch_invariant=False)
    assert bench.planned_splits(w3, 152) == 1  # 512 units: splitting never pays
    assert bench.planned_splits(w4, 152) == 4  # 64 units: segments of 3, 1, 1, 2 sevenths
    one = W.make_problem([16384], 1, 2, seed=1, batch_invariant=False)
    assert bench.planned_splits(one, 152) == 8
    one.batch_invariant = True
    assert bench.planned_splits(one, 152) == 1
    one.batch_invariant = False
    force_split(3)
    assert bench.planned_splits(one, 152) == 3


def test_reference_arm_json_line():
    """`bench.py --impl reference` runs the oracle on the host and prints one JSON line
    with the contract's keys (no GPU needed)."""
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "1", "--steps", "2",
                        "--warmup", "3", "--ref-units", "1"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "tokens/s"
    assert line["higher_is_better"] is True and line["n_gpus"] == 1 and line["steps"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["gpu_launches"] == 0
    assert line["config"]["workload"] == "w1_single_256"


def test_default_line_is_workload4_with_extras():
    """Without --workload the headline is the long-context workload (2 x 65536, fp32
    states, batch_invariant off) and the other full-size workloads ride along."""
    a = bench.parse_args([])
    assert a.workload == 4 and a.extras and not a.shard and a.warmup >= 3
    assert [(k, w) for k, w, _ in bench.EXTRAS] == [("w4_batch_invariant", 4), ("w3", 3), ("w5", 5)]
    assert not bench.parse_args(["--workload", "3"]).extras
    assert not bench.parse_args(["--no-extras"]).extras
    assert bench.parse_args(["--shard", "--gpus", "2"]).shard


def test_config_names_the_parallelism():
    p = W.make_workload(2)
    assert bench.config_of(p, 2, 1)["parallelism"].startswith("replicas x1")
    c = bench.config_of(p, 2, 4, shard=True)
    assert c["parallelism"].startswith("sequence shards x4") and c["workload"] == p.name
