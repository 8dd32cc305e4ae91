"""CPU tests of the benchmark's host logic: the multi-rank reduction (gloo,
world size 2), the clock-record parser and the CPU-baseline leg."""

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

WORKER = r"""
import os, sys, json
sys.path.insert(0, {root!r})
import torch, torch.distributed as dist
import bench
dist.init_process_group("gloo")
r = dist.get_rank()
t = bench.reduce_max(1.5 + r, dist.get_world_size())
bench.barrier(dist.get_world_size())
print(json.dumps({{"rank": r, "max": t}}))
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_reduce_max_over_two_gloo_ranks(tmp_path):
    script = tmp_path / "w.py"
    script.write_text(WORKER.format(root=ROOT))
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, str(script)], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=120) for p in procs]
    for p, (o, e) in zip(procs, outs):
        assert p.returncode == 0, e
    res = [json.loads(o.strip().splitlines()[-1]) for o, _ in outs]
    assert all(r["max"] == 2.5 for r in res)


def test_reduce_max_single_process_is_identity():
    assert bench.reduce_max(3.25, 1) == 3.25


def test_clock_summary_parses_nvidia_smi_csv():
    cs = bench.ClockSampler(0)
    cs.lines = [
        "0, 1965, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 1800, 2070, 1390.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 1900, 2070, 1200.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbage",
    ]
    s = cs.summary()
    assert s["sm_mhz"] == 1900 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] == 3


def test_cpu_baseline_leg_is_bounded_and_reports_cores():
    from block_sparse_attention_tra_gb300 import workloads

    w = workloads.TraWorkload("tiny", 1, 2, 256, 64, 1.0, 2.0, "bf16")
    host = workloads.workload_inputs(w)
    cb = bench.cpu_baseline(w, host, budget_s=0.2)
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0
    wn = workloads.NsaWorkload("tiny", 1, 16, 1, 256, 64, 64, 4)
    cb = bench.cpu_baseline(wn, workloads.workload_inputs(wn), budget_s=0.2)
    assert cb["value"] > 0


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3", "--workload", "tra_f32_B1_H2_T256_D64"], capture_output=True, text=True,
                       timeout=600, env=dict(os.environ, PYTHONPATH=ROOT))
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and "sample" in d["cpu_baseline"]
    # exactly the GPU arm's workload description (the sample note lives under cpu_baseline)
    import bench
    from block_sparse_attention_tra_gb300 import workloads

    assert d["config"] == bench.workload_config(workloads.TRA_WORKLOADS["tra_f32_B1_H2_T256_D64"], 1)
    # the step time is the measured time of the sampled work: steps x ms_per_step is the timed region
    assert d["ms_per_step"] > 0 and d["value"] == d["cpu_baseline"]["value"]


def test_clock_records_that_reject_a_measurement():
    import bench

    # a power cap under a dense tensor load is normal and kept
    assert not bench.clocks_rejected({"sm_mhz": 1927.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]})
    assert not bench.clocks_rejected({"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []})
    # hardware or thermal slowdowns are rejected
    for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"):
        assert bench.clocks_rejected({"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [r, "sw_power_cap"]})
    # clocks stuck well below the maximum with no reason: a leftover clock lock
    assert bench.clocks_rejected({"sm_mhz": 1200.0, "sm_max_mhz": 2070.0, "reasons": []})
    # no samples (no nvidia-smi): nothing to judge
    assert not bench.clocks_rejected({"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]})


def test_shard_range_covers_every_unit_once():
    from block_sparse_attention_tra_gb300 import workloads

    for units in (0, 1, 5, 64, 1000, 1023):
        for world in (1, 2, 3, 4, 7, 8):
            slices = [workloads.shard_range(units, world, r) for r in range(world)]
            assert slices[0][0] == 0 and slices[-1][1] == units
            assert all(a[1] == b[0] for a, b in zip(slices, slices[1:]))
            sizes = [e - s for s, e in slices]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        workloads.shard_range(8, 2, 2)


SHARD_WORKER = r"""
import os, sys, json
sys.path.insert(0, {root!r})
import numpy as np, torch, torch.distributed as dist
from block_sparse_attention_tra_gb300 import workloads
from oracle import tra as otra
dist.init_process_group("gloo")
r, n = dist.get_rank(), dist.get_world_size()
# this rank's slice of a batch-sharded problem, as bench.py draws it, and the
# oracle's output on it; rank 0 gathers every slice
B, H, T, D = 1, 2, 40, 16
q, k, v = workloads.tra_inputs(B, H, T, D, "f32", seed=workloads.shard_seed(r))
o = torch.from_numpy(otra.tra_forward(q.double().numpy(), k.double().numpy(), v.double().numpy(), 0.5, 1.5))
parts = [torch.zeros_like(o) for _ in range(n)] if r == 0 else None
dist.gather(o, parts, dst=0)
qs = [torch.zeros_like(q) for _ in range(n)] if r == 0 else None
dist.gather(q, qs, dst=0)
ks = [torch.zeros_like(k) for _ in range(n)] if r == 0 else None
dist.gather(k, ks, dst=0)
vs = [torch.zeros_like(v) for _ in range(n)] if r == 0 else None
dist.gather(v, vs, dst=0)
if r == 0:
    # the global problem: the slices stacked along the batch; its oracle output
    # equals the gathered per-rank outputs, and the slices differ
    Q, K, V = (torch.cat(x, 0).double().numpy() for x in (qs, ks, vs))
    full = otra.tra_forward(Q, K, V, 0.5, 1.5)
    ok = bool(np.array_equal(full, torch.cat(parts, 0).numpy())) and not torch.equal(qs[0], qs[1])
    print(json.dumps({{"ok": ok}}))
dist.destroy_process_group()
"""


def test_batch_sharded_ranks_partition_the_global_problem(tmp_path):
    script = tmp_path / "s.py"
    script.write_text(SHARD_WORKER.format(root=ROOT))
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, str(script)], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=180) for p in procs]
    for p, (o, e) in zip(procs, outs):
        assert p.returncode == 0, e
    assert json.loads(outs[0][0].strip().splitlines()[-1])["ok"]
