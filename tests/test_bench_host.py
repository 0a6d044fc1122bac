"""Host-side logic of bench.py (CPU only): the rank launcher behind
``--gpus N``, the clock-record parser and the oracle's thread count.

``python bench.py --gpus N`` without an outside launcher must start N ranks
itself (one per GPU) that agree on the world size; here the same launch command
runs a stub rank script over gloo instead of the GPU step.
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

STUB = r'''
import json, os, sys
import torch
import torch.distributed as dist
dist.init_process_group("gloo")
t = torch.ones(1)
dist.all_reduce(t)
out = os.path.join(os.path.dirname(os.path.abspath(__file__)), f"rank{dist.get_rank()}.json")
with open(out, "w") as f:
    json.dump({"rank": dist.get_rank(), "n_gpus": dist.get_world_size(), "sum": int(t.item()),
               "argv": sys.argv[1:]}, f)
dist.destroy_process_group()
'''


def test_rank_launcher_starts_n_ranks(tmp_path):
    stub = tmp_path / "stub_rank.py"
    stub.write_text(STUB)
    cmd = bench.rank_launch_cmd(2, str(stub), ["--steps", "3"])
    env = {k: v for k, v in os.environ.items()
           if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=240, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads((tmp_path / f"rank{i}.json").read_text()) for i in range(2)]
    assert sorted(x["rank"] for x in lines) == [0, 1]
    assert all(x["n_gpus"] == 2 and x["sum"] == 2 for x in lines)
    assert all(x["argv"] == ["--steps", "3"] for x in lines)


def test_bench_relaunches_itself_without_a_launcher(monkeypatch):
    seen = {}

    def fake_call(cmd):
        seen["cmd"] = cmd
        return 0

    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    monkeypatch.setattr(bench.subprocess, "call", fake_call)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--gpus", "4", "--steps", "5"])
    with pytest.raises(SystemExit) as e:
        bench.main()
    assert e.value.code == 0
    cmd = seen["cmd"]
    assert "--nproc-per-node=4" in cmd and "torch.distributed.run" in cmd
    assert cmd[-4:] == ["--gpus", "4", "--steps", "5"]
    assert os.path.samefile(cmd[-5], os.path.join(ROOT, "bench.py"))
    assert cmd[cmd.index("--master-addr") + 1] == "127.0.0.1"


def test_clock_sampler_keeps_only_this_gpu():
    c = bench.ClockSampler("abcd-1234")
    c.lines = [
        "GPU-abcd-1234, 2070, 2070, 0x0, Not Active, Not Active, Not Active, Not Active",
        "GPU-ffff-0000, 900, 2070, 0x0, Active, Not Active, Not Active, Not Active",
        "GPU-abcd-1234, 2060, 2070, 0x4, Not Active, Not Active, Not Active, Active",
    ]
    s = c.summary()
    assert s["samples"] == 2 and s["sm_mhz"] == 2065 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]
    # a single visible GPU whose UUID torch reports differently is still taken
    c1 = bench.ClockSampler("zzzz")
    c1.lines = ["GPU-abcd-1234, 1500, 2070, 0x0, Not Active, Not Active, Not Active, Not Active"]
    assert c1.summary()["samples"] == 1


def test_threads_used_rounds_and_floors():
    assert bench.threads_used(0.2) == 1
    assert bench.threads_used(1.4) == 1
    assert bench.threads_used(11.6) == 12


def test_traffic_hash_follows_the_kernels_own_sources(tmp_path, monkeypatch):
    """A committed DRAM-traffic figure stays valid while the captured kernel's
    translation unit and the headers it includes are unchanged, and only then."""
    csrc = tmp_path / "sequential_rnn_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "a.cu").write_text('#include "b.h"\nint a;\n')
    (csrc / "b.h").write_text('#include "c.h"\n')
    (csrc / "c.h").write_text("// c\n")
    (csrc / "d.cu").write_text("int d;\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.tu_source_hash("a.cu")
    (csrc / "d.cu").write_text("int d2;\n")          # another kernel: no effect
    assert bench.tu_source_hash("a.cu") == h0
    (csrc / "c.h").write_text("// c changed\n")      # an included header: invalidates
    assert bench.tu_source_hash("a.cu") != h0


def test_single_thread_oracle_baseline_keeps_one_thread_busy():
    """The cpu_baseline's one-thread figure really runs the oracle on one thread."""
    one = bench.oracle_rate_single_thread("lstm_f32_1x64_b4_t256", 32, 0.5)
    assert one is not None and one["value"] > 0 and one["reps"] >= 1
    assert one["busy"] < 1.5, one
