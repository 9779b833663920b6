"""The benchmark's multi-rank host logic on CPU (gloo, two ranks): each rank
runs an independent replica, the job's time is the slowest rank's, value is
all ranks' tokens over that time, and only rank 0 prints. (The GPU leg's
kernels need a GPU; the reduction, token accounting and the reference arm's
rank handling do not.)"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, local = bench.dist_env()
    ms = bench.slowest_rank_ms(1.0 + rank, w, "cpu")  # rank 1 is the slow one
    out[rank] = (r, w, local, ms, bench.job_tokens_per_s(w, 8192, ms))
    dist.barrier()
    dist.destroy_process_group()


def test_slowest_rank_and_job_throughput_gloo():
    world, port = 2, _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        r, w, local, ms, tps = res[rank]
        assert (r, w, local) == (rank, world, rank)
        assert ms == 2.0  # the maximum over ranks, on every rank
        assert tps == pytest.approx(world * 8192 / 2e-3)


def test_single_rank_needs_no_process_group():
    assert bench.slowest_rank_ms(3.5, 1, "cpu") == 3.5
    assert bench.job_tokens_per_s(1, 100, 1.0) == pytest.approx(1e5)


def test_reference_arm_under_torchrun_prints_once():
    """bench.py --impl reference with two ranks: rank 0 runs the oracle on the
    host cores and prints one JSON line; rank 1 exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "1", "--workload", "switch_top1_toy"]
    p = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2
    assert rec["value"] > 0 and rec["cpu_baseline"]["kind"] == "oracle"


@pytest.mark.parametrize("workload", ["hier_16x64_e1024", "balanced_top2_e64"])
def test_reference_arm_widened_workloads(workload):
    """The oracle legs of the hierarchical and balanced workloads (reduced T)
    print one well-formed JSON line on one rank."""
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
           "--warmup", "1", "--cpu-sample", "2", "--tokens", "256", "--workload", workload]
    p = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["config"]["workload"] == workload
    assert rec["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_training_step():
    """bench.py --backward --impl reference: the oracle's forward and backward
    on a bounded token sample print one well-formed JSON line."""
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--backward",
           "--steps", "1", "--warmup", "1", "--workload", "noisy_top4_e16"]
    p = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["value"] > 0
    assert "fwd+bwd" in rec["metric"] and rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["config"]["workload"] == "noisy_top4_e16"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0


def test_traffic_record_keys_on_code_not_comments():
    """The measured expert-GEMM traffic is reported only for the kernel code
    it was captured on: comment and blank-line edits keep the key, a code
    edit changes it, and the recorded key is the current source's."""
    src = "// note\nint f(int a) {  // why\n  /* more\n text */ return a + 1;\n}\n\n"
    same = "int f(int a) {\n\n  return a + 1;   // other words\n}\n"
    other = "int f(int a) {\n  return a + 2;\n}\n"
    assert bench._code_only(src) == bench._code_only(same)
    assert bench._code_only(src) != bench._code_only(other)
    rec = bench.FFN_TRAFFIC["top2_large_experts"]
    assert rec["source"] == bench.ffn_source_hash()
    assert bench.measured_traffic(bench.wl.WORKLOADS["top2_large_experts"]) == rec["bytes"]
