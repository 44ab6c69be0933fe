"""Host-side logic of bench.py, on CPU: the multi-rank helpers under a
world-size-2 gloo group, and the reference arm's JSON line."""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import torch.distributed as dist
    r, wsz, _ = bench.dist_setup(use_cuda=False)
    assert (r, wsz) == (rank, world)
    bench.barrier(None)
    seed = bench.replica_seed(1005, r)
    elapsed = 1.0 + r  # rank 1 is the slow one
    mx = bench.max_over_ranks(elapsed)
    thr = bench.aggregate_throughput(256 * 10, wsz, mx)
    q.put((r, seed, mx, thr))
    dist.destroy_process_group()


def test_two_rank_gloo_helpers():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get() for _ in range(2))
    seeds = {r[1] for r in res}
    assert len(seeds) == 2                       # each rank its own replica
    assert all(r[2] == 2.0 for r in res)         # the slowest rank's time everywhere
    assert all(abs(r[3] - 2 * 2560 / 2.0) < 1e-9 for r in res)


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "tiny", "--steps", "3", "--warmup", "1"], capture_output=True, text=True, timeout=600,
                       env={**os.environ, "CUDA_VISIBLE_DEVICES": ""})
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == bench.UNIT and d["metric"] == bench.METRIC
    assert d["value"] > 0 and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert "processes at once" in d["cpu_baseline"]["sample"] and d["cpu_baseline"]["write_chunk_gbs"] > 0
    # the same workload description as our arm prints for the same arguments
    args = bench.argparse.Namespace(workload="tiny", batch=0)
    from int4_token_head_gb300 import synthetic
    assert d["config"] == bench.bench_config(args, synthetic.make_workload("tiny"), 1)


def test_gpus_flag_launches_ranks_itself():
    """`bench.py --gpus 2` without torchrun starts two ranks itself; for the
    reference arm rank 0 alone prints the line, which reports both ranks."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--workload", "tiny", "--steps", "2", "--warmup", "1"], capture_output=True, text=True,
                       timeout=600, env={**os.environ, "CUDA_VISIBLE_DEVICES": ""})
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["config"]["parallelism"] == "replicas x2"


def test_gpus_flag_without_enough_gpus_fails_cleanly():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--steps", "1"],
                       capture_output=True, text=True, timeout=300, env={**os.environ, "CUDA_VISIBLE_DEVICES": ""})
    assert r.returncode != 0 and "needs 2 visible GPUs" in r.stderr


def test_reference_arm_nonzero_rank_exits_quietly():
    env = {**os.environ, "RANK": "1", "WORLD_SIZE": "2", "CUDA_VISIBLE_DEVICES": ""}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "tiny", "--steps", "2"], capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_clock_sampler_parses_nvidia_smi_lines():
    s = bench.ClockSampler("0")
    s.proc = type("P", (), {"terminate": lambda self: None, "wait": lambda self, timeout=None: 0})()
    s.thread = type("T", (), {"join": lambda self, timeout=None: None})()
    s.lines = ["0, 1900, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Active",
               "0, 1950, 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active",
               "garbage"]
    c = s.stop()
    assert c["sm_mhz"] == 1925 and c["sm_max_mhz"] == 2070 and c["reasons"] == ["sw_power_cap"]


def test_kernel_names_and_recorded_traffic():
    # the bench names the kernel it times: INT4 head size 128 has its own entry point
    assert bench.decode_kernel_name(128) == "decode_kernel_i4d128"
    assert bench.decode_kernel_name(128, int8=True) == "decode_kernel"
    assert bench.decode_kernel_name(96) == "decode_kernel"
    assert bench.prefill_kernel_name(192) == "prefill_ws_kernel"
    assert bench.prefill_kernel_name(256) == "prefill_kernel"
    # a committed traffic record is reported only for the sources it was taken on
    rec = bench.recorded_traffic("decode", "long")
    assert rec is None or rec > 9.0e9
    assert bench.recorded_traffic("decode", "no-such-workload") is None


def test_source_sha_depends_on_every_file(tmp_path):
    a, b = tmp_path / "a.cuh", tmp_path / "b.cuh"
    a.write_bytes(b"one")
    b.write_bytes(b"two")
    h = bench.source_sha([str(a), str(b)])
    assert len(h) == 16 and h != bench.source_sha([str(a)])
    b.write_bytes(b"three")
    assert bench.source_sha([str(a), str(b)]) != h
