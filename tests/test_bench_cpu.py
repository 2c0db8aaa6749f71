"""bench.py on the host: the reference arm (the CPU oracle), its JSON line,
and the multi-rank path (torchrun, gloo, two ranks) -- no GPU needed."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _json_lines(text):
    return [json.loads(l) for l in text.splitlines() if l.startswith("{")]


def test_reference_arm_prints_one_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "1",
                        "--steps", "2", "--warmup", "3", "--ref-step-seconds", "0.2"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    d = lines[0]
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "pairs/s"
    assert d["higher_is_better"] is True and d["steps"] == 2 and d["warmup"] == 3
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["config"]["workload"].startswith("tiny_sparse")


def test_reference_arm_under_torchrun_two_ranks():
    """Rank 0 alone runs and prints; the other rank exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--gpus", "2", "--impl", "reference", "--config", "1", "--steps", "1", "--warmup", "3",
           "--ref-step-seconds", "0.2"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1 and lines[0]["n_gpus"] == 2


def _max_worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        got = bench.all_max(1.5 + rank, world)   # rank 1 is the slowest
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo():
    """The timed region is the max over ranks of each rank's own time."""
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_max_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(2))
    assert res == {0: 2.5, 1: 2.5}


def test_workload_numbers_config3():
    sys.path.insert(0, ROOT)
    import bench
    import workloads as W
    w = W.make_config(3)
    pairs, flops, b, comp = bench.workload_numbers(w)
    assert pairs == 805_437_440 and flops == 2 * 512 * pairs
    assert b["k_gathered"] == 6_292_480 * 1024 and b["q"] == 4096 * 128 * 1024
    assert abs(sum(b.values()) - 7.0496e9) < 1e6
    # compulsory: each tensor once; key j is visible to rows >= j only, so a
    # few of the last keys are never picked
    assert "k_gathered" not in comp and 4000 * 1024 <= comp["k_unique"] <= 4096 * 1024
    assert abs(sum(comp.values()) - 0.6104e9) < 2e6
    # the binding bound is the tensor one: 824.8 GFLOP at the measured peak
    # takes longer than moving the compulsory bytes
    r = bench.roofline_block(flops, sum(comp.values()), 0.7e-3, 6791.4, 1869.3, "measured")
    assert r["bound"] == "tensor" and abs(r["frac"] - flops / 0.7e-3 / 1e12 / 1869.3) < 1e-12
    assert r["frac"] < 1.0


def test_workload_numbers_dense_unique_keys():
    sys.path.insert(0, ROOT)
    import bench
    import workloads as W
    w = W.make_config(2)
    pairs, flops, b, comp = bench.workload_numbers(w)
    assert pairs == 2 * (512 * 513 // 2) * 16
    assert comp["k_unique"] == 2 * 512 * 1024 and comp["out"] == 2 * 512 * 512 * 4


def test_profiled_traffic_follows_the_kernel_and_its_source(tmp_path, monkeypatch):
    """The roofline's DRAM traffic is read from the summary of the kernel the
    L1-norm launch ran, and only while that summary was taken on the
    kernel's current source and on the same workload."""
    import bench

    class Info:
        def __init__(self, pairs):
            self.info = type("I", (), {"cta_pairs": pairs})()

    assert bench.l1_kernel_name(Info(76)) == "smla_pair_kernel"
    assert bench.l1_kernel_name(Info(0)) == "smla_fused_kernel"
    for kernel, (path, srcs) in bench.KERNELS.items():
        assert all(os.path.exists(s) for s in srcs), kernel
        summary = tmp_path / f"{kernel}.txt"
        monkeypatch.setitem(bench.KERNELS, kernel, (str(summary), srcs))
        body = "# comment: not a field\nworkload: wl\nkernel_sha256_16: {}\ndram_bytes_per_launch: 1234\n"
        summary.write_text(body.format(bench.kernel_sha(kernel)))
        assert bench.profiled_traffic("wl", kernel) == 1234.0
        assert bench.profiled_traffic("other", kernel) is None
        summary.write_text(body.format("0" * 16))
        assert bench.profiled_traffic("wl", kernel) is None
    # the two kernels hash different sources
    assert bench.kernel_sha("smla_pair_kernel") != bench.kernel_sha("smla_fused_kernel")
