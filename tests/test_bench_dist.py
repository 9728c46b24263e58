"""The benchmark's multi-process host logic on CPU with gloo (world size 2):
max-over-ranks timing, whole-job aggregation, per-rank seeds, and the
torchrun launch of the reference arm (rank 0 prints one line, rank 1
prints nothing and exits 0)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        m = bench.reduce_max(1.5 + rank)
        bench.barrier()
        out.put((rank, m, bench.rank_seed(0, rank)))
    finally:
        dist.destroy_process_group()


def test_reduce_max_and_seeds_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [m for _, m, _ in res] == [2.5, 2.5]
    assert res[0][2] != res[1][2]


def test_aggregate_is_whole_job():
    # Two ranks each doing 1e12 FLOPs, slowest in 0.5 s: 4 TFLOPS in total.
    assert bench.aggregate(1e12, 2, 0.5) == pytest.approx(4.0)
    f, b = bench.step_flops(dict(B=8, H=16, N=8192, d=128, causal=False))
    assert f == 4 * 8 * 16 * 8192 ** 2 * 128 and b == 2.5 * f
    f, _ = bench.step_flops(dict(B=4, H=32, N=4096, d=128, causal=True))
    assert f == 0.5 * 4 * 4 * 32 * 4096 ** 2 * 128


def test_torchrun_reference_arm_two_ranks():
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--gpus", "2",
           "--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]


@pytest.mark.parametrize("N,causal", [(1, False), (1, True), (200, False), (200, True),
                                      (385, True), (385, False)])
def test_visible_pairs_brute_force(N, causal):
    import torch
    from io_aware_exact_02_gb300 import synth
    nb = -(-N // 128)
    mask = synth.draw_block_mask(nb, 0.5, seed=N, diagonal=False).tolist()
    want = sum(1 for i in range(N) for j in range(N)
               if mask[i // 128][j // 128] and (not causal or j <= i))
    assert bench.visible_pairs(mask, N, causal) == want
