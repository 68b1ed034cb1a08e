"""The N > 1 launch of bench.py, on CPU: two gloo ranks (127.0.0.1) check the
max-over-ranks timing and the whole-job throughput; the reference arm under
a two-rank launch runs on rank 0 only, and rank 1 exits 0 without output."""
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


def _rank(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank,
                            world_size=world)
    try:
        # rank r: step 1 + r ms, end to end 5 - r ms
        ms, e2e = bench.max_over_ranks([1.0 + rank, 5.0 - rank])
        out.put((rank, ms, e2e, bench.job_gbs(2e6, ms, world)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo():
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(out.get(timeout=10) for _ in range(2))
    for rank, ms, e2e, gbs in res:
        assert ms == 2.0 and e2e == 5.0  # the slowest rank's times, on every rank
        assert gbs == pytest.approx(2 * 2e6 / 2e-3 / 1e9)  # both ranks' bytes over the max time


def test_single_rank_max_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 4.0]) == [3.0, 4.0]
    assert bench.job_gbs(1e9, 1000.0, 1) == pytest.approx(1.0)


@pytest.mark.parametrize("rank", [0, 1])
def test_reference_arm_runs_on_rank_0_only(rank):
    env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0", "--cpu-budget", "0.2",
                        "--workload", "gemv_960"],
                       env=env, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    if rank == 1:
        assert lines == []
    else:
        d = json.loads(lines[-1])
        assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
        assert d["e2e"]["h2d_bytes_per_step"] == 0
