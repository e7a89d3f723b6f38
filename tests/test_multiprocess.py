"""The N > 1 host path of bench.py on CPU: two gloo ranks (world_size 2) run
the rendezvous, the barrier and the max-over-ranks reduction that bench.py uses
to time a step.  The path has no data-path collective (heads are independent
across ranks), so this is the whole multi-process logic."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, local = bench.dist_setup()
    bench.barrier(w)
    got = bench.max_over_ranks(10.0 + r, w)   # each rank's "step time"
    bench.barrier(w)
    q.put((r, w, local, got))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_step_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[0] for o in out] == [0, 1]
    assert all(o[1] == 2 for o in out)
    assert all(o[3] == 11.0 for o in out)   # max over ranks of 10 + rank


def test_bench_gpus_flag_starts_the_ranks_itself():
    """`bench.py --gpus 2` without an outer launcher starts two ranks through
    torch.distributed.run (gloo rendezvous on 127.0.0.1).  The oracle arm runs on CPU, so the
    spawn path is exercised here without a GPU: rank 0 prints one line that reports both
    ranks, the other rank exits 0 without work."""
    import json
    import subprocess
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                          "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    # the reference arm's line carries the same metric, unit and workload as the main arm's
    import bench
    assert line["metric"] == bench.METRIC and line["unit"] == "TFLOPS" and line["higher_is_better"] is True
    assert line["config"]["workload"] == bench.WORKLOAD_NAME
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
