"""The multi-rank path of bench.py on CPU: two gloo ranks launched the way
torchrun launches them (RANK / WORLD_SIZE / MASTER_ADDR in the environment);
each rank's timing is reduced to the maximum over ranks."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    w, r, lr = bench.dist_env()
    dist.init_process_group("gloo", rank=r, world_size=w)
    try:
        mine = 10.0 + 7.5 * r                 # a slower rank 1
        results[r] = (w, r, lr, bench.max_over_ranks(mine, w, "cpu"))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time():
    ctx = torch.multiprocessing.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        got = dict(results)
    assert got[0] == (2, 0, 0, 17.5)
    assert got[1] == (2, 1, 1, 17.5)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.25, 1, "cpu") == 3.25


def test_reference_arm_prints_one_contract_line():
    # bench.py --impl reference times the CPU oracle (the reference arm) and
    # prints one JSON line with the contract's keys; on a tiny shape here
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2", "--warmup", "3",
                        "--shape", "64,48,80"], cwd=root, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert (d["steps"], d["warmup"], d["n_gpus"]) == (2, 3, 1)
    assert d["config"]["M"] == 64 and d["config"]["N"] == 48 and d["config"]["K"] == 80
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
