"""Host-side logic of bench.py without a GPU: the multi-rank timing reduction over gloo, and the
reference (oracle) arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier()
        slowest = bench.max_over_ranks(1.0 + rank)  # rank r "took" 1 + r seconds
        value = bench.weak_scaling_value(100.0, 1.0 + rank)
        out[rank] = (slowest, value)
    finally:
        torch.distributed.destroy_process_group()


def test_two_rank_timing_reduction_over_gloo():
    world, port = 2, _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    for rank in range(world):
        slowest, value = out[rank]
        assert slowest == 2.0  # max over ranks
        assert value == world * 100.0 / 2.0  # all ranks' units over the slowest rank's time


def test_reference_arm_prints_one_json_line():
    env = dict(os.environ, PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_traffic_entries_ignore_comment_edits():
    """The source hash that keys the committed DRAM traffic per kernel covers the code only: a comment edit
    keeps it, a code edit changes it (bench.py then reports the traffic as null)."""
    sys.path.insert(0, ROOT)
    import bench
    code = "int f(int x) {  // doubles x\n    /* body */ return 2 * x;\n}\n"
    assert bench._code_only(code) == bench._code_only(code.replace("doubles x", "twice x").replace("body", "b"))
    assert bench._code_only(code) != bench._code_only(code.replace("2 * x", "3 * x"))
