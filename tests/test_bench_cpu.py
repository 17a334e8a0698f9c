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


def _split_rank_main(rank, world, port, out):
    """One rank of the head split: its slice of a small problem through the oracle (standing in for the GPU
    library on CPU ranks); the test alone gathers the slices to compare them with the unsplit run."""
    sys.path.insert(0, ROOT)
    from gated_delta_rule_27_gb300 import shard, workloads
    from oracle import oracle
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        H = 5
        inp = workloads.prefill_inputs([23, 0, 17], H=H, d=16, dtype=torch.float32, seed=91, s0_std=0.3)
        lo, hi = shard.head_range(H, world, rank)
        part = [shard.take_heads(x, lo, hi, 1).double().numpy() for x in (inp.q, inp.k, inp.v, inp.g, inp.beta)]
        S0 = shard.take_heads(inp.S0, lo, hi, 1).double().numpy()
        o, S, _ = oracle.run(*part, inp.cu_seqlens.numpy(), S0=S0, threads=1)
        gathered = [None] * world
        torch.distributed.all_gather_object(gathered, (lo, hi, o, S))
        if rank == 0:
            o_full, S_full, _ = oracle.run(*(x.double().numpy() for x in (inp.q, inp.k, inp.v, inp.g, inp.beta)),
                                           inp.cu_seqlens.numpy(), S0=inp.S0.double().numpy(), threads=1)
            import numpy as np
            spans = [(a, b) for a, b, _, _ in gathered]
            o_cat = np.concatenate([x for _, _, x, _ in gathered], axis=1)
            S_cat = np.concatenate([x for _, _, _, x in gathered], axis=1)
            out["spans"] = spans
            out["same"] = bool(np.array_equal(o_cat, o_full) and np.array_equal(S_cat, S_full))
    finally:
        torch.distributed.destroy_process_group()


def test_head_split_over_two_gloo_ranks_concatenates_to_the_unsplit_run():
    world, port = 2, _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_split_rank_main, args=(world, port, out), nprocs=world, join=True)
    assert out["spans"] == [(0, 3), (3, 5)]
    assert out["same"]  # every chain is independent: the split changes no bit


def test_head_ranges_cover_every_head_once():
    sys.path.insert(0, ROOT)
    from gated_delta_rule_27_gb300 import shard
    for H in (1, 5, 16, 32, 33):
        for world in (1, 2, 3, 4, 8):
            spans = [shard.head_range(H, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == H
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            assert max(b - a for a, b in spans) - min(b - a for a, b in spans) <= 1
