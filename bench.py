"""Benchmark of libkda on GB300: chunked prefill tokens/s and decode step time.

One step = one kda_prefill_chunked pass over the prefill workload (B=1,
H=16, T=4096, d=128, bf16 q/k/v, fp32 gates, chunk 64, zero S0), the
configuration the headline metric is quoted on.  In the same run, and
reported under their own keys, the packed-varlen workload (8 documents,
H=32), the long-context workload (B=2, H=32, T=65536, one pass), the decode
workload (256 sequences x 32 heads, fp32 state of 512 MiB, 1000 pre-generated
steps) and the indexed decode over a state pool are timed.  Prints ONE JSON
line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl libkda|reference]
  python bench.py --profile-case prefill|varlen|long|decode|decode-n64|conv [--repeat R]   (untimed, for ncu)
  python bench.py --compare-plans      (pass time of each tensor-core launch plan, one JSON line each)

Timing: CUDA events on the launching stream, L2 flushed (a 256 MB write)
before every timed prefill step (the prefill inputs, 101 MB, would otherwise
sit in the 129 MB L2); the decode state (512 MiB) is larger than L2.
Under torchrun (N > 1) the heads are split across ranks with no collective on
the data path: the problem has 16 N heads and rank r owns heads
[16 r, 16 (r + 1)) (weak scaling); value = all ranks' tokens x heads / 16 over
the slowest rank's time.  `--impl reference` times the fp64 CPU oracle on the
same workload instead.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from gated_delta_rule_27_gb300 import workloads  # noqa: E402

METRIC = "KDA prefill tokens/s and decode step µs (state GB/s) on 1 GB300, % of roofline"
WORKLOAD = "prefill"
DESCRIPTION = {
    "prefill": "prefill B=1 H=16 T=4096 d_k=d_v=128 chunk=64 bf16 q/k/v fp32 g/beta zero S0",
    "varlen": "packed varlen: 8 documents with seeded lengths U[128,8192], H=32, d=128, chunk 64, bf16 q/k/v, "
              "fp32 g/beta, state reset per document",
    "long": "long context B=2 H=32 T=65536 d=128 chunk 64 bf16, one prefill pass",
}
PREFILL_BYTES_PER_TOKEN_HEAD = 3 * 128 * 2 + 128 * 4 + 4 + 128 * 2  # q,k,v bf16 + g fp32 + beta + o bf16
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(
        os.environ.get("LOCAL_RANK", "0"))


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS if k in p}, "measured (MEASURED_PEAKS.json)"
    return dict(FALLBACK_PEAKS), "fallback (no MEASURED_PEAKS.json on this box)"


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="kda_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) < 9:
                        continue
                    try:
                        sm.append(float(parts[1]))
                        smax.append(float(parts[2]))
                    except ValueError:
                        continue
                    for n, v in zip(names, parts[5:9]):
                        if v.lower() == "active":
                            reasons.add(n)
            os.unlink(self.path)
        except OSError:
            pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# profile summaries committed under profiles/ (ncu DRAM traffic per launch)
# ---------------------------------------------------------------------------
def _code_only(text: str) -> str:
    """C++ source without comments and with whitespace collapsed, so that an edit to a comment does not
    count as a change of the kernel (the sources hold no string literal with a comment marker)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def source_hash(kernel_file: str) -> str:
    """Hash of the code (comments excluded) of a kernel's source file and the two shared headers."""
    h = hashlib.sha256()
    for rel in (kernel_file, "gated_delta_rule_27_gb300/csrc/kda_internal.cuh",
                "gated_delta_rule_27_gb300/csrc/kda_tc.cuh"):
        p = os.path.join(ROOT, rel)
        if os.path.exists(p):
            with open(p, encoding="utf-8") as f:
                h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


KERNEL_SOURCES = {
    "prefill_prepare_simt": "gated_delta_rule_27_gb300/csrc/kda_prefill_simt.cu",
    "prefill_state_simt": "gated_delta_rule_27_gb300/csrc/kda_prefill_simt.cu",
    "chunk_index": "gated_delta_rule_27_gb300/csrc/kda_prefill_simt.cu",
    "prefill_prepare_tc": "gated_delta_rule_27_gb300/csrc/kda_prefill_tc.cu",
    "prefill_state_tc": "gated_delta_rule_27_gb300/csrc/kda_prefill_tc.cu",
    "prefill_output_tc": "gated_delta_rule_27_gb300/csrc/kda_prefill_tc.cu",
    "prefill_chain_tc": "gated_delta_rule_27_gb300/csrc/kda_prefill_tc.cu",
    "prefill_pipe_tc": "gated_delta_rule_27_gb300/csrc/kda_prefill_tc.cu",
    "prefill_state_fold_tc": "gated_delta_rule_27_gb300/csrc/kda_prefill_tc.cu",
    "out_gated_norm": "gated_delta_rule_27_gb300/csrc/kda_prefill_simt.cu",
    "decode_step": "gated_delta_rule_27_gb300/csrc/kda_decode.cu",
}


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from profiles/traffic.json, or None if absent or the kernel changed since."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path) or kernel not in KERNEL_SOURCES:
        return None
    with open(path) as f:
        table = json.load(f)
    entry = table.get("%s/%s" % (kernel, workload))
    if not entry or entry.get("source_hash") != source_hash(KERNEL_SOURCES[kernel]):
        return None
    return float(entry["dram_bytes_per_launch"])


# ---------------------------------------------------------------------------
# libkda arm
# ---------------------------------------------------------------------------
def new_events(n):
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in evs:
        e.record()  # materialise the underlying cudaEvent_t
    return evs


def bench_prefill(libkda, steps, warmup, dev, rank, name=WORKLOAD, head_block=0):
    """Times kda_prefill_chunked on one prefill workload: `steps` plain calls, each after an L2 flush and
    bracketed by events, then the same number of profiled calls for the per-kernel split."""
    w = workloads.WORKLOADS[name]
    inp = workloads.workload_prefill(name, device=dev, head_block=head_block)
    q, k, v, g, beta, cu = inp.q, inp.k, inp.v, inp.g, inp.beta, inp.cu_seqlens
    T, H, d = q.shape
    N = inp.num_seqs
    o = torch.empty((T, H, d), dtype=v.dtype, device=dev)
    S_final = torch.empty((N, H, d, d), dtype=torch.float32, device=dev)
    ws = libkda.new_workspace(T, N, H, d, d, libkda.KDA_BF16, w["chunk"], dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    nk = libkda.PREFILL_MAX_KERNELS + 1
    per_step = [new_events(nk) for _ in range(steps)]
    names = None

    def one(evs):
        return libkda.kda_prefill_chunked_profiled(q, k, v, g, beta, cu, o, evs, S_final=S_final, workspace=ws,
                                                   chunk_size=w["chunk"])

    def plain():
        libkda.kda_prefill_chunked(q, k, v, g, beta, cu, o, S_final=S_final, workspace=ws, chunk_size=w["chunk"])

    warm_ev = new_events(nk)
    for _ in range(warmup):
        flush.zero_()
        plain()
        flush.zero_()
        one(warm_ev)
    torch.cuda.synchronize()
    # the timed steps: plain calls, an event on each side of every call (after its L2 flush)
    step_ev = [new_events(2) for _ in range(steps)]
    barrier()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("kda prefill timed: " + name)
    t_wall = time.perf_counter()
    for i in range(steps):
        flush.zero_()
        step_ev[i][0].record()
        plain()
        step_ev[i][1].record()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    barrier()
    torch.cuda.synchronize()
    wall_s = time.perf_counter() - t_wall
    step_ms = [step_ev[i][0].elapsed_time(step_ev[i][1]) for i in range(steps)]
    # the per-kernel split: the same number of calls with an event before each kernel
    torch.cuda.nvtx.range_push("kda prefill per-kernel split: " + name)
    for i in range(steps):
        flush.zero_()
        names = one(per_step[i])
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    n = len(names)
    kern_ms = {names[j]: [per_step[i][j].elapsed_time(per_step[i][j + 1]) for i in range(steps)] for j in range(n)}
    token_heads = T * H
    alg_bytes = PREFILL_BYTES_PER_TOKEN_HEAD * token_heads + N * H * d * d * 4
    return dict(name=name, T=T, H=H, d=d, N=N, chunk=w["chunk"], step_ms=step_ms, kern_ms=kern_ms, names=names,
                wall_s=wall_s, launches=n * steps, inp=inp, alg_bytes=alg_bytes)


def bench_host_overhead(libkda, dev, inp, calls=400):
    """Host time of one call into the C ABI (argument checks, cached launch set-up, the launches themselves),
    measured around the raw ctypes call with pointers marshalled once, next to the cost of a ctypes call that
    does nothing (kda_status_string) and of the Python wrapper.  The device is drained every 8 calls, outside
    the timed calls, so that the launch queue never fills."""
    lib = libkda.load()
    T, H, d = inp.q.shape
    N = inp.num_seqs
    o = torch.empty_like(inp.v)
    S = torch.empty((N, H, d, d), device=dev)
    ws = libkda.new_workspace(T, N, H, d, d, libkda.KDA_BF16, 64, dev)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    pre = (p(inp.q), p(inp.k), p(inp.v), p(inp.g), p(inp.beta), p(inp.cu_seqlens), N, T, H, d, d, libkda.KDA_BF16,
           64, None, p(o), p(S), p(ws), ws.numel() * ws.element_size(), st)
    dq = torch.zeros((N, H, d), dtype=torch.bfloat16, device=dev)
    dg = torch.zeros((N, H, d), dtype=torch.float32, device=dev)
    db = torch.zeros((N, H), dtype=torch.float32, device=dev)
    do = torch.empty_like(dq)
    dec = (p(dq), p(dq), p(dq), p(dg), p(db), N, H, d, d, libkda.KDA_BF16, p(S), p(do), st)

    def timed(fn):
        out = []
        for i in range(calls):
            if i % 8 == 0:
                torch.cuda.synchronize()
            t0 = time.perf_counter_ns()
            fn()
            out.append((time.perf_counter_ns() - t0) * 1e-3)
        torch.cuda.synchronize()
        return statistics.median(out[calls // 8:])

    def prefill_raw():
        if lib.kda_prefill_chunked(*pre) != libkda.KDA_OK:
            raise RuntimeError("kda_prefill_chunked failed")

    def decode_raw():
        if lib.kda_decode_step(*dec) != libkda.KDA_OK:
            raise RuntimeError("kda_decode_step failed")

    res = {"prefill_call_us": timed(prefill_raw), "decode_call_us": timed(decode_raw),
           "ctypes_floor_us": timed(lambda: lib.kda_status_string(0)),
           "prefill_python_wrapper_us": timed(lambda: libkda.kda_prefill_chunked(
               inp.q, inp.k, inp.v, inp.g, inp.beta, inp.cu_seqlens, o, S_final=S, workspace=ws))}
    res["note"] = ("median host wall time per call (time.perf_counter_ns around the call, launches included, "
                   "device drained every 8 calls outside the timed calls); the *_call_us figures call the C ABI "
                   "through ctypes with pre-marshalled pointers")
    return res


def compare_plans(libkda, dev, reps=8):
    """Pass time of each tensor-core launch plan, forced through the test hook, on the prefill workload and on
    single documents of 4096 tokens with 8, 24 and 32 heads, L2 flushed before every pass."""
    flush = torch.empty(64 << 20, device=dev)
    cases = [("prefill", workloads.workload_prefill("prefill", device=dev))]
    for H in (8, 24, 32):
        cases.append(("single document T=4096 H=%d" % H,
                      workloads.prefill_inputs([4096], H=H, d=128, dtype=torch.bfloat16, seed=3, device=dev)))
    plans = [("auto", libkda.PLAN_AUTO), ("three", libkda.PLAN_THREE), ("chain", libkda.PLAN_CHAIN),
             ("pipe", libkda.PLAN_PIPE)]
    out = []
    try:
        for name, inp in cases:
            T, H, d = inp.q.shape
            N = inp.num_seqs
            o = torch.empty_like(inp.v)
            S = torch.empty((N, H, d, d), device=dev)
            ws = libkda.new_workspace(T, N, H, d, d, libkda.KDA_BF16, 64, dev)
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(libkda.PREFILL_MAX_KERNELS + 1)]
            for e in evs:
                e.record()
            for pname, plan in plans:
                libkda.testing_set_plan(plan)
                tot, per = [], {}
                for rep in range(reps):
                    flush.zero_()
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record()
                    libkda.kda_prefill_chunked(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.cu_seqlens, o, S_final=S,
                                               workspace=ws)
                    b.record()
                    flush.zero_()
                    names = libkda.kda_prefill_chunked_profiled(inp.q, inp.k, inp.v, inp.g, inp.beta,
                                                                inp.cu_seqlens, o, evs, S_final=S, workspace=ws)
                    torch.cuda.synchronize()
                    if rep >= 2:
                        tot.append(a.elapsed_time(b) * 1e3)
                        for j, n in enumerate(names):
                            per.setdefault(n, []).append(evs[j].elapsed_time(evs[j + 1]) * 1e3)
                out.append({"case": name, "plan": pname, "us": round(statistics.median(tot), 1),
                            "kernels_us": {n: round(statistics.median(t), 1) for n, t in per.items()}})
    finally:
        libkda.testing_set_plan(libkda.PLAN_AUTO)
    return out


def bench_e2e(libkda, steps, warmup, dev, inp):
    """The prefill through the C ABI from pinned HOST buffers, every step's host->device copy of its inputs and
    device->host copy of its results (o, S_final) inside the timed region.  Steps are independent requests and
    are pipelined with two sets of device and host buffers: step i's inputs are copied in (three copy streams)
    while step i-1 computes and step i-2's results are copied out."""
    w = workloads.WORKLOADS[WORKLOAD]
    host = [x.to("cpu").pin_memory() for x in (inp.q, inp.k, inp.v, inp.g, inp.beta, inp.cu_seqlens)]
    T, H, d = inp.q.shape
    N = inp.num_seqs
    nb = 2
    dbuf = [[torch.empty_like(x, device=dev) for x in host] for _ in range(nb)]
    o = [torch.empty((T, H, d), dtype=inp.v.dtype, device=dev) for _ in range(nb)]
    S_final = [torch.empty((N, H, d, d), dtype=torch.float32, device=dev) for _ in range(nb)]
    o_h = [torch.empty((T, H, d), dtype=inp.v.dtype).pin_memory() for _ in range(nb)]
    S_h = [torch.empty((N, H, d, d), dtype=torch.float32).pin_memory() for _ in range(nb)]
    ws = libkda.new_workspace(T, N, H, d, d, libkda.KDA_BF16, w["chunk"], dev)
    h2d = sum(x.numel() * x.element_size() for x in host)
    d2h = o_h[0].numel() * o_h[0].element_size() + S_h[0].numel() * S_h[0].element_size()
    # inputs travel on three copy streams with about equal bytes each (g; q and k; v, beta, cu_seqlens),
    # so that several copy engines work at once
    groups = [[3], [0, 1], [2, 4, 5]]
    s_in = [torch.cuda.Stream(dev) for _ in groups]
    s_comp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    in_done = [[torch.cuda.Event() for _ in groups] for _ in range(nb)]
    comp_done = [torch.cuda.Event() for _ in range(nb)]
    out_done = [torch.cuda.Event() for _ in range(nb)]

    def step(i, compute=True):
        b = i % nb
        for gi, (sg, members) in enumerate(zip(s_in, groups)):
            with torch.cuda.stream(sg):
                if i >= nb:
                    sg.wait_event(comp_done[b])  # the compute of step i - 2 has read this input set
                for m in members:
                    dbuf[b][m].copy_(host[m], non_blocking=True)
                in_done[b][gi].record(sg)
        for e in in_done[b]:
            s_comp.wait_event(e)
        if i >= nb:
            s_comp.wait_event(out_done[b])  # step i - 2's results have left this output set
        if compute:
            libkda.kda_prefill_chunked(*dbuf[b], o[b], S_final=S_final[b], workspace=ws, chunk_size=w["chunk"],
                                       stream=s_comp)
        comp_done[b].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[b])
            o_h[b].copy_(o[b], non_blocking=True)
            S_h[b].copy_(S_final[b], non_blocking=True)
            out_done[b].record(s_out)

    def timed(compute):
        for i in range(warmup):
            step(i, compute)
        torch.cuda.synchronize()
        ev = new_events(2)
        ev[0].record(s_in[0])
        for sg in s_in[1:]:
            sg.wait_event(ev[0])
        for i in range(steps):
            step(i, compute)
        ev[1].record(s_out)
        torch.cuda.synchronize()
        return ev[0].elapsed_time(ev[1]) / steps

    ms = timed(True)
    # the same copies in the same pipeline without the prefill: the host link's floor for this step
    copy_ms = timed(False)
    return dict(ms=ms, copy_ms=copy_ms, h2d=h2d, d2h=d2h, tokens=T)


def bench_decode(libkda, warmup, dev):
    """The decode workload as specified: 1000 successive steps whose inputs are all generated on the device
    beforehand (about 10.5 GB), each step timed alone with events; the median is reported."""
    w = workloads.WORKLOADS["decode"]
    N, H, d, steps = w["N"], w["H"], w["d"], w["steps"]
    dec = workloads.decode_inputs(steps, N, H, d, w["dtype"], seed=workloads.workload_seed("decode"), device=dev)
    S = dec.S0.clone()
    o = torch.empty((N, H, d), dtype=w["dtype"], device=dev)
    args = lambda t: (dec.q[t], dec.k[t], dec.v[t], dec.g[t], dec.beta[t])
    for t in range(warmup):
        libkda.kda_decode_step(*args(t), S, o)
    S.copy_(dec.S0)
    torch.cuda.synchronize()
    evs = [new_events(2) for _ in range(steps)]
    torch.cuda.nvtx.range_push("kda decode timed: 1000 steps")
    for i in range(steps):
        evs[i][0].record()
        libkda.kda_decode_step(*args(i), S, o)
        evs[i][1].record()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    us = [e[0].elapsed_time(e[1]) * 1e3 for e in evs]
    state_bytes = N * H * d * d * 4
    io_bytes = N * H * (3 * d * 2 + d * 4 + 4 + d * 2)
    first = workloads.DecodeInputs(*(x[:4] for x in (dec.q, dec.k, dec.v, dec.g, dec.beta)), dec.S0,
                                   dec.extreme_steps[:0])
    del dec
    return dict(us=us, state_bytes=state_bytes, io_bytes=io_bytes, N=N, H=H, d=d, launches=steps, dec=first)


def bench_decode_indexed(libkda, steps, warmup, dev):
    """Indexed decode over a state pool: 256 of 512 slots (a seeded random choice) active, 32 heads, d = 128."""
    slots, active, H, d = 512, 256, 32, 128
    gen = torch.Generator(device="cpu").manual_seed(workloads.BASE_SEED + 11)
    idx = torch.randperm(slots, generator=gen)[:active].to(torch.int32).to(dev)
    pool = torch.empty((slots, H, d, d), device=dev).normal_(0.0, 0.1)
    n_in = 16
    dec = workloads.decode_inputs(n_in, active, H, d, torch.bfloat16, seed=workloads.BASE_SEED + 12, device=dev)
    o = torch.empty((active, H, d), dtype=torch.bfloat16, device=dev)
    args = lambda t: (dec.q[t % n_in], dec.k[t % n_in], dec.v[t % n_in], dec.g[t % n_in], dec.beta[t % n_in])
    for t in range(warmup):
        libkda.kda_decode_step_indexed(*args(t), idx, pool, o)
    torch.cuda.synchronize()
    evs = [new_events(2) for _ in range(steps)]
    for i in range(steps):
        evs[i][0].record()
        libkda.kda_decode_step_indexed(*args(i), idx, pool, o)
        evs[i][1].record()
    torch.cuda.synchronize()
    us = statistics.median([e[0].elapsed_time(e[1]) * 1e3 for e in evs])
    nbytes = 2 * active * H * d * d * 4 + active * H * (3 * d * 2 + d * 4 + 4 + d * 2) + active * 4
    return dict(us=us, bytes=nbytes, slots=slots, active=active, H=H, d=d, steps=steps)


def bench_sublayer(steps, warmup, dev):
    """Whole-sublayer timing with synthetic weights (measurement only): the stages around the recurrence --
    projections (cuBLAS bf16 GEMMs and the gate activations), short convolution, recurrence with the fused
    normalisations, output projection -- each bracketed by events, for the prefill workload's shape and for
    one decode step of the decode workload's shape.  Hidden size H * d.  The stages made of many small
    launches (projections, convolution, output projection) are replayed from CUDA graphs, so that their
    intervals are device time rather than the host's launch latency; the recurrence is enqueued while the GPU
    is still busy with the stages before it."""
    from gated_delta_rule_27_gb300 import libkda, sublayer
    stages = ["projections", "short_conv", "recurrence", "output_projection"]
    out = {}
    cases = (("prefill", 1, 4096, 16), ("decode", 256, 1, 32))

    def graph_of(fn):
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            fn()
        torch.cuda.current_stream(dev).wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        return g

    for name, N, T, H in cases:
        d = 128
        D = H * d
        R = T * N if name == "prefill" else N
        w = sublayer.synthetic_weights(D, H, d, seed=workloads.BASE_SEED + 21, device=dev)
        gen = torch.Generator(device="cpu").manual_seed(workloads.BASE_SEED + 22)
        flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
        x = torch.randn((R, D), generator=gen).to(torch.bfloat16).to(dev)
        b = sublayer.Buffers(R, N, H, d, dev)
        y = torch.empty((R, D), dtype=torch.bfloat16, device=dev)
        HD = H * d
        if name == "prefill":
            cu = workloads.cu_from_lengths([T], device=dev)
            ws = libkda.new_workspace(T, 1, H, d, d, libkda.KDA_BF16, 64, dev)

            def conv():
                for src, cw, dst, st in ((b.q, w.conv_q, b.qc, b.conv_state[0]), (b.k, w.conv_k, b.kc,
                                                                                 b.conv_state[1]),
                                         (b.v, w.conv_v, b.vc, b.conv_state[2])):
                    libkda.kda_short_conv_prefill(src, cw, cu, dst, conv_state_out=st)

            def rec():
                libkda.kda_prefill_chunked_ex(b.qc.view(T, H, d), b.kc.view(T, H, d), b.vc.view(T, H, d),
                                              b.g.view(T, H, d), b.beta, cu, b.o, S_final=b.S, workspace=ws,
                                              qk_l2norm=True, qk_eps=1e-6, out_gate=b.z.view(T, H, d),
                                              out_weight=w.out_weight, out_eps=1e-6)
        else:
            b.S.normal_(0.0, 0.1)
            for st in b.conv_state:
                st.zero_()

            def conv():
                for src, cw, st, dst in ((b.q, w.conv_q, b.conv_state[0], b.qc), (b.k, w.conv_k, b.conv_state[1],
                                                                                 b.kc),
                                         (b.v, w.conv_v, b.conv_state[2], b.vc)):
                    libkda.kda_short_conv_decode(src, cw, st, dst)

            def rec():
                libkda.kda_decode_step_ex(b.qc.view(N, H, d), b.kc.view(N, H, d), b.vc.view(N, H, d),
                                          b.g.view(N, H, d), b.beta, b.S, b.o, qk_l2norm=True, qk_eps=1e-6,
                                          out_gate=b.z.view(N, H, d), out_weight=w.out_weight, out_eps=1e-6)

        proj = lambda: sublayer._project(x, w, b)
        outp = lambda: torch.matmul(b.o.view(R, HD), w.W_o, out=y)
        for _ in range(warmup):
            proj(); conv(); rec(); outp()
        g_proj, g_conv, g_out = graph_of(proj), graph_of(conv), graph_of(outp)
        per = {k: [] for k in stages}
        for _ in range(steps):
            ev = new_events(5)
            torch.cuda.synchronize()
            flush.zero_()
            ev[0].record()
            g_proj.replay()
            ev[1].record()
            g_conv.replay()
            ev[2].record()
            rec()
            ev[3].record()
            g_out.replay()
            ev[4].record()
            torch.cuda.synchronize()
            for j, k in enumerate(stages):
                per[k].append(ev[j].elapsed_time(ev[j + 1]))
        ms = {k: statistics.median(v) for k, v in per.items()}
        total = sum(ms.values())
        conv_bytes = 3 * R * HD * 2 * 2 + (3 * 2 * N * (sublayer.CONV_W - 1) * HD * 4 if name == "decode" else
                                            3 * N * (sublayer.CONV_W - 1) * HD * 4)
        out[name] = {"shape": "N=%d T=%d H=%d d=%d hidden=%d bf16, synthetic weights" % (N, T, H, d, D),
                     "ms": {k: round(v, 5) for k, v in ms.items()}, "total_ms": total,
                     "recurrence_share": ms["recurrence"] / total,
                     "short_conv_gbs": conv_bytes / (ms["short_conv"] * 1e-3) / 1e9,
                     "note": "projections are cuBLAS GEMMs (q, k, v, decay gate, write gate, output gate) plus "
                             "torch gate activations; short_conv, recurrence (with the q/k L2 norm and the gated "
                             "output norm fused) are libkda kernels; buffers allocated once; L2 flushed before "
                             "every step; projections, convolution and output projection replayed from CUDA "
                             "graphs"}
    return out


def barrier():
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.barrier()


def max_over_ranks(x: float) -> float:
    """The slowest rank's value (timing control plane only; no data-path collective)."""
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        return float(t.item())
    return x


def weak_scaling_value(units_per_rank: float, seconds_per_rank: float) -> float:
    """Whole-job throughput: every rank processes its own copy of the workload, the job ends with the
    slowest rank."""
    world = torch.distributed.get_world_size() if torch.distributed.is_initialized() else 1
    return world * units_per_rank / max_over_ranks(seconds_per_rank)


def cpu_baseline_prefill(inp, budget_s=10.0, heads=None):
    """The fp64 oracle on a prefill workload (all heads, or the first `heads` of them as a bounded sample),
    repeated until ~budget_s; the value is scaled to tokens/s of the whole workload."""
    from oracle import oracle
    H = inp.q.shape[1]
    hs = H if heads is None else min(heads, H)
    f = lambda x: x[:, :hs].detach().to("cpu", torch.float64).contiguous().numpy()
    args = [f(x) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta)]
    cu = inp.cu_seqlens.cpu().numpy()
    threads = min(oracle.default_threads(), inp.num_seqs * hs)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.run(*args, cu, threads=threads)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= 50:
            break
    what = "the full workload" if hs == H else "heads 0..%d of %d of the workload" % (hs - 1, H)
    return dict(value=reps * inp.total_tokens * hs / H / el, unit="tokens/s", cores=threads, kind="oracle",
                sample="%s (%d tokens x %d heads), %d repetition(s) in %.1f s; scaled to all %d heads"
                       % (what, inp.total_tokens, hs, reps, el, H))


def cpu_baseline_decode(dec, steps=4):
    from oracle import oracle
    import numpy as np
    N, H, d = dec.S0.shape[0], dec.S0.shape[1], dec.S0.shape[2]
    f = lambda x: x.detach().to("cpu", torch.float64).numpy()
    S = f(dec.S0)
    threads = oracle.default_threads()
    cu = np.arange(N + 1)
    t0 = time.perf_counter()
    for t in range(steps):
        _, S, _ = oracle.run(f(dec.q[t]), f(dec.k[t]), f(dec.v[t]), f(dec.g[t]), f(dec.beta[t]), cu, S0=S,
                             threads=threads)
    el = time.perf_counter() - t0
    return dict(value=el / steps * 1e6, unit="us/step", cores=threads, kind="oracle",
                sample="%d decode steps over all %d x %d chains" % (steps, N, H))


def prefill_summary(pf, pk, pk_src, world):
    """Per-pass figures of one prefill workload: time, throughput, roofline of the pass and of its dominant
    kernel."""
    T, H, N, d = pf["T"], pf["H"], pf["N"], pf["d"]
    hbm = pk["hbm_gbs"]
    ms = max_over_ranks(statistics.mean(pf["step_ms"]))
    token_heads = T * H
    kern_avg = {n: statistics.mean(v) for n, v in pf["kern_ms"].items()}
    dom = max(kern_avg, key=kern_avg.get)
    # the path's unavoidable bytes, each counted in the kernel that moves it: the inputs are read by the
    # preparation, the final state written by the state pass, o written by the output pass (the chain
    # kernel writes both; the SIMT path's state pass writes both); records between kernels do not count
    read_bytes = (3 * d * 2 + d * 4 + 4) * token_heads  # q, k, v, g, beta
    s_bytes = N * H * d * d * 4
    o_bytes = d * 2 * token_heads
    if "prepare" in dom:
        dom_bytes = read_bytes
    elif "output" in dom:
        dom_bytes = o_bytes
    elif "chain" in dom:
        dom_bytes = s_bytes + o_bytes
    elif "state" in dom:
        dom_bytes = s_bytes + (o_bytes if "simt" in dom else 0)
    else:
        dom_bytes = pf["alg_bytes"]
    achieved = dom_bytes / (kern_avg[dom] * 1e-3) / 1e9
    roofline = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "traffic": ncu_traffic(dom, pf["name"]), "algorithmic_bytes": dom_bytes,
                "avg_launch_ms": kern_avg[dom], "peak_source": pk_src,
                "kernels_ms": {n: round(m, 5) for n, m in kern_avg.items()}}
    pass_bw = pf["alg_bytes"] / (ms * 1e-3) / 1e9
    pass_roofline = {"bound": "hbm", "algorithmic_bytes": pf["alg_bytes"], "achieved": pass_bw, "peak": hbm,
                     "unit": "GB/s", "frac": pass_bw / hbm, "roofline_us": pf["alg_bytes"] / (hbm * 1e9) * 1e6}
    return dict(ms=ms, tokens_per_s=world * T * H / pf["H"] / (ms * 1e-3), roofline=roofline,
                pass_roofline=pass_roofline)


def run_libkda(args):
    from gated_delta_rule_27_gb300 import libkda, shard
    rank, world, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    libkda.load()
    pk, pk_src = peaks()
    # head split: the problem has 16 * world heads; this rank owns block `rank` of 16 of them
    H_block = workloads.WORKLOADS[WORKLOAD]["H"]
    lo, hi = shard.head_range(H_block * world, world, rank)
    assert (lo, hi) == (rank * H_block, (rank + 1) * H_block)

    with ClockSampler(local) as clk:
        pf = bench_prefill(libkda, args.steps, args.warmup, dev, rank, head_block=rank)
        dc = bench_decode(libkda, max(args.warmup, 3), dev)
    clocks = clk.summary()
    others = {}
    if not args.headline_only:
        for name in ("varlen", "long"):
            steps = min(args.steps, 10 if name == "varlen" else 5)
            others[name] = bench_prefill(libkda, steps, 3, dev, rank, name=name, head_block=rank)
        di = bench_decode_indexed(libkda, 50, 3, dev)
        sub = bench_sublayer(min(args.steps, 10), 3, dev)
    e2e = bench_e2e(libkda, args.steps, args.warmup, dev, pf["inp"])
    host = bench_host_overhead(libkda, dev, pf["inp"])

    T = pf["T"]
    summ = prefill_summary(pf, pk, pk_src, world)
    ms_per_step = summ["ms"]
    value = world * T * pf["N"] / (ms_per_step * 1e-3)
    hbm = pk["hbm_gbs"]

    us = sorted(dc["us"])
    dec_us = statistics.median(us)
    dec_bytes = 2 * dc["state_bytes"] + dc["io_bytes"]
    dec_gbs = dec_bytes / (dec_us * 1e-6) / 1e9
    decode = {"workload": "decode N=256 H=32 d=128 bf16 q/k/v, fp32 state 512 MiB, 1000 pre-generated steps "
                          "(5% extreme gates), each timed alone",
              "us_per_step_median": dec_us, "us_per_step_mean": statistics.mean(us),
              "state_gbs": 2 * dc["state_bytes"] / (dec_us * 1e-6) / 1e9,
              "roofline": {"bound": "hbm", "kernel": "decode_step", "achieved": dec_gbs, "peak": hbm, "unit": "GB/s",
                           "frac": dec_gbs / hbm, "frac_of_8tbs": dec_gbs / 8000.0, "algorithmic_bytes": dec_bytes,
                           "traffic": ncu_traffic("decode_step", "decode"), "peak_source": pk_src},
              "steps": len(us), "gpu_launches": dc["launches"]}

    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": DESCRIPTION[WORKLOAD], "global_batch": world * pf["N"], "seq_len": T,
                       "heads": pf["H"] * world, "d": pf["d"], "chunk": pf["chunk"],
                       "l2": "flushed (256 MB write) before every timed prefill step",
                       "parallelism": ("head split: rank r owns heads [16r, 16r+16) of %d, no collective"
                                       % (16 * world)) if world > 1 else "single-gpu"},
            "roofline": summ["roofline"], "pass_roofline": summ["pass_roofline"], "decode": decode,
            "e2e": {"value": world * e2e["tokens"] / (max_over_ranks(e2e["ms"]) * 1e-3), "unit": "tokens/s",
                    "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                    "ms_per_step": e2e["ms"], "copy_only_ms_per_step": e2e["copy_ms"],
                    "link_gbs": (e2e["h2d"] + e2e["d2h"]) / (e2e["copy_ms"] * 1e-3) / 1e9,
                    "frac_of_copy_floor": e2e["copy_ms"] / e2e["ms"],
                    "note": "pinned host inputs copied in and o, S_final copied out every step; consecutive "
                            "steps pipelined on copy-in / compute / copy-out streams"},
            "host_overhead": host, "gpu_launches": pf["launches"], "clocks": clocks,
            "wall_s_timed_region": pf["wall_s"]}
    for name, p in others.items():
        ps = prefill_summary(p, pk, pk_src, world)
        line[name] = {"workload": DESCRIPTION[name], "tokens": p["T"], "documents": p["N"], "heads": p["H"],
                      "ms_per_pass": ps["ms"], "tokens_per_s": ps["tokens_per_s"], "steps": len(p["step_ms"]),
                      "pass_roofline": ps["pass_roofline"], "roofline": ps["roofline"]}
    if not args.headline_only:
        di_gbs = di["bytes"] / (di["us"] * 1e-6) / 1e9
        line["decode_indexed"] = {
            "workload": "indexed decode: %d of %d pool slots active (seeded random), H=%d, d=%d, bf16"
                        % (di["active"], di["slots"], di["H"], di["d"]),
            "us_per_step_median": di["us"], "steps": di["steps"],
            "roofline": {"bound": "hbm", "achieved": di_gbs, "peak": hbm, "unit": "GB/s", "frac": di_gbs / hbm,
                         "algorithmic_bytes": di["bytes"], "peak_source": pk_src}}
        line["sublayer"] = sub
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_prefill(pf["inp"])
        line["decode"]["cpu_baseline"] = cpu_baseline_decode(dc["dec"])
        for name, p in others.items():
            line[name]["cpu_baseline"] = cpu_baseline_prefill(p["inp"], budget_s=5.0, heads=4)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from oracle import oracle
    inp = workloads.workload_prefill(WORKLOAD, device="cpu")
    f = lambda x: x.detach().to(torch.float64).numpy()
    a = [f(x) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta)]
    cu = inp.cu_seqlens.numpy()
    threads = min(oracle.default_threads(), inp.num_seqs * inp.q.shape[1])
    for _ in range(args.warmup):
        oracle.run(*a, cu, threads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.run(*a, cu, threads=threads)
    el = time.perf_counter() - t0
    value = args.steps * inp.total_tokens / el
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "prefill B=1 H=16 T=4096 d_k=d_v=128 chunk=64 bf16 q/k/v fp32 g/beta zero S0",
                   "global_batch": inp.num_seqs, "seq_len": inp.total_tokens, "heads": inp.q.shape[1], "d": 128,
                   "parallelism": "cpu threads over (sequence, head) chains"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": "the full prefill workload per step, %d step(s)" % args.steps},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_profile_case(case: str, repeat: int):
    """Untimed launches of one workload, for an external profiler (ncu) to capture.

    'prefill', 'varlen' and 'long' run that prefill workload through kda_prefill_chunked; 'decode' runs decode
    steps of the decode workload's size (256 x 32 heads, 512 MiB of state; one-pass captures such as DRAM bytes);
    'decode-n64' runs them over a quarter of its sequences (64 x 32 heads, 128 MiB of state), small enough for a
    many-pass capture; 'conv' runs the sublayer's short convolutions (prefill and decode).
    """
    from gated_delta_rule_27_gb300 import libkda
    torch.cuda.set_device(0)
    if case in ("prefill", "varlen", "long"):
        inp = workloads.workload_prefill(case, device="cuda")
        T, N = inp.total_tokens, inp.num_seqs
        H, d = inp.q.shape[1], inp.q.shape[2]
        o = torch.empty_like(inp.v)
        S = torch.empty((N, H, d, d), device="cuda")
        ws = libkda.new_workspace(T, N, H, d, d, libkda.KDA_BF16, 64, "cuda")
        for _ in range(repeat):
            libkda.kda_prefill_chunked(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.cu_seqlens, o, S_final=S,
                                       workspace=ws)
    elif case == "conv":
        # the sublayer's short convolutions: q, k, v of the prefill workload's shape (4096 tokens x 2048
        # channels) and of one decode step of the decode workload's shape (256 sequences x 4096 channels)
        gen = torch.Generator(device="cpu").manual_seed(workloads.BASE_SEED + 23)
        for R, C, step in ((4096, 2048, False), (256, 4096, True)):
            x = torch.randn((R, C), generator=gen).to(torch.bfloat16).to("cuda")
            w = torch.randn((C, 4), generator=gen).to("cuda")
            y = torch.empty_like(x)
            st = torch.zeros((1 if not step else R, 3, C), device="cuda")
            cu = workloads.cu_from_lengths([R], device="cuda")
            for _ in range(repeat):
                for _ in range(3):
                    if step:
                        libkda.kda_short_conv_decode(x, w, st, y)
                    else:
                        libkda.kda_short_conv_prefill(x, w, cu, y, conv_state_out=st)
    else:
        n = 64 if case == "decode-n64" else 256
        dec = workloads.decode_inputs(repeat, n, 32, 128, torch.bfloat16, seed=workloads.workload_seed("decode"),
                                      device="cuda")
        S = dec.S0.clone()
        o = torch.empty((n, 32, 128), dtype=torch.bfloat16, device="cuda")
        for t in range(repeat):
            libkda.kda_decode_step(dec.q[t], dec.k[t], dec.v[t], dec.g[t], dec.beta[t], S, o)
    torch.cuda.synchronize()
    print(json.dumps({"profile_case": case, "repeat": repeat, "status": "ok"}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["libkda", "reference"], default="libkda")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--headline-only", action="store_true",
                    help="time only the prefill and decode workloads (skip varlen, long, indexed decode)")
    ap.add_argument("--profile-case", choices=["prefill", "varlen", "long", "decode", "decode-n64", "conv"], default=None,
                    help="run untimed launches of one workload for a profiler, print a status line, exit")
    ap.add_argument("--repeat", type=int, default=3)
    ap.add_argument("--compare-plans", action="store_true",
                    help="print the pass time of every tensor-core launch plan (one JSON line each) and exit")
    args = ap.parse_args()
    if args.profile_case:
        run_profile_case(args.profile_case, args.repeat)
        return
    if args.compare_plans:
        from gated_delta_rule_27_gb300 import libkda
        torch.cuda.set_device(0)
        libkda.load()
        for row in compare_plans(libkda, torch.device("cuda", 0)):
            print(json.dumps(row), flush=True)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_libkda(args)


if __name__ == "__main__":
    main()
