"""Benchmark of the gated-delta-rule forward library on one (or N) GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Headline workload: KDA prefill with per-channel decay, 2 sequences x 16384 tokens, 32 heads,
d=128, bf16 q/k/v, fp32 state ~N(0, 0.02), chunk 64 ("kda_prefill", the largest of the
single-GPU workloads).  A step is one kda_prefill_fwd call over that batch (every stage of
the prefill path); the metric is prefill tokens/s.  The Gated DeltaNet prefill
("gdn_prefill"), the ragged GQA prefill, the decode step (256 sequences x 32 heads) and the
speculative-decode verification (a 4-token window plus the fold of the accepted prefix) are
measured in the same run and reported under "also".

Multi-GPU: every rank runs an independent replica on its own batch of the same sizes
(another seed per rank; sequences never interact, so nothing is exchanged); value = all ranks'
tokens / the slowest rank's time.
`--impl reference` times the fp64 CPU oracle on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "prefill tokens/s"
UNIT = "tokens/s"
L2_BYTES = 129e6


# ----------------------------------------------------------------------------- accounting

def prefill_algorithmic_bytes(p) -> dict:
    """Bytes the method must move once: inputs read, o written, touched states read+written."""
    qkv = 2 if p.qkv_dtype == "bf16" else 4
    st = 2 if p.state_dtype == "bf16" else 4
    T, HK, HV, d = p.total_tokens, p.num_k_heads, p.num_v_heads, p.d_k
    g_elems = T * HV * (d if p.decay_kind == "per_channel" else 1)
    live = int(np.count_nonzero(p.lengths))
    return dict(q=T * HK * d * qkv, k=T * HK * d * qkv, v=T * HV * d * qkv, beta=T * HV * 4,
                g=g_elems * 4, o=T * HV * d * 4, state=2 * live * HV * d * d * st)


def decode_algorithmic_bytes(dp) -> dict:
    qkv = 2 if dp.qkv_dtype == "bf16" else 4
    st = 2 if dp.state_dtype == "bf16" else 4
    B, HK, HV, d = dp.num_seqs, dp.num_k_heads, dp.num_v_heads, dp.d_k
    g_elems = B * HV * (d if dp.decay_kind == "per_channel" else 1)
    return dict(q=B * HK * d * qkv, k=B * HK * d * qkv, v=B * HV * d * qkv, beta=B * HV * 4,
                g=g_elems * 4, o=B * HV * d * 4, state=2 * B * HV * d * d * st)


def tc_executed_flops(p) -> dict:
    """Tensor-core FLOPs the two tensor-core kernels issue per launch (d = 128, C = 64), as
    issued (an M = 128 MMA of which 64 rows are used counts in full): front per (chunk, value
    head) the A-GEMM (three passes for per-channel decay) and the two M=128 N=64 K=64 products
    K_end^T TB and [*; A_qk] TB; chain per chunk and value tile of 64 columns [K~; Q~] S
    (K = 128), Kb E' and A1o E' (K = 64 each)."""
    chunks = sum((int(n) + 63) // 64 for n in p.lengths) * p.num_v_heads
    agemm = 2 * 128 * 64 * 128 * (3 if p.decay_kind == "per_channel" else 1)
    front = agemm + 2 * (2 * 128 * 64 * 64)
    chain = 2 * (2 * 128 * 64 * 128 + 2 * (2 * 128 * 64 * 64))
    return {"tc_front": float(front * chunks), "tc_chain": float(chain * chunks)}


def prefill_flops(p) -> float:
    """Chunk-form multiply-adds x 2 per token and value head (d_k = d_v = d)."""
    d, C = p.d_k, p.chunk
    macs = 3 * d * d + 2.5 * C * d + C * C / 6.0
    return 2.0 * macs * p.total_tokens * p.num_v_heads


# The prefill kernels in launch order, with the part of the algorithmic traffic each
# one carries.  Tensor-core path: the chunk-parallel front kernel reads the chunk-local
# inputs (q, k, beta, g); the chain kernel reads v, writes o and reads/writes the states
# (the chunk records between them are overhead, not algorithmic traffic).  CUDA-core
# path: the chunk-parallel kernel reads every input once; the scan writes o and
# reads/writes the states.
PREFILL_STAGES = {
    True: [("plan", ()), ("tc_front", ("q", "k", "beta", "g")), ("tc_chain", ("v", "o", "state"))],
    False: [("plan", ()), ("chunk_local", ("q", "k", "v", "beta", "g")),
            ("state_scan", ("o", "state"))],
}
# the single-kernel form (KDA_FLAG_COMPACT), by decay kind (per-channel: True)
COMPACT_STAGES = {
    True: [("plan", ()), ("tc_range_scan", ("g",)), ("tc_prefill", ("q", "k", "v", "beta", "o", "state"))],
    False: [("plan", ()), ("tc_prefill", ("q", "k", "v", "beta", "g", "o", "state"))],
}


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of a kernel on a
# workload, from an ncu capture of the kernel as it is built now (see profiles/); a kernel
# without a capture of its current build has no entry and is reported as null.
# The prefill entries: launches 7 and 8 of
#   ncu --metrics gpu__time_duration.sum,dram__bytes_read.sum,dram__bytes_write.sum --clock-control none
#       -k regex:"tc_front|tc_chain" -s 6 -c 2 python bench.py --profile prefill --workload W --steps 1 --warmup 3
NCU_TRAFFIC = {("decode_step", "kda_decode"): 547441408 + 480736768,
               ("verify_window", "kda_verify"): 579015936 + 57849088,
               ("fold_accepted", "kda_verify"): 453014272 + 364333056,
               ("conv_kernel", "gdn_prefill"): 358.74e6,
               ("tc_front", "kda_prefill"): 1118451968 + 905703424,
               ("tc_chain", "kda_prefill"): 1220631040 + 504979200,
               ("tc_front", "gdn_prefill"): 138534656 + 182024192,
               ("tc_chain", "gdn_prefill"): 308361728 + 103951616}


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d.get("hbm_gbs"), "bf16_tflops": d.get("bf16_tflops"),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (SM clock, throttle reasons) while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- distributed

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = os.environ.get("KDA_BENCH_BACKEND", "nccl")
        dist.init_process_group(backend=backend)
    return rank, world, local


def reduce_max(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate(units_per_rank: float, seconds: float, world: int, device=None) -> tuple:
    """Whole-job throughput: all ranks' units over the slowest rank's time (weak scaling)."""
    slowest = reduce_max(seconds, world, device)
    return units_per_rank * world / slowest, slowest


# ----------------------------------------------------------------------------- CPU side

def cpu_model() -> str:
    """The host CPU as /proc/cpuinfo names it (x86 "model name", or the Arm implementer and
    part numbers), with the count of online cores."""
    name = None
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
        for key in ("model name", "Model", "cpu model"):
            for line in info.splitlines():
                if line.split(":")[0].strip() == key:
                    name = line.split(":", 1)[1].strip()
                    break
            if name:
                break
        if not name:
            impl = [ln.split(":")[1].strip() for ln in info.splitlines() if ln.startswith("CPU implementer")]
            part = [ln.split(":")[1].strip() for ln in info.splitlines() if ln.startswith("CPU part")]
            if impl and part:
                name = f"Arm implementer {impl[0]} part {part[0]}"
    except OSError:
        pass
    return f"{name or 'unknown CPU'}, {os.cpu_count()} cores online"


def cpu_oracle_prefill(p, pair_fraction: float = 1.0, threads=None):
    """Times the fp64 oracle on (a seeded subset of) the workload's (sequence, head) pairs."""
    import oracle
    npairs = p.num_seqs * p.num_v_heads
    mask = np.zeros(npairs, np.uint8)
    take = max(1, int(round(npairs * pair_fraction)))
    mask[np.random.Generator(np.random.PCG64(7)).permutation(npairs)[:take]] = 1
    threads = threads or oracle.default_threads()
    t0 = time.perf_counter()
    oracle.run(p, pair_mask=mask, nthreads=threads)
    dt = time.perf_counter() - t0
    # tokens-equivalent: the sampled pairs' token-head work over the workload's heads
    lengths = p.lengths
    tok_heads = float(sum(lengths[i // p.num_v_heads] for i in np.flatnonzero(mask)))
    return tok_heads / p.num_v_heads / dt, dt, threads, take, npairs


def reference_arm(args, rank, world):
    if rank != 0:
        return
    p = workloads.workload(args.workload)
    frac = 0.25 if args.workload != "tiny_gdn" else 1.0
    for _ in range(args.warmup):
        cpu_oracle_prefill(p, frac)
    tok, secs = 0.0, 0.0
    for _ in range(args.steps):
        r, dt, threads, take, npairs = cpu_oracle_prefill(p, frac)
        tok += r * dt            # token-equivalents of this step's sample
        secs += dt
    value = tok / secs if secs > 0 else 0.0
    sample = (f"{take} of {npairs} (sequence, value head) pairs of {args.workload} per step, "
              f"fp64, {threads} threads on {cpu_model()}")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * secs / max(args.steps, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(p),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_config(p) -> dict:
    return {"workload": p.name, "num_seqs": p.num_seqs, "total_tokens": p.total_tokens,
            "num_k_heads": p.num_k_heads, "num_v_heads": p.num_v_heads, "d_k": p.d_k,
            "d_v": p.d_v, "decay": p.decay_kind, "qkv_dtype": p.qkv_dtype,
            "state_dtype": p.state_dtype, "chunk": p.chunk}


# ----------------------------------------------------------------------------- GPU side

def time_prefill(p, dev, steps, warmup, compact=False):
    import torch
    import gated_delta_rule_deltanet_gb300 as kda
    from workloads import torch_io
    t = torch_io.prefill_inputs(p, dev)
    T, HV, d = p.total_tokens, p.num_v_heads, p.d_v
    out = torch.empty((T, HV, d), dtype=torch.float32, device=dev)
    params = kda.kda._prefill_params(t["q"], t["k"], t["v"], t["beta"], t["log_decay"],
                                     t["input_row_offsets"], t["slot_idx"], t["state_pool"],
                                     p.chunk, p.scale, True, False, compact=compact)
    ws = torch.empty(max(kda.workspace_size(params), 1), dtype=torch.uint8, device=dev)
    stages = (COMPACT_STAGES[p.decay_kind == "per_channel"] if compact
              else PREFILL_STAGES[kda.uses_tensor_cores(params)])

    def step():
        kda.prefill(**t, chunk=p.chunk, scale=p.scale, out=out, workspace=ws, compact=compact)

    for _ in range(warmup):
        step()
    nst = len(stages) + 1
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nst)] for _ in range(steps)]
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for s in range(steps):
        kda.set_stage_events(evs[s])
        step()
    end.record()
    kda.set_stage_events([])
    torch.cuda.synchronize()
    total_ms = start.elapsed_time(end)
    stage_ms = [float(np.mean([evs[s][i].elapsed_time(evs[s][i + 1]) for s in range(steps)]))
                for i in range(nst - 1)]
    # device span of each step (first stage event to last): free of host gaps between steps
    span_ms = float(np.mean([evs[s][0].elapsed_time(evs[s][nst - 1]) for s in range(steps)]))
    return total_ms / steps, stage_ms, t, out, stages, span_ms


def time_prefill_e2e(p, dev, steps, warmup):
    """Through the public API with host buffers: every step uploads its inputs from pinned host
    memory, makes the call and reads its outputs back into pinned host memory, all inside the
    timed region.  Consecutive steps are double-buffered as a serving loop would run them:
    step i's upload (one stream) overlaps step i - 1's call (the compute stream) and the
    download of step i - 2's outputs (a third stream); the calls stay in order on the compute
    stream, since each updates the state pool the next one reads."""
    import torch
    import gated_delta_rule_deltanet_gb300 as kda
    from workloads import torch_io
    host = {"q": torch_io.tensor(p.q, p.qkv_dtype, pin=True),
            "k": torch_io.tensor(p.k, p.qkv_dtype, pin=True),
            "v": torch_io.tensor(p.v, p.qkv_dtype, pin=True),
            "beta": torch_io.tensor(p.beta, "f32", pin=True),
            "log_decay": torch_io.tensor(p.g, "f32", pin=True),
            "input_row_offsets": torch_io.index(p.offsets).pin_memory(),
            "slot_idx": torch_io.index(p.slot_idx).pin_memory()}
    pool = torch_io.tensor(p.pool, p.state_dtype, dev)
    devb = [{k: torch.empty_like(v, device=dev) for k, v in host.items()} for _ in range(2)]
    T, HV, d = p.total_tokens, p.num_v_heads, p.d_v
    out = [torch.empty((T, HV, d), dtype=torch.float32, device=dev) for _ in range(2)]
    out_host = [torch.empty((T, HV, d), dtype=torch.float32).pin_memory() for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = out_host[0].numel() * out_host[0].element_size()
    params = kda.kda._prefill_params(devb[0]["q"], devb[0]["k"], devb[0]["v"], devb[0]["beta"],
                                     devb[0]["log_decay"], devb[0]["input_row_offsets"],
                                     devb[0]["slot_idx"], pool, p.chunk, p.scale, True, False)
    ws = torch.empty(max(kda.workspace_size(params), 1), dtype=torch.uint8, device=dev)
    comp = torch.cuda.current_stream(dev)
    s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    up_done, comp_done, down_done = [None, None], [None, None], [None, None]

    def step(i):
        b = i % 2
        with torch.cuda.stream(s_up):
            if comp_done[b] is not None:        # the call of step i - 2 has read devb[b]
                s_up.wait_event(comp_done[b])
            for k in host:
                devb[b][k].copy_(host[k], non_blocking=True)
            up_done[b] = torch.cuda.Event()
            up_done[b].record(s_up)
        comp.wait_event(up_done[b])
        if down_done[b] is not None:            # out[b] of step i - 2 is downloaded
            comp.wait_event(down_done[b])
        kda.prefill(**devb[b], state_pool=pool, chunk=p.chunk, scale=p.scale, out=out[b],
                    workspace=ws, stream=comp)
        comp_done[b] = torch.cuda.Event()
        comp_done[b].record(comp)
        with torch.cuda.stream(s_down):
            s_down.wait_event(comp_done[b])
            out_host[b].copy_(out[b], non_blocking=True)
            down_done[b] = torch.cuda.Event()
            down_done[b].record(s_down)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(comp)
    s_up.wait_stream(comp)                      # nothing of the timed steps starts before `start`
    s_down.wait_stream(comp)
    for i in range(steps):
        step(i)
    for e in down_done:
        comp.wait_event(e)
    end.record(comp)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps, h2d, d2h


def time_decode(dp, dev, steps, warmup):
    import torch
    import gated_delta_rule_deltanet_gb300 as kda
    from workloads import torch_io
    t = torch_io.decode_inputs(dp, dev)
    B, HV, d = dp.num_seqs, dp.num_v_heads, dp.d_v
    out = torch.empty((B, HV, d), dtype=torch.float32, device=dev)

    def step(s):
        i = s % dp.steps
        kda.decode_step(t["q"][i], t["k"][i], t["v"][i], t["beta"][i], t["log_decay"][i],
                        t["slot_idx"], t["state_pool"], out=out)

    for s in range(warmup):
        step(s)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for s in range(steps):
        step(s)
    end.record()
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps


def time_gdp_prefill(p, dev, steps, warmup):
    """Gated DeltaProduct prefill (virtual-sequence expansion, prefill, gather), resident inputs."""
    import torch
    import gated_delta_rule_deltanet_gb300 as kda
    from workloads import torch_io
    t = torch_io.prefill_inputs(p, dev)
    out = torch.empty((p.total_tokens, p.num_v_heads, p.d_v), dtype=torch.float32, device=dev)
    ws = None

    def step():
        nonlocal ws
        kda.gdp_prefill(t["q"], t["k"], t["v"], t["beta"], t["log_decay"], t["input_row_offsets"],
                        t["slot_idx"], t["state_pool"], chunk=p.chunk, scale=p.scale, out=out,
                        workspace=ws)

    p_ws = kda.kda._gdp_params(t["q"], t["k"], t["v"], t["beta"], t["log_decay"], p.num_seqs,
                               t["slot_idx"], t["state_pool"], p.chunk, p.scale, True, False,
                               False, False)[2]
    ws = torch.empty(max(p_ws, 1), dtype=torch.uint8, device=dev)
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(steps):
        step()
    end.record()
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps


def backward_algorithmic_bytes(p) -> float:
    """Bytes the backward must move once: q, k, v, beta, g, d_o and the initial and final-state
    gradients of the touched slots read, the initial states read, dq, dk, dv, dbeta, dg and
    the initial-state gradients written (fp32 gradients)."""
    T, HK, HV, D = p.total_tokens, p.num_k_heads, p.num_v_heads, p.d_k
    es = 2 if p.qkv_dtype == "bf16" else 4
    gw = D if p.decay_kind == "per_channel" else 1
    states = p.num_seqs * HV * D * D
    reads = T * (2 * HK * D + HV * D) * es + T * HV * 4 * (1 + gw) + T * HV * D * 4 \
        + states * ((2 if p.state_dtype == "bf16" else 4) + 4)
    writes = T * (2 * HK * D + HV * D) * 4 + T * HV * 4 * (1 + gw) + states * 4
    return float(reads + writes)


def time_prefill_bwd(p, dev, steps, warmup, compact=False):
    """The backward pass on resident inputs and output gradients (CUDA events); `compact`
    runs it in the bounded workspace (KDA_FLAG_COMPACT)."""
    import torch
    import gated_delta_rule_deltanet_gb300 as kda
    from workloads import torch_io
    t = torch_io.prefill_inputs(p, dev)
    gen = torch.Generator(device="cpu").manual_seed(5)
    d_o = torch.randn((p.total_tokens, p.num_v_heads, p.d_v), generator=gen).to(dev)
    d_state = torch.randn(tuple(p.pool.shape), generator=gen).to(dev)
    d_state0 = torch.zeros_like(d_state)
    params = kda.kda._prefill_params(t["q"], t["k"], t["v"], t["beta"], t["log_decay"],
                                     t["input_row_offsets"], t["slot_idx"], t["state_pool"],
                                     p.chunk, p.scale, True, False, compact=compact)
    import ctypes
    n = ctypes.c_size_t(0)
    kda.load().kda_prefill_bwd_workspace_size(ctypes.byref(params), ctypes.byref(n))
    ws = torch.empty(max(int(n.value), 1), dtype=torch.uint8, device=dev)

    def step():
        kda.prefill_bwd(t["q"], t["k"], t["v"], t["beta"], t["log_decay"],
                        t["input_row_offsets"], t["slot_idx"], t["state_pool"], d_o, d_state,
                        chunk=p.chunk, scale=p.scale, d_state0=d_state0, workspace=ws,
                        compact=compact)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(steps):
        step()
    end.record()
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps, int(n.value)


CONV_WIDTH = 4


def conv_algorithmic_bytes(p) -> float:
    """The front end on a prefill's shapes: x read and y written once ([T, conv_dim] in the
    q/k/v dtype), the gate pre-activations read and the gates written (fp32), the weights."""
    T, HK, HV, d = p.total_tokens, p.num_k_heads, p.num_v_heads, p.d_k
    es = 2 if p.qkv_dtype == "bf16" else 4
    cd = (2 * HK + HV) * d
    gw = d if p.decay_kind == "per_channel" else 1
    return float(2 * T * cd * es + 2 * T * HV * (1 + gw) * 4 + cd * (CONV_WIDTH + 1) * 4)


def time_conv_gates(p, dev, steps, warmup):
    """The front end (short causal conv + SiLU + gates) on the prefill's shapes and offsets,
    conv state in a slot pool, resident inputs (CUDA events)."""
    import torch
    import gated_delta_rule_deltanet_gb300 as kda
    from workloads import torch_io
    T, HK, HV, d = p.total_tokens, p.num_k_heads, p.num_v_heads, p.d_k
    cd = (2 * HK + HV) * d
    gen = torch.Generator(device="cpu").manual_seed(7)
    dt = torch.bfloat16 if p.qkv_dtype == "bf16" else torch.float32
    x = torch.randn((T, cd), generator=gen).to(dt).to(dev)
    w = (torch.randn((cd, CONV_WIDTH), generator=gen) * 0.5).to(dev)
    a = torch.randn((T, HV, d) if p.decay_kind == "per_channel" else (T, HV), generator=gen).to(dev)
    b = torch.randn((T, HV), generator=gen).to(dev)
    state = torch.zeros((p.num_slots, cd, CONV_WIDTH - 1), dtype=dt, device=dev)
    off = torch_io.index(p.offsets, dev)
    slots = torch_io.index(p.slot_idx, dev)

    def step():
        kda.conv_gates(x, w, a, b, num_k_heads=HK, num_v_heads=HV, d=d,
                       input_row_offsets=off, slot_idx=slots, conv_state=state)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(steps):
        step()
    end.record()
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps


VERIFY_WINDOW = 4


def verify_problem():
    """Speculative-decode verification on the decode workload's shape: 256 sequences x
    32 heads, d=128, bf16 q/k/v, per-channel decay, fp32 pool, a window of 4 draft tokens."""
    return workloads.make_problem("kda_verify", num_seqs=256, lengths=[VERIFY_WINDOW] * 256,
                                  num_k_heads=32, num_v_heads=32, d=128, qkv_dtype="bf16",
                                  state_dtype="f32", decay_kind="per_channel", chunk=64,
                                  zero_state=False, seed=2006)


def verify_algorithmic_bytes(p, accepted) -> dict:
    """Verify reads the state once and every window token's inputs, writes o and one
    record per token; the fold reads and writes the state of every sequence with at least
    one accepted token (the others are left alone) and reads the accepted records."""
    accepted = np.asarray(accepted)
    accepted_total, touched = int(accepted.sum()), int(np.count_nonzero(accepted))
    B, HK, HV, d, W = p.num_seqs, p.num_k_heads, p.num_v_heads, p.d_k, VERIFY_WINDOW
    rec = 3 * d if p.decay_kind == "per_channel" else 2 * d + 4
    st = 2 if p.state_dtype == "bf16" else 4
    g = d if p.decay_kind == "per_channel" else 1
    tok = B * W
    verify = (B * HV * d * d * st + tok * (2 * HK * d * 2 + HV * d * 2 + HV * 4 + HV * g * 4
                                           + HV * d * 4 + HV * rec * 4))
    fold = 2 * touched * HV * d * d * st + accepted_total * HV * rec * 4
    return {"verify_window": float(verify), "fold_accepted": float(fold)}


def time_verify(dev, steps, warmup):
    import torch
    import gated_delta_rule_deltanet_gb300 as kda
    from workloads import torch_io
    p = verify_problem()
    t = torch_io.prefill_inputs(p, dev)
    B, HV, d = p.num_seqs, p.num_v_heads, p.d_v
    out = torch.empty((B * VERIFY_WINDOW, HV, d), dtype=torch.float32, device=dev)
    acc_host = np.arange(B, dtype=np.int32) % (VERIFY_WINDOW + 1)   # 0..W accepted, mean W/2
    acc = torch.tensor(acc_host, device=dev)
    ring = None
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]

    def step(e=None):
        nonlocal ring
        if e:
            e[0].record()
        _, ring = kda.verify_window(t["q"], t["k"], t["v"], t["beta"], t["log_decay"],
                                    t["slot_idx"], t["state_pool"], window=VERIFY_WINDOW,
                                    out=out, ring=ring)
        if e:
            e[1].record()
        kda.fold_accepted(ring, acc, t["slot_idx"], t["state_pool"], window=VERIFY_WINDOW)
        if e:
            e[2].record()

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    for s in range(steps):
        step(ev[s])
    torch.cuda.synchronize()
    if kda.get_device_error() != 0:
        raise RuntimeError("verify/fold raised a device error")
    ms_v = sum(e[0].elapsed_time(e[1]) for e in ev) / steps
    ms_f = sum(e[1].elapsed_time(e[2]) for e in ev) / steps
    total = sum(e[0].elapsed_time(e[2]) for e in ev) / steps
    return p, total, {"verify_window": ms_v, "fold_accepted": ms_f}, acc_host


def prefill_rooflines(p, stage_ms, stages, span_ms, peaks, tensor_cores) -> tuple:
    """The dominant kernel's roofline (its share of the algorithmic bytes over its own
    CUDA-event time) and the whole path's (all algorithmic bytes over the step's device span)."""
    abytes = prefill_algorithmic_bytes(p)
    dom = int(np.argmax(stage_ms))
    name, parts = stages[dom]
    dom_bytes = float(sum(abytes[x] for x in parts))
    achieved = dom_bytes / (stage_ms[dom] / 1e3) / 1e9
    tflops = tc_executed_flops(p) if tensor_cores else {}
    roofline = {"bound": "hbm", "kernel": name, "achieved": achieved, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                "traffic": NCU_TRAFFIC.get((name, p.name)),
                "peak_source": peaks["source"], "kernel_ms": stage_ms[dom],
                "algorithmic_bytes_per_launch": dom_bytes,
                "stage_ms": {n: m for (n, _), m in zip(stages, stage_ms)},
                "tensor_tflops": tflops[name] / (stage_ms[dom] / 1e3) / 1e12 if name in tflops else None,
                "tensor_peak_tflops": peaks["bf16_tflops"]}
    path_bytes = float(sum(abytes.values()))
    path = {"algorithmic_bytes": path_bytes, "achieved_gbs": path_bytes / (span_ms / 1e3) / 1e9,
            "frac_hbm": path_bytes / (span_ms / 1e3) / 1e9 / peaks["hbm_gbs"],
            "flops": prefill_flops(p)}
    return roofline, path


def ours_arm(args, rank, world, local):
    import torch
    import gated_delta_rule_deltanet_gb300 as kda
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    kda.load()
    peaks = load_peaks()
    p = workloads.workload(args.workload, replica=rank)

    # timed region: K prefill steps on resident inputs (inputs > L2, no flush needed)
    barrier(world)
    clocks = ClockSampler(local)
    clocks.start()
    ms, stage_ms, t_dev, _, stages, span_ms = time_prefill(p, dev, args.steps, args.warmup)
    tensor_cores = stages is PREFILL_STAGES[True]
    clk = clocks.stop()
    barrier(world)
    tokens = p.total_tokens
    value, slowest_s = aggregate(tokens * args.steps, ms * args.steps / 1e3, world, dev)
    ms_per_step = 1e3 * slowest_s / args.steps
    del t_dev
    roofline, path_roofline = prefill_rooflines(p, stage_ms, stages, ms_per_step, peaks, tensor_cores)

    # end to end through the public API with host buffers: the median of three runs, since the
    # host link is shared with the rest of the machine
    e2e_runs = [time_prefill_e2e(p, dev, max(3, min(args.steps // 2, 200)), 3) for _ in range(3)]
    e2e_ms = float(np.median([r[0] for r in e2e_runs]))
    h2d, d2h = e2e_runs[0][1], e2e_runs[0][2]
    e2e_value, _ = aggregate(tokens, e2e_ms / 1e3, world, dev)

    also = []
    if not args.no_decode:
        for wname in ("gdn_prefill", "kda_prefill", "ragged_gqa_kda"):
            if wname == p.name:
                continue
            wp = workloads.workload(wname, replica=rank)
            # 30 steps of well under a millisecond to a millisecond: a host stall between two
            # steps would dominate the wall-clock mean, so the line reports the mean device
            # span of a step
            _, wst, wt, _, wstages, wms = time_prefill(wp, dev, 30, 3)
            del wt
            wroof, wpath = prefill_rooflines(wp, wst, wstages, wms, peaks,
                                             wstages is PREFILL_STAGES[True])
            wval, _ = aggregate(float(wp.total_tokens), wms / 1e3, world, dev)
            also.append({"workload": wname, "metric": "prefill tokens/s", "value": wval,
                         "unit": "tokens/s", "ms_per_step": wms, "roofline": wroof,
                         "path_roofline": wpath})

        dp = workloads.workload("kda_decode", replica=rank)
        dms = time_decode(dp, dev, max(args.steps, 20), max(args.warmup, 3))
        dbytes = float(sum(decode_algorithmic_bytes(dp).values()))
        dval, _ = aggregate(1.0, dms / 1e3, world, dev)      # one step per dms
        also.append({"workload": "kda_decode", "metric": "decode steps/s", "value": dval,
                     "unit": "steps/s", "ms_per_step": dms,
                     "tokens_per_s": dval * dp.num_seqs,
                     "roofline": {"bound": "hbm", "kernel": "decode_step",
                                  "achieved": dbytes / (dms / 1e3) / 1e9,
                                  "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                  "frac": dbytes / (dms / 1e3) / 1e9 / peaks["hbm_gbs"],
                                  "algorithmic_bytes_per_launch": dbytes,
                                  "traffic": NCU_TRAFFIC.get(("decode_step", "kda_decode"))}})
        vp, vms, vstage, vacc = time_verify(dev, max(args.steps, 20), max(args.warmup, 3))
        vbytes = verify_algorithmic_bytes(vp, vacc)
        vval, _ = aggregate(float(vp.num_seqs * VERIFY_WINDOW), vms / 1e3, world, dev)
        vroof = {}
        for vk in ("verify_window", "fold_accepted"):
            vroof[vk] = {"bound": "hbm", "kernel": vk,
                         "achieved": vbytes[vk] / (vstage[vk] / 1e3) / 1e9,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": vbytes[vk] / (vstage[vk] / 1e3) / 1e9 / peaks["hbm_gbs"],
                         "algorithmic_bytes_per_launch": vbytes[vk],
                         "traffic": NCU_TRAFFIC.get((vk, "kda_verify"))}
        also.append({"workload": "kda_verify (256 seq x 32 heads, d=128, window 4, "
                                 "accepted 0..4 per sequence)",
                     "metric": "verified draft tokens/s", "value": vval, "unit": "tokens/s",
                     "ms_per_step": vms, "stage_ms": vstage,
                     "roofline": vroof["verify_window"], "fold_roofline": vroof["fold_accepted"]})

        gp = workloads.workload("gdp_prefill", replica=rank)
        gms = time_gdp_prefill(gp, dev, 30, 3)
        gval, _ = aggregate(float(gp.total_tokens), gms / 1e3, world, dev)
        also.append({"workload": "gdp_prefill (Gated DeltaProduct, 4 x 4096 tokens x 2 substeps, "
                                 "16 heads, d=128, bf16, scalar decay)",
                     "metric": "prefill tokens/s", "value": gval, "unit": "tokens/s",
                     "ms_per_step": gms, "virtual_tokens_per_s": gval * gp.n_h})

        bp = workloads.workload("gdn_prefill")
        bms, bws = time_prefill_bwd(bp, dev, 10, 3)
        bval, _ = aggregate(float(bp.total_tokens), bms / 1e3, world, dev)
        bbytes = backward_algorithmic_bytes(bp)
        also.append({"workload": f"{bp.name} backward (kda_prefill_bwd)",
                     "metric": "backward tokens/s", "value": bval, "unit": "tokens/s",
                     "ms_per_step": bms, "workspace_bytes": bws,
                     "path_roofline": {"algorithmic_bytes": bbytes,
                                       "achieved_gbs": bbytes / (bms / 1e3) / 1e9,
                                       "frac_hbm": bbytes / (bms / 1e3) / 1e9
                                       / peaks["hbm_gbs"]}})
        # the bounded-workspace form on gdn_prefill and on kda_prefill
        for cp in (bp, workloads.workload("kda_prefill", replica=rank)):
            cms_, cws_ = time_prefill_bwd(cp, dev, 3, 3, compact=True)
            cval_, _ = aggregate(float(cp.total_tokens), cms_ / 1e3, world, dev)
            also.append({"workload": f"{cp.name} backward, bounded workspace "
                                     "(kda_prefill_bwd, KDA_FLAG_COMPACT)",
                         "metric": "backward tokens/s", "value": cval_, "unit": "tokens/s",
                         "ms_per_step": cms_, "workspace_bytes": cws_})

        cms = time_conv_gates(bp, dev, 50, 3)
        cval, _ = aggregate(float(bp.total_tokens), cms / 1e3, world, dev)
        cbytes = conv_algorithmic_bytes(bp)
        also.append({"workload": f"{bp.name} front end (kda_conv_gates_fwd: conv width "
                                 f"{CONV_WIDTH} + SiLU over [Q | K | V], gates)",
                     "metric": "tokens/s", "value": cval, "unit": "tokens/s", "ms_per_step": cms,
                     "roofline": {"bound": "hbm", "kernel": "conv_gates (three launches)",
                                  "achieved": cbytes / (cms / 1e3) / 1e9,
                                  "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                  "frac": cbytes / (cms / 1e3) / 1e9 / peaks["hbm_gbs"],
                                  "traffic": NCU_TRAFFIC.get(("conv_kernel", bp.name))}})

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        import oracle
        rate, dt, threads, take, npairs = cpu_oracle_prefill(p, 1.0)
        one = max(1, npairs // 32)
        rate1, dt1, _, take1, _ = cpu_oracle_prefill(p, one / npairs, threads=1)
        cpu = {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"{take} of {npairs} (sequence, value head) pairs of {p.name} "
                         f"(the whole workload), fp64, {threads} threads, {dt:.1f} s",
               "one_thread": {"value": rate1, "unit": UNIT, "cores": 1,
                              "sample": f"{take1} of {npairs} pairs, 1 thread, {dt1:.1f} s"},
               "cpu": cpu_model()}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f16" if tensor_cores else "f32",
                "qkv_dtype": p.qkv_dtype, "mma_operands": "f16" if tensor_cores else None,
                "accumulate": "f32", "state_dtype": p.state_dtype, "data": "synthetic",
                "config": {**workload_config(p),
                           "l2": f"inputs larger than L2 ({path_roofline['algorithmic_bytes'] / 1e6:.0f} "
                                 f"MB moved per step vs 129 MB L2); no flush"},
                "path_roofline": path_roofline,
                "roofline": roofline, "cpu_baseline": cpu,
                "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
                "gpu_launches": len(stages) * args.steps,
                "clocks": clk, "also": also}
        print(json.dumps(line), flush=True)


def profile_arm(args):
    """W + K steps of one piece, for an ncu capture (no JSON line; nothing reported here is
    a bench value): `prefill` on --workload, `decode` on kda_decode, `verify` on the
    256-sequence window of 4 plus the fold, `backward` on --workload."""
    import torch
    import gated_delta_rule_deltanet_gb300 as kda
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    kda.load()
    if args.profile == "prefill":
        ms, stage_ms, _, _, stages, _ = time_prefill(workloads.workload(args.workload), dev, args.steps,
                                                     args.warmup, compact=args.compact)
        print("stages: " + ", ".join(f"{n} {m:.4f} ms" for (n, _), m in zip(stages, stage_ms)))
    elif args.profile == "decode":
        ms = time_decode(workloads.workload("kda_decode"), dev, args.steps, args.warmup)
    elif args.profile == "backward":
        ms = time_prefill_bwd(workloads.workload(args.workload), dev, args.steps, args.warmup,
                              compact=args.compact)[0]
    else:
        _, ms, vstage, _ = time_verify(dev, args.steps, args.warmup)
        print("stages: " + ", ".join(f"{n} {m:.4f} ms" for n, m in vstage.items()))
    print(f"profile {args.profile}: {args.warmup} + {args.steps} steps, {ms:.4f} ms per step")


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="kda_prefill",
                    choices=[w for w in workloads.WORKLOADS if w != "kda_decode"])
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--compact", action="store_true",
                    help="with --profile prefill or backward: the single-kernel / bounded-workspace form")
    ap.add_argument("--profile", choices=["prefill", "decode", "verify", "backward"],
                    help="run W + K steps of one piece for a profiler, print no JSON line")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_setup()
    try:
        if args.profile:
            profile_arm(args)
        elif args.impl == "reference":
            reference_arm(args, rank, world)
        else:
            ours_arm(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
