"""Benchmark of the linear-attention hot path on one GB300 (or N replicas).

Headline (the JSON line's value): prefill throughput, tokens/s = B*H*N / s, on
the bf16 workload B=4 H=8 N=4096 dk=dv=64 (inputs N(0,1), fp32 state and
accumulation).  One step = one la_prefill call over that batch (phi, the
intra-chunk scores, the masked score-value product, the inter-chunk read, the
normalisation, the state update and carry, the final state).  The same run
measures the other workloads of the path and reports them under "extra":
the long streaming prefill (B=1 H=16 N=65536), the decode step (B=256 H=32
dk=dv=128, 100 consecutive steps as one CUDA graph, HBM GB/s), the delta-rule
memory (B=8 H=16 N=8192 dk=dv=128) and the small fp32 case (B=1 H=1 N=256).

Timing: W untimed warm-up steps, then exactly K steps bracketed by a barrier
and torch.cuda.synchronize(), timed with CUDA events on the launching stream.
The K steps are captured once as a CUDA graph (one kernel node per step) and
replayed, so the device runs them back to back instead of waiting on the
host's per-call launch work; the average launch duration is the timed region
divided by K (one kernel per step).  The step inputs rotate over four buffer
sets (about 340 MB, more than the 129 MB L2) so that no step finds its inputs
in L2.  The e2e number goes through the public API call by call, host
overhead included.  Clocks are sampled with nvidia-smi while the GPU
measurements run.

--impl reference times the fp64 CPU oracle on the host cores instead (a
bounded sample of the same workload per step), printing the same JSON line
with "impl": "reference".
"""
from __future__ import annotations

import argparse
import hashlib
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

METRIC = ("linear-attn prefill tokens/s (B*H*N/s) at dk=dv=64/128; "
          "decode-step HBM GB/s")
PREFILL_BYTES_PER_TOKEN = 640  # q,k,v bf16 at d=64 (384 B) + o fp32 (256 B)


def _args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None,
                   help="timed steps (default 10000 prefill calls, about 0.3 s of device time, "
                        "so that the clock samples taken every 100 ms fall inside the timed "
                        "region; 200 oracle samples for --impl reference)")
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-extra", action="store_true",
                   help="headline workload only (no long/decode/delta/e2e/cpu)")
    p.add_argument("--only", default="",
                   help="comma list of extra workloads to run "
                        "(long,decode,delta,pr1,gated,decay,rbw,nc,backward,prefill128,rbw128,nc128,"
                        "decay128)")
    p.add_argument("--profile-backward", type=int, default=0, metavar="CALLS",
                   help="run CALLS plain la_prefill_backward calls and exit (for ncu)")
    p.add_argument("--profile-order", type=int, default=0, metavar="MODE",
                   help="with --profile N: la_prefill_variant calls in read order MODE "
                        "(1 read before write, 2 non-causal) instead of la_prefill")
    p.add_argument("--profile-decay", type=int, default=0, metavar="CALLS",
                   help="run CALLS plain decayed-prefill calls and exit (for ncu)")
    p.add_argument("--profile-decode", type=int, default=0, metavar="CALLS",
                   help="run CALLS plain decode steps of the decode workload (B=256 H=32 "
                        "dk=dv=128, random fp32 state) and exit (for ncu)")
    p.add_argument("--profile-delta", type=int, default=0, metavar="CALLS",
                   help="run CALLS plain delta_prefill calls of the delta workload and exit "
                        "(for profilers)")
    p.add_argument("--profile", type=int, default=0, metavar="CALLS",
                   help="run CALLS plain (non-graph) prefill calls of the headline workload on "
                        "the same rotating buffer sets and exit: the command profilers run")
    p.add_argument("--profile-workload", default="prefill", choices=["prefill", "long", "prefill128"],
                   help="workload that --profile runs (default: the headline prefill)")
    args = p.parse_args()
    if args.steps is None:
        args.steps = 200 if args.impl == "reference" else 10000
    return args


# --------------------------------------------------------------------------
# distributed plumbing (one process per GPU; replicas, no collective on the
# data path -- only the barrier and the max over ranks of the timed region)

def _dist_init(n):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    return rank, world


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, world, max_ms, steps):
    """Whole-job throughput: the units every rank processed in `steps` steps,
    over the slowest rank's time (weak scaling: each rank runs its own
    replica of the workload)."""
    return units_per_rank * world * steps / (max_ms * 1e-3)


# --------------------------------------------------------------------------
# clocks

class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons (read only)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id=None):
        self.proc = None
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if bus_id:
            cmd += ["-i", bus_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    rows.append(dict(sm=float(parts[1]), smax=float(parts[2]),
                                     util=float(parts[4]), hw=parts[6], hwt=parts[7],
                                     swt=parts[8], swp=parts[9]))
                except ValueError:
                    continue
        os.unlink(self.file.name)
        if not rows:
            return None
        load = [r for r in rows if r["util"] >= 50] or rows
        reasons = set()
        for r in load:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in load),
                "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows),
                "samples_under_load": len([r for r in rows if r["util"] >= 50])}


# --------------------------------------------------------------------------
# measured peaks and committed ncu counters

def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, "fallback"


def tensor_fractions(d, chunk, tokens, ms, bf16_peak):
    """Contraction work of the chunked prefill against the bf16 tensor peak.
    Per token, with full C x C tiles as executed: scores 2 C d, masked P V
    2 C d, inter-chunk read 2 d d, state update 2 d d; causal-only counts
    half of the C x C tiles.  The path is HBM-bound at these sizes, so these
    fractions are reported beside the HBM roofline, not as the bound."""
    executed = (4 * chunk * d + 4 * d * d) * tokens
    causal = (2 * chunk * d + 4 * d * d) * tokens
    t = ms * 1e-3
    return {"flop_per_token_executed": 4 * chunk * d + 4 * d * d,
            "flop_per_token_causal": 2 * chunk * d + 4 * d * d,
            "tflops_executed": executed / t / 1e12, "tflops_causal": causal / t / 1e12,
            "frac_executed": executed / t / 1e12 / bf16_peak,
            "frac_causal": causal / t / 1e12 / bf16_peak, "peak_tflops": bf16_peak}


def _kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fixed_state_recurrent_gb300", "csrc")
    for name in ("prefill_prefix64.cu", "prefill_tc_common.cuh", "tc_primitives.cuh"):
        p = os.path.join(csrc, name)
        if os.path.exists(p):
            with open(p, "rb") as f:
                h.update(f.read())
    return h.hexdigest()


# Kernel launches per la_prefill call on the headline workload: the d = 64
# tensor-core path runs the prefix and output kernels.
PREFILL_LAUNCHES_PER_CALL = 2


def _committed_traffic(tokens):
    """dram bytes of one la_prefill call (its two kernels) from the committed
    ncu counters (profiles/prefill_d64_bf16_ncu.json), scaled to `tokens`, or
    None when the kernel sources changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "prefill_d64_bf16_ncu.json")
    try:
        with open(path, encoding="utf-8") as f:
            rec = json.load(f)
        if rec["kernel_source_sha256"] != _kernel_source_hash():
            return None
        return float(rec["dram_bytes_per_token"]) * tokens
    except (OSError, KeyError, ValueError, TypeError):
        return None


# --------------------------------------------------------------------------
# workloads

def _device_inputs(w, seed, device):
    from fixed_state_recurrent_gb300 import inputs
    q, k, v = inputs.la_inputs(w.B, w.H, w.N, w.dk, w.dv, w.dtype, seed, w.scale)
    return q.to(device), k.to(device), v.to(device)


def _timed(fn, steps, stream, world, per_launch=True):
    """Run fn(i) for i in range(steps) on `stream`; returns (total_ms, list of
    per-step ms) with events on that stream, max over ranks for the total."""
    import torch
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    _barrier(world)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        evs[0].record(stream)
        for i in range(steps):
            fn(i)
            if per_launch or i == steps - 1:
                evs[i + 1].record(stream)
    torch.cuda.synchronize()
    _barrier(world)
    total = evs[0].elapsed_time(evs[steps])
    per = [evs[i].elapsed_time(evs[i + 1]) for i in range(steps)] if per_launch else []
    return _max_over_ranks(total, world), per


def bench_prefill(api, w, steps, warmup, rank, world, sets=4):
    """K la_prefill calls over rotating buffer sets, captured once as a CUDA
    graph (one kernel node per step) so that the timed region measures the
    device back to back rather than the host's launch rate; the K-step graph
    is replayed once, bracketed by events on its stream."""
    import torch
    dev = torch.device("cuda")
    bufs = []
    for r in range(sets):
        q, k, v = _device_inputs(w, w.seed + 1000 * rank + r, dev)
        o = torch.empty((w.B, w.H, w.N, w.dv), device=dev)
        S = torch.empty((w.B, w.H, w.dk, w.dv), device=dev)
        z = torch.empty((w.B, w.H, w.dk), device=dev)
        bufs.append((q, k, v, o, S, z))
    ws = api.workspace(w.B, w.H, w.N, w.dk, w.dv, w.dtype, 0, dev)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())

    def step(i):
        q, k, v, o, S, z = bufs[i % sets]
        api.prefill(q, k, v, o=o, S_N=S, z_N=z, ws=ws)

    with torch.cuda.stream(stream):
        for i in range(warmup):
            step(i)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(steps):
                step(i)
        graph.replay()  # untimed: the first replay uploads the graph
    total, _ = _timed(lambda i: graph.replay(), 1, stream, world, per_launch=False)
    status = api.read_device_status(ws, stream)
    if status != 0:
        raise RuntimeError(f"prefill kernel reported device status {status}")
    return total, [total / steps] * steps


def _graph_ms(step, steps, stream, world):
    """Device ms per call of `step(i)`: `steps` calls captured as one CUDA
    graph on `stream` (after the caller's warm-up calls), replayed once
    untimed, then once between events; max over ranks."""
    import torch
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            for i in range(steps):
                step(i)
        graph.replay()
    total, _ = _timed(lambda i: graph.replay(), 1, stream, world, per_launch=False)
    return total / steps


def profile_calls(api, w, calls, sets=4):
    """`calls` plain la_prefill calls over the rotating buffer sets of
    bench_prefill, launched one by one (no graph), for profilers."""
    import torch
    dev = torch.device("cuda")
    bufs = []
    for r in range(sets):
        q, k, v = _device_inputs(w, w.seed + r, dev)
        bufs.append((q, k, v, torch.empty((w.B, w.H, w.N, w.dv), device=dev),
                     torch.empty((w.B, w.H, w.dk, w.dv), device=dev),
                     torch.empty((w.B, w.H, w.dk), device=dev)))
    ws = api.workspace(w.B, w.H, w.N, w.dk, w.dv, w.dtype, 0, dev)
    for i in range(calls):
        q, k, v, o, S, z = bufs[i % sets]
        api.prefill(q, k, v, o=o, S_N=S, z_N=z, ws=ws)
    torch.cuda.synchronize()
    if api.read_device_status(ws) != 0:
        raise RuntimeError("prefill kernel reported a nonzero device status")
    print(f"profiled {calls} prefill calls", flush=True)


def profile_delta_calls(api, calls):
    """`calls` plain delta_prefill calls of the delta workload, for profilers."""
    import torch
    from fixed_state_recurrent_gb300 import inputs
    w = inputs.WORKLOADS["delta"]
    dev = torch.device("cuda")
    k, v, beta = inputs.delta_inputs(w.B, w.H, w.N, w.dk, w.dv, w.dtype, w.seed, device=dev)
    reads = torch.empty((w.B, w.H, w.N, w.dv), device=dev)
    S = torch.empty((w.B, w.H, w.dk, w.dv), device=dev)
    for _ in range(calls):
        api.delta_prefill(k, v, beta, reads=reads, S_N=S)
    torch.cuda.synchronize()
    print(f"profiled {calls} delta calls", flush=True)


def profile_decode_calls(api, calls):
    """`calls` plain decode steps on the decode workload's shapes (B=256 H=32
    dk=dv=128, bf16 tokens); the state is random fp32 (the DRAM traffic of a
    step does not depend on its values), for profilers."""
    import torch
    from fixed_state_recurrent_gb300 import inputs
    w = inputs.WORKLOADS["decode"]
    dev = torch.device("cuda")
    B, H, d = w.B, w.H, w.dk
    g = torch.Generator(device=dev).manual_seed(w.seed)
    S = torch.randn((B, H, d, d), generator=g, device=dev)
    z = torch.rand((B, H, d), generator=g, device=dev) * 100 + 1
    qs, ks, vs = inputs.decode_step_inputs(B, H, d, d, calls, torch.bfloat16, w.seed, device=dev)
    o = torch.empty((B, H, d), device=dev)
    for t in range(calls):
        api.decode_step(qs[t], ks[t], vs[t], S, z, o=o)
    torch.cuda.synchronize()
    print(f"profiled {calls} decode steps", flush=True)


def profile_decay_calls(api, calls, sets=4, wname="prefill"):
    """`calls` plain decayed-prefill calls (la_prefill_variant, alpha ~ U(0.9, 1))
    on the headline prefill shape (or another prefill workload) over rotating
    input sets, for profilers."""
    import torch
    w = inputs_mod().WORKLOADS[wname]
    dev = torch.device("cuda")
    bufs = []
    for r in range(sets):
        q, k, v = _device_inputs(w, w.seed + r, dev)
        g = torch.Generator(device=dev).manual_seed(6 + 17 * r)
        bufs.append((q, k, v, 0.9 + 0.1 * torch.rand((w.B, w.H, w.N), generator=g, device=dev)))
    for i in range(calls):
        q, k, v, alpha = bufs[i % sets]
        api.prefill_variant(q, k, v, alpha, 0)
    torch.cuda.synchronize()
    print(f"profiled {calls} decayed prefill calls", flush=True)


def profile_order_calls(api, calls, mode, sets=4, wname="prefill"):
    """`calls` plain la_prefill_variant calls in another read order (no decay)
    on a prefill workload over rotating input sets, for profilers."""
    import torch
    w = inputs_mod().WORKLOADS[wname]
    dev = torch.device("cuda")
    bufs = [_device_inputs(w, w.seed + r, dev) for r in range(sets)]
    for i in range(calls):
        q, k, v = bufs[i % sets]
        api.prefill_variant(q, k, v, None, mode)
    torch.cuda.synchronize()
    print(f"profiled {calls} read-order {mode} calls", flush=True)


def profile_backward_calls(api, calls):
    """`calls` plain la_prefill_backward calls on the headline prefill shape
    (bf16 inputs, dO ~ N(0,1)), for profilers."""
    import torch
    w = inputs_mod().WORKLOADS["prefill"]
    dev = torch.device("cuda")
    q, k, v = _device_inputs(w, w.seed, dev)
    g = torch.Generator(device=dev).manual_seed(9)
    dO = torch.randn((w.B, w.H, w.N, w.dv), generator=g, device=dev)
    for _ in range(calls):
        api.prefill_backward(q, k, v, dO)
    torch.cuda.synchronize()
    print(f"profiled {calls} backward calls", flush=True)


def bench_decode(api, rank, world, reps=3):
    """100 consecutive decode steps captured in one CUDA graph; the state comes
    from a 1024-token prefix run through la_prefill."""
    import torch
    from fixed_state_recurrent_gb300 import inputs
    w = inputs.WORKLOADS["decode"]
    dev = torch.device("cuda")
    B, H, d, P, T = w.B, w.H, w.dk, w.N, w.steps
    S = torch.empty((B, H, d, d), device=dev)
    z = torch.empty((B, H, d), device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed + 1000 * rank)
    step = 32
    for b0 in range(0, B, step):  # prefix prefilled 32 sequences at a time
        pq = inputs.gaussian((step, H, P, d), g, torch.bfloat16, device=dev)
        pk = inputs.gaussian((step, H, P, d), g, torch.bfloat16, device=dev)
        pv = inputs.gaussian((step, H, P, d), g, torch.bfloat16, device=dev)
        api.prefill(pq, pk, pv, S_N=S[b0:b0 + step], z_N=z[b0:b0 + step])
        del pq, pk, pv
    qs, ks, vs = inputs.decode_step_inputs(B, H, d, d, T, torch.bfloat16,
                                           w.seed + 1000 * rank, device=dev)
    o = torch.empty((T, B, H, d), device=dev)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        api.decode_step(qs[0], ks[0], vs[0], S, z, o=o[0])  # warm (caches attributes)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for t in range(T):
                api.decode_step(qs[t], ks[t], vs[t], S, z, o=o[t])
        graph.replay()
        graph.replay()
    times = []
    for _ in range(reps):
        ms, _ = _timed(lambda i: graph.replay(), 1, stream, world, per_launch=False)
        times.append(ms)
    ms = min(times)
    bytes_per_head = 2 * d * d * 4 + 2 * d * 4 + 3 * d * 2 + d * 4
    bytes_step = bytes_per_head * B * H
    us_step = ms * 1e3 / T
    return {"workload": "decode: B=256 H=32 dk=dv=128, 100 steps in one CUDA graph, "
                        "state from a 1024-token bf16 prefix",
            "us_per_step": us_step, "hbm_gbs": bytes_step / (us_step * 1e-6) / 1e9,
            "bytes_per_step": bytes_step, "reps": reps, "launches_per_rep": T}


def bench_delta(api, rank, world, reps=3):
    import torch
    from fixed_state_recurrent_gb300 import inputs
    w = inputs.WORKLOADS["delta"]
    dev = torch.device("cuda")
    k, v, beta = inputs.delta_inputs(w.B, w.H, w.N, w.dk, w.dv, w.dtype,
                                     w.seed + 1000 * rank, device=dev)
    reads = torch.empty((w.B, w.H, w.N, w.dv), device=dev)
    S = torch.empty((w.B, w.H, w.dk, w.dv), device=dev)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    fn = lambda i: api.delta_prefill(k, v, beta, reads=reads, S_N=S)
    with torch.cuda.stream(stream):
        fn(0)
    ms, per = _timed(fn, reps, stream, world)
    ms_call = min(per)
    tokens = w.B * w.H * w.N
    flops = 4.0 * w.dk * w.dv * tokens
    # algorithmic HBM bytes: k, v (bf16) and beta (fp32) in, reads (fp32) out,
    # per token; the final state (fp32) per head
    nbytes = tokens * (2 * w.dk + 2 * w.dv + 4 + 4 * w.dv) + w.B * w.H * w.dk * w.dv * 4
    return {"workload": "delta: B=8 H=16 N=8192 dk=dv=128, unit bf16 keys, bf16 values, "
                        "sigmoid beta", "ms_per_call": ms_call,
            "tokens_per_s": tokens / (ms_call * 1e-3),
            "fp32_tflops": flops / (ms_call * 1e-3) / 1e12,
            "bytes_per_call": nbytes, "hbm_gbs": nbytes / (ms_call * 1e-3) / 1e9}


def bench_gated_delta(api, rank, world, reps=3):
    """gated_delta_prefill on the delta workload with alpha ~ U(0.9, 1): the
    chunked tensor-core kernel with decay factors (bf16, dk = dv = 128)."""
    import torch
    from fixed_state_recurrent_gb300 import inputs
    w = inputs.WORKLOADS["delta"]
    dev = torch.device("cuda")
    k, v, beta = inputs.delta_inputs(w.B, w.H, w.N, w.dk, w.dv, w.dtype,
                                     w.seed + 1000 * rank, device=dev)
    g = torch.Generator(device=dev).manual_seed(5 + rank)
    alpha = 0.9 + 0.1 * torch.rand((w.B, w.H, w.N), generator=g, device=dev)
    reads = torch.empty((w.B, w.H, w.N, w.dv), device=dev)
    S = torch.empty((w.B, w.H, w.dk, w.dv), device=dev)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    fn = lambda i: api.gated_delta_prefill(k, v, beta, alpha, reads=reads, S_N=S)
    with torch.cuda.stream(stream):
        fn(0)
    _, per = _timed(fn, reps, stream, world)
    ms = min(per)
    tokens = w.B * w.H * w.N
    return {"workload": "gated delta: B=8 H=16 N=8192 dk=dv=128, bf16 keys and values, "
                        "alpha ~ U(0.9, 1), sigmoid beta", "ms_per_call": ms,
            "tokens_per_s": tokens / (ms * 1e-3),
            "fp32_tflops": 4.0 * w.dk * w.dv * tokens / (ms * 1e-3) / 1e12}


def bench_decay_prefill(api, rank, world, reps=12, sets=4, wname="prefill"):
    """la_prefill_variant, write-then-read with a per-token decay, on the
    headline prefill shape (wname "prefill") or its d = 128 twin
    ("prefill128"), on the tensor cores (the heads split over the SMs with a
    workspace), over `sets` rotating input/output sets (> L2)."""
    import torch
    w = inputs_mod().WORKLOADS[wname]
    dev = torch.device("cuda")
    bufs = []
    for r in range(sets):
        q, k, v = _device_inputs(w, w.seed + 1000 * rank + r, dev)
        g = torch.Generator(device=dev).manual_seed(6 + rank + 17 * r)
        alpha = 0.9 + 0.1 * torch.rand((w.B, w.H, w.N), generator=g, device=dev)
        bufs.append((q, k, v, alpha, torch.empty((w.B, w.H, w.N, w.dv), device=dev),
                     torch.empty((w.B, w.H, w.dk, w.dv), device=dev),
                     torch.empty((w.B, w.H, w.dk), device=dev)))
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())

    def fn(i):
        q, k, v, alpha, o, S, z = bufs[i % sets]
        api.prefill_variant(q, k, v, alpha, 0, o=o, S_N=S, z_N=z)

    with torch.cuda.stream(stream):
        for i in range(sets):
            fn(i)
    _, per = _timed(fn, reps, stream, world)
    ms_calls = statistics.median(per)
    ms = _graph_ms(fn, 4 * sets, stream, world)
    # algorithmic bytes: q, k, v bf16 in, o fp32 out, alpha (4 B/token), final state
    b = (2 * (w.dk + w.dk + w.dv) + 4 * w.dv + 4) * w.tokens + w.B * w.H * (w.dk * w.dv + w.dk) * 4
    hbm_peak, _, kind = _peaks()
    return {"workload": f"decayed prefill: B={w.B} H={w.H} N={w.N} dk=dv={w.dk} bf16, "
                        "alpha ~ U(0.9, 1), write then read", "ms_per_call": ms,
            "ms_per_python_call": ms_calls,
            "timing": f"{4 * sets} calls in one CUDA graph, replayed (device time per call); "
                      "ms_per_python_call: median of back-to-back calls from Python",
            "tokens_per_s": w.tokens / (ms * 1e-3), "hbm_gbs": b / (ms * 1e-3) / 1e9,
            "hbm_frac": b / (ms * 1e-3) / 1e9 / hbm_peak, "peak_kind": f"of {kind}",
            "l2": f"{sets} rotating input/output sets"}


def bench_backward(api, rank, world, reps=5):
    """la_prefill_backward on the headline prefill shape (dO ~ N(0,1)): tensor
    cores, every chunk independent from per-chunk state tiles over every SM (the
    default, with a workspace); the one-block-per-head sweeps beside it."""
    import torch
    w = inputs_mod().WORKLOADS["prefill"]
    dev = torch.device("cuda")
    q, k, v = _device_inputs(w, w.seed + 1000 * rank, dev)
    g = torch.Generator(device=dev).manual_seed(7 + rank)
    dO = torch.randn((w.B, w.H, w.N, w.dv), generator=g, device=dev)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    fn = lambda i: api.prefill_backward(q, k, v, dO)
    fh = lambda i: api.prefill_backward(q, k, v, dO, ws=False)
    with torch.cuda.stream(stream):
        for i in range(3):
            fn(i)
            fh(i)
    _, per = _timed(fn, reps, stream, world)
    ms_calls = statistics.median(per)
    ms = _graph_ms(fn, reps, stream, world)
    ms_head = _graph_ms(fh, reps, stream, world)
    # algorithmic bytes: q, k, v (bf16) and dO (fp32) in, dq, dk, dv (fp32) out
    b = (3 * 2 * w.dk + 4 * w.dv + 4 * (2 * w.dk + w.dv)) * w.tokens
    hbm_peak, _, kind = _peaks()
    return {"workload": "backward: B=4 H=8 N=4096 dk=dv=64 bf16 inputs, dO ~ N(0,1), "
                        "gradients of q, k, v, S0, z0", "ms_per_call": ms,
            "ms_per_call_one_block_per_head": ms_head, "ms_per_python_call": ms_calls,
            "timing": f"{reps} calls in one CUDA graph, replayed (device time per call); "
                      "ms_per_python_call: median of back-to-back calls from Python",
            "tokens_per_s": w.tokens / (ms * 1e-3), "hbm_gbs": b / (ms * 1e-3) / 1e9,
            "hbm_frac": b / (ms * 1e-3) / 1e9 / hbm_peak, "peak_kind": f"of {kind}"}


def bench_order_prefill(api, rank, world, mode, reps=12, sets=4, wname="prefill"):
    """la_prefill_variant in read-before-write or non-causal order (no decay)
    on the headline prefill shape (wname "prefill") or its d = 128 twin
    ("prefill128"), on the tensor cores (read before write: la_prefill's
    launches with a strict mask; non-causal: the piece totals, then one product
    per chunk against the head's final state), over `sets` rotating
    input/output sets."""
    import torch
    w = inputs_mod().WORKLOADS[wname]
    dev = torch.device("cuda")
    bufs = []
    for r in range(sets):
        q, k, v = _device_inputs(w, w.seed + 1000 * rank + r, dev)
        bufs.append((q, k, v, torch.empty((w.B, w.H, w.N, w.dv), device=dev),
                     torch.empty((w.B, w.H, w.dk, w.dv), device=dev),
                     torch.empty((w.B, w.H, w.dk), device=dev)))
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())

    def fn(i):
        q, k, v, o, S, z = bufs[i % sets]
        api.prefill_variant(q, k, v, None, mode, o=o, S_N=S, z_N=z)

    with torch.cuda.stream(stream):
        for i in range(sets):
            fn(i)
    _, per = _timed(fn, reps, stream, world)
    ms_calls = statistics.median(per)
    ms = _graph_ms(fn, 4 * sets, stream, world)
    b = (2 * (w.dk + w.dk + w.dv) + 4 * w.dv) * w.tokens  # q, k, v bf16 in, o fp32 out
    hbm_peak, _, kind = _peaks()
    order = "read-before-write" if mode == api.LA_MODE_READ_BEFORE_WRITE else "non-causal"
    return {"workload": f"{order} prefill: B={w.B} H={w.H} N={w.N} dk=dv={w.dk} bf16",
            "ms_per_call": ms, "ms_per_python_call": ms_calls,
            "timing": f"{4 * sets} calls in one CUDA graph, replayed (device time per call); "
                      "ms_per_python_call: median of back-to-back calls from Python",
            "tokens_per_s": w.tokens / (ms * 1e-3), "hbm_gbs": b / (ms * 1e-3) / 1e9,
            "hbm_frac": b / (ms * 1e-3) / 1e9 / hbm_peak, "peak_kind": f"of {kind}",
            "l2": f"{sets} rotating input/output sets"}


def inputs_mod():
    from fixed_state_recurrent_gb300 import inputs
    return inputs


def bench_simple_prefill(api, wname, rank, world, steps=20):
    """la_prefill on another workload, timed like the headline: `steps` calls
    over rotating buffer sets captured as one CUDA graph and replayed, so the
    figure is device time per call (the host's call path is not in it)."""
    import torch
    from fixed_state_recurrent_gb300 import inputs
    w = inputs.WORKLOADS[wname]
    total, _ = bench_prefill(api, w, steps, 3, rank, world)
    ms = total / steps
    res = {"workload": f"{wname}: B={w.B} H={w.H} N={w.N} dk={w.dk} dv={w.dv} "
                       f"{'bf16' if w.dtype == torch.bfloat16 else 'fp32'}",
           "ms_per_call": ms, "tokens_per_s": w.tokens / (ms * 1e-3),
           "timing": f"{steps} calls in one CUDA graph, rotating buffer sets"}
    if w.dtype == torch.bfloat16:
        per_token = 2 * (w.dk + w.dk + w.dv) + 4 * w.dv  # q, k, v bf16 in, o fp32 out
        b = per_token * w.tokens + w.B * w.H * (w.dk * w.dv + w.dk) * 4
        res["hbm_gbs"] = b / (ms * 1e-3) / 1e9
        res["hbm_frac"] = b / (ms * 1e-3) / 1e9 / _peaks()[0]
    return res


def bench_e2e(api, w, steps, warmup, rank, world, lanes=2):
    """Same metric through the public API from pinned HOST buffers: each step
    copies its q, k, v host->device, runs la_prefill and copies its o, S, z
    back.  Consecutive steps alternate over `lanes` streams, each with its own
    device buffers and workspace, so that one step's device->host copies and
    the next step's host->device copies use the link's two directions at once
    (the way a serving loop overlaps requests); every step still moves all of
    its own bytes inside the timed region."""
    import torch
    from fixed_state_recurrent_gb300 import inputs
    dev = torch.device("cuda")
    q, k, v = inputs.la_inputs(w.B, w.H, w.N, w.dk, w.dv, w.dtype, w.seed + 1000 * rank)
    hq, hk, hv = (x.pin_memory() for x in (q, k, v))
    need = api.prefill_workspace_bytes(w.B, w.H, w.N, w.dk, w.dv, w.dtype)
    lane_bufs = []
    for _ in range(lanes):  # every lane owns its device buffers and its pinned host results
        lane_bufs.append(dict(
            q=torch.empty_like(q, device=dev), k=torch.empty_like(k, device=dev),
            v=torch.empty_like(v, device=dev),
            o=torch.empty((w.B, w.H, w.N, w.dv), device=dev),
            S=torch.empty((w.B, w.H, w.dk, w.dv), device=dev),
            z=torch.empty((w.B, w.H, w.dk), device=dev),
            ho=torch.empty((w.B, w.H, w.N, w.dv)).pin_memory(),
            hS=torch.empty((w.B, w.H, w.dk, w.dv)).pin_memory(),
            hz=torch.empty((w.B, w.H, w.dk)).pin_memory(),
            ws=torch.zeros(need, dtype=torch.uint8, device=dev),
            stream=torch.cuda.Stream()))
    main = torch.cuda.current_stream()

    def step(i):
        L = lane_bufs[i % lanes]
        with torch.cuda.stream(L["stream"]):
            L["q"].copy_(hq, non_blocking=True)
            L["k"].copy_(hk, non_blocking=True)
            L["v"].copy_(hv, non_blocking=True)
            api.prefill(L["q"], L["k"], L["v"], o=L["o"], S_N=L["S"], z_N=L["z"], ws=L["ws"])
            L["ho"].copy_(L["o"], non_blocking=True)
            L["hS"].copy_(L["S"], non_blocking=True)
            L["hz"].copy_(L["z"], non_blocking=True)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    _barrier(world)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(main)
    for L in lane_bufs:
        L["stream"].wait_stream(main)
    for i in range(steps):
        step(i)
    for L in lane_bufs:
        main.wait_stream(L["stream"])
    t1.record(main)
    torch.cuda.synchronize()
    _barrier(world)
    total = _max_over_ranks(t0.elapsed_time(t1), world)
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv))
    L = lane_bufs[0]
    d2h = sum(x.numel() * x.element_size() for x in (L["ho"], L["hS"], L["hz"]))
    return total, h2d, d2h


def cpu_baseline(w, target_s=10.0):
    """The fp64 oracle, as it stands, on the host cores: token recurrence over
    the whole prefill workload, repeated until about target_s of CPU time."""
    import torch
    import oracle
    from fixed_state_recurrent_gb300 import inputs
    q, k, v = inputs.la_inputs(w.B, w.H, w.N, w.dk, w.dv, w.dtype, w.seed, w.scale)
    f = lambda t: t.to(torch.float64).numpy()
    q, k, v = f(q), f(k), f(v)
    cores = oracle.default_threads()
    done, t0 = 0, time.perf_counter()
    while True:
        oracle.la_recurrent(q, k, v, threads=cores)
        done += 1
        el = time.perf_counter() - t0
        if el >= target_s or done >= 20:
            break
    return {"value": done * w.tokens / el, "unit": "tokens/s", "cores": cores,
            "kind": "oracle",
            "sample": f"fp64 C oracle token recurrence over the whole prefill workload "
                      f"(B={w.B} H={w.H} N={w.N} d={w.dk}, {w.tokens} tokens) x {done}, "
                      f"{el:.1f} s, threads over heads"}


# --------------------------------------------------------------------------

def run_reference(args):
    """The reference arm: the fp64 oracle on the host cores, the whole prefill
    workload (all 32 heads, threads over the heads) per step."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import torch
    import oracle
    from fixed_state_recurrent_gb300 import inputs
    oracle.build()
    w = inputs.WORKLOADS["prefill"]
    q, k, v = inputs.la_inputs(w.B, w.H, w.N, w.dk, w.dv, w.dtype, w.seed, w.scale)
    heads = w.B * w.H
    f = lambda t: t.reshape(w.B * w.H, 1, w.N, -1)[:heads].to(torch.float64).numpy()
    q, k, v = f(q), f(k), f(v)
    cores = oracle.default_threads()
    for _ in range(args.warmup):
        oracle.la_recurrent(q, k, v, threads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.la_recurrent(q, k, v, threads=cores)
    el = time.perf_counter() - t0
    tokens = heads * w.N * args.steps
    value = tokens / el
    sample = (f"fp64 C oracle token recurrence over the whole prefill workload per step "
              f"({heads} heads x {w.N} tokens), threads over heads")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el * 1e3 / max(args.steps, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "prefill: B=4 H=8 N=4096 dk=dv=64, bf16 q,k,v ~ N(0,1), "
                                   "fp32 state/accumulate, zero initial state",
                       "B": w.B, "H": w.H, "N": w.N, "dk": w.dk, "dv": w.dv},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = _args()
    if args.impl == "reference":
        run_reference(args)
        return
    import torch
    from fixed_state_recurrent_gb300 import build, api, inputs
    rank, world = _dist_init(args.gpus)
    if rank == 0 or world == 1:
        build.build()
    _barrier(world)
    api.load()
    dev = torch.device("cuda")
    props = torch.cuda.get_device_properties(dev)
    bus = getattr(props, "pci_bus_id", None)
    bus_id = None
    if isinstance(bus, int) and hasattr(props, "pci_domain_id"):
        bus_id = f"{props.pci_domain_id:08X}:{bus:02X}:{props.pci_device_id:02X}.0"
    sampler = ClockSampler(bus_id)
    time.sleep(0.3)

    w = inputs.WORKLOADS["prefill"]
    if args.profile_backward:
        profile_backward_calls(api, args.profile_backward)
        sampler.stop()
        return
    if args.profile_decay:
        profile_decay_calls(api, args.profile_decay, wname=args.profile_workload)
        sampler.stop()
        return
    if args.profile_decode:
        profile_decode_calls(api, args.profile_decode)
        sampler.stop()
        return
    if args.profile_delta:
        profile_delta_calls(api, args.profile_delta)
        sampler.stop()
        return
    if args.profile and args.profile_order:
        profile_order_calls(api, args.profile, args.profile_order, wname=args.profile_workload)
        sampler.stop()
        return
    if args.profile:
        profile_calls(api, inputs.WORKLOADS[args.profile_workload], args.profile)
        sampler.stop()
        return
    total_ms, per = bench_prefill(api, w, args.steps, args.warmup, rank, world)
    ms_step = total_ms / args.steps
    value = job_throughput(w.tokens, world, total_ms, args.steps)

    extra = {}
    e2e = None
    wanted = set(x for x in args.only.split(",") if x) or {"long", "decode", "delta", "pr1",
                                                             "gated", "decay", "rbw", "nc", "backward",
                                                             "prefill128", "rbw128", "nc128", "decay128"}
    if not args.no_extra:
        if "long" in wanted:
            extra["long"] = bench_simple_prefill(api, "long", rank, world)
        if "decode" in wanted:
            extra["decode"] = bench_decode(api, rank, world)
        if "delta" in wanted:
            extra["delta"] = bench_delta(api, rank, world)
        if "pr1" in wanted:
            extra["pr1"] = bench_simple_prefill(api, "pr1", rank, world)
        if "prefill128" in wanted:
            extra["prefill_d128"] = bench_simple_prefill(api, "prefill128", rank, world)
        if "gated" in wanted:
            extra["gated_delta"] = bench_gated_delta(api, rank, world)
        if "decay" in wanted:
            extra["decay_prefill"] = bench_decay_prefill(api, rank, world)
        if "decay128" in wanted:
            extra["decay_prefill_d128"] = bench_decay_prefill(api, rank, world, wname="prefill128")
        if "rbw" in wanted:
            extra["rbw_prefill"] = bench_order_prefill(api, rank, world, api.LA_MODE_READ_BEFORE_WRITE)
        if "nc" in wanted:
            extra["noncausal_prefill"] = bench_order_prefill(api, rank, world, api.LA_MODE_NONCAUSAL)
        if "rbw128" in wanted:
            extra["rbw_prefill_d128"] = bench_order_prefill(api, rank, world, api.LA_MODE_READ_BEFORE_WRITE,
                                                            wname="prefill128")
        if "nc128" in wanted:
            extra["noncausal_prefill_d128"] = bench_order_prefill(api, rank, world, api.LA_MODE_NONCAUSAL,
                                                                  wname="prefill128")
        if "backward" in wanted:
            extra["backward"] = bench_backward(api, rank, world)
        e_steps = min(max(args.steps // 4, 20), 200)  # at least 20 steps whatever --steps is
        e_ms, h2d, d2h = bench_e2e(api, w, e_steps, 3, rank, world)
        e2e = {"value": w.tokens * world / (e_ms * 1e-3 / e_steps), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": e_steps}
    clocks = sampler.stop()

    hbm_peak, _, peak_kind = _peaks()
    algo_bytes = PREFILL_BYTES_PER_TOKEN * w.tokens + w.B * w.H * (w.dk * w.dv + w.dk) * 4
    launch_ms = statistics.mean(per)
    achieved = algo_bytes / (launch_ms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved / hbm_peak, "traffic": _committed_traffic(w.tokens),
                "peak_kind": f"of {peak_kind}",
                "algorithmic_bytes_per_launch": algo_bytes,
                "launch_ms_mean": launch_ms, "launch_ms_min": min(per),
                "tensor": tensor_fractions(w.dk, 128, w.tokens, launch_ms, _peaks()[1])}
    if "decode" in extra:
        extra["decode"]["hbm_frac"] = extra["decode"]["hbm_gbs"] / hbm_peak
    for name in ("long", "prefill_d128"):
        if name in extra and "hbm_gbs" in extra[name]:
            extra[name]["hbm_frac"] = extra[name]["hbm_gbs"] / hbm_peak
            ew = inputs.WORKLOADS["prefill128" if name == "prefill_d128" else name]
            extra[name]["tensor"] = tensor_fractions(ew.dk, 128, ew.tokens,
                                                     extra[name]["ms_per_call"], _peaks()[1])
    if "delta" in extra:
        extra["delta"]["hbm_frac"] = extra["delta"]["hbm_gbs"] / hbm_peak

    cpu = None
    if rank == 0 and world == 1 and not args.no_extra:
        cpu = cpu_baseline(w)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16", "data": "synthetic",
                "config": {"workload": "prefill: B=4 H=8 N=4096 dk=dv=64, bf16 q,k,v ~ N(0,1), "
                                       "fp32 state/accumulate, zero initial state",
                           "B": w.B, "H": w.H, "N": w.N, "dk": w.dk, "dv": w.dv,
                           "chunk": 128, "parallelism": f"replicas x{world}",
                           "l2": "4 rotating input/output buffer sets (~340 MB > 129 MB L2)"},
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": args.steps * PREFILL_LAUNCHES_PER_CALL, "clocks": clocks,
                "extra": extra}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
