"""Benchmark of the gated delta rule hot path on GB300.

One step is one gdr_chunk_fwd call (chunked prefill) over the B=4, H=16,
T=4096, d_k=d_v=128 bf16 workload, with inputs resident in HBM. The decode row
of the hot path (gdr_decode_step over 256 sequences x 32 heads, fp32 state of
537 MB) is timed in the same run and reported under "decode"; the other prefill
workloads (packed varying lengths, one long sequence with d_v = 256, the tiny fp32
case) under "varlen", "long" and "tiny". Every workload also runs a sustained stretch
of back-to-back calls (about 2 s) with the clocks sampled.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gdr|reference]

Prints ONE JSON line on rank 0. Under torchrun (N > 1) every rank runs an
independent replica of the workload (the path needs no collective); the time
is the max over ranks and `value` counts the tokens of all ranks.
`--impl reference` times the float64 CPU oracle (the reference arm) instead.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from gated_delta_rule_03_gb300 import inputs  # noqa: E402

METRIC = "GDN prefill tokens/s (H=16,d=128,bf16); decode state GB/s vs HBM peak"
PREFILL_WORKLOAD = "prefill_bf16"  # the headline workload; --workload picks another
DECODE_WORKLOAD = "decode_bf16"


# ----------------------------------------------------------------------------- helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def prefill_bytes(inp):
    """Algorithmic HBM bytes of one prefill call: read q, k, v and the gates, write o,
    write S_final (and read S0 when given)."""
    esz = 2 if inp.dtype == "bf16" else 4
    per_token_head = (2 * inp.dk + 2 * inp.dv) * esz
    gates = (inp.log_alpha.numel() + inp.beta.numel()) * 4  # one or d_k forget rates, beta
    state = inp.num_seqs * inp.H * inp.dk * inp.dv * 4
    return (inp.total_tokens * inp.H * per_token_head + gates +
            state * (2 if inp.S0 is not None else 1))


def prefill_flops(inp):
    """Algorithmic flops of one prefill call: the chunk count of "Attention as Matrix
    Algebra", section 8, 4 C d_k + 3 C d_v + 6 d_k d_v per token-head."""
    C = inp.chunk
    return inp.total_tokens * inp.H * (4 * C * inp.dk + 3 * C * inp.dv + 6 * inp.dk * inp.dv)


def decode_bytes(N, H, dk, dv, esz=2):
    """Algorithmic HBM bytes of one decode step: the fp32 state read and written once,
    plus q, k, v, o and the two gates."""
    return N * H * (2 * dk * dv * 4 + (2 * dk + 2 * dv) * esz + 8)


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch from an ncu capture summarised in profiles/traffic.txt. A
    record holds while the kernel's source files (and the shared internal header) are
    unchanged since the capture; otherwise the traffic is unknown (None)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        for line in f:
            fields = dict(kv.split("=", 1) for kv in line.split() if "=" in kv)
            if fields.get("kernel") != kernel or fields.get("workload") != workload:
                continue
            if fields.get("source_sha") == source_sha(fields.get("source", "")):
                return float(fields["dram_bytes_per_launch"])
    return None


def source_sha(names):
    """Hash of the CUDA source files a kernel is built from (comma-separated names) plus
    the internal header every kernel includes."""
    csrc = os.path.join(ROOT, "gated_delta_rule_03_gb300", "csrc")
    h = hashlib.sha256()
    for fn in [n for n in names.split(",") if n] + ["internal.h"]:
        path = os.path.join(csrc, fn)
        if not os.path.exists(path):
            return None
        with open(path, "rb") as f:
            h.update(fn.encode() + f.read())
    return h.hexdigest()[:16]


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples taken while the GPU works."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, local_rank):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        self.index = vis.split(",")[local_rank] if vis else str(local_rank)
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", self.index, "-lms", "50"], stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        with open(self.file.name) as f:
            rows = [r.strip().split(", ") for r in f if r.strip()]
        os.unlink(self.file.name)
        sm, reasons, smax = [], set(), None
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax = float(r[2])
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_model():
    """The host CPU's model name (from /proc/cpuinfo or lscpu), for the baseline records."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":", 1)[0].strip().lower()
                if key in ("model name", "cpu model", "hardware") and ":" in line:
                    val = line.split(":", 1)[1].strip()
                    if val:
                        return val
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=5).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return "unknown"


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def timed_calls(fn, steps, stream, world, device, per_call=True):
    """Run fn() `steps` times on `stream` between a barrier and a synchronize on both
    sides; return (total ms max over ranks, mean per-call ms from per-call events)."""
    barrier(world)
    torch.cuda.synchronize(device)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(steps)] if per_call else []
    with torch.cuda.stream(stream):
        start.record(stream)
        for i in range(steps):
            if per_call:
                pairs[i][0].record(stream)
            fn()
            if per_call:
                pairs[i][1].record(stream)
        end.record(stream)
    torch.cuda.synchronize(device)
    barrier(world)
    total = max_over_ranks(start.elapsed_time(end), world, device)
    mean_call = (sum(a.elapsed_time(b) for a, b in pairs) / steps) if per_call else None
    return total, mean_call


def sustained_calls(fn, stream, device, local_rank, seconds, est_ms):
    """Back-to-back calls of fn() for about `seconds` on `stream`, with nvidia-smi sampling
    the clocks meanwhile: a stretch long enough for an outside sampler to see the GPU
    busy. Returns the calls, the CUDA-event time and the clock samples."""
    calls = int(min(max(seconds * 1e3 / max(est_ms, 1e-3), 1), 500_000))
    clocks = ClockSampler(local_rank)
    clocks.start()
    torch.cuda.synchronize(device)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(calls):
            fn()
        end.record(stream)
    torch.cuda.synchronize(device)
    ms = start.elapsed_time(end)
    return {"calls": calls, "seconds": ms / 1e3, "ms_per_call": ms / calls,
            "clocks": clocks.stop()}


# ----------------------------------------------------------------------------- arms

def oracle_prefill_sample(inp):
    """Float64 views of the workload for the oracle, prepared outside any timing."""
    f = lambda t: t.to(torch.float64).numpy()
    cu = None if inp.cu_seqlens is None else inp.cu_seqlens.numpy().astype(np.int64)
    return dict(q=f(inp.q), k=f(inp.k), v=f(inp.v), log_alpha=f(inp.log_alpha),
                beta=f(inp.beta), S0=None if inp.S0 is None else f(inp.S0), cu_seqlens=cu,
                num_seqs=inp.num_seqs)


def cpu_baseline(inp, seconds, name, heads=None, gpu_out=None):
    """The oracle, as it stands, on this host's cores: repeat the full workload (or only
    the given heads of it) until `seconds` have passed (at least once). With a subset of
    heads the rate is scaled to the workload's H heads (the heads are independent and
    equal in work) and the per-head rate is reported beside it. gpu_out: the timed call's
    (o, S_final) for the same heads, as float64 arrays; the oracle's result is compared
    with them (max |gpu - oracle| / max |oracle|, the tests' measure) under "parity"."""
    import oracle
    args = oracle_prefill_sample(inp)
    nh = inp.H
    if heads is not None:
        sel = list(heads)
        nh = len(sel)
        for key in ("q", "k", "v", "log_alpha", "beta"):
            args[key] = np.ascontiguousarray(args[key][:, sel])
        if args["S0"] is not None:
            args["S0"] = np.ascontiguousarray(args["S0"][:, sel])
    threads = oracle.default_threads()
    reps, t0 = 0, time.perf_counter()
    while True:
        ref = oracle.forward(**args, threads=threads)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds or reps >= 1000:
            break
    token_heads = inp.total_tokens * nh * reps
    out = {"value": token_heads / inp.H / el, "unit": "tokens/s", "cores": threads,
           "cpu_model": cpu_model(), "kind": "oracle"}
    what = f"full {name} workload" if heads is None else \
        f"{name} workload, heads {sel[0]}-{sel[-1]} of {inp.H} (rate scaled to all heads)"
    out["sample"] = (f"{what} ({inp.num_seqs} sequences, {inp.total_tokens} tokens, "
                     f"H={nh}, d_k={inp.dk}, d_v={inp.dv}) x {reps} repetitions, "
                     f"{el:.1f} s, float64 token loop")
    if heads is not None:
        out["per_head_token_rate"] = token_heads / nh / el
    if gpu_out is not None:
        err = lambda g, r: float(np.abs(g - r).max() / max(np.abs(r).max(), 1e-300))
        out["parity"] = {"o_rel_err": err(gpu_out[0], ref[0]), "S_rel_err": err(gpu_out[1], ref[1]),
                         "tolerance": 1e-4 if inp.dtype == "f32" else 2e-2,
                         "heads": "all" if heads is None else list(heads)}
    return out


def host_outputs(o, S, heads=None):
    """The call's o and S_final (the given heads only) as float64 host arrays."""
    if heads is not None:
        o, S = o[:, list(heads)], S[:, list(heads)]
    return (o.to(torch.float64).cpu().numpy(), S.to(torch.float64).cpu().numpy())


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    inp = inputs.workload_prefill(args.workload, decay=args.decay)
    sample = oracle_prefill_sample(inp)
    threads = oracle.default_threads()
    for _ in range(args.warmup):
        oracle.forward(**sample, threads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.forward(**sample, threads=threads)
    el = time.perf_counter() - t0
    value = inp.total_tokens * args.steps / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(inp, args.workload),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads,
                         "cpu_model": cpu_model(), "kind": "oracle",
                         "sample": f"each step: the full {args.workload} workload, "
                                   f"float64 token loop on {threads} host threads"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(inp, name):
    equal = len(set(inp.seq_lens)) == 1
    if inp.log_alpha.dim() == 3:
        name += " with one forget rate per key channel"

    lens = f"T={inp.seq_lens[0]}" if equal else f"T in {min(inp.seq_lens)}..{max(inp.seq_lens)} " \
                                                 f"packed ({inp.total_tokens} tokens)"
    s0 = "S0=0" if inp.S0 is None else "S0 ~ N(0, 0.02^2)"
    return {"workload": f"{name}: B={inp.num_seqs} H={inp.H} {lens} "
                        f"d_k={inp.dk} d_v={inp.dv} chunk={inp.chunk} {inp.dtype} q/k/v/o, fp32 "
                        f"gates and state, {s0}",
            "global_batch": inp.num_seqs,
            "seq_len": inp.seq_lens[0] if equal else inp.total_tokens // inp.num_seqs,
            "heads": inp.H, "l2": "inputs larger than L2 (no flush)", "parallelism": "replicas"}


# the other prefill workloads, timed in the same run as the headline one
# (key, workload, heads the CPU baseline runs (None: all), forget-rate granularity)
SIDE_WORKLOADS = (("varlen", "varlen_bf16", None, "head"), ("long", "long_bf16", (0, 1), "head"),
                  ("tiny", "tiny_fp32", None, "head"),
                  ("channel", "prefill_bf16", (0, 1), "channel"))


def bench_prefill_workload(name, args, device, stream, world, local, peaks, cpu_heads=None,
                           decay="head"):
    """One prefill workload: per-call CUDA-event timing over the driver's --steps, a
    sustained stretch of back-to-back calls with the clocks sampled, the roofline of the
    call (HBM and tensor fractions), the recorded DRAM traffic and the oracle on the host."""
    from gated_delta_rule_03_gb300 import chunk_fwd, chunk_fwd_workspace_size, ops
    inp = inputs.workload_prefill(name, decay=decay)
    d = lambda t: None if t is None else t.to(device)
    q, k, v, la, b = d(inp.q), d(inp.k), d(inp.v), d(inp.log_alpha), d(inp.beta)
    S0, cu = d(inp.S0), d(inp.cu_seqlens)
    o = torch.empty((inp.total_tokens, inp.H, inp.dv), dtype=q.dtype, device=device)
    S = torch.empty((inp.num_seqs, inp.H, inp.dk, inp.dv), dtype=torch.float32, device=device)
    ws = torch.empty(chunk_fwd_workspace_size(inp.num_seqs, inp.total_tokens, inp.H, inp.dk,
                                              inp.dv, inp.chunk, q.dtype, decay),
                     dtype=torch.uint8, device=device)

    def step():
        chunk_fwd(q, k, v, la, b, S0=S0, cu_seqlens=cu, num_seqs=inp.num_seqs, chunk=inp.chunk,
                  o=o, S_final=S, workspace=ws, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    total_ms, call_ms = timed_calls(step, args.steps, stream, world, device)
    sus = sustained_calls(step, stream, device, local, args.sustained_seconds, call_ms)
    varlen = cu is not None
    schedule = ops.chunk_fwd_schedule(inp.num_seqs, inp.total_tokens, inp.H, inp.dk, inp.dv,
                                      q.dtype, varlen=varlen, decay=decay)
    main_kernel = ops.chunk_fwd_main_kernel(inp.dk, inp.dv, q.dtype, schedule=schedule,
                                            decay=decay)
    launches = ops.chunk_fwd_kernel_launches(inp.num_seqs, inp.total_tokens, inp.H, inp.dk,
                                             inp.dv, q.dtype, varlen=varlen, decay=decay)
    traffic_key = name + ("" if decay == "head" else "_channel")
    nbytes, flops = prefill_bytes(inp), prefill_flops(inp)
    achieved = nbytes / (call_ms / 1e3) / 1e9
    tflops = flops / (call_ms / 1e3) / 1e12
    out = {
        "workload": workload_config(inp, name)["workload"],
        "tokens_per_s": world * inp.total_tokens * args.steps / (total_ms / 1e3),
        "ms_per_call": total_ms / args.steps, "steps": args.steps,
        "schedule": schedule, "dtype": ops.chunk_fwd_compute_dtype(inp.dk, inp.dv, q.dtype, decay),
        "roofline": {"kernel": main_kernel, "bound": "hbm", "achieved": achieved,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                     "traffic": recorded_traffic(main_kernel, traffic_key),
                     "algorithmic_bytes_per_launch": nbytes, "launch_ms": call_ms,
                     "tensor": {"achieved": tflops, "peak": peaks["bf16_tflops"],
                                "unit": "TFLOP/s", "frac": tflops / peaks["bf16_tflops"],
                                "algorithmic_flops_per_launch": flops}},
        "sustained": sus,
        "gpu_launches": launches * (args.steps + sus["calls"]),
        "cpu_baseline": None,
    }
    if inp.dtype == "f32":
        out["roofline"]["note"] = ("latency-bound: 512 token-heads in 8 chunks; reported, no "
                                   "roofline target")
    cpu = world == 1 and not args.no_cpu_baseline
    gpu_out = host_outputs(o, S, cpu_heads) if cpu else None
    del q, k, v, la, b, S0, cu, o, S, ws
    torch.cuda.empty_cache()
    if cpu:
        out["cpu_baseline"] = cpu_baseline(inp, min(args.cpu_seconds, 3.0), traffic_key,
                                           heads=cpu_heads, gpu_out=gpu_out)
    return out


def run_gdr(args):
    from gated_delta_rule_03_gb300 import chunk_fwd, chunk_fwd_workspace_size, decode_step, ops
    world, rank, local = dist_env()
    if world > 1:
        torch.distributed.init_process_group("nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    stream = torch.cuda.Stream(device)
    peaks = load_peaks()

    inp = inputs.workload_prefill(args.workload, decay=args.decay)
    d = lambda t: None if t is None else t.to(device)
    q, k, v, la, b = d(inp.q), d(inp.k), d(inp.v), d(inp.log_alpha), d(inp.beta)
    S0, cu = d(inp.S0), d(inp.cu_seqlens)
    o = torch.empty((inp.total_tokens, inp.H, inp.dv), dtype=q.dtype, device=device)
    S = torch.empty((inp.num_seqs, inp.H, inp.dk, inp.dv), dtype=torch.float32, device=device)
    ws = torch.empty(chunk_fwd_workspace_size(inp.num_seqs, inp.total_tokens, inp.H, inp.dk,
                                              inp.dv, inp.chunk, q.dtype, args.decay),
                     dtype=torch.uint8, device=device)

    def step():
        chunk_fwd(q, k, v, la, b, S0=S0, cu_seqlens=cu, num_seqs=inp.num_seqs, chunk=inp.chunk,
                  o=o, S_final=S, workspace=ws, stream=stream)

    clocks = ClockSampler(local)
    clocks.start()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    total_ms, call_ms = timed_calls(step, args.steps, stream, world, device)
    clock_info = clocks.stop()
    # a sustained stretch of the same call (its own clock samples), long enough for an
    # outside sampler to see the GPU busy; `value` stays the timed --steps above
    sustained = sustained_calls(step, stream, device, local, args.sustained_seconds, call_ms)

    tokens = inp.total_tokens
    value = world * tokens * args.steps / (total_ms / 1e3)
    kernel_launches = ops.chunk_fwd_kernel_launches(inp.num_seqs, inp.total_tokens, inp.H, inp.dk,
                                                    inp.dv, q.dtype, varlen=cu is not None,
                                                    decay=args.decay)
    schedule = ops.chunk_fwd_schedule(inp.num_seqs, inp.total_tokens, inp.H, inp.dk, inp.dv,
                                      q.dtype, varlen=cu is not None, decay=args.decay)
    main_kernel = ops.chunk_fwd_main_kernel(inp.dk, inp.dv, q.dtype, schedule=schedule,
                                            decay=args.decay)
    bytes_call = prefill_bytes(inp)
    achieved = bytes_call / (call_ms / 1e3) / 1e9
    workload_key = args.workload + ("" if args.decay == "head" else "_channel")
    traffic = recorded_traffic(main_kernel, workload_key)

    # end to end through the public API: every step copies its inputs in from pinned host
    # memory and its results (o and the final state) back out. Steps are pipelined over
    # three streams with two device copies of the inputs and outputs: the copy-in of step
    # i + 1 and the copy-out of step i - 1 run while step i computes.
    pin = lambda t: None if t is None else t.pin_memory()
    host_in = [pin(t) for t in (inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, inp.S0)
               if t is not None]
    dev_in = [[torch.empty(t.shape, dtype=t.dtype, device=device) for t in host_in]
              for _ in range(2)]
    dev_out = [(torch.empty_like(o), torch.empty_like(S)) for _ in range(2)]
    host_out = [(torch.empty(o.shape, dtype=o.dtype).pin_memory(),
                 torch.empty(S.shape, dtype=S.dtype).pin_memory()) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of buffer set b landed
    ev_done = [torch.cuda.Event() for _ in range(2)]  # the call on set b finished
    ev_out = [torch.cuda.Event() for _ in range(2)]   # the outputs of set b copied out

    def e2e_steps(n):
        for i in range(n):
            bset = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:  # the call two steps back has read this set's inputs
                    s_in.wait_event(ev_done[bset])
                for h, dv in zip(host_in, dev_in[bset]):
                    dv.copy_(h, non_blocking=True)
                ev_in[bset].record(s_in)
            stream.wait_event(ev_in[bset])
            if i >= 2:  # this set's outputs of two steps back are out
                stream.wait_event(ev_out[bset])
            qd, kd, vd, lad, bd = dev_in[bset][:5]
            s0d = dev_in[bset][5] if inp.S0 is not None else None
            chunk_fwd(qd, kd, vd, lad, bd, S0=s0d, cu_seqlens=cu, num_seqs=inp.num_seqs,
                      chunk=inp.chunk, o=dev_out[bset][0], S_final=dev_out[bset][1],
                      workspace=ws, stream=stream)
            ev_done[bset].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[bset])
                host_out[bset][0].copy_(dev_out[bset][0], non_blocking=True)
                host_out[bset][1].copy_(dev_out[bset][1], non_blocking=True)
                ev_out[bset].record(s_out)

    e2e_steps(min(args.warmup, 3))
    torch.cuda.synchronize(device)
    barrier(world)
    e2e_start, e2e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_start.record(s_in)
    stream.wait_event(e2e_start)
    s_out.wait_event(e2e_start)
    e2e_steps(args.steps)
    s_out.wait_event(ev_done[(args.steps - 1) % 2])
    e2e_end.record(s_out)
    torch.cuda.synchronize(device)
    barrier(world)
    e2e_ms = max_over_ranks(e2e_start.elapsed_time(e2e_end), world, device)
    e2e_value = world * tokens * args.steps / (e2e_ms / 1e3)

    decode = None
    if not args.no_decode:
        decode = run_decode(args, decode_step, device, stream, world, peaks, local)

    side = {}
    if not args.no_side and args.decay == "head":
        for key, name, heads, decay in SIDE_WORKLOADS:
            if (name, decay) != (args.workload, args.decay):
                side[key] = bench_prefill_workload(name, args, device, stream, world, local,
                                                   peaks, cpu_heads=heads, decay=decay)

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(inp, args.cpu_seconds, workload_key, gpu_out=host_outputs(o, S))

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ops.chunk_fwd_compute_dtype(inp.dk, inp.dv, q.dtype, args.decay),
        "data": "synthetic",
        "config": workload_config(inp, args.workload),
        "roofline": {"kernel": main_kernel, "bound": "hbm", "achieved": achieved,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                     "algorithmic_bytes_per_launch": bytes_call,
                     "launch_ms": call_ms, "peak_source": peaks["source"],
                     # the other bound, for the same call: the chunk form's flops against
                     # the measured bf16 burst peak (the binding one is the HBM fraction)
                     "tensor": {"achieved": prefill_flops(inp) / (call_ms / 1e3) / 1e12,
                                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                                "frac": prefill_flops(inp) / (call_ms / 1e3) / 1e12 /
                                        peaks["bf16_tflops"],
                                "algorithmic_flops_per_launch": prefill_flops(inp)},
                     "timing": "CUDA events around each gdr_chunk_fwd call on its stream"},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms / args.steps,
                "pipeline": "two device sets of inputs and outputs on three streams: the "
                            "copy-in of step i+1 and the copy-out of step i-1 overlap step i"},
        "gpu_launches": kernel_launches * args.steps,
        "clocks": clock_info,
        "sustained": sustained,
        "decode": decode,
    }
    line.update(side)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def cpu_decode_baseline(dec, seconds, seqs=8):
    """The oracle's decode step on this host's cores over a bounded sample: the first
    `seqs` sequences (all heads) of the workload, its steps cycled until `seconds` pass."""
    import oracle
    sel = slice(0, seqs)
    f = lambda t: t.to(torch.float64).numpy()
    steps = [(f(dec.q[s])[sel], f(dec.k[s])[sel], f(dec.v[s])[sel], f(dec.log_alpha[s])[sel],
              f(dec.beta[s])[sel]) for s in range(dec.steps)]
    S = f(dec.S)[sel]
    threads = oracle.default_threads()
    calls, t0 = 0, time.perf_counter()
    while True:
        _, S = oracle.decode(*steps[calls % dec.steps], S, threads=threads)
        calls += 1
        el = time.perf_counter() - t0
        if el >= seconds or calls >= 10000:
            break
    state_bytes = 2 * seqs * dec.H * dec.dk * dec.dv * 4  # fp32 state read + written, as on the GPU
    return {"value": state_bytes * calls / el / 1e9, "unit": "GB/s (fp32 state read + written)",
            "cores": threads, "cpu_model": cpu_model(), "kind": "oracle",
            "sample": f"{seqs} of {dec.N} sequences x {dec.H} heads, {calls} decode steps, "
                      f"{el:.1f} s, float64"}


def run_decode(args, decode_step, device, stream, world, peaks, local=0):
    w = inputs.WORKLOADS[DECODE_WORKLOAD]
    decay = getattr(args, "decay", "head")
    dec = inputs.workload_decode(DECODE_WORKLOAD, decay=decay)
    S = dec.S.to(device)
    qs, ks, vs = dec.q.to(device), dec.k.to(device), dec.v.to(device)
    las, bs = dec.log_alpha.to(device), dec.beta.to(device)
    o = torch.empty((dec.N, dec.H, dec.dv), dtype=qs.dtype, device=device)
    it = [0]

    def step():
        s = it[0] % dec.steps
        decode_step(qs[s], ks[s], vs[s], las[s], bs[s], S, o=o, stream=stream)
        it[0] += 1

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            step()
    calls = max(dec.steps, args.steps)
    total_ms, call_ms = timed_calls(step, calls, stream, world, device)
    sus = sustained_calls(step, stream, device, local, args.sustained_seconds, call_ms)
    nbytes = decode_bytes(dec.N, dec.H, dec.dk, dec.dv)
    if decay == "channel":  # d_k fp32 rates per (n, h) instead of one
        nbytes += dec.N * dec.H * (dec.dk - 1) * 4
    state_bytes = 2 * dec.N * dec.H * dec.dk * dec.dv * 4
    achieved = nbytes / (call_ms / 1e3) / 1e9
    rates = "" if decay == "head" else ", one forget rate per key channel"
    return {"workload": f"{DECODE_WORKLOAD}: N={w['N']} H={w['H']} d_k={w['dk']} d_v={w['dv']}, "
                        f"{dec.steps} distinct steps cycled, fp32 state "
                        f"{state_bytes // 2 / 1e6:.0f} MB{rates}",
            "calls": calls, "ms_per_step": total_ms / calls,
            "state_gbs": world * state_bytes * calls / (total_ms / 1e3) / 1e9,
            "roofline": {"kernel": "decode_step_kernel", "bound": "hbm", "achieved": achieved,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"],
                         "traffic": recorded_traffic("decode_step_kernel", DECODE_WORKLOAD)
                         if decay == "head" else None,
                         "algorithmic_bytes_per_launch": nbytes, "launch_ms": call_ms},
            "sustained": sus,
            "gpu_launches": calls + sus["calls"],
            "cpu_baseline": (cpu_decode_baseline(dec, min(args.cpu_seconds, 5.0))
                             if world == 1 and not args.no_cpu_baseline else None)}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["gdr", "reference"], default="gdr")
    ap.add_argument("--workload", choices=["prefill_bf16", "varlen_bf16", "long_bf16"],
                    default=PREFILL_WORKLOAD,
                    help="prefill workload of the step (default: the headline prefill_bf16)")
    ap.add_argument("--decay", choices=["head", "channel"], default="head",
                    help="forget rates: one per head (default), or one per key channel")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--sustained-seconds", type=float, default=2.0,
                    help="length of each workload's stretch of back-to-back calls")
    ap.add_argument("--no-side", action="store_true",
                    help="skip the other prefill workloads (varlen, long, tiny)")
    ap.add_argument("--only", choices=["all", "decode"], default="all",
                    help="'decode' runs only the decode timing (for profiling that kernel)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.only == "decode":
        return run_decode_only(args)
    return run_gdr(args)


def run_decode_only(args):
    """Only the decode timing, printed as its own JSON object (a profiling aid; the
    benchmark line proper comes from the default mode)."""
    from gated_delta_rule_03_gb300 import decode_step
    world, rank, local = dist_env()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    stream = torch.cuda.Stream(device)
    out = run_decode(args, decode_step, device, stream, 1, load_peaks(), local)
    print(json.dumps({"decode": out}), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
