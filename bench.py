#!/usr/bin/env python
"""Throughput of the KATA chunked-state forward at the long-context workload
(B=1, H=8, T=131072, p=64, d_v=64, C=128, bf16, associative-scan prefix).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one kata_forward_chunked call over the whole workload (every
step of the path: normalise, lift, intra-chunk scores, state build, inter-
chunk prefix, readout, normalisation).  Inputs are resident in HBM and
larger than L2 (403 MB), so no L2 flush is needed between steps.  Prints one
JSON line on rank 0.  Under torchrun every rank runs its own replica of the
workload (independent sequences, no collective on the data path): weak
scaling, value = all ranks' tokens / max-over-ranks time.

--impl reference times the fp64 CPU oracle (the only reference this method
has) on a bounded sample of the same workload on the host cores.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from kernelized_linear_attention_03_b300 import binding as kb  # noqa: E402
from kernelized_linear_attention_03_b300 import inputs  # noqa: E402

METRIC = "KATA chunked fwd tokens/s at T=131072 (1 B300); % tensor-core peak"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
                  "sm_max_mhz": 2032.0}
SMS = 148
FP32_LANES_PER_SM = 128
DECODE_B, DECODE_H = 64, 16  # decode batch: sequences x heads, one new token each
LIFTS = {"sigma": 1, "multi": 2}  # block-lift families (KATA-Sigma-g, KATA-M-g)
BLOCK_FORMS = ("chunked_block", "quadratic_block", "decode_block")


def load_peaks():
    if os.path.exists(PEAKS_FILE):
        with open(PEAKS_FILE) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    d = dict(FALLBACK_PEAKS)
    d["source"] = "fallback"
    return d


# ---------------------------------------------------------------- work model
def flops_forward(w):
    """Algorithmic flops of one chunked forward: per head-token
    4 n (dv+1) (state build + readout, normaliser column included) plus
    (C+1)(p+dv) (causal intra-chunk scores and their value product)."""
    return w.B * w.H * w.T * (4 * w.n * (w.dv + 1) + (w.C + 1) * (w.p + w.dv))


def lift_dim(family, p, g):
    """Width of a block lift: KATA-Sigma-g m(m+1)/2, KATA-M-g g m(m+1)/2 (m = p/g)."""
    m = p // g
    return m * (m + 1) // 2 * (1 if family == LIFTS["sigma"] else g)


# DRAM bytes per launch of the dominant kernel (dram__bytes_read.sum + dram__bytes_write.sum from
# one ncu pass with --clock-control none) for the configurations they were captured on; the summary
# under profiles/ gives the command.  An entry is dropped whenever its kernel changes.
MEASURED_TRAFFIC = {
    ("chunked", "c4_T131072_p64_bf16", "chunked_tc"): 1.36e9 + 431.20e6,
}


def kernel_work(name, w, form="chunked", lift=None):
    """(kind, algorithmic amount per forward call) of a library kernel.  `lift`
    = (family, g) for the block-lift forms."""
    bht = w.B * w.H * w.T
    if lift is not None:
        family, g = lift
        n, m = lift_dim(family, w.p, g), w.p // g
        pairs = g * g if family == LIFTS["sigma"] else g  # block dot products per score
        if name == "block_states_simt":
            return "flop", bht * 2 * n * (w.dv + 1)
        if name == "block_output_simt":
            # prefix readout with the normaliser column, and the causal local half with block scores
            return "flop", bht * (2 * n * (w.dv + 1) + (w.C + 1) * (pairs * m + w.dv))
        if name == "block_quadratic_simt":
            return "flop", bht * (w.T + 1) * (pairs * m + w.dv)
        if name in ("scan_tree", "scan_sequential"):
            return "byte", 2 * w.B * w.H * w.NC * n * (w.dv + 1) * 4
        if name == "decode_step_block":
            elem = 4 if w.dtype == "fp32" else 2
            return "byte", w.B * w.H * (2 * n * (w.dv + 1) * 4 + (2 * w.p + 2 * w.dv) * elem)
        if name == "chunked_tc":
            # the fused KATA-Sigma-g forward: state build and readout with the normaliser column
            return "flop", bht * 4 * n * (w.dv + 1)
        if name == "intra_tc":
            # the causal local half with block scores
            return "flop", bht * (w.C + 1) * (pairs * m + w.dv)
        return None, 0
    if name in ("chunk_states_simt",):
        return "flop", bht * 2 * w.n * (w.dv + 1)
    if name in ("chunk_output_simt",):
        return "flop", bht * (2 * w.n * (w.dv + 1) + (w.C + 1) * (w.p + w.dv))
    if name in ("scan_tree", "scan_sequential"):
        return "byte", 2 * w.B * w.H * w.NC * w.n * (w.dv + 1) * 4
    if name in ("quadratic_tc", "quadratic_simt", "quadratic_gated_tc"):
        # causal half of the flash-style form: (T+1)(p+dv) per head-token
        return "flop", bht * (w.T + 1) * (w.p + w.dv)
    if name == "states_tc" and form == "chunk_state_scan":
        # every chunk state is written once (fp32), the keys and values read once
        return "byte", w.B * w.H * w.NC * w.n * (w.dv + 1) * 4 + bht * (w.p + w.dv) * 2
    if name == "chunked_tc":
        # the fused forward: state build and readout with the normaliser column
        return "flop", bht * 4 * w.n * (w.dv + 1)
    if name == "normalize":
        # fp32 numerator rows and denominators read, o written
        return "byte", bht * (w.dv * 4 + 4 + w.dv * 2)
    if name == "intra_tc":
        # the causal intra-chunk half of the forward
        return "flop", bht * (w.C + 1) * (w.p + w.dv)
    if name == "states_tc" and form == "gated":
        # the gated form's chunk states (each key lift weighted by its decay)
        return "flop", bht * 2 * w.n * (w.dv + 1)
    if name == "states_tc":
        # segment start states: recomputed work, no algorithmic share
        return "flop", 0
    if name == "backward_query_simt" or name == "backward_key_simt":
        # prefix readout and its gradient (normaliser column included), two passes over the
        # causal local half at the backward's 64-token chunks
        return "flop", bht * (4 * w.n * (w.dv + 1) + 2 * 65 * (w.p + w.dv))
    if name == "backward_gstates_simt" or name == "gated_states_simt":
        return "flop", bht * 2 * w.n * (w.dv + 1)
    if name in ("backward_rows_simt", "backward_cols_simt"):
        # flash-style backward: two passes over the causal half per query (rows) or key (columns)
        return "flop", bht * 2 * (w.T + 1) * (w.p + w.dv)
    if name == "gated_output_simt":
        return "flop", bht * (2 * w.n * (w.dv + 1) + (w.C + 1) * (w.p + w.dv))
    if name in ("gated_scan", "backward_reverse_scan"):
        nc = w.NC if name == "gated_scan" else (w.T + 63) // 64
        return "byte", 2 * w.B * w.H * nc * w.n * (w.dv + 1) * 4
    if name == "gate_decay":
        # the gates read, each token's decay to its chunk's end written
        return "byte", bht * 8
    if name == "gate_prefix":
        # the gates read, the per-token log-gate sums and last zero gates written
        return "byte", bht * 12
    if name == "decode_step":
        # state and normaliser read and written once, the token's q, k, v read, o written
        elem = 4 if w.dtype == "fp32" else 2
        return "byte", w.B * w.H * (2 * w.n * (w.dv + 1) * 4 + (2 * w.p + 2 * w.dv) * elem)
    return None, 0


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, device):
        self.samples = []
        self.proc = None
        self.thread = None
        sel = []
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            pass
        self.cmd = ["nvidia-smi", *sel, "--query-gpu=" + ",".join(self.FIELDS),
                    "--format=csv,noheader,nounits", "-lms", "100"]

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == len(self.FIELDS):
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=5)

    def summary(self, t0, t1):
        inside = [s for (t, s) in self.samples if t0 <= t <= t1] or [s for (_, s) in self.samples]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(s[0]) for s in inside if num(s[0]) is not None]
        smax = [num(s[1]) for s in inside if num(s[1]) is not None]
        reasons = set()
        for s in inside:
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                  "sw_power_cap"), s[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        power = [num(s[2]) for s in inside if num(s[2]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(inside),
                "power_w_median": statistics.median(power) if power else None}


# ---------------------------------------------------------------- distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- CPU oracle
def oracle_sample(w, q, k, v, T_s, nthreads):
    """Run the fp64 oracle's chunked form on the first T_s tokens of every
    head; return seconds."""
    import oracle
    qs, ks, vs = (t[:, :, :T_s].double().cpu().numpy() for t in (q, k, v))
    t0 = time.perf_counter()
    oracle.forward_chunked(qs, ks, vs, w.C, oracle.SCAN_TREE, nthreads=nthreads)
    return time.perf_counter() - t0


def oracle_threads(w):
    try:
        cores = len(os.sched_getaffinity(0))
    except AttributeError:
        cores = os.cpu_count() or 1
    return max(1, min(cores, w.B * w.H))


def sample_len(w, q, k, v, seconds, nthreads):
    """Tokens per head for an oracle sample of about `seconds` (multiple of C),
    calibrated on a short sample long enough that the per-call overhead does
    not dominate."""
    T_c = min(w.T, 8 * w.C)
    t_cal = max(oracle_sample(w, q, k, v, T_c, nthreads), 1e-3)
    T_s = int(T_c * seconds / t_cal)
    return max(w.C, min(w.T, T_s // w.C * w.C))


def cpu_baseline(w, q, k, v, seconds=15.0):
    nthreads = oracle_threads(w)
    T_s = sample_len(w, q, k, v, seconds, nthreads)
    dt = oracle_sample(w, q, k, v, T_s, nthreads)
    return {"value": w.B * T_s / dt, "unit": "tokens/s", "cores": nthreads, "kind": "oracle",
            "sample": f"fp64 oracle chunked form (C={w.C}, tree prefix) on the first {T_s} tokens "
                      f"of all {w.B * w.H} heads of {w.name}; {dt:.1f} s"}


# ---------------------------------------------------------------- main arms
def run_reference(args, world, rank):
    if rank != 0:
        return
    w = inputs.HEADLINE
    q, k, v = inputs.make(w, "cpu")
    nthreads = oracle_threads(w)
    budget = 150.0
    per_step = max(1.0, budget / max(1, args.steps + args.warmup))
    T_s = sample_len(w, q, k, v, per_step, nthreads)
    for _ in range(args.warmup):
        oracle_sample(w, q, k, v, w.C, nthreads)
    times = [oracle_sample(w, q, k, v, T_s, nthreads) for _ in range(args.steps)]
    total = sum(times)
    value = args.steps * w.B * T_s / total
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "impl": "reference",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "p": w.p, "dv": w.dv, "C": w.C,
                   "scan_mode": "tree", "sample_tokens_per_head": T_s},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": nthreads, "kind": "oracle",
                         "sample": f"each step: fp64 oracle chunked form on the first {T_s} tokens of "
                                   f"all {w.B * w.H} heads of {w.name}"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, world, rank, local):
    dev = torch.device("cuda", torch.cuda.current_device())
    w0 = {x.name.split("_")[0]: x for x in inputs.WORKLOADS}[args.workload]
    w = inputs.Workload(w0.name, w0.B, w0.H, w0.T, w0.p, w0.dv, w0.C, w0.dtype, w0.kind, seed=rank)
    if args.form in ("decode", "decode_block"):
        # a serving batch of one-token steps with the workload's head shape:
        # 64 sequences x 16 heads, each head's state n x (dv+1) fp32 (above L2 at p >= 32)
        w = inputs.Workload(f"decode_B{DECODE_B}_H{DECODE_H}_p{w0.p}_dv{w0.dv}_{w0.dtype}", DECODE_B, DECODE_H, 1,
                            w0.p, w0.dv, w0.C, w0.dtype, w0.kind, seed=rank)
    mode = kb.KATA_SCAN_TREE if args.scan == "tree" else kb.KATA_SCAN_SEQUENTIAL
    lift = (LIFTS[args.lift], args.g) if args.form in BLOCK_FORMS else None
    q, k, v = inputs.make(w, dev)
    o = torch.empty_like(v)
    ws_bytes = kb.kata_chunked_workspace_bytes(q.dtype, w.B, w.H, w.T, w.p, w.dv, w.C)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    if args.form == "chunked":
        def step():
            kb.kata_forward_chunked(q, k, v, w.C, mode, o=o, workspace=ws, stream=stream)
    elif args.form == "quadratic":
        def step():
            kb.kata_forward_quadratic(q, k, v, o=o, C=w.C, stream=stream)
    elif args.form == "chunk_state_scan":
        Sp = torch.empty((w.B, w.H, w.NC, w.n, w.dv), dtype=torch.float32, device=dev)
        zp = torch.empty((w.B, w.H, w.NC, w.n), dtype=torch.float32, device=dev)

        def step():
            kb.kata_chunk_state_scan(k, v, w.C, mode, S_prefix=Sp, z_prefix=zp, stream=stream)
    elif args.form == "decode":
        qt, kt, vt = (x[:, :, 0].contiguous() for x in (q, k, v))
        S = torch.zeros((w.B, w.H, w.n, w.dv), dtype=torch.float32, device=dev)
        z = torch.zeros((w.B, w.H, w.n), dtype=torch.float32, device=dev)
        ot = torch.empty_like(vt)

        def step():
            kb.kata_decode_step(qt, kt, vt, S, z, o=ot, stream=stream)
    elif args.form == "decode_block":
        qt, kt, vt = (x[:, :, 0].contiguous() for x in (q, k, v))
        nl = lift_dim(lift[0], w.p, lift[1])
        S = torch.zeros((w.B, w.H, nl, w.dv), dtype=torch.float32, device=dev)
        z = torch.zeros((w.B, w.H, nl), dtype=torch.float32, device=dev)
        ot = torch.empty_like(vt)

        def step():
            kb.kata_decode_step_block(qt, kt, vt, S, z, lift[0], lift[1], o=ot, stream=stream)
    elif args.form in ("backward", "backward_quadratic"):
        g = torch.Generator(device=dev).manual_seed(rank)
        dO = torch.randn(v.shape, generator=g, device=dev).to(v.dtype)
        dq, dk, dvv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        bform = "chunked" if args.form == "backward" else "quadratic"
        lib = kb.load()
        need = (lib.kata_backward_chunked_workspace_bytes(w.B, w.H, w.T, w.p, w.dv) if bform == "chunked"
                else lib.kata_backward_quadratic_workspace_bytes(w.B, w.H, w.T))
        wsg = torch.empty(max(1, need), dtype=torch.uint8, device=dev)

        def step():
            kb.kata_backward(q, k, v, dO, dq, dk, dvv, workspace=wsg, stream=stream, form=bform)
    elif args.form == "quadratic_gated":
        g = torch.Generator(device=dev).manual_seed(rank)
        gate = torch.rand((w.B, w.H, w.T), generator=g, device=dev) * 0.1 + 0.9
        wsq = torch.empty(max(1, kb.load().kata_quadratic_gated_workspace_bytes(kb._dtype_code(q), w.B, w.H, w.T)),
                          dtype=torch.uint8, device=dev)

        def step():
            kb.kata_forward_quadratic_gated(q, k, v, gate, o=o, workspace=wsq, stream=stream)
    elif args.form == "gated":
        g = torch.Generator(device=dev).manual_seed(rank)
        gate = torch.rand((w.B, w.H, w.T), generator=g, device=dev) * 0.1 + 0.9
        wsg = torch.empty(max(1, kb.load().kata_chunked_gated_workspace_bytes(kb._dtype_code(q), w.B, w.H, w.T, w.p,
                                                                               w.dv, w.C)),
                          dtype=torch.uint8, device=dev)

        def step():
            kb.kata_forward_chunked_gated(q, k, v, gate, w.C, o=o, workspace=wsg, stream=stream)
    elif args.form == "chunked_block":
        wsb = torch.empty(max(1, kb.kata_chunked_block_workspace_bytes(q.dtype, lift[0], lift[1], w.B, w.H, w.T,
                                                                       w.p, w.dv, w.C)),
                          dtype=torch.uint8, device=dev)

        def step():
            kb.kata_forward_chunked_block(q, k, v, w.C, lift[0], lift[1], mode, o=o, workspace=wsb, stream=stream)
    elif args.form == "quadratic_block":
        def step():
            kb.kata_forward_quadratic_block(q, k, v, lift[0], lift[1], o=o, stream=stream)
    else:  # scan of given chunk states
        g = torch.Generator(device=dev).manual_seed(rank)
        S_loc = torch.randn((w.B, w.H, w.NC, w.n, w.dv), generator=g, device=dev)
        z_loc = torch.rand((w.B, w.H, w.NC, w.n), generator=g, device=dev)
        Sp, zp = torch.empty_like(S_loc), torch.empty_like(z_loc)

        def step():
            kb.kata_scan_states(S_loc, z_loc, mode, S_prefix=Sp, z_prefix=zp, stream=stream)

    for _ in range(args.warmup):
        step()
    kb.kata_get_device_status(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = ClockSampler(dev)
    clocks.start()
    kb.kata_trace_start(args.steps * 16 + 16)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    wall0 = time.time()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    trace = kb.kata_trace_stop()
    barrier(world)
    clocks.stop()
    kb.kata_get_device_status(stream)
    ms = e0.elapsed_time(e1) / args.steps
    ms_max = max_over_ranks(ms, world)
    tokens = w.B * w.T
    value = world * tokens / (ms_max / 1e3)

    # dominant kernel from the live trace
    peaks = load_peaks()
    per = {}
    for name, t in trace:
        per.setdefault(name, []).append(t)
    dom = max(per, key=lambda n: sum(per[n]))
    kind, amount = kernel_work(dom, w, args.form, lift)
    calls_per_step = len(per[dom]) / args.steps
    dom_ms_per_call = sum(per[dom]) / args.steps  # all launches of it in one forward
    if kind == "flop":
        achieved = amount / (dom_ms_per_call / 1e3) / 1e12
        if dom.endswith("_simt"):
            peak = SMS * FP32_LANES_PER_SM * 2 * peaks.get("sm_max_mhz", 2032.0) * 1e6 / 1e12
            bound, unit = "alu", "TFLOP/s"
        else:
            peak = peaks["bf16_tflops"]
            bound, unit = "tensor", "TFLOP/s"
    else:
        achieved = amount / (dom_ms_per_call / 1e3) / 1e9
        peak, bound, unit = peaks["hbm_gbs"], "hbm", "GB/s"
    roof = {"kernel": dom, "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak,
            "traffic": args.traffic if args.traffic is not None else MEASURED_TRAFFIC.get((args.form, w.name, dom)),
            "peak_source": peaks["source"],
            "launches_per_step": calls_per_step,
            "ms_per_step_in_kernel": dom_ms_per_call,
            "share_of_step": dom_ms_per_call / ms}
    kernels = {n: {"launches": len(t), "ms_total": sum(t), "share": sum(t) / max(1e-9, sum(x for _, x in trace))}
               for n, t in per.items()}
    alg_tflops = flops_forward(w) / (ms / 1e3) / 1e12

    if args.form != "chunked":
        if rank == 0:
            label = f"{args.form} {args.lift}{args.g}" if lift else args.form
            line = {"metric": f"KATA {label} {w.name}: tokens/s (1 B300)", "value": value, "unit": "tokens/s",
                    "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
                    "higher_is_better": True, "form": args.form, "roofline": roof, "kernels": kernels,
                    "gpu_launches": len(trace), "clocks": clocks.summary(wall0, wall1),
                    "config": {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "p": w.p, "dv": w.dv, "C": w.C,
                               "n": lift_dim(lift[0], w.p, lift[1]) if lift else w.n, "scan_mode": args.scan,
                               "lift": f"{args.lift}{args.g}" if lift else "full"}}
            print(json.dumps(line), flush=True)
        return

    # end to end through the C ABI with host buffers.  The heads stream
    # through: one copy stream brings each head's rows in, in order, and each
    # head's forward (its own call, on its own stream) starts as soon as its
    # rows have landed, its output going back on the same stream.
    qh, kh, vh = (t.cpu().pin_memory() for t in (q, k, v))
    oh = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    qd, kd, vd = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh))
    d2h = oh.numel() * oh.element_size()
    nh = w.B * w.H
    heads = lambda t: t.view(nh, 1, 1, w.T, t.shape[-1])
    qh_, kh_, vh_, oh_ = heads(qh), heads(kh), heads(vh), heads(oh)
    qd_, kd_, vd_, od_ = heads(qd), heads(kd), heads(vd), heads(o)
    copy_in = torch.cuda.Stream(device=dev)
    hstreams = [torch.cuda.Stream(device=dev) for _ in range(nh)]
    landed = [torch.cuda.Event() for _ in range(nh)]
    ws1 = kb.kata_chunked_workspace_bytes(q.dtype, 1, 1, w.T, w.p, w.dv, w.C)
    wsh = [torch.empty(max(ws1, 1), dtype=torch.uint8, device=dev) for _ in range(nh)]

    def e2e_step():
        copy_in.wait_stream(stream)
        for h in range(nh):
            with torch.cuda.stream(copy_in):
                qd_[h].copy_(qh_[h], non_blocking=True)
                kd_[h].copy_(kh_[h], non_blocking=True)
                vd_[h].copy_(vh_[h], non_blocking=True)
                landed[h].record(copy_in)
        for h in range(nh):
            sh = hstreams[h]
            sh.wait_stream(stream)
            sh.wait_event(landed[h])
            kb.kata_forward_chunked(qd_[h], kd_[h], vd_[h], w.C, mode, o=od_[h], workspace=wsh[h], stream=sh)
            with torch.cuda.stream(sh):
                oh_[h].copy_(od_[h], non_blocking=True)
        for sh in hstreams:
            stream.wait_stream(sh)

    e2e_steps = max(1, min(args.steps, 5))
    e2e_step()
    torch.cuda.synchronize()
    # which kernels one end-to-end step runs (single-head calls may cut each
    # head into segments: a segment-state prepass and a scan of their totals)
    kb.kata_trace_start(4096)
    e2e_step()
    torch.cuda.synchronize()
    e2e_names = sorted({n for n, _ in kb.kata_trace_stop()})
    barrier(world)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world)
    e2e = {"value": world * tokens / (e2e_ms / 1e3), "unit": "tokens/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
           "calls": f"one kata_forward_chunked call per head ({nh} calls)", "kernels": e2e_names,
           "segment_prepass": "states_tc" in e2e_names,
           "scan_ran": any(n.startswith("scan") for n in e2e_names)}

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if not dom.endswith("_simt") else "f32",
        "data": "synthetic: seeded N(0,1) draws, q/k put on the unit sphere",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "p": w.p, "dv": w.dv, "C": w.C,
                   "n": w.n, "scan_mode_requested": args.scan,
                   "segment_prepass": "states_tc" in per, "scan_ran": any(n.startswith("scan") for n in per),
                   "inputs": "bf16",
                   "l2": f"inputs larger than L2 ({(h2d) / 1e6:.0f} MB), no flush",
                   "parallelism": f"replicas x{world}"},
        "algorithmic_tflops": alg_tflops,
        "pct_bf16_peak": 100.0 * alg_tflops / peaks["bf16_tflops"],
        "roofline": roof,
        "kernels": kernels,
        "gpu_launches": len(trace),
        "e2e": e2e,
        "clocks": clocks.summary(wall0, wall1),
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, q, k, v)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="c4", choices=["c1", "c2", "c3", "c4", "c5"])
    ap.add_argument("--scan", default="tree", choices=["tree", "sequential"])
    ap.add_argument("--traffic", type=float, default=None,
                    help="dram bytes per call of the dominant kernel from an ncu capture")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--form", default="chunked",
                    choices=["chunked", "quadratic", "quadratic_gated", "scan", "chunk_state_scan", "decode", "backward",
                             "backward_quadratic", "gated"] + list(BLOCK_FORMS),
                    help="entry point timed (the contract's line is the chunked forward)")
    ap.add_argument("--lift", default="sigma", choices=sorted(LIFTS), help="block-lift family of the *_block forms")
    ap.add_argument("--g", type=int, default=2, help="number of blocks of the *_block forms")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
