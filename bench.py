"""Benchmark: MoE-layer forward tokens/s on one GB300 (or N independent replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-cpu-baseline]

A step is one full forward pass of the layer (router GEMM, routing, dispatch,
gate-up GEMM with SwiGLU, down GEMM, weighted combine) over
one batch of the workload's seeded synthetic tokens, through the C ABI
(moe_layer_forward), inputs resident in HBM.  Rank 0 prints one JSON line.

Multi-GPU: one process per GPU (torchrun), each runs an independent replica
of the layer on its own batch ("replicas only": the layer has no exchange
step on one node with every expert resident); value = all ranks' tokens /
the slowest rank's time.

--impl reference times the CPU oracle (single thread) on a bounded sample of
the same workload: routing and dispatch of the whole batch plus the expert FFN
of a sample of kept rows, extrapolated by the kept-row count.
"""
from __future__ import annotations

import argparse
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
sys.path.insert(0, ROOT)

from token_level_top_gb300 import moe, synth  # noqa: E402

METRIC = "MoE-layer tokens/s at Mixtral shape (top-2); % of BF16 tensor / HBM roofline"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "mixtral_prefill"
CLOCK_LEAD_S = 0.25  # untimed lead-in for clock samples when the timed region is short
CHUNK = 256  # tokens per routing chunk; a batch of one chunk routes and dispatches in one kernel


BACKWARD_KERNELS = 12  # prep, pad, four GEMMs, SwiGLU backward, router backward, dh, dW_r (two), bias sum


def kernels_per_step(T, quant=None, norm=0, hidden=0):
    """Kernels of this library one layer step launches."""
    # router GEMM, row gather, gate-up, down, combine + route and dispatch:
    # one fused kernel for a single chunk, else route + dispatch replay + finish;
    # FP8: the activation rows are quantised between the two expert GEMMs;
    # router variants: the normalisation before the router GEMM, the
    # two-layer router's second layer after it
    # (NVFP4 likewise: its token-row quantiser replaces the gather, the
    # activation rows are quantised between the GEMMs)
    return 5 + (1 if T <= CHUNK else 3) + (1 if quant else 0) + (1 if norm else 0) + (1 if hidden else 0)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=synth.CONFIG_ORDER)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other workloads measured after the main one (the 'workloads' key)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--nvfp4-weights", action="store_true",
                    help="expert GEMMs in NVFP4: e2m1 weights with e4m3 scales per 16 elements and a row "
                         "scale (moe_quantize_w13_nvfp4 / moe_quantize_nvfp4), token and activation rows "
                         "likewise on the fly")
    ap.add_argument("--fp8-weights", action="store_true",
                    help="expert GEMMs in e4m3: weights quantised per row once (moe_quantize_fp8), "
                         "token and activation rows per row on the fly")
    ap.add_argument("--backward", action="store_true",
                    help="time a training step of the layer: the forward, then moe_layer_backward "
                         "(dL/dout drawn once; every gradient written each step)")
    ap.add_argument("--graph", action="store_true",
                    help="time replays of one step captured in a CUDA graph (the same kernels, "
                         "without per-launch host overhead); the stage split comes from eager steps")
    ap.add_argument("--tau", type=float, default=1.0, help="router temperature")
    ap.add_argument("--router-norm", default="none", choices=["none", "layer", "l2"],
                    help="normalise the token rows before the router (LayerNorm or L2)")
    ap.add_argument("--router-hidden", type=int, default=0,
                    help="H > 0: the two-layer router silu(x W1^T) W2^T with H hidden units "
                         "(-1: H = 2E)")
    return ap.parse_args()


def dist_setup(n):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""

    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev_index: int):
        self.dev = dev_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50",
                                          "-i", str(self.dev)], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self, t_begin=None, t_end=None):
        """Summary of the samples taken between the wall-clock times t_begin and t_end."""
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        import datetime
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                except ValueError:
                    continue
                if t_begin is not None and not (t_begin <= ts <= t_end):
                    continue
                rows.append(parts[1:])
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "power_w_median": statistics.median(power) if power else None,
                "samples": len(rows), "window": "timed region only"}


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu capture of this kernel and
    workload, or None when there is none or the kernel source changed since."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        recs = json.load(fh)
    # a capture of the kernel on this workload ("<kernel> @ <workload>"), or its only one
    rec = recs.get(f"{kernel} @ {workload}") or recs.get(kernel)
    if not rec or rec.get("workload") != workload:
        return None
    h = hashlib.sha256()
    for f in rec["sources"]:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    if h.hexdigest()[:16] != rec["source_sha256_16"]:
        return None
    return rec["dram_bytes_per_launch"]


SUSTAINED_AFTER_S = 2.0   # a timed region at least this long is held to the sustained peak


# nominal dense tensor rates relative to bf16 (2.25 PFLOP/s): e4m3 4.5, NVFP4 13.5
QUANT_RATIO = {None: 1.0, "fp8": 2.0, "nvfp4": 6.0}
# weight bytes per element: codes, plus e4m3 block scales per 16 for NVFP4
QUANT_BYTES = {None: 2.0, "fp8": 1.0, "nvfp4": 0.5 + 1.0 / 16}
QUANT_DTYPE = {None: "bf16", "fp8": "e4m3 expert weights and activations (fp32 row scales), fp32 accumulate",
               "nvfp4": "NVFP4 expert weights and activations (e2m1, e4m3 scales per 16, fp32 row scales), "
                        "fp32 accumulate"}


def tensor_peak(peaks, peak_kind, timed_s, quant=None):
    """(TFLOP/s, description): the measured bf16 burst peak for a timed region shorter
    than SUSTAINED_AFTER_S, the sustained one (a seconds-long loop under the power cap)
    for a longer one; for e4m3 MMAs times 2, the nominal e4m3 / bf16 ratio."""
    if timed_s < SUSTAINED_AFTER_S or "bf16_tflops_sustained" not in peaks:
        v, kind = float(peaks["bf16_tflops"]), (f"{peak_kind} bf16 burst (timed region "
                                               f"{timed_s:.2f} s < {SUSTAINED_AFTER_S:.0f} s)")
    else:
        v, kind = float(peaks["bf16_tflops_sustained"]), (f"{peak_kind} bf16 sustained (timed region "
                                                          f"{timed_s:.2f} s)")
    if quant:
        r = QUANT_RATIO[quant]
        v, kind = r * v, kind + f" x {r:g}, the nominal {quant} / bf16 ratio"
    return v, kind


def layer_inputs(shape, device="cuda"):
    h, wr, bias, usage = synth.router_inputs(shape)
    w1, w3, w2 = synth.expert_weights(shape, device=device)
    L = dict(h=h.to(device), wr=wr.to(device), w1=w1, w3=w3, w2=w2,
             bias=None if bias is None else bias.to(device),
             usage=None if usage is None else usage.to(device))
    L["w13"] = moe.pack_w13(w1, w3)
    return L


def oracle_inputs(h, wr, bias, usage, w1, w3, w2):
    """The oracle's inputs (bf16 bit patterns and float arrays), converted once."""
    return dict(h=synth.bf16_bits(h), wr=synth.bf16_bits(wr),
                bias=None if bias is None else bias.cpu().numpy(),
                usage=None if usage is None else usage.cpu().numpy(),
                w1=synth.bf16_bits(w1), w3=synth.bf16_bits(w3), w2=synth.bf16_bits(w2))


def oracle_sample(shape, X, budget_s=12.0, seed=0):
    """Time the oracle: route + dispatch of the whole batch, then the expert FFN
    of sampled kept rows until ~budget_s; extrapolate the FFN by kept rows."""
    import oracle
    C = oracle.capacity(shape.T, shape.k, shape.E, shape.cf, shape.capacity)
    t0 = time.perf_counter()
    r = oracle.route(shape.k, h=X["h"], wr=X["wr"], bias=X["bias"], usage=X["usage"], lam=shape.lam)
    d = oracle.dispatch(r["scores"], shape.k, C)
    t_rd = time.perf_counter() - t0
    kept = int(d["offsets"][-1])
    rng = np.random.default_rng(seed)
    order = rng.permutation(kept)
    rows, t_ffn = 0, 0.0
    while rows < kept and (rows == 0 or (t_rd + t_ffn) < budget_s):
        i = int(order[rows])
        t1 = time.perf_counter()
        oracle.expert_slots(X["h"], X["w1"], X["w3"], X["w2"], d["assign"], d["perm"], i, i + 1)
        t_ffn += time.perf_counter() - t1
        rows += 1
    t_total = t_rd + (t_ffn / max(rows, 1)) * kept
    return dict(t_route_dispatch=t_rd, ffn_rows=rows, kept=kept, t_ffn_sample=t_ffn,
                t_total=t_total, tokens_per_s=shape.T / t_total)


REF_BUDGET_S = 90.0    # wall-clock bound of the reference (oracle) arm's timed steps
STEP_MIN_S = 0.5


def reference_plan(steps: int, warmup: int):
    """(seconds per step, steps to time) for the reference arm: the budget split
    over warm-up and timed steps, at least STEP_MIN_S each, and fewer timed steps
    than asked (at least one) when that is needed to stay within REF_BUDGET_S."""
    per_step = max(STEP_MIN_S, REF_BUDGET_S / max(steps + warmup, 1))
    if (warmup + steps) * per_step > REF_BUDGET_S:
        steps = max(1, int(REF_BUDGET_S / per_step) - warmup)
    return per_step, steps


def host_cpu():
    """The host the oracle is timed on: architecture, CPU model (as /proc/cpuinfo
    or lscpu names it) and the number of cores the OS reports."""
    import platform
    model = None
    try:
        with open("/proc/cpuinfo") as fh:
            for ln in fh:
                key = ln.split(":")[0].strip().lower()
                if key in ("model name", "cpu model", "hardware"):
                    model = ln.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    if model is None:
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=5).stdout
            for ln in out.splitlines():
                if ln.lower().startswith("model name"):
                    model = ln.split(":", 1)[1].strip()
                    break
        except (OSError, subprocess.SubprocessError):
            pass
    return {"machine": platform.machine(), "model": model, "nproc": os.cpu_count()}


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle   # this arm never loads the CUDA library
    shape = synth.CONFIGS[args.workload]
    h, wr, bias, usage = synth.router_inputs(shape)
    w1, w3, w2 = synth.expert_weights(shape, device="cpu")
    # Each step times route + dispatch of the whole batch (about 0.1 s on the
    # prefill shape) and at least one expert row (about 0.3 s), so a step takes
    # at least STEP_MIN_S; the whole run is held to about REF_BUDGET_S by giving
    # each step budget / (W + K) and, when even STEP_MIN_S per step is too long,
    # timing fewer steps than asked (the line gives both counts).
    per_step, steps = reference_plan(args.steps, args.warmup)
    X = oracle_inputs(h, wr, bias, usage, w1, w3, w2)
    vals = []
    for i in range(args.warmup + steps):
        res = oracle_sample(shape, X, budget_s=per_step, seed=i)
        if i >= args.warmup:
            vals.append(res)
    v = statistics.median(r["tokens_per_s"] for r in vals)
    sample = (f"per step: route+dispatch of all {shape.T} tokens, expert FFN of "
              f"{vals[-1]['ffn_rows']} of {vals[-1]['kept']} kept rows, extrapolated by kept rows")
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world,
            "steps": steps, "steps_requested": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * shape.T / v, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(shape, capacity_fn=oracle.capacity),
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": sample, "host": host_cpu()},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_config(shape, router=None, graph=False, capacity_fn=None):
    extra = {"router": router} if router else {}
    if graph:
        extra["launch"] = "CUDA graph replay of one step"
    cap = (capacity_fn or moe.capacity)(shape.T, shape.k, shape.E, shape.cf, shape.capacity)
    return {**extra, "workload": shape.name, "T": shape.T, "d_model": shape.d, "E": shape.E, "k": shape.k,
            "d_ff": shape.F, "cf": shape.cf, "lambda": shape.lam,
            "capacity": cap,
            "parallelism": "replicas", "l2": "inputs larger than L2: every step streams "
            f"{3 * shape.E * shape.F * shape.d * 2 / 1e9:.2f} GB of expert weights"}


def run_ours(args, rank, world, local):
    assert torch.cuda.is_available(), "the CUDA path needs a GPU (there is no CPU fallback)"
    from token_level_top_gb300 import build
    if world == 1 or rank == 0:
        build.build()
    barrier(world)
    moe.lib()
    shape = synth.CONFIGS[args.workload]
    L = layer_inputs(shape)
    want_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    # the oracle reads the unpacked W1/W3 from host memory; the device keeps only W13
    host_w = (L["w1"].cpu(), L["w3"].cpu(), L["w2"].cpu()) if want_cpu else None
    del L["w1"], L["w3"]
    torch.cuda.empty_cache()
    if args.fp8_weights and args.nvfp4_weights:
        raise SystemExit("--fp8-weights and --nvfp4-weights exclude each other")
    quant = "fp8" if args.fp8_weights else ("nvfp4" if args.nvfp4_weights else None)
    quantized = quant is not None
    if quant == "fp8":   # e4m3 expert weights, one fp32 scale per weight row
        L["w13"] = moe.quantize_fp8(L["w13"])
        L["w2"] = moe.quantize_fp8(L["w2"])
    elif quant == "nvfp4":
        L["w13"] = moe.quantize_w13_nvfp4(L["w13"])
        L["w2"] = moe.quantize_nvfp4(L["w2"])
    if quant:
        want_cpu = False
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    norm = {"none": moe.NORM_NONE, "layer": moe.NORM_LAYER, "l2": moe.NORM_L2}[args.router_norm]
    hidden = 2 * shape.E if args.router_hidden < 0 else args.router_hidden
    variant = norm != moe.NORM_NONE or hidden > 0 or args.tau != 1.0
    router_desc = None
    wr, bias = L["wr"], L["bias"]
    if variant:   # the router variants: their own seeded weights, the bias in the Router
        # no bias and no LayerNorm shift: the experts' loads stay as even as
        # with the workload's own router, so that the dispatch does the same work
        rw = synth.router_variant_weights(shape.d, shape.E, hidden, norm == moe.NORM_LAYER,
                                          seed=shape.seed + 11, bias=False, beta=False)
        if not hidden and not norm:
            rw["w"], rw["bias"] = L["wr"].cpu(), (None if L["bias"] is None else L["bias"].cpu())
        wr = moe.Router(**{n: (None if v is None else v.cuda()) for n, v in rw.items()})
        bias = None
        router_desc = {"tau": args.tau, "norm": args.router_norm, "hidden": hidden}
    bwd = args.backward
    if bwd and (quantized or norm or hidden):
        raise SystemExit("--backward runs with bf16 experts and the linear router")
    flags = {None: 0, "fp8": moe.FLAG_FP8, "nvfp4": moe.FLAG_NVFP4}[quant] | (moe.FLAG_BACKWARD if bwd else 0)
    cfg = moe.Config.of(shape, flags=flags, tau=args.tau, router_norm=norm,
                        norm_eps=1e-5 if norm == moe.NORM_LAYER else 1e-12, router_hidden=hidden)
    ws = moe.workspace(cfg)
    dout = None
    if bwd:   # dL/dout ~ N(0, 1), bf16, drawn once
        dout = torch.randn(shape.T, shape.d, generator=torch.Generator().manual_seed(shape.seed + 3))
        dout = dout.to(torch.bfloat16).cuda()
    out = torch.empty(shape.T, shape.d, dtype=torch.bfloat16, device="cuda")
    # kept rows of this batch (routing is deterministic, identical every step)
    _, aux = moe.layer_forward(cfg, ws, L["h"], wr, L["w13"], L["w2"], bias, L["usage"],
                               aux=True, out=out)
    counts = aux["counts"].cpu()
    kept = int(counts.sum().item())
    active = int((counts > 0).sum().item())
    st = moe.device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st} ({moe.STATUS.get(st)})")

    def step(evs=None, bev=None):
        moe.layer_forward(cfg, ws, L["h"], wr, L["w13"], L["w2"], bias, L["usage"],
                          stage_events=evs, out=out)
        if bwd:
            moe.layer_backward(cfg, ws, L["h"], L["wr"], L["w13"], L["w2"], dout)
            if bev is not None:
                bev.record()

    graph = None
    if args.graph:   # one step captured once (after an eager warm-up on the capture stream)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            step()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
    run = graph.replay if graph is not None else step

    w0 = torch.cuda.Event(enable_timing=True)
    w1 = torch.cuda.Event(enable_timing=True)
    w0.record()
    for _ in range(args.warmup):
        run()
    w1.record()
    torch.cuda.synchronize()
    step_ms = w0.elapsed_time(w1) / max(args.warmup, 1)
    stage_evs = [[torch.cuda.Event(enable_timing=True) for _ in range(moe.NUM_STAGES + 1)]
                 for _ in range(min(args.steps, 50))]
    bwd_evs = [torch.cuda.Event(enable_timing=True) if bwd else None for _ in range(min(args.steps, 50))]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    # A timed region shorter than a few sampling intervals may hold no clock
    # sample: identical untimed steps run for CLOCK_LEAD_S just before it, and
    # the samples are taken over both.
    lead = 0
    if args.steps * step_ms < 1e3 * CLOCK_LEAD_S:
        lead = int(1e3 * CLOCK_LEAD_S / max(step_ms, 1e-3)) + 1
    wall0 = time.time()
    for _ in range(lead):
        run()
    # the timed steps carry no stage events (their host-side recording would slow the
    # launch-bound batches); the stage split comes from instrumented steps afterwards
    t0.record()
    for i in range(args.steps):
        run()
    t1.record()
    torch.cuda.synchronize()
    wall1 = time.time()
    barrier(world)
    time.sleep(0.2)   # let the sampler flush its last lines
    clk = clocks.stop(wall0, wall1)
    if clk is not None and lead:
        clk["window"] = (f"timed region and the {lead} identical untimed steps "
                         f"(~{CLOCK_LEAD_S:.2f} s) run just before it")
    ms = t0.elapsed_time(t1)
    ms_max = max_over_ranks(ms, world)
    st = moe.device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st} ({moe.STATUS.get(st)}) after the timed region")
    n_stage = min(args.steps, 50)   # the stage split: eager steps with events, after the timed region
    for i in range(n_stage):
        step(stage_evs[i], bwd_evs[i])
    torch.cuda.synchronize()
    stage_ms = {n: statistics.mean(stage_evs[i][j].elapsed_time(stage_evs[i][j + 1])
                                   for i in range(n_stage))
                for j, n in enumerate(moe.STAGE_NAMES)}
    if bwd:
        stage_ms["backward"] = statistics.mean(stage_evs[i][-1].elapsed_time(bwd_evs[i])
                                               for i in range(n_stage))

    # end to end from pinned host memory: every step copies its input in and its result back
    h_host = L["h"].cpu().pin_memory()
    o_host = torch.empty(shape.T, shape.d, dtype=torch.bfloat16).pin_memory()
    h_dev = torch.empty_like(L["h"])

    dh_host = torch.empty(shape.T, shape.d, dtype=torch.float32).pin_memory() if bwd else None
    # Every mode keeps two batches in flight the same way; the plain layer goes through the
    # library's host-buffer call, the others through the binding with explicit copies.
    wss = [ws, moe.workspace(cfg)]
    o_hosts = [o_host, torch.empty_like(o_host).pin_memory()]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    h_devs = [h_dev, torch.empty_like(h_dev)]
    outs = [out, torch.empty_like(out)]
    dh_hosts = [dh_host, torch.empty_like(dh_host).pin_memory()] if bwd else None

    def e2e_one(i):
        j = i % 2
        if not (bwd or quantized or variant):
            moe.layer_forward_host_async(cfg, wss[j], h_host, L["wr"], L["w13"], L["w2"], o_hosts[j], L["bias"],
                                         L["usage"])
            return
        h_devs[j].copy_(h_host, non_blocking=True)
        moe.layer_forward(cfg, wss[j], h_devs[j], wr, L["w13"], L["w2"], bias, L["usage"], out=outs[j])
        if bwd:   # dL/dh back to the host
            g = moe.layer_backward(cfg, wss[j], h_devs[j], L["wr"], L["w13"], L["w2"], dout)
            dh_hosts[j].copy_(g["dh"], non_blocking=True)
        else:
            o_hosts[j].copy_(outs[j], non_blocking=True)

    def e2e_run(n):
        torch.cuda.current_stream().synchronize()
        for i in range(n):
            with torch.cuda.stream(streams[i % 2]):
                e2e_one(i)
        for st_ in streams:
            st_.synchronize()

    e2e_run(2)
    barrier(world)
    te0 = time.perf_counter()
    e2e_run(args.e2e_steps)
    te = max_over_ranks(time.perf_counter() - te0, world)

    peaks, peak_kind = load_peaks()
    d, F, T = shape.d, shape.F, shape.T
    roof, expert_tflops, weight_gbs = expert_roofline(shape, kept, active, stage_ms, peaks, peak_kind,
                                                      ms_max * 1e-3, quant)
    peak_tf = tensor_peak(peaks, peak_kind, ms_max * 1e-3, quant)[0]
    bwd_line = None
    if bwd:
        # the backward's GEMM work on the kept rows: W2^T dout (2 d F), dx (2 2F d), dW2
        # (2 d F), dW13 (2 2F d) per row (g and u are kept by the forward); each expert's
        # rows are rounded up to the 128-row tile, which the GEMMs also compute
        bflops = 12.0 * kept * d * F
        sec_b = stage_ms["backward"] * 1e-3
        rows_pad = int(sum((int(c) + 127) // 128 * 128 for c in counts.tolist()))
        bwd_line = {"stage_ms": stage_ms["backward"], "algorithmic_tflop": bflops / 1e12,
                    "achieved_tflops": bflops / sec_b / 1e12, "peak": peak_tf,
                    "frac": bflops / sec_b / 1e12 / peak_tf, "padded_rows": rows_pad, "kept_rows": kept,
                    "gemms": "this library's tcgen05 grouped GEMM (bf16 in, fp32 accumulate)",
                    "kernels": "this library's: prep, pad, SwiGLU backward, router backward, dh, dW_r, bias sum"}
    value = world * T * args.steps / (ms_max * 1e-3)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": QUANT_DTYPE[quant],
        "data": "synthetic",
        "config": workload_config(shape, router_desc, graph is not None),
        "roofline": roof,
        "expert_gemm_tflops": expert_tflops,
        "weight_stream_gbs": weight_gbs,
        "stages_ms": stage_ms, "kept_rows": kept,
        "clocks": clk,
        "e2e": ({"value": world * T * args.e2e_steps / te, "unit": UNIT,
                 "h2d_bytes_per_step": T * d * 2, "d2h_bytes_per_step": T * d * (4 if bwd else 2),
                 "overlap": ("two workspaces on two streams" +
                             (" (moe_layer_forward_host_async)" if not (bwd or quantized or variant) else ""))}
                if args.e2e_steps > 0 else None),
        "gpu_launches": (kernels_per_step(shape.T, quant, norm, hidden) + (BACKWARD_KERNELS if bwd else 0))
        * args.steps,
    }
    if bwd:
        line["metric"] = METRIC + " (training step: forward + backward)"
        line["backward"] = bwd_line
    if want_cpu:
        X = oracle_inputs(L["h"].cpu(), L["wr"].cpu(), None if L["bias"] is None else L["bias"].cpu(),
                          None if L["usage"] is None else L["usage"].cpu(), *host_w)
        res = oracle_sample(shape, X)
        line["cpu_baseline"] = {
            "value": res["tokens_per_s"], "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": (f"route+dispatch of all {T} tokens ({res['t_route_dispatch']:.2f} s), "
                       f"expert FFN of {res['ffn_rows']} of {res['kept']} kept rows "
                       f"({res['t_ffn_sample']:.1f} s), extrapolated by kept rows"),
            "host": host_cpu()}
    plain = not (quantized or bwd or variant or graph is not None)
    if plain and not args.no_workloads:
        del L, ws, wss, h_devs, outs
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        line["workloads"] = {}
        for name, wq in SIDE_WORKLOADS:
            if name == shape.name and not wq:
                continue
            line["workloads"][name + (f"_{wq}" if wq else "")] = side_workload(name, wq, peaks, peak_kind)
            torch.cuda.empty_cache()
    if rank == 0:
        print(json.dumps(line), flush=True)


def expert_roofline(shape, kept, active, stage_ms, peaks, peak_kind, timed_s, quant):
    """Roofline of the dominant expert GEMM (gate-up or down) of one layer step: its
    algorithmic work per launch -- kept rows only, every active expert's weights read
    once -- over its mean CUDA-event duration; plus the two expert GEMMs' TFLOP/s and
    weight-streaming GB/s together."""
    d, F = shape.d, shape.F
    flops = {"gate_up": 2.0 * kept * d * 2 * F, "down": 2.0 * kept * F * d}
    wb = QUANT_BYTES[quant]   # bytes per weight element (+ 4 per weight row for the row scales)
    rs = 4 if quant else 0
    # (quantised: the GEMMs read activation rows of the same width; the act
    # quantisation pass between them is timed in the down stage)
    bytes_ = {"gate_up": active * 2.0 * F * (d * wb + rs) + kept * d * wb + kept * F * 2,
              "down": active * 1.0 * d * (F * wb + rs) + kept * F * wb + kept * d * 2}
    dom = max(("gate_up", "down"), key=lambda n: stage_ms[n])
    peak_tf, tf_kind = tensor_peak(peaks, peak_kind, timed_s, quant)
    peak_bw = float(peaks["hbm_gbs"])
    intensity = (flops["gate_up"] + flops["down"]) / (bytes_["gate_up"] + bytes_["down"])
    sec = stage_ms[dom] * 1e-3
    if intensity * 1e9 >= peak_tf * 1e12 / peak_bw:     # above the ridge: tensor bound
        roof = {"bound": "tensor", "achieved": flops[dom] / sec / 1e12, "peak": peak_tf,
                "unit": "TFLOP/s", "peak_kind": tf_kind}
    else:
        roof = {"bound": "hbm", "achieved": bytes_[dom] / sec / 1e9, "peak": peak_bw,
                "unit": "GB/s", "peak_kind": f"{peak_kind} HBM copy bandwidth"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    kname = ("moe_gemm_nvfp4_kernel" if quant == "nvfp4" else "moe_gemm_kernel") + \
        f" ({dom.replace('_', '-')}{', e4m3' if quant == 'fp8' else ''})"
    roof["traffic"] = recorded_traffic(kname, shape.name)
    roof["kernel"] = kname
    roof["algorithmic_per_launch"] = {"flop": flops[dom], "bytes": bytes_[dom]}
    gemm_s = (stage_ms["gate_up"] + stage_ms["down"]) * 1e-3
    expert_tflops = (flops["gate_up"] + flops["down"]) / gemm_s / 1e12
    weight_gbs = 3.0 * active * F * d * wb / gemm_s / 1e9
    return roof, expert_tflops, weight_gbs


# The other workloads, measured after the main one in the same run (eager steps
# over a ~0.2 s timed region, and CUDA-graph replays for the launch-bound batches
# of one routing chunk), each with its dominant expert GEMM's roofline.
SIDE_WORKLOADS = [("mixtral_decode", None), ("mixtral_decode", "fp8"), ("mixtral_decode", "nvfp4"),
                  ("fine_grained", None), ("skewed", None), ("tiny", None), ("mixtral_prefill", None),
                  ("mixtral_prefill", "fp8"), ("mixtral_prefill", "nvfp4")]
SIDE_TIMED_S = 0.2


def side_workload(name, quant, peaks, peak_kind):
    shape = synth.CONFIGS[name]
    L = layer_inputs(shape)
    del L["w1"], L["w3"]
    if quant == "fp8":
        L["w13"] = moe.quantize_fp8(L["w13"])
        L["w2"] = moe.quantize_fp8(L["w2"])
    elif quant == "nvfp4":
        L["w13"] = moe.quantize_w13_nvfp4(L["w13"])
        L["w2"] = moe.quantize_nvfp4(L["w2"])
    cfg = moe.Config.of(shape, flags={None: 0, "fp8": moe.FLAG_FP8, "nvfp4": moe.FLAG_NVFP4}[quant])
    ws = moe.workspace(cfg)
    out = torch.empty(shape.T, shape.d, dtype=torch.bfloat16, device="cuda")
    _, aux = moe.layer_forward(cfg, ws, L["h"], L["wr"], L["w13"], L["w2"], L["bias"], L["usage"],
                               aux=True, out=out)
    counts = aux["counts"].cpu()
    kept, active = int(counts.sum().item()), int((counts > 0).sum().item())

    def step(evs=None):
        moe.layer_forward(cfg, ws, L["h"], L["wr"], L["w13"], L["w2"], L["bias"], L["usage"],
                          stage_events=evs, out=out)

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(5):
        step()
    e1.record()
    torch.cuda.synchronize()
    steps = int(min(400, max(20, 1e3 * SIDE_TIMED_S / max(e0.elapsed_time(e1) / 5, 1e-3))))
    e0.record()
    for i in range(steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    st = moe.device_status(ws)
    if st != 0:
        raise RuntimeError(f"{name}: device status {st} ({moe.STATUS.get(st)})")
    n_stage = min(steps, 50)   # the stage split from instrumented steps after the timed ones
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(moe.NUM_STAGES + 1)] for _ in range(n_stage)]
    for i in range(n_stage):
        step(evs[i])
    torch.cuda.synchronize()
    stage_ms = {n: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(n_stage))
                for j, n in enumerate(moe.STAGE_NAMES)}
    roof, tflops, wgbs = expert_roofline(shape, kept, active, stage_ms, peaks, peak_kind, ms * 1e-3, quant)
    res = {"tokens_per_s": shape.T * steps / (ms * 1e-3), "ms_per_step": ms / steps, "steps": steps,
           "dtype": QUANT_DTYPE[quant],
           "kept_rows": kept, "stages_ms": stage_ms, "roofline": roof, "expert_gemm_tflops": tflops,
           "weight_stream_gbs": wgbs, "weight_stream_frac_of_hbm": wgbs / float(peaks["hbm_gbs"]),
           "gpu_launches": kernels_per_step(shape.T, quant) * steps,
           "config": {k: v for k, v in workload_config(shape).items() if k != "l2"}}
    if shape.T <= CHUNK:   # launch-bound: the same step replayed from a CUDA graph
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            step()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        for _ in range(3):
            g.replay()
        e0.record()
        for _ in range(steps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        res["ms_per_step_graph"] = e0.elapsed_time(e1) / steps
        res["tokens_per_s_graph"] = shape.T * steps / (e0.elapsed_time(e1) * 1e-3)
        res["gpu_launches"] += kernels_per_step(shape.T, quant) * (steps + 3)
        del g
    del L, ws, out
    return res


def main():
    args = parse()
    rank, world, local = dist_setup(args.gpus)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_ours(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
