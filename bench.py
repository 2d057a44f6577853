"""Benchmark of the routed-MoE layer on GB300.

Default workload: the decode / verify slice E=384, H=7168, I=576, top-6, MXFP4 weights with
MXFP8 activations, swiglu limit 7; one step = one layer call at each decode batch size
M in {1,2,3,4,5,6,7,8,10,12,14,16} (last 25 % of rows are CUDA-graph padding, id -1).
Metric: tokens/s (valid rows per second of layer time).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--det]

Timing: every layer call is a CUDA graph replay whose kernels run between two event-record
nodes of the same graph; before them (outside the events) a 512 MB buffer is written and
another 512 MB read, which flushes L2 and leaves it clean; the routing set rotates over 8
pre-generated sets per M.  The step time is the sum of its calls' event times.  The dominant kernel is timed by event-record nodes inside the same graphs.
Under torchrun each rank runs the same workload on its own GPU (replicas; weak scaling);
rank 0 prints one JSON line with the max time over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from synth import moe_inputs as S  # noqa: E402

DECODE_CFG = "decode_w4a8"
N_ROUTING_SETS = 8
FLUSH_BYTES = 512 << 20
EXPERT_BYTES_W13 = {"decode_w4a8": 2 * 576 * 7168 // 2 + 2 * 576 * 7168 // 32}   # codes + E8M0
EXPERT_BYTES_W2 = {"decode_w4a8": 7168 * 576 // 2 + 7168 * 576 // 32}
# the dominant kernel of the decode ladder (every call has M <= 16: 16-token tiles)
FC1_KERNEL = "fc1_stream_kernel<16>"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--det", action="store_true", help="deterministic combine")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-prefill", action="store_true", help="skip the prefill ladder report")
    p.add_argument("--no-modes", action="store_true",
                   help="skip the report of the other weight / activation formats")
    p.add_argument("--profile", type=int, default=0, metavar="M",
                   help="profiling case: eager layer calls at decode size M (no timing)")
    p.add_argument("--profile-calls", type=int, default=4)
    p.add_argument("--profile-cfg", default="",
                   help="profiling case of another synthetic config (e.g. w4a16_nvfp4)")
    p.add_argument("--cpu-baseline-worker", action="store_true", help=argparse.SUPPRESS)
    p.add_argument("--sample-m", type=str, default="1,2", help=argparse.SUPPRESS)
    return p.parse_args()


class L2Flush:
    """Before each timed call: write a 512 MB buffer (larger than the 129 MB L2, so nothing the
    call reads is left in L2), then read a second 512 MB buffer, so that the lines L2 holds when
    the call starts are clean: otherwise the call's own reads would first have to write back
    the ~100 MB of dirty lines the flush left (measured: 3-9 us per decode call), a cost of the
    flush, not of the layer."""

    def __init__(self, torch):
        self.w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
        self.r = torch.ones(FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    def __call__(self, v=1):
        self.w.fill_(v & 0xFF)
        return self.r.amax()


def valid_rows(ids):
    return int(((ids >= 0)).any(axis=1).sum())


def distinct_experts(ids, E):
    v = ids[(ids >= 0) & (ids < E)]
    return int(np.unique(v).size)


# ---------------------------------------------------------------------------------- oracle arm

def oracle_sample(cfg, ck, m_list, sets):
    """Time the fp64 oracle on one call per M in m_list; returns (tokens, seconds)."""
    from oracle import moe as O
    tok, sec = 0, 0.0
    for i, M in enumerate(m_list):
        x, ids, w = S.make_inputs(cfg, M, seed=cfg.seed_base + 100 * M + sets[i % len(sets)])
        t0 = time.perf_counter()
        O.moe_forward(ck, x, ids, w, cfg.swiglu_limit)
        sec += time.perf_counter() - t0
        tok += valid_rows(ids)
    return tok, sec


def cpu_baseline_worker(args):
    cfg = S.CONFIGS[DECODE_CFG]
    ck = S.make_checkpoint(cfg)
    m_list = [int(v) for v in args.sample_m.split(",")]
    tok, sec = oracle_sample(cfg, ck, m_list, [0])
    print(json.dumps({"tokens": tok, "seconds": sec}))


def run_cpu_baseline(m_list="1,2,3,4,5,6,7,8,10,12,14,16"):
    # the oracle as it stands: numpy fp64 with its default BLAS threading (all host cores)
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-baseline-worker",
                        "--sample-m", m_list], capture_output=True, text=True, timeout=900)
    if r.returncode != 0:
        return None
    d = json.loads(r.stdout.strip().splitlines()[-1])
    cores = os.cpu_count() or 1
    return {"value": d["tokens"] / d["seconds"], "unit": "tokens/s", "cores": cores,
            "kind": "oracle",
            "sample": f"one layer call at each M in {{{m_list}}} of the decode workload "
                      f"({d['tokens']} valid tokens, {d['seconds']:.1f} s; numpy fp64, default "
                      f"BLAS threading over the {cores} host cores)"}


def reference_arm(args, rank, world):
    """The oracle timed as the reference implementation (rank 0 only)."""
    if rank != 0:
        return
    cfg = S.CONFIGS[DECODE_CFG]
    ck = S.make_checkpoint(cfg)
    tok_total, sec_total = 0, 0.0
    for s in range(args.warmup + args.steps):
        tok, sec = oracle_sample(cfg, ck, [1], [s % N_ROUTING_SETS])
        if s >= args.warmup:
            tok_total += tok
            sec_total += sec
    value = tok_total / sec_total
    line = {
        "impl": "reference", "metric": "decode MoE layer tokens/s", "value": value,
        "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sec_total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "decode_w4a8 sample: one call at M=1 per step (E=384, H=7168, "
                               "I=576, top-6, MXFP4/MXFP8)"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": os.cpu_count() or 1,
                         "kind": "oracle",
                         "sample": "one M=1 decode call per step, rotating routing sets (numpy "
                                   "fp64, default BLAS threading over the host cores)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


# ---------------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples every 50 ms from before the warm-up to after the timed region; the
    summary keeps the samples whose timestamps fall inside the marked timed region."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def start(self):
        self.t0 = time.time()

    def stop(self):
        self.t1 = time.time()

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        import datetime
        rows = [r.split(",") for r in (self.out or "").strip().splitlines() if r.strip()]
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                ts = datetime.datetime.strptime(r[0].strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
                mx = float(r[2])
                if self.t0 is not None and not (self.t0 <= ts <= self.t1):
                    continue
                sm.append(float(r[1]))
                for n, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(n)
            except (ValueError, IndexError):
                continue
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm),
                "window_s": None if self.t0 is None else round(self.t1 - self.t0, 3)}


# ---------------------------------------------------------------------------------- our arm

def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def kernel_source_hash(ent, root=ROOT, read=None):
    """sha256 over the source text that defines a kernel: each listed file whole, or, for a file
    that also holds other kernels, only its `spans` ([start marker, end marker) pairs, "" = the
    file's start), which cover the kernel, everything before it in the file and its host launch
    code.  None when a marker is missing."""
    import hashlib
    if read is None:
        def read(src):
            with open(os.path.join(root, src), "rb") as f:
                return f.read()
    h = hashlib.sha256()
    for src in ent["sources"]:
        text = read(src)
        spans = ent.get("spans", {}).get(src)
        if not spans:
            h.update(text)
            continue
        for a, b in spans:
            i = text.find(a.encode()) if a else 0
            j = text.find(b.encode(), max(i, 0))
            if i < 0 or j < 0:
                return None
            h.update(text[i:j])
    return h.hexdigest()


def kernel_traffic(kernel):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, or None when the kernel
    source changed since the counters were taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.txt")) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    ent = d.get(kernel)
    if not ent:
        return None
    try:
        if kernel_source_hash(ent) != ent["sha256"]:
            return None
    except OSError:
        return None
    return ent


def reduce_over_ranks(step_ms: float, tokens: int, world: int, device=None):
    """Whole-job numbers of a replicated run: the slowest rank's time and the tokens of all
    ranks (each rank processes its own batches; there is no data-path collective)."""
    if world <= 1:
        return step_ms, tokens
    import torch
    import torch.distributed as dist
    t = torch.tensor([step_ms], dtype=torch.float64, device=device)
    n = torch.tensor([tokens], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t.item()), int(n.item())


def profile_case(args):
    """A case for ncu: the decode / prefill layer (E=384, H=7168, I=576, top-6) called eagerly
    `--profile-calls` times at M = `--profile`, each call on its own routing set (the decode
    recipe up to M = 16, the uniform prefill recipe beyond)."""
    import torch

    from serving_route_count_gb300 import MoELayer, build
    build.build()
    cfg = S.CONFIGS[args.profile_cfg or DECODE_CFG]
    ck = S.make_checkpoint(cfg)
    M = args.profile
    icfg = cfg if (M <= 16 or args.profile_cfg) else S.CONFIGS[PREFILL_CFG]
    layer = MoELayer(ck, cfg.topk, M, cfg.swiglu_limit, args.det)
    del ck
    for c in range(args.profile_calls):
        x, ids, w = S.make_inputs(icfg, M, seed=icfg.seed_base + 100 * M + c)
        xt = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).cuda()
        layer(xt, torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    st, code = layer.device_error()
    print(json.dumps({"profile_case": M, "calls": args.profile_calls, "device_error": code}))


PREFILL_CFG = "prefill_w4a8"
PREFILL_M = (128, 512, 2048, 4096)
EXPERT_BYTES = 2 * 576 * 7168 // 2 + 2 * 576 * 7168 // 32 + 7168 * 576 // 2 + 7168 * 576 // 32


def prefill_report(stream, flush, hbm_peak):
    """Secondary report: whole-call times of the prefill ladder (E=384, H=7168, I=576, top-6,
    uniform routing, atomic combine), each call a CUDA graph replayed after an L2 flush, with the
    fraction of the HBM roofline (touched expert bytes) and of the dense FP8 tensor peak."""
    import torch
    from serving_route_count_gb300 import MoELayer
    cfg = S.CONFIGS[PREFILL_CFG]
    ck = S.make_checkpoint(cfg)
    layer = MoELayer(ck, cfg.topk, max(PREFILL_M), cfg.swiglu_limit, 0)
    del ck
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except (OSError, ValueError):
        pass
    # dense FP8 (kind::mxf8f6f4) peak: the measured bf16 GEMM rate x the nominal FP8/bf16 ratio 2
    fp8_peak = 2.0 * float(peaks.get("bf16_tflops", 1900.0))
    out = {}
    for M in PREFILL_M:
        x, ids, w = S.make_inputs(cfg, M)
        xt = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).cuda()
        it = torch.from_numpy(ids).cuda()
        wt = torch.from_numpy(w).cuda()
        ot = torch.empty((M, cfg.H), dtype=torch.bfloat16, device="cuda")
        torch.cuda.synchronize()          # inputs copied before the side stream reads them
        with torch.cuda.stream(stream):
            layer(xt, it, wt, ot)
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                layer(xt, it, wt, ot)
        ts = []
        for c in range(7):
            with torch.cuda.stream(stream):
                flush(c)
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                g.replay()
                b.record(stream)
            stream.synchronize()
            if c >= 2:
                ts.append(a.elapsed_time(b) * 1e-3)
        sec = float(np.median(ts))
        distinct = distinct_experts(ids, cfg.E)
        slots = int(((ids >= 0) & (ids < cfg.E)).sum())
        flops = 2.0 * slots * (2 * cfg.I * cfg.H + cfg.H * cfg.I)
        out[str(M)] = {"us": round(sec * 1e6, 1), "tokens_per_s": round(M / sec),
                       "hbm_frac": round(distinct * EXPERT_BYTES / sec / 1e9 / hbm_peak, 3),
                       "tflops": round(flops / sec / 1e12, 1),
                       "fp8_dense_frac": round(flops / sec / 1e12 / fp8_peak, 3)}
    layer.close()
    return {"workload": "prefill_w4a8: E=384 H=7168 I=576 top-6, MXFP4 x MXFP8, uniform "
                        "routing, atomic combine; one graph replay per M after an L2 flush",
            "fp8_dense_peak_tflops": fp8_peak, "calls": out}


# The other weight formats (E=256, H=6144, I=512, top-8): per-expert bytes of the checkpoint
# format each call must stream (fc1 2I x H plus fc2 H x I elements).
MODE_CFGS = ("w4a16_nvfp4", "w4a8_nvfp4", "w4a4_nvfp4", "hybrid_nvfp4_nf3", "hybrid_mxfp4_nf3")
MODE_M = (1, 64, 2048)


def _mode_expert_bytes(kind, I, H):
    n = 3 * I * H                                # elements of one expert's two matrices
    if kind == "nf3":
        return n * 3 // 8 + n // 32              # 3-bit codes, E4M3 per 32
    if kind == "mxfp4":
        return n // 2 + n // 32                  # E2M1, E8M0 per 32
    return n // 2 + n // 16                      # NVFP4: E2M1, E4M3 per 16 (+ globals)


def modes_report(stream, flush, hbm_peak):
    """Secondary report: whole-call times of the other weight / activation formats at decode,
    mid and prefill sizes (one graph replay per M after an L2 flush), with the fraction of the
    HBM roofline over the touched experts' bytes, the dense tensor rate (2 x 3 x I x H flops per
    routed slot) and, for W4A4 (`kind::mxf4nvf4`), its fraction of the dense FP4 peak."""
    import torch
    from serving_route_count_gb300 import MoELayer
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except (OSError, ValueError):
        pass
    # dense FP4 peak: the measured bf16 GEMM rate x the nominal FP4 / bf16 ratio 13.5 / 2.25 = 6
    fp4_peak = 6.0 * float(peaks.get("bf16_tflops", 1900.0))
    out = {}
    for name in MODE_CFGS:
        cfg = S.CONFIGS[name]
        ck = S.make_checkpoint(cfg)
        layer = MoELayer(ck, cfg.topk, max(MODE_M), cfg.swiglu_limit, 0)
        res = {}
        for M in MODE_M:
            x, ids, w = S.make_inputs(cfg, M)
            xt = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).cuda()
            it = torch.from_numpy(ids).cuda()
            wt = torch.from_numpy(w).cuda()
            ot = torch.empty((M, cfg.H), dtype=torch.bfloat16, device="cuda")
            torch.cuda.synchronize()      # inputs copied before the side stream reads them
            with torch.cuda.stream(stream):
                layer(xt, it, wt, ot)
                stream.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    layer(xt, it, wt, ot)
            ts = []
            for c in range(6):
                with torch.cuda.stream(stream):
                    flush(c)
                    a = torch.cuda.Event(enable_timing=True)
                    b = torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    g.replay()
                    b.record(stream)
                stream.synchronize()
                if c >= 2:
                    ts.append(a.elapsed_time(b) * 1e-3)
            sec = float(np.median(ts))
            touched = np.unique(ids[(ids >= 0) & (ids < cfg.E)])
            if ck.quant == "hybrid":
                kept = "mxfp4" if ck.nv.quant == "mxfp4" else "nvfp4"
                nbytes = sum(_mode_expert_bytes(kept if ck.tier[e] == S.TIER_NVFP4 else "nf3",
                                                cfg.I, cfg.H) for e in touched)
            else:
                nbytes = len(touched) * _mode_expert_bytes("nvfp4", cfg.I, cfg.H)
            slots = int(((ids >= 0) & (ids < cfg.E)).sum())
            tflops = 2.0 * 3 * cfg.I * cfg.H * slots / sec / 1e12
            res[str(M)] = {"us": round(sec * 1e6, 1), "tokens_per_s": round(M / sec),
                           "hbm_frac": round(nbytes / sec / 1e9 / hbm_peak, 3),
                           "tflops": round(tflops, 1)}
            if name == "w4a4_nvfp4":
                res[str(M)]["fp4_dense_frac"] = round(tflops / fp4_peak, 4)
        layer.close()
        del ck
        out[name] = res
    return {"workload": "E=256 H=6144 I=512 top-8 (Zipf 0.8 routing for the hybrids), atomic "
                        "combine; one graph replay per M after an L2 flush; hbm_frac over the "
                        "touched experts' checkpoint-format bytes",
            "fp4_dense_peak_tflops": round(fp4_peak, 1),
            "fp4_peak_basis": "measured bf16 dense rate x nominal FP4/bf16 ratio 6 (13.5 / 2.25)",
            "calls": out}


def our_arm(args, rank, world):
    import torch
    import torch.distributed as dist

    from serving_route_count_gb300 import MoELayer, build, moe_plan_set_profile_events
    from serving_route_count_gb300 import moe_call_launches, moe_profile_stage_names

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    build.build()
    cfg = S.CONFIGS[DECODE_CFG]
    ck = S.make_checkpoint(cfg)
    m_list = list(cfg.m_list)
    max_m = max(m_list)
    layer = MoELayer(ck, cfg.topk, max_m, cfg.swiglu_limit, args.det)
    stages = moe_profile_stage_names(layer.plan)
    dom = "fc1"
    dom_i = stages.index(dom)

    # inputs: per M, N_ROUTING_SETS routing sets (+ x), device resident; one graph per (M, set)
    stream = torch.cuda.Stream()
    try:   # event-record nodes inside graphs (torch.cuda.Event(external=True))
        torch.cuda.Event(enable_timing=True, external=True)
        in_graph_events = True
    except TypeError:
        in_graph_events = False
    flush_graph = L2Flush(torch) if in_graph_events else None
    calls = []   # (M, set, graph, x, ids, w, out, prof_events, tokens, distinct)
    for M in m_list:
        for s in range(N_ROUTING_SETS):
            x, ids, w = S.make_inputs(cfg, M, seed=cfg.seed_base + 100 * M + s + 1000 * rank)
            xt = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).cuda()
            it = torch.from_numpy(ids).cuda()
            wt = torch.from_numpy(w).cuda()
            ot = torch.empty((M, cfg.H), dtype=torch.bfloat16, device="cuda")
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)]
            for ev in evs:   # torch creates the CUDA event on first record
                ev.record()
            calls.append(dict(M=M, set=s, x=xt, ids=it, w=wt, out=ot, ev=evs,
                              tokens=valid_rows(ids), distinct=distinct_experts(ids, cfg.E),
                              ids_np=ids, x_np=x, w_np=w))
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for c in calls:   # eager warm-up of each shape
            layer(c["x"], c["ids"], c["w"], c["out"])
        stream.synchronize()
        # two graphs per call: the timed one - the L2 flush, then the layer call between two
        # event-record nodes, so the events time the call's kernels on the device and not the
        # host's graph launch - and one with an event record between stages (which breaks the
        # launch chain) for the per-kernel durations
        for c in calls:
            g = torch.cuda.CUDAGraph()
            if in_graph_events:
                c["ea"] = torch.cuda.Event(enable_timing=True, external=True)
                c["eb"] = torch.cuda.Event(enable_timing=True, external=True)
            with torch.cuda.graph(g, stream=stream):
                if in_graph_events:
                    flush_graph()
                    c["ea"].record(stream)
                layer(c["x"], c["ids"], c["w"], c["out"])
                if in_graph_events:
                    c["eb"].record(stream)
            c["graph"] = g
            moe_plan_set_profile_events(layer.plan, c["ev"])
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                layer(c["x"], c["ids"], c["w"], c["out"])
            c["graph_ev"] = g
            moe_plan_set_profile_events(layer.plan, [])
    torch.cuda.synchronize()
    flush = L2Flush(torch)

    def step(si, stage_events=False):
        """One ladder pass; with stage_events the instrumented graphs run and the fc1 stage
        durations are returned instead of whole-call times."""
        tot_ms, dom_ms, dom_bytes, toks = 0.0, 0.0, 0.0, 0
        pairs, per_call = [], []
        with torch.cuda.stream(stream):
            for mi, M in enumerate(m_list):
                c = calls[mi * N_ROUTING_SETS + (si % N_ROUTING_SETS)]
                if in_graph_events and not stage_events:
                    c["graph"].replay()          # flush + events inside the graph
                    pairs.append((c["ea"], c["eb"], c))
                    continue
                flush(si)
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                (c["graph_ev"] if stage_events else c["graph"]).replay()
                b.record(stream)
                pairs.append((a, b, c))
        stream.synchronize()
        for a, b, c in pairs:
            tot_ms += a.elapsed_time(b)
            per_call.append((c["M"], a.elapsed_time(b)))
            if stage_events:
                dom_ms += c["ev"][dom_i].elapsed_time(c["ev"][dom_i + 1])
                dom_bytes += c["distinct"] * EXPERT_BYTES_W13[DECODE_CFG] + c["M"] * cfg.H
            toks += c["tokens"]
        return tot_ms, dom_ms, dom_bytes, toks, per_call

    tot_ms = dom_ms = dom_bytes = 0.0
    toks = 0
    with ClockSampler(local) as clk:
        for si in range(args.warmup):
            step(si)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        clk.start()
        per_m = {}
        for si in range(args.steps):
            a, _, _, d, pc = step(args.warmup + si)
            tot_ms += a
            toks += d
            for M, ms in pc:
                per_m.setdefault(M, []).append(ms)
        torch.cuda.synchronize()
        clk.stop()
        # fc1 durations: the same calls again through the stage-instrumented graphs
        for si in range(max(3, args.steps // 4)):
            _, b, c, _, _ = step(args.warmup + si, stage_events=True)
            dom_ms += b
            dom_bytes += c
    tot_ms, all_toks = reduce_over_ranks(tot_ms, toks, world, device="cuda")
    if world > 1:
        dist.barrier()
    clocks = clk.summary()

    # end to end: host (pinned) buffers through moe_run_host, copies inside the timed region
    e2e_ms, e2e_tok, h2d, d2h = 0.0, 0, 0, 0
    host = []
    for mi, M in enumerate(m_list):
        c = calls[mi * N_ROUTING_SETS]
        # one pinned buffer [x | ids | weights]: moe_run_host moves it up in one copy
        xb, kb = M * cfg.H * 2, M * cfg.topk * 4
        packed = torch.empty(xb + 2 * kb, dtype=torch.uint8).pin_memory()
        packed[:xb].copy_(torch.from_numpy(c["x_np"].view(np.uint8).reshape(-1)))
        packed[xb:xb + kb].copy_(torch.from_numpy(c["ids_np"].view(np.uint8).reshape(-1)))
        packed[xb + kb:].copy_(torch.from_numpy(c["w_np"].view(np.uint8).reshape(-1)))
        xh = packed[:xb].view(torch.bfloat16).view(M, cfg.H)
        ih = packed[xb:xb + kb].view(torch.int32).view(M, cfg.topk)
        wh = packed[xb + kb:].view(torch.float32).view(M, cfg.topk)
        oh = torch.empty((M, cfg.H), dtype=torch.bfloat16).pin_memory()
        host.append((xh, ih, wh, oh, c["tokens"]))
    for xh, ih, wh, oh, _ in host:   # warm-up
        layer.run_host(xh, ih, wh, oh, stream=stream)
    e2e_steps = max(3, args.steps // 2)
    for _ in range(e2e_steps):
        for xh, ih, wh, oh, tk in host:
            flush()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            layer.run_host(xh, ih, wh, oh, stream=stream)
            e2e_ms += 1e3 * (time.perf_counter() - t0)
            e2e_tok += tk
    h2d = sum(xh.numel() * 2 + ih.numel() * 4 + wh.numel() * 4 for xh, ih, wh, _, _ in host)
    d2h = sum(oh.numel() * 2 for *_, oh, _ in host)

    if rank != 0:
        return
    peak, peak_kind = measured_peaks()
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    traffic = kernel_traffic(FC1_KERNEL)
    launches_per_step = sum(moe_call_launches(layer.plan, M) for M in m_list)
    cpu = None if args.no_cpu_baseline else run_cpu_baseline()
    line = {
        "metric": "decode MoE layer tokens/s",
        "value": all_toks / (tot_ms * 1e-3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": tot_ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "mxfp4 x mxfp8 (fp32 accumulate)",
        "data": "synthetic",
        "config": {
            "workload": "decode_w4a8: E=384 H=7168 I=576 top-6, MXFP4 weights / MXFP8 "
                        "activations, M ladder 1..16 (one call each per step), last 25% rows "
                        "padding, swiglu limit 7",
            "combine": "deterministic" if args.det else "atomic",
            "tokens_per_step": toks // args.steps,
            "timing": ("CUDA graph per call: L2 flush (a 512 MB write, then a 512 MB read so "
                       "the L2 lines are clean), then the layer's kernels between two "
                       "event-record nodes (device time of the call, without the host's graph "
                       "launch); 8 routing sets rotated per M"
                       if in_graph_events else
                       "CUDA graph per call, CUDA events around each replay; L2 flushed (512 MB "
                       "write, then 512 MB read) before each call, outside the events; 8 "
                       "routing sets rotated per M"),
            "parallelism": f"replicas x{world}",
        },
        "roofline": {
            "kernel": dom,
            "bound": "hbm",
            "achieved": achieved,
            "peak": peak,
            "peak_kind": peak_kind,
            "unit": "GB/s",
            "frac": achieved / peak,
            "traffic": None if traffic is None else traffic["bytes_per_launch"],
            "traffic_kernel": FC1_KERNEL,
            "traffic_workload": None if traffic is None else traffic["workload"],
            "traffic_algorithmic_bytes": None if traffic is None
            else traffic["algorithmic_bytes_per_launch"],
            "algorithmic_bytes": "distinct touched experts x (w13 codes + E8M0 scales = "
                                 f"{EXPERT_BYTES_W13[DECODE_CFG]} B) + x rows",
            "kernel_ms_per_ladder_pass": dom_ms / max(3, args.steps // 4),
            "kernel_timing": "CUDA events around fc1 inside graphs of the same calls (separate "
                             "replays: an event between kernels breaks the launch chain)",
        },
        "stages": stages,
        # mean device time of one call at each M of the ladder, over the timed steps
        "calls_us": {str(M): round(statistics.mean(v) * 1e3, 1) for M, v in sorted(per_m.items())},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_tok / (e2e_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "api": "moe_run_host (one pinned host buffer [x | ids | weights], one H2D copy "
                       "+ run, finalize storing into the pinned output + sync)"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "prefill": None if args.no_prefill else prefill_report(stream, flush, peak),
        "modes": None if args.no_modes else modes_report(stream, flush, peak),
    }
    print(json.dumps(line))


def main():
    args = parse()
    if args.cpu_baseline_worker:
        cpu_baseline_worker(args)
        return
    if args.profile:
        profile_case(args)
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        import torch.distributed as dist
        if args.impl == "reference":
            if rank != 0:
                return
        else:
            dist.init_process_group("nccl")
    if args.impl == "reference":
        reference_arm(args, rank, world)
        return
    our_arm(args, rank, world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
