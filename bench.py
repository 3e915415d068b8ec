"""Benchmark: MoE route -> dispatch -> expert -> combine tokens/s on GB300.

One step = one pass of the whole path (route, dispatch, SwiGLU expert FFN,
combine) over one batch of N = W*T synthetic tokens.  Default workload:
Mixtral-like (W=8 slots, T=2048, H=4096, E=8, k=2, I=14336).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--fused]
    python bench.py --impl reference ...   # the CPU oracle on a bounded sample

Prints one JSON line.  With N > 1 (torchrun, one rank per GPU) every rank runs
an independent replica of the workload (the path has no inter-GPU exchange on
one box) and the value is the tokens of all ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE dispatch+expert+combine tokens/s on 1 GB300; % HBM / bf16 tensor roofline"
UNIT = "tokens/s"


def parse(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--config", default="mixtral")
    p.add_argument("--fused", action="store_true", help="single-launch pipeline")
    p.add_argument("--with-router", action="store_true",
                   help="start each step from the token activations: the router GEMM produces the logits")
    p.add_argument("--dedup", action="store_true",
                   help="rank-deduplicated dispatch (staged pipeline only)")
    p.add_argument("--fp8", action="store_true",
                   help="FP8 dispatch with per-token scales (staged pipeline only)")
    p.add_argument("--weights-in-ffn", action="store_true",
                   help="routing weights applied in the expert epilogue, unweighted combine")
    p.add_argument("--unfused", action="store_true",
                   help="stage-by-stage launches even for a workload defined as fused")
    p.add_argument("--tokens-per-slot", type=int, default=0,
                   help="override T (smaller cases for profiler captures)")
    p.add_argument("--world", type=int, default=0, help="override W")
    p.add_argument("--experts", type=int, default=0, help="override E")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-per-workload", action="store_true",
                   help="skip the record of the other workloads (the default run adds it to the headline line)")
    p.add_argument("--workload", default="moe", choices=["moe", "linear_a2a"],
                   help="linear_a2a: the GEMM + all-to-all workload on the same heap, fused vs split")
    return p.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, world: int, device) -> float:
    """The slowest rank's time (every rank gets it)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


L2_BYTES = 129 * 2**20


def l2_statement(cfg: dict) -> str:
    """Whether one step's inputs alone exceed the 129 MB L2 (no flush needed)."""
    wbytes = 3 * cfg["num_experts"] * cfg["hidden"] * cfg["inter"] * 2
    n = cfg["world"] * cfg["tokens_per_slot"]
    xbytes = n * cfg["hidden"] * 2 + n * cfg["num_experts"] * 4
    if wbytes + xbytes > L2_BYTES:
        return f"inputs larger than L2 (expert weights {wbytes / 2**20:.0f} MB, L2 129 MB); not flushed"
    return (f"working set {(wbytes + xbytes) / 2**20:.1f} MB fits in L2 and is not flushed: "
            "a small-case timing, not a roofline measurement")


def workload_config(name: str, cfg: dict, fused: bool, weights_in_ffn: bool = False,
                    with_router: bool = False) -> dict:
    import moe_synth as ms
    n = cfg["world"] * cfg["tokens_per_slot"]
    return {"workload": ms.CONFIG_TITLES.get(name, name), "preset": name,
            "world_slots": cfg["world"], "tokens_per_slot": cfg["tokens_per_slot"],
            "tokens_per_step": n, "hidden": cfg["hidden"], "inter": cfg["inter"],
            "experts": cfg["num_experts"], "topk": cfg["topk"], "fused": bool(fused),
            "weights_in_ffn": bool(weights_in_ffn), "with_router": bool(with_router),
            "l2": l2_statement(cfg),
            "parallelism": "replicas"}


def algorithmic(cfg: dict, experts_hit: int) -> dict:
    """Work the method must do per step (what a perfect kernel moves or computes)."""
    n = cfg["world"] * cfg["tokens_per_slot"]
    k, H, I, E = cfg["topk"], cfg["hidden"], cfg["inter"], cfg["num_experts"]
    P = n * k
    return {
        "route_bytes": n * E * 4 + n * k * 8,
        "dispatch_bytes": n * H * 2 * (1 + k),
        "ffn_flops": 6 * P * H * I,
        # weights of every expert that received a row, the dispatched rows, h
        # written and read once, y written once
        "ffn_bytes": experts_hit * 3 * H * I * 2 + P * H * 2 + 2 * P * I * 2 + P * H * 2,
        "combine_bytes": P * H * 2 + n * H * 2,
    }


class ClockSampler:
    """nvidia-smi clock / throttle samples every 20 ms.  The sampler starts
    before the warm-up (so the timed steps follow the warm-up with no idle
    gap); mark() brackets the timed region on the host clock and the summary
    keeps only the samples taken inside it."""
    Q = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.window = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def mark(self, t0: float, t1: float):
        self.window = (t0, t1)

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    @staticmethod
    def _when(stamp: str):
        import datetime
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(stamp.strip(), fmt).timestamp()
            except ValueError:
                pass
        return None

    def summary(self):
        if not getattr(self, "lines", None):
            return None
        sm, mx, power, reasons, outside = [], None, [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            if self.window is not None:
                t = self._when(f[0])
                if t is not None and not (self.window[0] <= t <= self.window[1]):
                    outside += 1
                    continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
                power.append(float(f[3]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_min_mhz": sm[0], "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None,
                "interval_ms": 20}


TRAFFIC_SOURCES = ("expert_ffn.cu", "gemm2sm.cuh", "symmoe_dev.cuh")


def code_of(src: str) -> str:
    """C/C++/CUDA source without its comments, each line's whitespace runs
    collapsed and blank lines dropped: what the compiler sees, so an edit to
    a comment leaves it unchanged and an edit to the code does not."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        elif c in "\"'":  # a string or character literal, copied whole
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        else:
            out.append(c)
            i += 1
    lines = (" ".join(line.split()) for line in "".join(out).splitlines())
    return "\n".join(line for line in lines if line)


def sources_code_sha256(files=TRAFFIC_SOURCES) -> str:
    """sha256 over the code (comments stripped) of the kernel sources a
    traffic record was captured from."""
    hsh = hashlib.sha256()
    for f in files:
        src = open(os.path.join(ROOT, "combine_symmetric_heap_gb300", "csrc", f), encoding="utf-8").read()
        hsh.update(code_of(src).encode())
    return hsh.hexdigest()


def traffic_record(workload: str, cfg: dict):
    """Per-step DRAM bytes of the expert FFN launches from the committed ncu
    summary, or None if it was captured for another workload or shape, or the
    code of any of its sources changed since."""
    import moe_synth as ms
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        rec = json.load(open(path))
        if rec.get("sources_code_sha256") != sources_code_sha256():
            return None
        if rec.get("workload") != workload or cfg != ms.CONFIGS.get(workload):
            return None
        return rec.get("traffic_bytes_per_step")
    except Exception:
        return None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return p["hbm_gbs"], p["bf16_tflops"], p["bf16_tflops_sustained"], "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# ---------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)
# ---------------------------------------------------------------------------

def oracle_sample_run(cfg: dict, tokens, weights: dict, weights_in_ffn: bool = False):
    """Time the oracle, as it stands, over a sample of tokens: routing of the
    sample, placement of its pairs, the SwiGLU FFN of every received row, and
    the combine.  ``weights[e]`` are the experts' bf16 bits (inputs, not timed
    as oracle work).  Returns seconds."""
    import numpy as np
    import moe_synth as ms
    import oracle
    lg = ms.logits_np(cfg, rows=tokens)
    xs = ms.x_np(cfg, rows=tokens)
    t0 = time.perf_counter()
    sample = dict(cfg, tokens_per_slot=len(tokens), world=1, num_experts=cfg["num_experts"])
    res = oracle.pipeline(lg, xs, dict(world=1, num_experts=cfg["num_experts"], topk=cfg["topk"]),
                          lambda e: weights[e], weights_in_ffn=weights_in_ffn)
    dt = time.perf_counter() - t0
    assert res["out"].shape == (len(tokens), cfg["hidden"])
    del sample
    return dt


def sample_weights(cfg: dict, tokens, device, skip=()):
    """Fresh host copies of the experts the sample tokens route to (input
    generation, outside any timed region)."""
    import numpy as np
    import moe_synth as ms
    import oracle
    idx, _ = oracle.route_topk(ms.logits_np(cfg, rows=tokens), cfg["topk"])
    out = {}
    for e in sorted(set(idx.reshape(-1).tolist()) - set(skip)):
        if device is not None:
            out[e] = tuple(ms.weight_expert_torch(cfg, nm, e, device).view(__import__("torch").int16)
                           .cpu().numpy().view(np.uint16) for nm in ("gate", "up", "down"))
        else:
            out[e] = tuple(ms.weight_np(cfg, nm, e) for nm in ("gate", "up", "down"))
    return out


def cores_used():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def get_cfg(args) -> dict:
    import moe_synth as ms
    cfg = dict(ms.CONFIGS[args.config])
    if args.tokens_per_slot:
        cfg["tokens_per_slot"] = args.tokens_per_slot
    if args.world:
        cfg["world"] = args.world
    if args.experts:
        cfg["num_experts"] = args.experts
    return cfg


def run_reference(args):
    rank, world, local = dist_env()
    if rank != 0:
        return 0
    import numpy as np
    import torch
    cfg = get_cfg(args)
    dev = torch.device("cuda", local) if torch.cuda.is_available() else None
    per_step = int(os.environ.get("SYMMOE_REF_TOKENS", "8"))
    n = cfg["world"] * cfg["tokens_per_slot"]
    rng = np.random.default_rng(0)
    times = []
    wts = {}
    for s in range(args.warmup + args.steps):
        tokens = np.sort(rng.choice(n, size=per_step, replace=False))
        wts.update(sample_weights(cfg, tokens, dev, skip=set(wts)))
        dt = oracle_sample_run(cfg, tokens, wts, bool(getattr(args, "weights_in_ffn", False)))
        if s >= args.warmup:
            times.append(dt)
    tot = sum(times)
    value = per_step * len(times) / tot
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(args.config, cfg, args.fused, getattr(args, "weights_in_ffn", False)),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores_used(), "threads": blas_threads(),
                         "kind": "oracle",
                         "sample": f"{per_step} random tokens of the workload per step (their "
                                   f"routing, placement, expert FFN rows and combine); expert "
                                   f"weights generated outside the timed region; fp64 numpy, "
                                   f"BLAS on {blas_threads()} threads"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

class Workload:
    """Device tensors of one configuration: the heap, the step's inputs and
    outputs, and the expert weights (which may be shared with another
    configuration of the same E, H, I: the weights depend on nothing else)."""

    def __init__(self, sm, cfg: dict, dev, with_router: bool = False, weights=None):
        import torch
        import moe_synth as ms
        self.cfg = cfg
        n, k, H = cfg["world"] * cfg["tokens_per_slot"], cfg["topk"], cfg["hidden"]
        self.n = n
        self.heap = sm.SymHeap(cfg, dev)
        self.logits = ms.logits_torch(cfg, dev)
        self.x = ms.x_torch(cfg, dev)
        self.weights = weights if weights is not None else ms.weights_torch(cfg, dev)
        self.wr = ms.router_weight_torch(cfg, dev) if with_router else None
        self.idx = torch.empty((n, k), dtype=torch.int32, device=dev)
        self.w = torch.empty((n, k), dtype=torch.float32, device=dev)
        self.out = torch.empty((n, H), dtype=torch.bfloat16, device=dev)


def weight_key(cfg: dict):
    return (cfg["num_experts"], cfg["hidden"], cfg["inter"])


def time_steps(wl: Workload, stream, steps: int, warmup: int, fused: int, wif=False, dedup=False,
               fp8=False, with_router=False, world=1, local=0, barrier=lambda: None, device=None):
    """W untimed warm-up steps, then K timed steps between CUDA events on the
    launching stream, with an event between stages (the staged step makes the
    four C-ABI calls moe_pipeline makes; the fused step is one launch).
    Returns the slowest rank's total ms, per-stage ms averages and the clocks
    sampled during the timed steps."""
    import torch
    heap = wl.heap
    wg, wu, wd = wl.weights
    stage_names = (["router"] if with_router else []) + (
        ["fused"] if fused else ["route", "dispatch", "expert_ffn", "combine"])
    nst = len(stage_names)
    stage_evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)] for _ in range(steps)]

    def step(i=None):
        ev = stage_evs[i] if i is not None else None
        calls = [lambda: heap.router_logits(wl.x, wl.wr, wl.logits, stream=stream)] if with_router else []
        if fused:
            calls.append(lambda: heap.pipeline(wl.logits, wl.x, wg, wu, wd, wl.idx, wl.w, wl.out, fused=1,
                                               weights_in_ffn=wif, stream=stream))
        else:
            calls += [lambda: heap.route_topk(wl.logits, wl.idx, wl.w, stream=stream),
                      lambda: heap.dispatch(wl.x, wl.idx, wl.w, dedup=dedup, fp8=fp8, stream=stream),
                      lambda: heap.expert_ffn(wg, wu, wd, weighted_rows=wif, stream=stream),
                      lambda: heap.combine(wl.idx, wl.w, wl.out, unweighted=wif, stream=stream)]
        for j, call in enumerate(calls):
            if ev:
                ev[j].record(stream)
            call()
        if ev:
            ev[nst].record(stream)

    with ClockSampler(local) as clk:
        for _ in range(max(warmup, 3)):
            step()
        torch.cuda.synchronize()
        assert heap.status(stream=stream) == 0, "device status word set during warm-up"
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        t0 = time.time()
        ev0.record(stream)
        for i in range(steps):
            step(i)
        ev1.record(stream)
        torch.cuda.synchronize()
        clk.mark(t0, time.time())
    barrier()
    ms_total = max_over_ranks(ev0.elapsed_time(ev1), world, device)
    assert heap.status(stream=stream) == 0, "device status word set during the timed steps"
    acc = [0.0] * nst
    for ev in stage_evs:
        for j in range(nst):
            acc[j] += ev[j].elapsed_time(ev[j + 1])
    return ms_total, dict(zip(stage_names, [a / steps for a in acc])), clk.summary()


def expert_counts(heap, cfg: dict):
    """Rows each expert received in the last dispatch (device -> host, outside
    any timed region)."""
    import numpy as np
    return np.concatenate([heap.cnt(d).cpu().numpy() for d in range(cfg["world"])]).astype(np.int64)


def per_expert_roof_s(cfg: dict, counts, tf_peak: float, hbm: float) -> float:
    """Sum over experts of max(flops_e / tensor peak, bytes_e / HBM): each
    expert's own binding roof, as if the experts ran one after another on the
    whole GPU.  Under a skewed routing the heavy experts are tensor-bound and
    the light ones weight-stream-bound; this roof does not let one regime's
    slack hide the other's time (the plain roof, max of the sums, is the
    tighter bound and stays the headline fraction)."""
    H, I = cfg["hidden"], cfg["inter"]
    t = 0.0
    for c in counts:
        c = int(c)
        if c == 0:
            continue
        flops = 6.0 * c * H * I
        bts = 3.0 * H * I * 2 + c * H * 2 * 2 + 2.0 * c * I * 2
        t += max(flops / (tf_peak * 1e12), bts / (hbm * 1e9))
    return t


def roofline_of(cfg: dict, counts, stages: dict, fused: int, ms_total: float, traffic=None) -> dict:
    """The dominant kernel's roofline entry: the expert FFN (staged) or the
    whole fused launch, against whichever measured peak binds its
    algorithmic work."""
    experts_hit = int((counts > 0).sum())
    alg = algorithmic(cfg, experts_hit)
    hbm, tf_burst, tf_sus, peak_src = peaks()
    long_region = ms_total > 1000.0
    tf_peak = tf_sus if long_region else tf_burst
    t_tensor = alg["ffn_flops"] / (tf_peak * 1e12)
    t_hbm = alg["ffn_bytes"] / (hbm * 1e9)
    bound = "tensor" if t_tensor >= t_hbm else "hbm"
    if fused:
        kern_s = stages["fused"] / 1e3
        kname = "moe_fused_kernel (whole step in one launch)"
        extra_bytes = alg["route_bytes"] + alg["dispatch_bytes"] + alg["combine_bytes"]
    else:
        kern_s = stages["expert_ffn"] / 1e3
        kname = "expert_gemm_kernel (gate/up SwiGLU + down launches)"
        extra_bytes = 0
    if bound == "tensor":
        achieved, peak, unit = alg["ffn_flops"] / kern_s / 1e12, tf_peak, "TFLOP/s"
        other = {"hbm_gbs": (alg["ffn_bytes"] + extra_bytes) / kern_s / 1e9, "hbm_peak": hbm}
        other["frac"] = other["hbm_gbs"] / hbm
    else:
        achieved, peak, unit = (alg["ffn_bytes"] + extra_bytes) / kern_s / 1e9, hbm, "GB/s"
        other = {"tflops": alg["ffn_flops"] / kern_s / 1e12, "tensor_peak": tf_peak}
        other["frac"] = other["tflops"] / tf_peak
    ideal_s = per_expert_roof_s(cfg, counts, tf_peak, hbm)
    return {"bound": bound, "kernel": kname, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "traffic": traffic,
            "peak_kind": f"{peak_src} " + ("bf16 " + ("sustained" if long_region else "burst")
                                           if bound == "tensor" else "HBM copy"),
            "algorithmic_per_step": {"flops": alg["ffn_flops"], "bytes": alg["ffn_bytes"] + extra_bytes,
                                     "experts_hit": experts_hit},
            "other_roof": other,
            "per_expert_roof": {"ideal_ms": 1e3 * ideal_s,
                                "frac": (ideal_s + (extra_bytes / (hbm * 1e9))) / kern_s}}


def stage_bandwidth(cfg: dict, stages: dict, fused: int) -> dict:
    n = cfg["world"] * cfg["tokens_per_slot"]
    alg = algorithmic(cfg, 0)
    hbm = peaks()[0]
    bw = {"hbm_peak_gbs": hbm}
    if not fused:
        bw["dispatch_gbs"] = alg["dispatch_bytes"] / (stages["dispatch"] / 1e3) / 1e9
        bw["combine_gbs"] = alg["combine_bytes"] / (stages["combine"] / 1e3) / 1e9
        bw["route_gbs"] = alg["route_bytes"] / (stages["route"] / 1e3) / 1e9
        bw["dispatch_frac"] = bw["dispatch_gbs"] / hbm
        bw["combine_frac"] = bw["combine_gbs"] / hbm
        bw["route_frac"] = bw["route_gbs"] / hbm
    del n
    return bw


def workload_summary(name: str, cfg: dict, fused: int, steps: int, ms_total: float, stages: dict,
                     clocks, counts, start: str = "from idle") -> dict:
    """One entry of the per-workload record."""
    n = cfg["world"] * cfg["tokens_per_slot"]
    rl = roofline_of(cfg, counts, stages, fused, ms_total)
    return {"workload": name, "fused": bool(fused), "steps": steps, "start": start,
            "tokens_per_s": n * steps / (ms_total / 1e3), "ms_per_step": ms_total / steps,
            "stages_ms": stages, "ffn_roof": {k: rl[k] for k in ("bound", "achieved", "peak", "unit", "frac",
                                                                 "peak_kind", "per_expert_roof", "other_roof")},
            "stage_bandwidth": stage_bandwidth(cfg, stages, fused), "clocks": clocks,
            "experts_hit": int((counts > 0).sum()), "max_expert_rows": int(counts.max())}


def run_ours(args):
    import torch
    import torch.distributed as dist
    import moe_synth as ms
    import combine_symmetric_heap_gb300 as sm

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = get_cfg(args)
    fused = 1 if (args.fused or (cfg.get("fused") and not args.unfused)) else 0
    wif = bool(getattr(args, "weights_in_ffn", False))
    dedup = bool(getattr(args, "dedup", False))
    fp8 = bool(getattr(args, "fp8", False))
    assert not ((dedup or fp8) and fused), "the deduplicated and FP8 dispatches run in the staged pipeline"
    assert not (dedup and fp8), "one dispatch variant at a time"
    with_router = bool(getattr(args, "with_router", False))
    n, k, H = cfg["world"] * cfg["tokens_per_slot"], cfg["topk"], cfg["hidden"]

    wl = Workload(sm, cfg, dev, with_router)
    heap = wl.heap
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            dist.barrier()

    # ---- timed region: K whole-path steps, device resident inputs
    ms_total, stages, clocks = time_steps(wl, stream, args.steps, args.warmup, fused, wif, dedup, fp8,
                                          with_router, world, local, barrier, dev)
    ms_step = ms_total / args.steps
    value = n * args.steps * world / (ms_total / 1e3)
    # the router is one GEMM launch, plus one reduction launch when it splits K
    router_launches = (1 + (heap.router_splits() > 1)) if with_router else 0
    launches_per_step = (1 if fused else 7) + router_launches

    counts = expert_counts(heap, cfg)
    roofline = roofline_of(cfg, counts, stages, fused, ms_total,
                           None if fused else traffic_record(args.config, cfg))
    stage_bw = stage_bandwidth(cfg, stages, fused)
    hbm, tf_burst, tf_sus, _ = peaks()
    if "router" in stages:
        # router GEMM: reads x [N,H] and Wr [E,H] (bf16), writes logits [N,E] (fp32)
        rbytes = n * H * 2 + cfg["num_experts"] * H * 2 + n * cfg["num_experts"] * 4
        rflops = 2.0 * n * H * cfg["num_experts"]
        rs = stages["router"] / 1e3
        tf_peak = tf_sus if ms_total > 1000.0 else tf_burst
        stage_bw["router_gbs"] = rbytes / rs / 1e9
        stage_bw["router_tflops"] = rflops / rs / 1e12
        stage_bw["router_frac"] = max(stage_bw["router_gbs"] / hbm, stage_bw["router_tflops"] / tf_peak)
        stage_bw["router_splits"] = heap.router_splits()

    if fp8:
        # a crossing row carries H code bytes and one 4-byte scale instead of 2H bytes
        stage_bw["fp8"] = {"cross_slot_bytes": n * k * (H + 4), "plain_cross_slot_bytes": n * k * H * 2}
    if dedup:
        # rows that cross to another slot: one per (token, distinct slot) instead of one per pair
        import numpy as np
        slots = np.sort(wl.idx.cpu().numpy() // (cfg["num_experts"] // cfg["world"]), axis=1)
        rows = int(n + (np.diff(slots, axis=1) != 0).sum())
        stage_bw["dedup"] = {"rows_crossing": rows, "pairs": n * k, "cross_slot_bytes": rows * H * 2,
                             "plain_cross_slot_bytes": n * k * H * 2}

    # ---- end to end through the public API with host buffers
    # Every step copies its inputs (logits, x) from pinned host memory and reads
    # its output back, as a serving loop does: the copies run on their own
    # streams, double-buffered, so step i+1's upload and step i-1's download
    # overlap step i's compute (the heap is reused, so the compute steps stay
    # in order on one stream).  Timed from the first upload to the last
    # download, over the same number of steps as the device-resident loop.
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e_loop(wl, stream, args.steps, fused, wif, dedup, fp8, with_router, world, barrier, dev)

    # ---- oracle on the host cores (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(cfg, dev, wif)

    # ---- every other workload (rank 0 prints; every rank runs them)
    per_workload = None
    if not args.no_per_workload and args.config == "mixtral" and not (with_router or dedup or fp8 or wif) \
            and not (args.tokens_per_slot or args.world or args.experts):
        per_workload = run_per_workload(sm, wl, args, stream, world, local, barrier, dev, fused, stages,
                                        ms_total, clocks, counts)
    del wl, heap
    torch.cuda.empty_cache()

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": dict(workload_config(args.config, cfg, fused, wif, with_router), dedup=dedup, fp8=fp8),
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
            "stages_ms": stages or None,
            "stage_bandwidth": stage_bw,
        }
        if per_workload is not None:
            line["per_workload"] = per_workload
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_e2e_loop(wl: Workload, stream, steps: int, fused: int, wif: bool, dedup: bool, fp8: bool,
                 with_router: bool, world: int, barrier, dev) -> dict:
    import torch
    heap = wl.heap
    wg, wu, wd = wl.weights
    logits, x, out = wl.logits, wl.x, wl.out
    lg_h = torch.empty(logits.shape, dtype=logits.dtype, pin_memory=True)
    x_h = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
    out_h = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
    lg_h.copy_(logits)
    x_h.copy_(x)
    lg_d = [torch.empty_like(logits) for _ in range(2)]
    x_d = [torch.empty_like(x) for _ in range(2)]
    out_d = [torch.empty_like(out) for _ in range(2)]
    s_up, s_down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    e_steps = max(3, steps)
    ev = lambda: torch.cuda.Event()
    computed = [None, None]  # step's compute done (buffers b consumed)
    downloaded = [None, None]  # step's output copied out (out_d[b] free)

    def run(nsteps):
        for i in range(nsteps):
            b = i & 1
            with torch.cuda.stream(s_up):
                if computed[b] is not None:
                    s_up.wait_event(computed[b])
                if not with_router:  # with the router the step starts from x alone
                    lg_d[b].copy_(lg_h, non_blocking=True)
                x_d[b].copy_(x_h, non_blocking=True)
                up = ev()
                up.record(s_up)
            stream.wait_event(up)
            if downloaded[b] is not None:
                stream.wait_event(downloaded[b])
            if with_router:
                heap.router_logits(x_d[b], wl.wr, lg_d[b], stream=stream)
            heap.pipeline(lg_d[b], x_d[b], wg, wu, wd, wl.idx, wl.w, out_d[b], fused=fused, weights_in_ffn=wif,
                          dedup=dedup, fp8=fp8, stream=stream)
            computed[b] = ev()
            computed[b].record(stream)
            with torch.cuda.stream(s_down):
                s_down.wait_event(computed[b])
                out_h[b].copy_(out_d[b], non_blocking=True)
                downloaded[b] = ev()
                downloaded[b].record(s_down)

    run(2)
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_up)
    run(e_steps)
    e1.record(s_down)
    torch.cuda.synchronize()
    barrier()
    e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    assert torch.equal(out_h[(e_steps - 1) & 1].view(torch.int16), out.cpu().view(torch.int16)), \
        "end-to-end output differs from the device-resident run"
    return {"value": wl.n * e_steps * world / (e_ms / 1e3), "unit": UNIT,
            "h2d_bytes_per_step": (0 if with_router else lg_h.numel() * 4) + x_h.numel() * 2,
            "d2h_bytes_per_step": out_h[0].numel() * 2, "steps": e_steps,
            "overlap": "uploads and downloads on their own streams, double-buffered"}


IDLE_BETWEEN_S = 1.5


def run_per_workload(sm, head: Workload, args, stream, world, local, barrier, dev, head_fused, head_stages,
                     head_ms, head_clocks, head_counts) -> list:
    """Every configuration of the path in one run: the headline workload's
    own numbers plus its other launch form, then Tiny, DeepSeek-V3-like,
    Skewed and Decode, each staged and as the fused single launch (Decode is
    defined as the fused launch; its staged form is the comparison).  Weights
    are shared between configurations of the same E, H, I."""
    import torch
    import moe_synth as ms
    steps = args.steps
    rec = [workload_summary(args.config, head.cfg, head_fused, steps, head_ms, head_stages, head_clocks,
                            head_counts, start="the headline's own timed steps")]
    # Every entry starts from the state the headline started from: an idle GPU
    # (the headline's timed steps follow only input generation and a short
    # warm-up).  Back-to-back load engages the power cap within ~0.25 s and
    # lowers the SM clock by up to a quarter; the clocks sampled during each
    # entry's timed steps are recorded beside it.
    idle = lambda: time.sleep(IDLE_BETWEEN_S)
    idle()
    ms_total, st, clk = time_steps(head, stream, steps, args.warmup, 1 - head_fused, world=world, local=local,
                                   barrier=barrier, device=dev)
    rec.append(workload_summary(args.config, head.cfg, 1 - head_fused, steps, ms_total, st, clk,
                                expert_counts(head.heap, head.cfg)))
    shared = {}
    for name in ("tiny", "deepseek", "skewed", "decode"):
        cfg = dict(ms.CONFIGS[name])
        key = weight_key(cfg)
        if key not in shared:
            shared.clear()
            torch.cuda.empty_cache()
            shared[key] = ms.weights_torch(cfg, dev)
        wl = Workload(sm, cfg, dev, weights=shared[key])
        forms = (1, 0) if cfg.get("fused") else (0, 1)
        for f in forms:
            torch.cuda.synchronize()
            idle()
            ms_total, st, clk = time_steps(wl, stream, steps, args.warmup, f, world=world, local=local,
                                           barrier=barrier, device=dev)
            rec.append(workload_summary(name, cfg, f, steps, ms_total, st, clk, expert_counts(wl.heap, cfg)))
        del wl
        torch.cuda.empty_cache()
    return rec


# ---------------------------------------------------------------------------
# CPU oracle timing legs
# ---------------------------------------------------------------------------

def _openblas_handles():
    """(set, get) functions of the OpenBLAS that numpy loaded, found by the
    library's exported thread-count calls (numpy wheels bundle OpenBLAS under
    a prefixed name); (None, None) if there is none."""
    import ctypes
    import numpy as np  # noqa: F401  (loads the BLAS)
    paths = set()
    try:
        for line in open("/proc/self/maps"):
            f = line.split()
            if len(f) >= 6 and "openblas" in f[-1].lower() and ".so" in f[-1]:
                paths.add(f[-1])
    except OSError:
        return None, None
    names = [("openblas_set_num_threads", "openblas_get_num_threads"),
             ("scipy_openblas_set_num_threads64_", "scipy_openblas_get_num_threads64_"),
             ("openblas_set_num_threads64_", "openblas_get_num_threads64_"),
             ("scipy_openblas_set_num_threads", "scipy_openblas_get_num_threads")]
    for pth in sorted(paths):
        try:
            L = ctypes.CDLL(pth)
        except OSError:
            continue
        for sname, gname in names:
            if hasattr(L, sname) and hasattr(L, gname):
                setf, getf = getattr(L, sname), getattr(L, gname)
                setf.argtypes, setf.restype = [ctypes.c_int], None
                getf.argtypes, getf.restype = [], ctypes.c_int
                return setf, getf
    return None, None


class OneCore:
    """BLAS limited to one thread and the calling thread pinned to one core
    (restored on exit); ``threads`` is the BLAS thread count in effect."""

    def __enter__(self):
        self.setf, self.getf = _openblas_handles()
        self.prev_threads = self.getf() if self.getf else None
        self.prev_aff = os.sched_getaffinity(0) if hasattr(os, "sched_getaffinity") else None
        if self.setf:
            self.setf(1)
        if self.prev_aff:
            os.sched_setaffinity(0, {min(self.prev_aff)})
        self.threads = self.getf() if self.getf else None
        return self

    def __exit__(self, *a):
        if self.setf and self.prev_threads:
            self.setf(self.prev_threads)
        if self.prev_aff:
            os.sched_setaffinity(0, self.prev_aff)


def blas_threads():
    _, getf = _openblas_handles()
    return getf() if getf else None


def oracle_stage_times(cfg: dict, dev) -> dict:
    """The oracle's route, count + placement, dispatched rows and combine on
    the full workload (seconds).  The combine runs on the dispatched rows as
    its expert rows: its time does not depend on their values.  The inputs
    come from the input generator (its device implementation, for speed:
    the same bits as its host one), outside the timed steps."""
    import numpy as np
    import torch
    import moe_synth as ms
    import oracle
    E, W, k = cfg["num_experts"], cfg["world"], cfg["topk"]
    lg = ms.logits_np(cfg)
    x = ms.x_torch(cfg, dev).view(torch.int16).cpu().numpy().view(np.uint16)
    t = {}
    t0 = time.perf_counter()
    idx, w = oracle.route_topk(lg, k)
    t["route"] = time.perf_counter() - t0
    t0 = time.perf_counter()
    pos, rp, _ = oracle.place_pairs(idx, w, E, W)
    t["count_place"] = time.perf_counter() - t0
    t0 = time.perf_counter()
    rows = oracle.dispatch_rows(x, rp, k)
    t["dispatch_rows"] = time.perf_counter() - t0
    t0 = time.perf_counter()
    oracle.combine(rows, idx, w, pos, E, W)
    t["combine"] = time.perf_counter() - t0
    return t


def cpu_baseline(cfg: dict, dev, wif: bool) -> dict:
    """The oracle as it stands on the host cores: a bounded token sample of
    the whole path at the BLAS's own thread count and on one core, plus its
    route / placement / dispatch / combine steps on the full workload on one
    core."""
    import numpy as np
    ntok = int(os.environ.get("SYMMOE_CPU_TOKENS", "64"))
    n, k = cfg["world"] * cfg["tokens_per_slot"], cfg["topk"]
    tokens = np.sort(np.random.default_rng(0).choice(n, size=ntok, replace=False))
    wts = sample_weights(cfg, tokens, dev)
    threads = blas_threads()
    dt = oracle_sample_run(cfg, tokens, wts, wif)
    with OneCore() as one:
        dt1 = oracle_sample_run(cfg, tokens, wts, wif)
        stages = oracle_stage_times(cfg, dev)
        t1 = one.threads
    return {"value": ntok / dt, "unit": UNIT, "cores": cores_used(), "threads": threads, "kind": "oracle",
            "sample": f"{ntok} random tokens of the workload (routing, placement, all {ntok * k} expert "
                      f"FFN rows, combine) in {dt:.1f} s; fp64 numpy, BLAS on {threads} threads",
            "one_core": {"value": ntok / dt1, "unit": UNIT, "threads": t1, "seconds": dt1,
                         "sample": "the same tokens, BLAS on one thread, pinned to one core"},
            "full_workload_one_core_s": stages}


def run_linear_a2a(args):
    """GEMM -> A2A and A2A -> GEMM on the config's W, T, H: the fused form
    against the split pipeline, alternating blocks of calls so both see the
    same clocks; CUDA events on the calling stream."""
    import torch
    import moe_synth as ms
    import combine_symmetric_heap_gb300 as sm
    rank, world, local = dist_env()
    if rank != 0:
        return 0
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = get_cfg(args)
    W, T, H = cfg["world"], cfg["tokens_per_slot"], cfg["hidden"]
    n = W * T
    heap = sm.SymHeap(cfg, dev)
    x = ms.x_torch(cfg, dev)
    z = ms.shards_torch(cfg, dev)
    w = ms.linear_weight_torch(cfg, dev)
    stream = torch.cuda.current_stream(dev)
    hbm, tf_burst, tf_sus, peak_src = peaks()
    flops = 2.0 * n * H * H
    # forms of each op: the fused one (the pages' LSA form), the split
    # pipeline, and for A2A -> GEMM the copy-engine form (the pages' SDMA form)
    forms = {"gemm_a2a": {"fused": lambda: heap.gemm_a2a(x, w, fused=True, stream=stream),
                          "split": lambda: heap.gemm_a2a(x, w, fused=False, stream=stream)},
             "a2a_gemm": {"fused": lambda: heap.a2a_gemm(z, w, fused=True, stream=stream),
                          "split": lambda: heap.a2a_gemm(z, w, fused=False, stream=stream),
                          "fused_copy_engines": lambda: heap.a2a_gemm(z, w, fused=True, copy_engines=True,
                                                                      stream=stream)}}
    steps, rounds = max(args.steps // 4, 5), 4
    out = {}
    with ClockSampler(local) as clk:
        for name, fs in forms.items():
            for call in fs.values():
                for _ in range(max(args.warmup, 3)):
                    call()
            torch.cuda.synchronize()
            times = {k: [] for k in fs}
            for _ in range(rounds):   # alternating blocks: every form sees the same clocks
                for k, call in fs.items():
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    for _ in range(steps):
                        call()
                    e1.record(stream)
                    torch.cuda.synchronize()
                    times[k].append(e0.elapsed_time(e1) / steps)
            assert heap.status(stream=stream) == 0, "device status word set"
            med = {k: sorted(v)[rounds // 2] for k, v in times.items()}
            tf = flops / (med["fused"] / 1e3) / 1e12
            out[name] = {**{f"{k}_ms": v for k, v in med.items()},
                         "speedup_pct": 100.0 * (med["split"] / med["fused"] - 1.0),
                         "fused_tflops": tf, "frac": tf / tf_burst,
                         "peak": f"{peak_src} bf16 burst {tf_burst} TFLOP/s",
                         "exchange_bytes": n * H * 2}
            if "fused_copy_engines" in med:
                out[name]["copy_engines_speedup_pct"] = 100.0 * (med["split"] / med["fused_copy_engines"] - 1.0)
    line = {"metric": "GEMM + all-to-all on the heap's slots: fused vs split, ms per call on 1 GB300",
            "impl": "ours", "workload": "linear_a2a", "n_gpus": 1, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"linear {H}x{H} over W={W} slots of T={T} tokens ({args.config} shape)",
                       "world_slots": W, "tokens_per_slot": T, "hidden": H,
                       "steps_per_block": steps, "blocks": rounds},
            **out, "clocks": clk.summary()}
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse()
    if args.workload == "linear_a2a":
        return run_linear_a2a(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
