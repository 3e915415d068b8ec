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


def parse():
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
    p.add_argument("--workload", default="moe", choices=["moe", "linear_a2a"],
                   help="linear_a2a: the GEMM + all-to-all workload on the same heap, fused vs split")
    return p.parse_args()


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
    """nvidia-smi clock / throttle samples during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

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

    def summary(self):
        if not getattr(self, "lines", None):
            return None
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


TRAFFIC_SOURCES = ("expert_ffn.cu", "gemm2sm.cuh", "symmoe_dev.cuh")


def sources_sha256(files=TRAFFIC_SOURCES) -> str:
    """sha256 over the kernel sources a traffic record was captured from."""
    hsh = hashlib.sha256()
    for f in files:
        hsh.update(open(os.path.join(ROOT, "combine_symmetric_heap_gb300", "csrc", f), "rb").read())
    return hsh.hexdigest()


def traffic_record(workload: str, cfg: dict):
    """Per-step DRAM bytes of the expert FFN launches from the committed ncu
    summary, or None if it was captured for another workload or shape, or any
    of its sources changed since."""
    import moe_synth as ms
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        rec = json.load(open(path))
        if rec.get("sources_sha256") != sources_sha256():
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
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores_used(), "kind": "oracle",
                         "sample": f"{per_step} random tokens of the workload per step (their "
                                   f"routing, placement, expert FFN rows and combine); expert "
                                   f"weights generated outside the timed region"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

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

    heap = sm.SymHeap(cfg, dev)
    logits = ms.logits_torch(cfg, dev)
    x = ms.x_torch(cfg, dev)
    wg, wu, wd = ms.weights_torch(cfg, dev)
    wr = ms.router_weight_torch(cfg, dev) if with_router else None
    idx = torch.empty((n, k), dtype=torch.int32, device=dev)
    w = torch.empty((n, k), dtype=torch.float32, device=dev)
    out = torch.empty((n, H), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            dist.barrier()

    # Stage-by-stage steps make the same four C-ABI calls that moe_pipeline
    # makes, with an event on the stream between stages, so every stage time
    # (and the expert FFN's roofline) is measured inside the timed region.
    # The fused step is one launch (plus the router's, when it is timed too).
    stage_names = (["router"] if with_router else []) + (
        ["fused"] if fused else ["route", "dispatch", "expert_ffn", "combine"])
    nst = len(stage_names)
    stage_evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)] for _ in range(args.steps)]

    def step(i=None):
        ev = stage_evs[i] if i is not None else None
        calls = [lambda: heap.router_logits(x, wr, logits, stream=stream)] if with_router else []
        if fused:
            calls.append(lambda: heap.pipeline(logits, x, wg, wu, wd, idx, w, out, fused=1,
                                               weights_in_ffn=wif, stream=stream))
        else:
            calls += [lambda: heap.route_topk(logits, idx, w, stream=stream),
                      lambda: heap.dispatch(x, idx, w, dedup=dedup, fp8=fp8, stream=stream),
                      lambda: heap.expert_ffn(wg, wu, wd, weighted_rows=wif, stream=stream),
                      lambda: heap.combine(idx, w, out, unweighted=wif, stream=stream)]
        for j, call in enumerate(calls):
            if ev:
                ev[j].record(stream)
            call()
        if ev:
            ev[nst].record(stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    assert heap.status(stream=stream) == 0, "device status word set during warm-up"

    # ---- timed region: K whole-path steps, device resident inputs
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        ev0.record(stream)
        for i in range(args.steps):
            step(i)
        ev1.record(stream)
        torch.cuda.synchronize()
    barrier()
    ms_total = max_over_ranks(ev0.elapsed_time(ev1), world, dev)
    assert heap.status(stream=stream) == 0, "device status word set during the timed steps"
    ms_step = ms_total / args.steps
    value = n * args.steps * world / (ms_total / 1e3)
    # the router is one GEMM launch, plus one reduction launch when it splits K
    router_launches = (1 + (heap.router_splits() > 1)) if with_router else 0
    launches_per_step = (1 if fused else 7) + router_launches

    # ---- stage times: averages over the timed steps (device time per stage)
    acc = [0.0] * nst
    for ev in stage_evs:
        for j in range(nst):
            acc[j] += ev[j].elapsed_time(ev[j + 1])
    stages = dict(zip(stage_names, [a / args.steps for a in acc]))

    experts_hit = int(sum(int((heap.cnt(d) > 0).sum().item()) for d in range(cfg["world"])))
    alg = algorithmic(cfg, experts_hit)
    hbm, tf_burst, tf_sus, peak_src = peaks()
    long_region = ms_total > 1000.0
    tf_peak = tf_sus if long_region else tf_burst
    # the expert FFN's binding roof: tensor time or HBM time at the measured peaks
    t_tensor = alg["ffn_flops"] / (tf_peak * 1e12)
    t_hbm = alg["ffn_bytes"] / (hbm * 1e9)
    bound = "tensor" if t_tensor >= t_hbm else "hbm"
    if fused:
        kern_s = stages["fused"] / 1e3  # one launch does the whole step
        kname = "moe_fused_kernel (whole step in one launch)"
        extra_bytes = alg["route_bytes"] + alg["dispatch_bytes"] + alg["combine_bytes"]
    else:
        kern_s = stages["expert_ffn"] / 1e3
        kname = "expert_gemm_kernel (gate/up SwiGLU + down launches)"
        extra_bytes = 0
    if bound == "tensor":
        achieved, peak, unit = alg["ffn_flops"] / kern_s / 1e12, tf_peak, "TFLOP/s"
        other = {"hbm_gbs": (alg["ffn_bytes"] + extra_bytes) / kern_s / 1e9, "hbm_peak": hbm}
    else:
        achieved, peak, unit = (alg["ffn_bytes"] + extra_bytes) / kern_s / 1e9, hbm, "GB/s"
        other = {"tflops": alg["ffn_flops"] / kern_s / 1e12, "tensor_peak": tf_peak}
    other["frac"] = (other.get("hbm_gbs", 0) / hbm) if bound == "tensor" else other["tflops"] / tf_peak
    roofline = {"bound": bound, "kernel": kname, "achieved": achieved, "peak": peak, "unit": unit,
                "frac": achieved / peak, "traffic": None if fused else traffic_record(args.config, cfg),
                "peak_kind": f"{peak_src} " + ("bf16 " + ("sustained" if long_region else "burst")
                                               if bound == "tensor" else "HBM copy"),
                "algorithmic_per_step": {"flops": alg["ffn_flops"], "bytes": alg["ffn_bytes"] + extra_bytes,
                                         "experts_hit": experts_hit},
                "other_roof": other}
    stage_bw = {"hbm_peak_gbs": hbm}
    if not fused:
        stage_bw["dispatch_gbs"] = alg["dispatch_bytes"] / (stages["dispatch"] / 1e3) / 1e9
        stage_bw["combine_gbs"] = alg["combine_bytes"] / (stages["combine"] / 1e3) / 1e9
        stage_bw["route_gbs"] = alg["route_bytes"] / (stages["route"] / 1e3) / 1e9
        stage_bw["dispatch_frac"] = stage_bw["dispatch_gbs"] / hbm
        stage_bw["combine_frac"] = stage_bw["combine_gbs"] / hbm
    if "router" in stages:
        # router GEMM: reads x [N,H] and Wr [E,H] (bf16), writes logits [N,E] (fp32)
        rbytes = n * H * 2 + cfg["num_experts"] * H * 2 + n * cfg["num_experts"] * 4
        rflops = 2.0 * n * H * cfg["num_experts"]
        rs = stages["router"] / 1e3
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
        slots = np.sort(idx.cpu().numpy() // (cfg["num_experts"] // cfg["world"]), axis=1)
        rows = int(n + (np.diff(slots, axis=1) != 0).sum())
        stage_bw["dedup"] = {"rows_crossing": rows, "pairs": n * k, "cross_slot_bytes": rows * H * 2,
                             "plain_cross_slot_bytes": n * k * H * 2}

    # ---- end to end through the public API with host buffers
    # Every step copies its inputs (logits, x) from pinned host memory and reads
    # its output back, as a serving loop does: the copies run on their own
    # streams, double-buffered, so step i+1's upload and step i-1's download
    # overlap step i's compute (the heap is reused, so the compute steps stay
    # in order on one stream).  Timed from the first upload to the last download.
    e2e = None
    if not args.no_e2e:
        lg_h = torch.empty(logits.shape, dtype=logits.dtype, pin_memory=True)
        x_h = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
        out_h = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
        lg_h.copy_(logits)
        x_h.copy_(x)
        lg_d = [torch.empty_like(logits) for _ in range(2)]
        x_d = [torch.empty_like(x) for _ in range(2)]
        out_d = [torch.empty_like(out) for _ in range(2)]
        s_up, s_down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        e_steps = max(3, min(args.steps, 30))
        ev = lambda: torch.cuda.Event()
        computed = [None, None]  # step's compute done (buffers b consumed)
        downloaded = [None, None]  # step's output copied out (out_d[b] free)

        def run_e2e(steps):
            for i in range(steps):
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
                    heap.router_logits(x_d[b], wr, lg_d[b], stream=stream)
                heap.pipeline(lg_d[b], x_d[b], wg, wu, wd, idx, w, out_d[b], fused=fused, weights_in_ffn=wif,
                              dedup=dedup, fp8=fp8, stream=stream)
                computed[b] = ev()
                computed[b].record(stream)
                with torch.cuda.stream(s_down):
                    s_down.wait_event(computed[b])
                    out_h[b].copy_(out_d[b], non_blocking=True)
                    downloaded[b] = ev()
                    downloaded[b].record(s_down)

        run_e2e(2)
        torch.cuda.synchronize()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_up)
        run_e2e(e_steps)
        e1.record(s_down)
        torch.cuda.synchronize()
        barrier()
        e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
        assert torch.equal(out_h[(e_steps - 1) & 1].view(torch.int16), out.cpu().view(torch.int16)), \
            "end-to-end output differs from the device-resident run"
        e2e = {"value": n * e_steps * world / (e_ms / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": (0 if with_router else lg_h.numel() * 4) + x_h.numel() * 2,
               "d2h_bytes_per_step": out_h[0].numel() * 2, "steps": e_steps,
               "overlap": "uploads and downloads on their own streams, double-buffered"}

    # ---- oracle on the host cores (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import numpy as np
        ntok = int(os.environ.get("SYMMOE_CPU_TOKENS", "64"))
        tokens = np.sort(np.random.default_rng(0).choice(n, size=ntok, replace=False))
        wts = sample_weights(cfg, tokens, dev)
        dt = oracle_sample_run(cfg, tokens, wts, wif)
        cpu = {"value": ntok / dt, "unit": UNIT, "cores": cores_used(), "kind": "oracle",
               "sample": f"{ntok} random tokens of the workload (routing, placement, all "
                         f"{ntok * k} expert FFN rows, combine) in {dt:.1f} s; fp64 numpy"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": dict(workload_config(args.config, cfg, fused, wif, with_router), dedup=dedup, fp8=fp8),
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk.summary(),
            "stages_ms": stages or None,
            "stage_bandwidth": stage_bw,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


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
