"""Shared helpers of the parity tests: small shapes that span several tiles and
ragged tails, the float tolerance, and runners for the CUDA path and the
oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

import moe_synth as ms
import oracle

# Float tolerance for bf16 outputs against the fp64 oracle: per element
# |gpu - ref| <= 2e-2 * max(1, |ref|), and relative L2 over the tensor <= 1e-2.
ATOL_REL = 2e-2
REL_L2 = 1e-2

SMALL = {
    "tiny": ms.CONFIGS["tiny"],
    # two 128-token tiles per expert with a ragged tail, 3 gate/up and 2 down feature tiles
    "ragged": dict(world=2, tokens_per_slot=200, hidden=256, num_experts=4, topk=2, inter=384),
    # several experts per slot, k = E/W
    "many": dict(world=4, tokens_per_slot=96, hidden=128, num_experts=16, topk=4, inter=128),
    # one slot holding every expert, k = E (every expert receives every token)
    "allk": dict(world=1, tokens_per_slot=130, hidden=128, num_experts=8, topk=8, inter=256),
    # k = 1, ~300 rows per expert: two token tiles (256 + ragged) per expert
    "multi": dict(world=1, tokens_per_slot=600, hidden=128, num_experts=2, topk=1, inter=256),
    # 32 slots (the most the deduplicated dispatch takes), two experts per slot
    "slots32": dict(world=32, tokens_per_slot=24, hidden=128, num_experts=64, topk=4, inter=128),
    # 64 slots of one expert each, 8 tokens per slot
    "slots64": dict(world=64, tokens_per_slot=8, hidden=256, num_experts=64, topk=2, inter=128),
}


# routing weights: fp32 expf on the GPU against the fp64 oracle
W_TOL = 2e-6


def checked_oracle_routing(cfg: dict, idx: torch.Tensor, w: torch.Tensor | None = None, seed: int = 0):
    """The oracle's routing of the generator's logits for ``cfg``.  The CUDA
    path's routing of the same logits (``idx``, ``w``) must match it: indices
    bit-exact, weights within W_TOL.  Returns the oracle's indices and
    weights (never the launch's) for the oracle calls that follow."""
    ridx, rw = oracle.route_topk(ms.logits_np(cfg, seed), cfg["topk"])
    assert np.array_equal(idx.cpu().numpy(), ridx), "routing indices differ from the oracle's"
    if w is not None:
        err = np.abs(w.cpu().numpy().astype(np.float64) - rw.astype(np.float64)).max(initial=0.0)
        assert err <= W_TOL, f"routing weights: max error {err}"
    return ridx, rw


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 bit patterns on the host."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_f64(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def assert_close(got_bits: np.ndarray, ref_f64: np.ndarray, what: str) -> dict:
    got = bf16_f64(got_bits)
    ref = np.asarray(ref_f64, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    diff = np.abs(got - ref)
    bound = ATOL_REL * np.maximum(1.0, np.abs(ref))
    bad = np.argwhere(diff > bound)
    assert bad.size == 0, f"{what}: {len(bad)} elements beyond tolerance, first {bad[:3].tolist()} " \
                          f"got {got[tuple(bad[0])]} ref {ref[tuple(bad[0])]}"
    nref = np.linalg.norm(ref)
    rel = np.linalg.norm(got - ref) / nref if nref > 0 else float(np.max(diff, initial=0.0))
    assert rel <= REL_L2, f"{what}: relative L2 {rel}"
    return {"max_abs": float(np.max(diff, initial=0.0)), "rel_l2": float(rel)}


def device_inputs(cfg: dict, dev, seed: int = 0):
    logits = ms.logits_torch(cfg, dev, seed)
    x = ms.x_torch(cfg, dev, seed)
    wg, wu, wd = ms.weights_torch(cfg, dev, seed)
    return logits, x, wg, wu, wd


def host_weight_fn(cfg: dict, seed: int = 0):
    cache = {}

    def fn(e):
        if e not in cache:
            cache[e] = tuple(ms.weight_np(cfg, nm, e, seed) for nm in ("gate", "up", "down"))
        return cache[e]
    return fn


def fresh_weight_fn(cfg: dict, device, seed: int = 0):
    """Expert weights for the oracle, generated afresh (never a buffer the
    CUDA path touched) by the input module's torch implementation on
    ``device`` -- fast for multi-GB experts -- and returned as host bits."""
    cache = {}

    def fn(e):
        if e not in cache:
            cache[e] = tuple(bits(ms.weight_expert_torch(cfg, nm, e, device, seed))
                             for nm in ("gate", "up", "down"))
        return cache[e]
    return fn


# Canaries: a byte pattern planted in the heap's guard bands (the bytes after
# every window that no call may touch) and checked after each call.  A kernel
# that stores past the end of a window (a row beyond capacity, a count it
# trusted) changes a band before anything else.
CANARY = 0xA5


def plant_canaries(heap) -> None:
    for start, length in heap.guard_bands():
        heap.buf[start:start + length].fill_(CANARY)


def assert_canaries(heap, what: str) -> None:
    torch.cuda.synchronize()
    bad = [(s, n) for s, n in heap.guard_bands() if not bool((heap.buf[s:s + n] == CANARY).all())]
    assert not bad, f"{what}: guard bands changed at {bad[:4]} (of {len(heap.guard_bands())})"


def run_gpu_stages(sm, cfg: dict, logits, x, wg, wu, wd, heap=None, idx=None, w=None):
    """route -> dispatch -> expert FFN -> combine, one call per stage.  On a
    heap it creates, canaries are planted first and checked after every call."""
    dev = x.device
    n, k = cfg["world"] * cfg["tokens_per_slot"], cfg["topk"]
    fresh = heap is None
    heap = heap or sm.SymHeap(cfg, dev)
    check = (lambda what: assert_canaries(heap, what)) if fresh else (lambda what: None)
    if fresh:
        plant_canaries(heap)
    if idx is None:
        idx = torch.empty((n, k), dtype=torch.int32, device=dev)
        w = torch.empty((n, k), dtype=torch.float32, device=dev)
        heap.route_topk(logits, idx, w)
        check("route")
    heap.dispatch(x, idx, w)
    check("dispatch")
    heap.expert_ffn(wg, wu, wd)
    check("expert FFN")
    out = torch.empty((n, cfg["hidden"]), dtype=torch.bfloat16, device=dev)
    heap.combine(idx, w, out)
    check("combine")
    torch.cuda.synchronize()
    return heap, idx, w, out
