"""Host-checked bounds of the CUDA path (a stand-in for a memory checker):

* counts in the heap's signal area that would send rows past a window's
  capacity -- written on the host after a normal dispatch, as a corrupted or
  stale signal area would hold them -- make the consumers skip that expert or
  slot, raise SYM_STATUS_OVERFLOW, and store nothing past the capacity;
* canaries in the guard bands after every window stay intact across every
  entry point on a small shape.

The corrupted counts exceed the capacity by only a few rows, so that even a
kernel without the checks would write inside the same heap allocation (the
guard band after the window), never outside it.
"""
import numpy as np
import pytest
import torch

import moe_synth as ms
import oracle
from _cases import (assert_canaries, assert_close, bits, checked_oracle_routing, device_inputs, fresh_weight_fn,
                    plant_canaries)

pytestmark = pytest.mark.gpu
DEV = "cuda"
CFG = dict(world=2, tokens_per_slot=64, hidden=256, num_experts=4, topk=2, inter=256)


@pytest.fixture(scope="module")
def sm():
    import combine_symmetric_heap_gb300 as m
    return m


def _dispatched(sm, cfg=CFG):
    logits, x, wg, wu, wd = device_inputs(cfg, DEV)
    n, k = cfg["world"] * cfg["tokens_per_slot"], cfg["topk"]
    heap = sm.SymHeap(cfg, DEV)
    plant_canaries(heap)
    idx = torch.empty((n, k), dtype=torch.int32, device=DEV)
    w = torch.empty((n, k), dtype=torch.float32, device=DEV)
    heap.route_topk(logits, idx, w)
    heap.dispatch(x, idx, w)
    torch.cuda.synchronize()
    assert heap.status() == 0
    return heap, idx, w, (wg, wu, wd)


def _y_of_expert(heap, e, e_loc):
    d, l = e // e_loc, e % e_loc
    o, c = int(heap.recv_off(d)[l]), int(heap.cnt(d)[l])
    return d, o, c


@pytest.mark.parametrize("excess", [1, 3])
def test_expert_rows_past_capacity_are_skipped(sm, excess):
    heap, idx, w, (wg, wu, wd) = _dispatched(sm)
    e_loc = CFG["num_experts"] // CFG["world"]
    e_bad = e_loc - 1                                 # last expert of slot 0
    d, o, c = _y_of_expert(heap, e_bad, e_loc)
    heap.cnt(d)[e_bad % e_loc] = heap.cap - o + excess  # its rows would end `excess` rows past cap
    heap.expert_ffn(wg, wu, wd)
    torch.cuda.synchronize()
    assert heap.status(clear=True) & sm.SYM_STATUS_OVERFLOW
    assert_canaries(heap, "expert FFN with a count past capacity")
    # the skipped expert stored nothing; every other expert matches the oracle
    assert int((heap.y(d)[o:o + c].view(torch.int16) != 0).sum()) == 0
    # every other expert against the oracle, on the oracle's own routing and
    # placement of the same logits (the launch's routing must equal it)
    ridx, rw = checked_oracle_routing(CFG, idx, w)
    E, W, k = CFG["num_experts"], CFG["world"], CFG["topk"]
    cnt, off, _ = oracle.count_experts(ridx, E, W)
    _, rp, _ = oracle.place_pairs(ridx, rw, E, W)
    wfn = fresh_weight_fn(CFG, DEV)
    x_bits = ms.x_np(CFG)
    for e in range(E):
        if e == e_bad:
            continue
        s, oe, ce = e // e_loc, int(off[e]), int(cnt[e])
        rows = x_bits[rp[s][oe:oe + ce] // k]
        _, _, ye = oracle.expert_ffn_rows(rows, *wfn(e))
        assert_close(bits(heap.y(s)[oe:oe + ce]), ye, f"expert {e} y")


def test_negative_count_and_offset_are_skipped(sm):
    heap, idx, w, (wg, wu, wd) = _dispatched(sm)
    heap.cnt(1)[0] = -5
    heap.recv_off(0)[1] = -256
    heap.expert_ffn(wg, wu, wd)
    torch.cuda.synchronize()
    assert heap.status(clear=True) & sm.SYM_STATUS_OVERFLOW
    assert_canaries(heap, "expert FFN with negative counts")


def test_total_past_capacity_skips_the_fallback_copy(sm):
    heap, idx, w, (wg, wu, wd) = _dispatched(sm)
    heap.expert_ffn(wg, wu, wd)
    torch.cuda.synchronize()
    assert heap.status() == 0
    W, H, cap = CFG["world"], CFG["hidden"], heap.cap
    y1_before = heap.y(1).clone()
    heap.total_recv(1)[0] = cap + 2                    # slot 1's total two rows past capacity
    dense = torch.full((W, cap, H), 1.0, dtype=torch.bfloat16, device=DEV)  # not the view: a staging copy
    out = torch.empty((W * CFG["tokens_per_slot"], H), dtype=torch.bfloat16, device=DEV)
    heap.combine(idx, w, out, expert_out=dense)
    torch.cuda.synchronize()
    assert heap.status(clear=True) & sm.SYM_STATUS_OVERFLOW
    assert_canaries(heap, "fallback combine with a total past capacity")
    assert torch.equal(heap.y(1).view(torch.int16), y1_before.view(torch.int16))   # slot 1 skipped
    t0 = int(heap.total_recv(0)[0])
    assert bool((heap.y(0)[:t0] == 1.0).all())                                    # slot 0 copied


def test_canaries_intact_across_every_entry_point(sm):
    """Every call on one heap, canaries checked after each: routing, the
    router GEMM, the plain / deduplicated / FP8 dispatch, the expert FFN (plain
    and weighted rows), the combine (view, fallback copy, unweighted), the
    staged and fused pipelines, and both GEMM + all-to-all directions."""
    cfg = CFG
    logits, x, wg, wu, wd = device_inputs(cfg, DEV)
    n, k, H = cfg["world"] * cfg["tokens_per_slot"], cfg["topk"], cfg["hidden"]
    heap = sm.SymHeap(cfg, DEV)
    plant_canaries(heap)
    idx = torch.empty((n, k), dtype=torch.int32, device=DEV)
    w = torch.empty((n, k), dtype=torch.float32, device=DEV)
    out = torch.empty((n, H), dtype=torch.bfloat16, device=DEV)
    lg = torch.empty_like(logits)
    wr = ms.router_weight_torch(cfg, DEV)
    wl = ms.linear_weight_torch(cfg, DEV)
    z = ms.shards_torch(cfg, DEV)
    calls = [
        ("router", lambda: heap.router_logits(x, wr, lg)),
        ("route", lambda: heap.route_topk(logits, idx, w)),
        ("dispatch", lambda: heap.dispatch(x, idx, w)),
        ("dispatch dedup", lambda: heap.dispatch(x, idx, w, dedup=True)),
        ("dispatch fp8", lambda: heap.dispatch(x, idx, w, fp8=True)),
        ("dispatch", lambda: heap.dispatch(x, idx, w)),
        ("expert FFN", lambda: heap.expert_ffn(wg, wu, wd)),
        ("expert FFN weighted", lambda: heap.expert_ffn(wg, wu, wd, weighted_rows=True)),
        ("combine unweighted", lambda: heap.combine(idx, w, out, unweighted=True)),
        ("combine fallback", lambda: heap.combine(idx, w, out, expert_out=heap.y(0).clone().repeat(2, 1))),
        ("pipeline staged", lambda: heap.pipeline(logits, x, wg, wu, wd, idx, w, out)),
        ("pipeline fused", lambda: heap.pipeline(logits, x, wg, wu, wd, idx, w, out, fused=1)),
        ("pipeline fused weighted", lambda: heap.pipeline(logits, x, wg, wu, wd, idx, w, out, fused=1,
                                                          weights_in_ffn=True)),
        ("pipeline dedup", lambda: heap.pipeline(logits, x, wg, wu, wd, idx, w, out, dedup=True)),
        ("pipeline fp8", lambda: heap.pipeline(logits, x, wg, wu, wd, idx, w, out, fp8=True)),
        ("gemm_a2a fused", lambda: heap.gemm_a2a(x, wl, fused=True)),
        ("gemm_a2a split", lambda: heap.gemm_a2a(x, wl, fused=False)),
        ("a2a_gemm fused", lambda: heap.a2a_gemm(z, wl, fused=True)),
        ("a2a_gemm split", lambda: heap.a2a_gemm(z, wl, fused=False)),
        ("a2a_gemm copy engines", lambda: heap.a2a_gemm(z, wl, fused=True, copy_engines=True)),
    ]
    for what, call in calls:
        call()
        assert_canaries(heap, what)
        assert heap.status() == 0, what
    # the pipeline still matches the oracle after all of that
    heap.pipeline(logits, x, wg, wu, wd, idx, w, out)
    ref = oracle.pipeline(ms.logits_np(cfg), ms.x_np(cfg), cfg, fresh_weight_fn(cfg, DEV))
    assert_close(bits(out), np.asarray(oracle.bf16_bits_to_f64(ref["out"])), "pipeline after every call")
