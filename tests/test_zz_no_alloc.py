"""The allocation-free dispatch layout call (moe_dispatch_layout_noalloc).

Some callers cannot allocate device memory: a plug-in whose host framework
hands it only its input and output buffers and owns every allocation, or a
process that fixes its device-memory footprint at start-up.  For them the
layout call keeps its scratch (the chunk histograms) in a library-owned
device array.  These tests check, through the C ABI, that two calls in a row
give exactly the counts, offsets, totals and receive rows that moe_dispatch
writes into a heap, and that too large a shape is refused.  This file is
collected last on purpose.
"""
import numpy as np
import pytest
import torch

import moe_synth as ms
import combine_symmetric_heap_gb300 as sm


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # E * ceil(N/128) histogram entries must fit in SYM_NOALLOC_HIST_MAX = 2^18
    big = dict(world=8, tokens_per_slot=1 << 14, num_experts=512, topk=8)
    A = 1 << 41  # never dereferenced: the size check comes first
    with pytest.raises(sm.SymmoeError) as ei:
        sm.moe_dispatch_layout_noalloc(big, A, A, A, A, A, stream=0)
    assert ei.value.code == sm.SYM_ENOSPACE


def _heap_layout(cfg, logits, dev):
    """Routing and the regular heap dispatch (the existing entry points)."""
    n, k = cfg["world"] * cfg["tokens_per_slot"], cfg["topk"]
    small = dict(cfg, hidden=128, inter=128)      # the layout does not depend on H or I
    heap = sm.SymHeap(small, dev)
    idx = torch.empty((n, k), dtype=torch.int32, device=dev)
    w = torch.empty((n, k), dtype=torch.float32, device=dev)
    x = torch.zeros((n, 128), dtype=torch.bfloat16, device=dev)
    heap.route_topk(logits, idx, w)
    heap.dispatch(x, idx, w)
    torch.cuda.synchronize()
    W = cfg["world"]
    cnt = torch.cat([heap.cnt(d) for d in range(W)]).cpu()
    off = torch.cat([heap.recv_off(d) for d in range(W)]).cpu()
    tot = torch.cat([heap.total_recv(d) for d in range(W)]).cpu()
    pos = torch.cat([heap.pos(d) for d in range(W)]).cpu()
    return idx, cnt, off, tot, pos


@pytest.mark.gpu
def test_noalloc_layout_matches_dispatch_on_two_calls():
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    results = []
    for name in ("deepseek", "skewed"):          # two calls in a row, different routings
        cfg = ms.CONFIGS[name]
        n, k, E, W = cfg["world"] * cfg["tokens_per_slot"], cfg["topk"], cfg["num_experts"], cfg["world"]
        idx, cnt_ref, off_ref, tot_ref, pos_ref = _heap_layout(cfg, ms.logits_torch(cfg, dev), dev)
        cnt = torch.full((E,), -7, dtype=torch.int32, device=dev)
        off = torch.full((E,), -7, dtype=torch.int32, device=dev)
        tot = torch.full((W,), -7, dtype=torch.int32, device=dev)
        pos = torch.full((n, k), -7, dtype=torch.int32, device=dev)
        sm.moe_dispatch_layout_noalloc(cfg, idx, cnt, off, tot, pos)
        torch.cuda.synchronize()
        assert torch.equal(cnt.cpu(), cnt_ref)
        assert torch.equal(off.cpu(), off_ref)
        assert torch.equal(tot.cpu(), tot_ref)
        assert torch.equal(pos.cpu(), pos_ref)
        results.append(cnt.cpu())
    # the skew changes the counts, so the second call really recomputed them
    assert not torch.equal(results[0], results[1])
