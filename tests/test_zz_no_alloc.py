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
    # calls in a row on different routings: the two full DeepSeek-V3-like
    # routings, then small odd shapes (a partial last chunk, a chunk count
    # that is not a multiple of 32, one expert per slot, a single slot)
    odd = [dict(world=8, tokens_per_slot=100, hidden=128, num_experts=8, topk=2, inter=128),
           dict(world=1, tokens_per_slot=77, hidden=128, num_experts=4, topk=3, inter=128)]
    for cfg in [ms.CONFIGS["deepseek"], ms.CONFIGS["skewed"]] + odd:
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


@pytest.mark.gpu
def test_noalloc_duplicate_expert_in_a_token():
    """A token that lists one expert twice: the expert counts it once and the
    later copy gets pos -1, so every placed pair has a row of its own.  The
    expected layout is the plain definition over the placed pairs: per
    expert, in (token, j) order, after the expert's receive offset."""
    dev = torch.device("cuda", 0)
    W, T, E, k = 4, 75, 16, 4
    n, e_loc = W * T, E // W
    rng = np.random.default_rng(5)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(n)]).astype(np.int32)
    for g in range(0, n, 7):                       # every 7th token repeats its first expert
        idx[g, 2] = idx[g, 0]
    want_pos = np.full((n, k), -1, dtype=np.int32)
    cnt_want = np.zeros(E, dtype=np.int64)
    for g in range(n):
        seen = set()
        for j in range(k):
            e = int(idx[g, j])
            if e not in seen:
                seen.add(e)
                cnt_want[e] += 1
    off_want = np.zeros(E, dtype=np.int64)
    tot_want = np.zeros(W, dtype=np.int64)
    for e in range(E):
        off_want[e] = tot_want[e // e_loc]
        tot_want[e // e_loc] += cnt_want[e]
    fill = np.zeros(E, dtype=np.int64)
    for g in range(n):
        seen = set()
        for j in range(k):
            e = int(idx[g, j])
            if e in seen:
                continue
            seen.add(e)
            want_pos[g, j] = off_want[e] + fill[e]
            fill[e] += 1
    shape = dict(world=W, tokens_per_slot=T, num_experts=E, topk=k)
    idx_d = torch.from_numpy(idx).to(dev)
    cnt = torch.full((E,), -7, dtype=torch.int32, device=dev)
    off = torch.full((E,), -7, dtype=torch.int32, device=dev)
    tot = torch.full((W,), -7, dtype=torch.int32, device=dev)
    pos = torch.full((n, k), -7, dtype=torch.int32, device=dev)
    for _ in range(2):
        sm.moe_dispatch_layout_noalloc(shape, idx_d, cnt, off, tot, pos)
        torch.cuda.synchronize()
        assert np.array_equal(cnt.cpu().numpy(), cnt_want)
        assert np.array_equal(off.cpu().numpy(), off_want)
        assert np.array_equal(tot.cpu().numpy(), tot_want)
        assert np.array_equal(pos.cpu().numpy(), want_pos)
    assert int(cnt_want.sum()) == int((want_pos >= 0).sum())
