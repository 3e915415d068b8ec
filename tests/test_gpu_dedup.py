"""The rank-deduplicated dispatch on the GPU: every window the expert FFN and
the combine read is bit-identical to the plain dispatch's, the staging rows
hold each slot's tokens once in the oracle's order, and the row sources are
the oracle's."""
import numpy as np
import pytest
import torch

import moe_synth as ms
import oracle
from _cases import SMALL, bits, checked_oracle_routing

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def sm():
    import combine_symmetric_heap_gb300 as m
    return m


def _dispatch(sm, cfg, dedup):
    n, k = cfg["world"] * cfg["tokens_per_slot"], cfg["topk"]
    heap = sm.SymHeap(cfg, DEV)
    x = ms.x_torch(cfg, DEV)
    lg = ms.logits_torch(cfg, DEV)
    idx = torch.empty((n, k), dtype=torch.int32, device=DEV)
    w = torch.empty((n, k), dtype=torch.float32, device=DEV)
    heap.route_topk(lg, idx, w)
    heap.dispatch(x, idx, w, dedup=dedup)
    torch.cuda.synchronize()
    assert heap.status() == 0
    return heap, idx, w, x


def _windows(heap, cfg):
    W = cfg["world"]
    out = []
    for d in range(W):
        t = int(heap.total_recv(d).item())
        out.append(dict(total=t, rx=heap.recv_x(d)[:t].clone(), rp=heap.recv_pair(d)[:t].clone(),
                        rw=heap.recv_w(d)[:t].clone(), pos=heap.pos(d).clone(), cnt=heap.cnt(d).clone(),
                        off=heap.recv_off(d).clone(), ready=heap.ready(d).clone()))
    return out


# the deduplicated dispatch takes up to 32 slots (one ballot bit per slot)
CASES = {name: cfg for name, cfg in SMALL.items() if cfg["world"] <= 32}
CASES["deepseek_small"] = dict(ms.CONFIGS["deepseek"], tokens_per_slot=64)


def test_dedup_refuses_more_than_32_slots(sm):
    cfg = SMALL["slots64"]
    assert cfg["world"] > 32
    n, k = cfg["world"] * cfg["tokens_per_slot"], cfg["topk"]
    heap = sm.SymHeap(cfg, DEV)
    x = ms.x_torch(cfg, DEV)
    idx = torch.zeros((n, k), dtype=torch.int32, device=DEV)
    idx[:, 1] = 1
    w = torch.full((n, k), 0.5, dtype=torch.float32, device=DEV)
    with pytest.raises(sm.SymmoeError) as err:
        heap.dispatch(x, idx, w, dedup=True)
    assert err.value.code == sm.SYM_EINVAL
    torch.cuda.synchronize()
    assert heap.status() == 0


@pytest.mark.parametrize("name", list(CASES))
def test_dedup_matches_plain_and_oracle(sm, name):
    cfg = CASES[name]
    E, W, k = cfg["num_experts"], cfg["world"], cfg["topk"]
    plain, idx, w, x = _dispatch(sm, cfg, False)
    a = _windows(plain, cfg)
    dd, idx2, _, _ = _dispatch(sm, cfg, True)
    assert torch.equal(idx, idx2)
    b = _windows(dd, cfg)
    for d in range(W):
        for key in a[d]:
            if key == "total":
                assert a[d][key] == b[d][key]
            else:
                assert torch.equal(a[d][key], b[d][key]), (name, d, key)
    # staging rows and row sources against the oracle
    # the oracle's own routing of the same logits (the launch's must equal it)
    idx_h, w_h = checked_oracle_routing(cfg, idx, w)
    toks = oracle.dedup_tokens(idx_h, E, W)
    pos, _, _ = oracle.place_pairs(idx_h, w_h, E, W)
    src = oracle.dedup_row_source(idx_h, E, W, pos)
    x_h = ms.x_np(cfg)
    for d in range(W):
        nt = len(toks[d])
        assert np.array_equal(bits(dd.y(d)[:nt]), x_h[toks[d]]), (name, d)
        rs = dd.h(d).view(-1).view(torch.int32)[:b[d]["total"]].cpu().numpy()
        assert np.array_equal(rs, src[d]), (name, d)
    # fewer rows crossed than pairs whenever a token has two experts on one slot
    assert sum(len(t) for t in toks) <= idx_h.size


@pytest.mark.parametrize("name", ["mixtral", "deepseek"])
def test_dedup_full_size_windows_identical(sm, name):
    cfg = ms.CONFIGS[name]
    plain, idx, w, x = _dispatch(sm, cfg, False)
    a = _windows(plain, cfg)
    del plain
    torch.cuda.empty_cache()
    dd, idx2, _, _ = _dispatch(sm, cfg, True)
    assert torch.equal(idx, idx2)
    b = _windows(dd, cfg)
    for d in range(cfg["world"]):
        for key in a[d]:
            if key != "total":
                assert torch.equal(a[d][key], b[d][key]), (name, d, key)


def test_dedup_pipeline_output_identical(sm):
    """dispatch (deduplicated) -> expert FFN -> combine gives the plain path's
    output bit for bit."""
    cfg = CASES["ragged"]
    n, H = cfg["world"] * cfg["tokens_per_slot"], cfg["hidden"]
    wg, wu, wd = ms.weights_torch(cfg, DEV)
    outs = []
    for dedup in (False, True):
        heap, idx, w, x = _dispatch(sm, cfg, dedup)
        out = torch.empty((n, H), dtype=torch.bfloat16, device=DEV)
        heap.expert_ffn(wg, wu, wd)
        heap.combine(idx, w, out)
        torch.cuda.synchronize()
        assert heap.status() == 0
        outs.append(out)
    assert torch.equal(outs[0], outs[1])
