"""The fused single-launch pipeline (moe_pipeline fused=1) against the
stage-by-stage launches and the oracle: same routing, layout and rows
bit-exact, identical bf16 outputs (same tile arithmetic), oracle tolerance,
and repeated launches on one heap (the kernel resets its own counters)."""
import numpy as np
import pytest
import torch

import moe_synth as ms
import oracle
from _cases import SMALL, assert_close, bf16_f64, bits, device_inputs, fresh_weight_fn, host_weight_fn

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def sm():
    import combine_symmetric_heap_gb300 as m
    return m


def _run(sm, cfg, inputs, fused, heap=None, reps=1):
    logits, x, wg, wu, wd = inputs
    n, k = cfg["world"] * cfg["tokens_per_slot"], cfg["topk"]
    heap = heap or sm.SymHeap(cfg, DEV)
    idx = torch.empty((n, k), dtype=torch.int32, device=DEV)
    w = torch.empty((n, k), dtype=torch.float32, device=DEV)
    outs = []
    for _ in range(reps):
        out = torch.full((n, cfg["hidden"]), float("nan"), dtype=torch.bfloat16, device=DEV)
        heap.pipeline(logits, x, wg, wu, wd, idx, w, out, fused=fused)
        outs.append(out)
    torch.cuda.synchronize()
    return heap, idx, w, outs


def _layout(heap, cfg):
    W = cfg["world"]
    return [torch.cat([heap.cnt(d) for d in range(W)]).cpu(),
            torch.cat([heap.recv_off(d) for d in range(W)]).cpu(),
            torch.cat([heap.total_recv(d) for d in range(W)]).cpu(),
            torch.cat([heap.pos(d) for d in range(W)]).cpu()]


@pytest.mark.parametrize("name", list(SMALL))
def test_fused_matches_unfused_and_oracle(sm, name):
    cfg = SMALL[name]
    inputs = device_inputs(cfg, DEV)
    hu, iu, wu_, ou = _run(sm, cfg, inputs, 0)
    hf, i_f, wf, of = _run(sm, cfg, inputs, 1, reps=3)
    assert hf.status() == 0 and hu.status() == 0
    assert torch.equal(i_f, iu) and torch.equal(wf.view(torch.int32), wu_.view(torch.int32))
    for a, b in zip(_layout(hf, cfg), _layout(hu, cfg)):
        assert torch.equal(a, b)
    for d in range(cfg["world"]):
        t = int(hu.total_recv(d).item())
        assert torch.equal(hf.recv_x(d)[:t].view(torch.int16), hu.recv_x(d)[:t].view(torch.int16))
        assert torch.equal(hf.recv_pair(d)[:t], hu.recv_pair(d)[:t])
        assert torch.equal(hf.h(d)[:t].view(torch.int16), hu.h(d)[:t].view(torch.int16))
        assert torch.equal(hf.y(d)[:t].view(torch.int16), hu.y(d)[:t].view(torch.int16))
    for o in of:                                   # three launches in a row
        assert torch.equal(o.view(torch.int16), ou[0].view(torch.int16))
    ref = oracle.pipeline(ms.logits_np(cfg), ms.x_np(cfg), cfg, host_weight_fn(cfg))
    assert np.array_equal(i_f.cpu().numpy(), ref["idx"])
    assert_close(bits(of[0]), bf16_f64(ref["out"]), f"{name} fused out")


def test_fused_and_unfused_share_a_heap(sm):
    cfg = SMALL["ragged"]
    inputs = device_inputs(cfg, DEV)
    heap, _, _, o1 = _run(sm, cfg, inputs, 1)
    _, _, _, o2 = _run(sm, cfg, inputs, 0, heap=heap)
    _, _, _, o3 = _run(sm, cfg, inputs, 1, heap=heap)
    assert heap.status() == 0
    assert torch.equal(o1[0].view(torch.int16), o2[0].view(torch.int16))
    assert torch.equal(o1[0].view(torch.int16), o3[0].view(torch.int16))


@pytest.mark.slow
@pytest.mark.parametrize("name", ["decode", "deepseek", "skewed", "mixtral"])
def test_fused_full_size(sm, name):
    """The workloads' full shapes: fused == unfused bit for bit, plus sampled
    tokens against the oracle."""
    cfg = ms.CONFIGS[name]
    inputs = device_inputs(cfg, DEV)
    hu, iu, _, ou = _run(sm, cfg, inputs, 0)
    del hu
    torch.cuda.empty_cache()
    hf, i_f, _, of = _run(sm, cfg, inputs, 1, reps=2)
    assert hf.status() == 0
    assert torch.equal(i_f, iu)
    for o in of:
        assert torch.equal(o.view(torch.int16), ou[0].view(torch.int16))
    if name == "decode":
        k = cfg["topk"]
        ridx, rw = oracle.route_topk(ms.logits_np(cfg), k)
        assert np.array_equal(i_f.cpu().numpy(), ridx)
        wfn = fresh_weight_fn(cfg, DEV)
        for g in (0, 517):
            acc = np.zeros(cfg["hidden"])
            for j in range(k):
                _, yb, _ = oracle.expert_ffn_rows(ms.x_np(cfg, rows=[g]), *wfn(int(ridx[g, j])))
                acc += float(rw[g, j]) * bf16_f64(yb[0])
            assert_close(bits(of[0][g]), bf16_f64(oracle.round_f64_to_bf16_bits(acc)), f"decode token {g}")
