"""Repeated full-size steps on one heap give the same output bit for bit.

The tile schedule is dynamic (pairs claim tiles in whatever order they free
up), the dispatch places rows through atomics on ready counters, and the fused
launch claims route, scatter, GEMM and combine work from counters.  None of
that may change a result: the receive order is fixed by (expert, source slot,
token), each output element is one tile's accumulation over K in a fixed
order, and the combine adds the k expert outputs of a token in j order.  So a
step repeated on the same inputs must reproduce its output exactly, whatever
the schedule of each launch; a race between roles (a tile read before its
inputs landed, a stale queue entry) would show up as a differing step."""
import pytest
import torch

import moe_synth as ms

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = "cuda"
REPS = 4

CASES = [("mixtral", {}), ("mixtral", {"fused": 1}), ("skewed", {}), ("skewed", {"fused": 1}),
         ("deepseek", {}), ("deepseek", {"fused": 1}), ("deepseek", {"dedup": True}),
         ("deepseek", {"fp8": True}), ("deepseek", {"fused": 1, "weights_in_ffn": True}),
         ("decode", {}), ("decode", {"fused": 1})]


@pytest.fixture(scope="module")
def sm():
    import combine_symmetric_heap_gb300 as m
    return m


@pytest.fixture(scope="module")
def weights():
    cache = {}

    def get(cfg):
        key = (cfg["num_experts"], cfg["hidden"], cfg["inter"])
        if key not in cache:
            cache.clear()
            torch.cuda.empty_cache()
            cache[key] = ms.weights_torch(cfg, DEV)
        return cache[key]
    yield get
    cache.clear()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name,mode", CASES, ids=[n + "-" + ("-".join(f"{a}" for a in m) or "staged")
                                                  for n, m in CASES])
def test_repeated_steps_bit_identical(sm, weights, name, mode):
    cfg = ms.CONFIGS[name]
    n, k, H = cfg["world"] * cfg["tokens_per_slot"], cfg["topk"], cfg["hidden"]
    wg, wu, wd = weights(cfg)
    heap = sm.SymHeap(cfg, DEV)
    logits, x = ms.logits_torch(cfg, DEV), ms.x_torch(cfg, DEV)
    idx = torch.empty((n, k), dtype=torch.int32, device=DEV)
    w = torch.empty((n, k), dtype=torch.float32, device=DEV)
    out = torch.empty((n, H), dtype=torch.bfloat16, device=DEV)
    heap.pipeline(logits, x, wg, wu, wd, idx, w, out, **mode)
    torch.cuda.synchronize()
    assert heap.status() == 0
    first_out, first_idx, first_w = out.clone(), idx.clone(), w.clone()
    for step in range(REPS):
        out.fill_(0)
        idx.fill_(-1)
        w.fill_(0)
        heap.pipeline(logits, x, wg, wu, wd, idx, w, out, **mode)
        torch.cuda.synchronize()
        assert heap.status() == 0, f"step {step}"
        assert torch.equal(idx, first_idx), f"step {step}: routing"
        assert torch.equal(w.view(torch.int32), first_w.view(torch.int32)), f"step {step}: weights"
        assert torch.equal(out.view(torch.int16), first_out.view(torch.int16)), f"step {step}: output"
    del heap
    torch.cuda.empty_cache()
