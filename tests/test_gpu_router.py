"""The router (gate) GEMM on the GPU against the oracle: fp32 logits within a
tolerance derived from fp32 accumulation (bf16 products are exact in fp32; an
H-term fp32 sum is off by at most about sqrt(H) ulps of its partial sums), and
the routing taken from the launch's logits against the oracle's routing of
the oracle's own logits: the same experts in the same order wherever the
largest k+1 logits are further apart than the logit tolerance, valid top-k
choices everywhere."""
import numpy as np
import pytest
import torch

import moe_synth as ms
import oracle
from _cases import SMALL

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def sm():
    import combine_symmetric_heap_gb300 as m
    return m


def _check_logits(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    diff = np.abs(got - ref)
    assert np.all(diff <= 1e-3 * np.maximum(1.0, np.abs(ref))), f"{what}: max diff {diff.max()}"
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert rel <= 1e-4, f"{what}: relative L2 {rel}"


def _check_routing(gi, ref, k, what):
    """Routing of the launch's logits (gi) against the oracle's routing of the
    oracle's logits (ref): logits differ within the logit tolerance, so the
    order is unique only where the largest k+1 oracle logits are further
    apart than twice that tolerance; there the experts and their order must
    be the oracle's.  Everywhere the picks must be k distinct experts whose
    oracle logits lie within the tolerance of the oracle's k largest."""
    ri, _ = oracle.route_topk(ref, k)
    ref = np.asarray(ref, dtype=np.float64)
    top = -np.sort(-ref, axis=1)[:, :k + 1]
    tol = 1e-3 * np.maximum(1.0, np.abs(top))
    # (with k = E there are only k values: their order is what must be clear)
    clear = np.all(top[:, :-1] - top[:, 1:] > 2 * (tol[:, :-1] + tol[:, 1:]), axis=1)
    assert clear.mean() >= 0.5, f"{what}: only {clear.mean():.2f} of the tokens have a unique top-k"
    assert np.array_equal(gi[clear], ri[clear]), f"{what}: routing differs where the top-k is unique"
    assert all(len(set(r.tolist())) == k for r in gi), f"{what}: repeated experts"
    chosen = np.take_along_axis(ref, gi.astype(np.int64), axis=1)
    assert np.all(np.abs(chosen - top[:, :k]) <= 2 * tol[:, :k] + 1e-12), f"{what}: a pick outside the top k"


def _run(sm, cfg):
    n = cfg["world"] * cfg["tokens_per_slot"]
    heap = sm.SymHeap(cfg, DEV)
    x = ms.x_torch(cfg, DEV)
    wr = ms.router_weight_torch(cfg, DEV)
    logits = torch.full((n, cfg["num_experts"]), float("nan"), dtype=torch.float32, device=DEV)
    heap.router_logits(x, wr, logits)
    torch.cuda.synchronize()
    assert heap.status() == 0
    return heap, logits


CASES = dict(SMALL)
CASES["wide_e"] = dict(world=3, tokens_per_slot=90, hidden=256, num_experts=300, topk=4, inter=128)
CASES["remainder"] = dict(world=2, tokens_per_slot=135, hidden=384, num_experts=8, topk=2, inter=128)
# few tiles and a long K: K is split across pairs (5 splits of 6, 6, 6, 6, 2 blocks on 152 SMs),
# two feature tiles and a ragged token tile
CASES["split_wide"] = dict(world=2, tokens_per_slot=300, hidden=1664, num_experts=300, topk=4, inter=128)
# 18 splits of 3 blocks with a last split of one block; a token tail of 8 rows
CASES["split_tail"] = dict(world=1, tokens_per_slot=520, hidden=3328, num_experts=24, topk=2, inter=128)


@pytest.mark.parametrize("name", list(CASES))
def test_router_small(sm, name):
    cfg = CASES[name]
    heap, logits = _run(sm, cfg)
    if name.startswith("split_"):
        assert heap.router_splits() > 1, "the case is meant to split K"
    ref = oracle.router_logits(ms.x_np(cfg), ms.router_weight_np(cfg))
    got = logits.cpu().numpy()
    _check_logits(got, ref, name)
    k = cfg["topk"]
    n = got.shape[0]
    idx = torch.empty((n, k), dtype=torch.int32, device=DEV)
    w = torch.empty((n, k), dtype=torch.float32, device=DEV)
    heap.route_topk(logits, idx, w)
    _check_routing(idx.cpu().numpy(), ref, k, name)


# on 152 SMs: one GEMM writing the logits; 2 K splits; 14 K splits of 8 blocks
@pytest.mark.parametrize("name,rows", [("mixtral", 256), ("deepseek", 128), ("decode", 128)])
def test_router_full_size_sampled(sm, name, rows):
    cfg = ms.CONFIGS[name]
    heap, logits = _run(sm, cfg)
    n = cfg["world"] * cfg["tokens_per_slot"]
    pick = np.sort(np.random.default_rng(2).choice(n, size=rows, replace=False))
    ref = oracle.router_logits(ms.x_np(cfg, rows=pick), ms.router_weight_np(cfg))
    _check_logits(logits[torch.from_numpy(pick).to(DEV)].cpu().numpy(), ref, name)
    assert torch.isfinite(logits).all()


def test_router_split_leaves_heap_usable(sm):
    """The K-split partials live in slot 0's y window before dispatch: a full
    dispatch -> expert -> combine after the router still matches the staged
    result taken without the router."""
    cfg = CASES["split_wide"]
    heap, logits = _run(sm, cfg)
    n, k, H = cfg["world"] * cfg["tokens_per_slot"], cfg["topk"], cfg["hidden"]
    x = ms.x_torch(cfg, DEV)
    wg, wu, wd = ms.weights_torch(cfg, DEV)
    idx = torch.empty((n, k), dtype=torch.int32, device=DEV)
    w = torch.empty((n, k), dtype=torch.float32, device=DEV)
    out1 = torch.empty((n, H), dtype=torch.bfloat16, device=DEV)
    heap.pipeline(logits, x, wg, wu, wd, idx, w, out1)
    fresh = sm.SymHeap(cfg, DEV)
    out2 = torch.empty_like(out1)
    fresh.pipeline(logits, x, wg, wu, wd, idx, w, out2)
    torch.cuda.synchronize()
    assert heap.status() == 0 and fresh.status() == 0
    assert torch.equal(out1, out2)

