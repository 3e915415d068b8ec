"""Edge cases of the CUDA path against the oracle, staged and fused: every pair
on two experts (all others empty), the largest E and k the ABI accepts, a
single expert, token counts that are not multiples of any tile or chunk."""
import numpy as np
import pytest
import torch

import moe_synth as ms
import oracle
from _cases import assert_close, bf16_f64, bits, device_inputs, fresh_weight_fn

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def sm():
    import combine_symmetric_heap_gb300 as m
    return m


def _oracle_from_idx(cfg, idx, w, wfn):
    """The oracle's dispatch -> expert -> combine for a given routing."""
    E, W, k = cfg["num_experts"], cfg["world"], cfg["topk"]
    cnt, off, tot = oracle.count_experts(idx, E, W)
    pos, rp, rw = oracle.place_pairs(idx, w, E, W)
    rx = oracle.dispatch_rows(ms.x_np(cfg), rp, k)
    h, y, ye = oracle.expert_ffn(rx, cnt, off, E, W, wfn)
    out = oracle.combine(y, idx, w, pos, E, W)
    return dict(cnt=cnt, off=off, tot=tot, pos=pos, rx=rx, y=y, y_exact=ye, out=out)


# routing weights: fp32 expf on the GPU against the fp64 oracle
W_TOL = 2e-6


def _check_fused_routing(lg_np, idx_out, w_out, idx_expected, k):
    """The fused launch's routing of ``lg_np`` against the oracle's routing of
    the same logits: indices bit-exact, weights within W_TOL.  Returns the
    oracle's weights (never the launch's)."""
    idx_o, w_o = oracle.route_topk(lg_np, k)
    assert np.array_equal(idx_o, np.asarray(idx_expected)), "oracle routing differs from the intended indices"
    assert np.array_equal(idx_out.cpu().numpy(), idx_o.astype(np.int32)), "fused routing indices"
    werr = np.abs(w_out.cpu().numpy().astype(np.float64) - w_o.astype(np.float64)).max()
    assert werr <= W_TOL, f"fused routing weights: max error {werr}"
    return w_o


def _run(sm, cfg, idx_np, w_np, fused):
    logits, x, wg, wu, wd = device_inputs(cfg, DEV)
    n, k = cfg["world"] * cfg["tokens_per_slot"], cfg["topk"]
    heap = sm.SymHeap(cfg, DEV)
    idx = torch.from_numpy(idx_np.astype(np.int32)).to(DEV)
    w = torch.from_numpy(w_np.astype(np.float32)).to(DEV)
    out = torch.empty((n, cfg["hidden"]), dtype=torch.bfloat16, device=DEV)
    if fused:
        # the fused launch routes from logits itself: feed logits that select idx
        lg = torch.full((n, cfg["num_experts"]), -30.0, dtype=torch.float32)
        for j in range(k):
            lg[torch.arange(n), torch.from_numpy(idx_np[:, j]).long()] = 10.0 - j * 1e-3
        idx_out = torch.empty_like(idx)
        w_out = torch.empty_like(w)
        heap.pipeline(lg.to(DEV), x, wg, wu, wd, idx_out, w_out, out, fused=1)
        torch.cuda.synchronize()
        # the oracle routes the same logits: its indices and weights are the
        # reference for the launch's own routing and feed the oracle's combine
        return heap, out, _check_fused_routing(lg.numpy(), idx_out, w_out, idx_np, k)
    heap.dispatch(x, idx, w)
    heap.expert_ffn(wg, wu, wd)
    heap.combine(idx, w, out)
    torch.cuda.synchronize()
    return heap, out, w_np


@pytest.mark.parametrize("fused", [0, 1])
def test_all_pairs_on_two_experts(sm, fused):
    cfg = dict(world=4, tokens_per_slot=150, hidden=256, num_experts=8, topk=2, inter=256)
    n = 600
    idx = np.tile(np.array([[0, 1]]), (n, 1))
    idx[::2] = [1, 0]                                  # order within a token varies
    w = np.tile(np.array([[0.75, 0.25]], dtype=np.float32), (n, 1))
    heap, out, w_used = _run(sm, cfg, idx, w, fused)
    assert heap.status() == 0
    ref = _oracle_from_idx(cfg, idx, w_used, fresh_weight_fn(cfg, DEV))
    assert ref["cnt"].tolist() == [600, 600, 0, 0, 0, 0, 0, 0]
    assert np.array_equal(heap.pos(0).cpu().numpy(), ref["pos"][:150])
    assert_close(bits(out), bf16_f64(ref["out"]), "two-expert out")


@pytest.mark.parametrize("fused", [0, 1])
def test_max_experts_and_topk(sm, fused):
    cfg = dict(world=8, tokens_per_slot=40, hidden=128, num_experts=1024, topk=32, inter=128)
    n, k = 320, 32
    lg = ms.logits_np(cfg)
    idx, w = oracle.route_topk(lg, k)
    heap, out, w_used = _run(sm, cfg, idx, w, fused)
    assert heap.status() == 0
    ref = _oracle_from_idx(cfg, idx, w_used, fresh_weight_fn(cfg, DEV))
    assert_close(bits(out), bf16_f64(ref["out"]), "E=1024 k=32 out")


@pytest.mark.parametrize("fused", [0, 1])
def test_single_expert_ragged_tokens(sm, fused):
    cfg = dict(world=1, tokens_per_slot=333, hidden=384, num_experts=1, topk=1, inter=384)
    n = 333
    idx = np.zeros((n, 1), dtype=np.int64)
    w = np.ones((n, 1), dtype=np.float32)
    heap, out, w_used = _run(sm, cfg, idx, w, fused)
    assert heap.status() == 0
    ref = _oracle_from_idx(cfg, idx, w_used, fresh_weight_fn(cfg, DEV))
    t = int(ref["tot"][0])
    assert_close(bits(heap.y(0)[:t]), ref["y_exact"][0], "single expert y")
    assert_close(bits(out), bf16_f64(ref["out"]), "single expert out")


def test_ragged_world_and_tokens_through_pipeline(sm):
    cfg = dict(world=3, tokens_per_slot=100, hidden=256, num_experts=6, topk=2, inter=128)
    logits, x, wg, wu, wd = device_inputs(cfg, DEV)
    n = 300
    heap = sm.SymHeap(cfg, DEV)
    outs = []
    for fused in (0, 1, 0):
        idx = torch.empty((n, 2), dtype=torch.int32, device=DEV)
        w = torch.empty((n, 2), dtype=torch.float32, device=DEV)
        out = torch.empty((n, cfg["hidden"]), dtype=torch.bfloat16, device=DEV)
        heap.pipeline(logits, x, wg, wu, wd, idx, w, out, fused=fused)
        outs.append(out)
    torch.cuda.synchronize()
    assert heap.status() == 0
    assert all(torch.equal(o.view(torch.int16), outs[0].view(torch.int16)) for o in outs)
    ref = oracle.pipeline(ms.logits_np(cfg), ms.x_np(cfg), cfg, fresh_weight_fn(cfg, DEV))
    assert_close(bits(outs[0]), bf16_f64(ref["out"]), "W=3 T=100 out")


@pytest.mark.parametrize("fused", [0, 1])
def test_remainder_rows_on_last_tile(sm, fused):
    """Row counts around the token-tile boundary: 256 + r rows with r <= 32 put
    the remainder on the one full tile (second MMA of the same weight stream),
    r = 33 gets a tile of its own; 16, 512 + 20 and 256 + 1 rows cover one
    short tile, a remainder behind two full tiles (a tile of its own) and the
    smallest remainder."""
    counts = [260, 288, 289, 16, 532, 257]
    cfg = dict(world=2, tokens_per_slot=sum(counts) // 2, hidden=256, num_experts=6, topk=1, inter=384)
    idx = np.repeat(np.arange(len(counts)), counts).reshape(-1, 1)
    rng = np.random.default_rng(7)
    idx = idx[rng.permutation(len(idx))]              # experts interleaved over the tokens
    w = np.ones_like(idx, dtype=np.float32)
    heap, out, w_used = _run(sm, cfg, idx, w, fused)
    assert heap.status() == 0
    ref = _oracle_from_idx(cfg, idx, w_used, fresh_weight_fn(cfg, DEV))
    assert ref["cnt"].tolist() == counts
    for d in range(cfg["world"]):
        t = int(ref["tot"][d])
        assert_close(bits(heap.y(d)[:t]), ref["y_exact"][d], f"slot {d} y")
    assert_close(bits(out), bf16_f64(ref["out"]), "remainder tiles out")


@pytest.mark.parametrize("fused", [0, 1])
def test_wide_rows(sm, fused):
    """H = 16384: the staged scatter moves a row in two register passes and the
    fused scatter's rows no longer fit a warp's share of the ring (plain-copy
    path); the combine streams a row in many passes."""
    cfg = dict(world=2, tokens_per_slot=24, hidden=16384, num_experts=4, topk=2, inter=128)
    lg = ms.logits_np(cfg)
    idx, w = oracle.route_topk(lg, cfg["topk"])
    heap, out, w_used = _run(sm, cfg, idx, w, fused)
    assert heap.status() == 0
    ref = _oracle_from_idx(cfg, idx, w_used, fresh_weight_fn(cfg, DEV))
    for d in range(cfg["world"]):
        t = int(ref["tot"][d])
        assert np.array_equal(bits(heap.recv_x(d)[:t]), ref["rx"][d])   # dispatched rows, bit-exact
    assert_close(bits(out), bf16_f64(ref["out"]), "H=16384 out")


@pytest.mark.parametrize("fused", [0, 1])
def test_grouped_token_tiles(sm, fused):
    """Gate/up token tiles of a heavy expert run in groups whose rows fit a
    fixed L2 budget (48 MiB: 6 token tiles of 256 rows at H = 16384): 3000
    rows make 12 tiles in two groups of 6, 1700 rows make groups of 6 and 1,
    100 rows one short tile.  Every row's result must not depend on the order."""
    counts = [3000, 1700, 100]
    cfg = dict(world=1, tokens_per_slot=sum(counts), hidden=16384, num_experts=3, topk=1, inter=128)
    idx = np.repeat(np.arange(len(counts)), counts).reshape(-1, 1)
    idx = idx[np.random.default_rng(11).permutation(len(idx))]
    w = np.ones_like(idx, dtype=np.float32)
    heap, out, w_used = _run(sm, cfg, idx, w, fused)
    assert heap.status() == 0
    ref = _oracle_from_idx(cfg, idx, w_used, fresh_weight_fn(cfg, DEV))
    assert ref["cnt"].tolist() == counts
    t = int(ref["tot"][0])
    assert_close(bits(heap.y(0)[:t]), ref["y_exact"][0], "grouped tiles y")
    assert_close(bits(out), bf16_f64(ref["out"]), "grouped tiles out")


@pytest.mark.parametrize("fused", [0, 1])
def test_grouped_down_tiles(sm, fused):
    """Down token tiles of a heavy expert run in groups whose h rows fit a
    fixed L2 budget (64 MiB: 8 token tiles of 256 rows at I = 16384): 2600
    rows make 11 tiles (10 full, one of 40 rows) in groups of 8 and 3, and a
    second expert of 90 rows keeps one short tile."""
    counts = [2600, 90]
    cfg = dict(world=1, tokens_per_slot=sum(counts), hidden=128, num_experts=2, topk=1, inter=16384)
    idx = np.repeat(np.arange(len(counts)), counts).reshape(-1, 1)
    idx = idx[np.random.default_rng(13).permutation(len(idx))]
    w = np.ones_like(idx, dtype=np.float32)
    heap, out, w_used = _run(sm, cfg, idx, w, fused)
    assert heap.status() == 0
    ref = _oracle_from_idx(cfg, idx, w_used, fresh_weight_fn(cfg, DEV))
    assert ref["cnt"].tolist() == counts
    t = int(ref["tot"][0])
    assert_close(bits(heap.y(0)[:t]), ref["y_exact"][0], "grouped down tiles y")
    assert_close(bits(out), bf16_f64(ref["out"]), "grouped down tiles out")


@pytest.mark.parametrize("fused", [0, 1])
@pytest.mark.parametrize("hidden,inter", [(65536, 128), (128, 65536)])
def test_largest_hidden_and_inter(sm, fused, hidden, inter):
    """The ABI's largest H and I: a dispatched / combined row of 8192 16-byte
    vectors (several passes of every copy loop) and K loops of 1024 blocks in
    the gate/up (H) or down (I) GEMM.  At H = 65536 the gate/up weights are
    scaled by 2^-3 (exact in bf16; about the 1/sqrt(H) of a trained layer):
    with sigma = 0.02 the gate and up values reach |h| ~ 200, where one bf16
    step of h is 1.0, and the tensor cores' fp32 accumulation over 4096 MMAs
    (its additions truncate) moves 0.02% of y past the per-element tolerance;
    a truncating-accumulator model of the same inputs gives the same count."""
    cfg = dict(world=2, tokens_per_slot=40, hidden=hidden, num_experts=2, topk=1, inter=inter)
    scale = 2.0 ** -3 if hidden >= 65536 else 1.0
    n, k = cfg["world"] * cfg["tokens_per_slot"], cfg["topk"]
    lg = ms.logits_np(cfg)
    idx_np, w_np = oracle.route_topk(lg, k)
    heap = sm.SymHeap(cfg, DEV)
    x = ms.x_torch(cfg, DEV)
    wg, wu, wd = ms.weights_torch(cfg, DEV)
    wg.mul_(scale)
    wu.mul_(scale)
    idx = torch.from_numpy(idx_np.astype(np.int32)).to(DEV)
    w = torch.from_numpy(w_np.astype(np.float32)).to(DEV)
    out = torch.empty((n, hidden), dtype=torch.bfloat16, device=DEV)
    if fused:
        idx_out, w_out = torch.empty_like(idx), torch.empty_like(w)
        heap.pipeline(torch.from_numpy(lg).to(DEV), x, wg, wu, wd, idx_out, w_out, out, fused=1)
        torch.cuda.synchronize()
        w_np = _check_fused_routing(lg, idx_out, w_out, idx_np, k)   # the oracle's own weights
    else:
        heap.dispatch(x, idx, w)
        heap.expert_ffn(wg, wu, wd)
        heap.combine(idx, w, out)
    torch.cuda.synchronize()
    assert heap.status() == 0
    base = fresh_weight_fn(cfg, DEV)

    def scaled(e):
        g, u, dn = base(e)
        sc = lambda b: oracle.round_f64_to_bf16_bits(oracle.bf16_bits_to_f64(b) * scale)
        return sc(g), sc(u), dn
    ref = _oracle_from_idx(cfg, idx_np, w_np, scaled)
    for d in range(cfg["world"]):
        t = int(ref["tot"][d])
        assert np.array_equal(bits(heap.recv_x(d)[:t]), ref["rx"][d])
        assert_close(bits(heap.y(d)[:t]), ref["y_exact"][d], f"H={hidden} I={inter} slot {d} y")
    assert_close(bits(out), bf16_f64(ref["out"]), f"H={hidden} I={inter} out")
