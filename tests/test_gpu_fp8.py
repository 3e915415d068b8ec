"""The FP8 dispatch on the GPU: E4M3 codes and per-token scales bit-exact
against the oracle (including rounding ties, subnormals and -0), the
dequantized receive rows bit-exact, the other windows identical to the bf16
dispatch, and the pipeline's output within the path's tolerance of the oracle
run on the dequantized rows."""
import numpy as np
import pytest
import torch

import moe_synth as ms
import oracle
from _cases import SMALL, assert_close, bits, bf16_f64, checked_oracle_routing, fresh_weight_fn

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def sm():
    import combine_symmetric_heap_gb300 as m
    return m


def _dispatch(sm, cfg, x, fp8, idx=None):
    n, k = cfg["world"] * cfg["tokens_per_slot"], cfg["topk"]
    heap = sm.SymHeap(cfg, DEV)
    w = torch.empty((n, k), dtype=torch.float32, device=DEV)
    if idx is None:
        idx = torch.empty((n, k), dtype=torch.int32, device=DEV)
        heap.route_topk(ms.logits_torch(cfg, DEV), idx, w)
    else:
        w.fill_(1.0 / k)
    heap.dispatch(x, idx, w, fp8=fp8)
    torch.cuda.synchronize()
    assert heap.status() == 0
    return heap, idx, w


def _check_slots(heap, cfg, idx_h, x_bits):
    """codes, scales and dequantized rows of every received row vs the oracle;
    idx_h: the routing as the test or the oracle made it (host array)"""
    E, W, k, H = cfg["num_experts"], cfg["world"], cfg["topk"], cfg["hidden"]
    pos, rp, _ = oracle.place_pairs(idx_h, np.ones(idx_h.shape, np.float32), E, W)
    codes, exps = oracle.quantize_rows_e4m3(x_bits)
    deq = oracle.dequantize_rows(codes, exps)
    for d in range(W):
        t = len(rp[d])
        g = rp[d] // k
        got_codes = heap.y(d).view(-1).view(torch.uint8)[:t * H].view(t, H).cpu().numpy()
        assert np.array_equal(got_codes, codes[g]), f"slot {d} codes"
        sc = heap.h(d).view(-1).view(torch.float32)[:t].cpu().numpy().astype(np.float64)
        assert np.array_equal(sc, np.exp2(exps[g].astype(np.float64))), f"slot {d} scales"
        assert np.array_equal(bits(heap.recv_x(d)[:t]), deq[g]), f"slot {d} rows"


@pytest.mark.parametrize("name", list(SMALL))
def test_fp8_dispatch_small(sm, name):
    cfg = SMALL[name]
    x = ms.x_torch(cfg, DEV)
    heap, idx, w = _dispatch(sm, cfg, x, True)
    _check_slots(heap, cfg, checked_oracle_routing(cfg, idx, w)[0], ms.x_np(cfg))
    plain, _, _ = _dispatch(sm, cfg, x, False)
    for d in range(cfg["world"]):
        t = int(plain.total_recv(d).item())
        assert int(heap.total_recv(d).item()) == t
        assert torch.equal(heap.recv_pair(d)[:t], plain.recv_pair(d)[:t])
        assert torch.equal(heap.recv_w(d)[:t], plain.recv_w(d)[:t])
        assert torch.equal(heap.pos(d), plain.pos(d))
        assert torch.equal(heap.ready(d), plain.ready(d))


def test_fp8_rounding_edges(sm):
    """Rows built from bf16 values on and between E4M3 steps: every tie, the
    subnormal range, values that round to zero (both signs), and amax values
    that pin the scale at 2^0, 2^5 and 2^-7."""
    cfg = dict(world=1, tokens_per_slot=6, hidden=1024, num_experts=1, topk=1, inter=128)
    table = np.array([oracle.e4m3_decode(c) for c in range(0x7F)])
    mids = (table[:-1] + table[1:]) / 2
    cand = np.concatenate([table, mids, mids * (1 + 2.0 ** -7), mids * (1 - 2.0 ** -7),
                           [2.0 ** -10, 2.0 ** -11, 3 * 2.0 ** -11]])
    cand_bits = oracle.round_f64_to_bf16_bits(cand)
    cand = oracle.bf16_bits_to_f64(cand_bits)
    rng = np.random.default_rng(8)
    rows = []
    for r, scale in enumerate([1.0, 32.0, 2.0 ** -7, 1.0, 32.0, 2.0 ** -7]):
        v = rng.choice(cand, size=1024) * rng.choice([-1.0, 1.0], size=1024)
        v[0] = 448.0                      # amax -> scale exactly `scale`
        rows.append(v * scale)
    xb = oracle.round_f64_to_bf16_bits(np.array(rows))
    x = torch.from_numpy(xb.view(np.int16)).to(DEV).view(torch.bfloat16)
    idx_h = np.zeros((6, 1), dtype=np.int32)
    heap, _, _ = _dispatch(sm, cfg, x, True, idx=torch.from_numpy(idx_h).to(DEV))
    _check_slots(heap, cfg, idx_h, xb)


def test_fp8_pipeline_matches_oracle_on_dequantized_rows(sm):
    cfg = SMALL["ragged"]
    n, k, H = cfg["world"] * cfg["tokens_per_slot"], cfg["topk"], cfg["hidden"]
    heap = sm.SymHeap(cfg, DEV)
    logits = ms.logits_torch(cfg, DEV)
    x = ms.x_torch(cfg, DEV)
    wg, wu, wd = ms.weights_torch(cfg, DEV)
    idx = torch.empty((n, k), dtype=torch.int32, device=DEV)
    w = torch.empty((n, k), dtype=torch.float32, device=DEV)
    out = torch.empty((n, H), dtype=torch.bfloat16, device=DEV)
    heap.pipeline(logits, x, wg, wu, wd, idx, w, out, fp8=True)
    torch.cuda.synchronize()
    assert heap.status() == 0
    codes, exps = oracle.quantize_rows_e4m3(ms.x_np(cfg))
    xq = oracle.dequantize_rows(codes, exps)
    ref = oracle.pipeline(ms.logits_np(cfg), xq, cfg, fresh_weight_fn(cfg, DEV))
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    assert_close(bits(out), bf16_f64(ref["out"]), "fp8 pipeline out")


@pytest.mark.parametrize("name", ["deepseek"])
def test_fp8_dispatch_full_size_sampled(sm, name):
    cfg = ms.CONFIGS[name]
    E, W, k, H = cfg["num_experts"], cfg["world"], cfg["topk"], cfg["hidden"]
    x = ms.x_torch(cfg, DEV)
    heap, idx, w = _dispatch(sm, cfg, x, True)
    idx_h, _ = checked_oracle_routing(cfg, idx, w)
    pos = np.stack([heap.pos(d).cpu().numpy().reshape(-1, k) for d in range(W)]).reshape(-1, k)
    rng = np.random.default_rng(12)
    toks = np.sort(rng.choice(idx_h.shape[0], size=24, replace=False))
    codes, exps = oracle.quantize_rows_e4m3(ms.x_np(cfg, rows=toks))
    deq = oracle.dequantize_rows(codes, exps)
    for i, g in enumerate(toks):
        for j in range(k):
            d = int(idx_h[g, j]) // (E // W)
            p = int(pos[g, j])
            assert np.array_equal(bits(heap.recv_x(d)[p]), deq[i]), (g, j)


def test_fp8_and_dedup_with_weights_in_ffn(sm):
    """The dispatch variants combine with the weights-in-epilogue variant in
    the staged pipeline: deduplicated gives the plain dispatch's output bit
    for bit; FP8 matches the oracle's weights-in-epilogue path on the
    dequantized rows."""
    cfg = SMALL["many"]
    n, k, H = cfg["world"] * cfg["tokens_per_slot"], cfg["topk"], cfg["hidden"]
    logits = ms.logits_torch(cfg, DEV)
    x = ms.x_torch(cfg, DEV)
    wg, wu, wd = ms.weights_torch(cfg, DEV)
    outs = {}
    for name, kw in [("plain", {}), ("dedup", {"dedup": True}), ("fp8", {"fp8": True})]:
        heap = sm.SymHeap(cfg, DEV)
        idx = torch.empty((n, k), dtype=torch.int32, device=DEV)
        w = torch.empty((n, k), dtype=torch.float32, device=DEV)
        out = torch.empty((n, H), dtype=torch.bfloat16, device=DEV)
        heap.pipeline(logits, x, wg, wu, wd, idx, w, out, weights_in_ffn=True, **kw)
        torch.cuda.synchronize()
        assert heap.status() == 0
        outs[name] = out
    assert torch.equal(outs["plain"], outs["dedup"])
    codes, exps = oracle.quantize_rows_e4m3(ms.x_np(cfg))
    ref = oracle.pipeline(ms.logits_np(cfg), oracle.dequantize_rows(codes, exps), cfg,
                          fresh_weight_fn(cfg, DEV), weights_in_ffn=True)
    assert_close(bits(outs["fp8"]), bf16_f64(ref["out"]), "fp8 + weights in the epilogue")
