"""Parity of the CUDA path (through the C ABI) with the CPU oracle on the same
seeded inputs: bit-exact routing indices, counts, offsets, receive rows and
dispatched rows; bf16 outputs within the stated float tolerance."""
import numpy as np
import pytest
import torch

import moe_synth as ms
import oracle
from _cases import (SMALL, W_TOL, assert_close, bf16_f64, bits, checked_oracle_routing, device_inputs,
                    fresh_weight_fn, host_weight_fn, run_gpu_stages)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sm():
    import combine_symmetric_heap_gb300 as m
    return m


DEV = "cuda"


# ----------------------------------------------------------------- inputs

def test_device_generator_matches_host():
    cfg = ms.CONFIGS["deepseek"]
    x = ms.x_torch(cfg, DEV)
    rows = np.array([0, 4095, 8191])
    assert np.array_equal(bits(x[torch.tensor(rows, device=DEV)]), ms.x_np(cfg, rows=rows))
    lg = ms.logits_torch(ms.CONFIGS["skewed"], DEV)
    assert np.array_equal(lg[:64].cpu().numpy(), ms.logits_np(ms.CONFIGS["skewed"], rows=np.arange(64)))
    wg, _, wd = ms.weights_torch(ms.CONFIGS["tiny"], DEV)
    assert np.array_equal(bits(wg[3]), ms.weight_np(ms.CONFIGS["tiny"], "gate", 3))
    assert np.array_equal(bits(wd[1]), ms.weight_np(ms.CONFIGS["tiny"], "down", 1))
    # a full-size expert generated on the device equals the host definition
    big = ms.CONFIGS["deepseek"]
    wexp = ms.weight_expert_torch(big, "up", 201, DEV)
    per = big["inter"] * big["hidden"]
    sel = np.arange(0, per, 997)
    host = ms.normal_bf16_np(0, ms.STREAM_WU, 201 * per + sel, ms.W_SIGMA)
    assert np.array_equal(bits(wexp).reshape(-1)[sel], host)


# ----------------------------------------------------------------- a1 route

@pytest.mark.parametrize("name", ["tiny", "mixtral", "deepseek", "skewed", "decode"])
def test_route_parity(sm, name):
    cfg = ms.CONFIGS[name]
    n, k = cfg["world"] * cfg["tokens_per_slot"], cfg["topk"]
    lg = ms.logits_torch(cfg, DEV)
    idx = torch.empty((n, k), dtype=torch.int32, device=DEV)
    w = torch.empty((n, k), dtype=torch.float32, device=DEV)
    small = dict(cfg, hidden=128, inter=128)  # routing does not touch H/I windows
    heap = sm.SymHeap(small, DEV)
    heap.route_topk(lg, idx, w)
    torch.cuda.synchronize()
    ridx, rw = oracle.route_topk(ms.logits_np(cfg), k)  # the generator's host copy of the same logits
    assert np.array_equal(idx.cpu().numpy(), ridx)
    assert np.max(np.abs(w.cpu().numpy().astype(np.float64) - rw)) <= 2e-6


@pytest.mark.parametrize("e,k", [(8, 2), (256, 8), (64, 5), (33, 3), (1024, 32)])
def test_route_ties_and_odd_expert_counts(sm, e, k):
    world = 1
    cfg = dict(world=world, tokens_per_slot=1000, hidden=128, inter=128, num_experts=e, topk=k)
    g = torch.Generator().manual_seed(e + k)
    lg = (torch.round(torch.randn(1000, e, generator=g) * 2) / 2).to(torch.float32)
    lg[0] = 0.25                                   # a token with all-equal logits
    heap = sm.SymHeap(cfg, DEV)
    idx = torch.empty((1000, k), dtype=torch.int32, device=DEV)
    w = torch.empty((1000, k), dtype=torch.float32, device=DEV)
    heap.route_topk(lg.to(DEV), idx, w)
    torch.cuda.synchronize()
    ridx, rw = oracle.route_topk(lg.numpy(), k)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    assert np.max(np.abs(w.cpu().numpy().astype(np.float64) - rw)) <= 2e-6
    assert np.all(w[0].cpu().numpy() == np.float32(1.0 / k))


# ----------------------------------------------------------------- a2/a3 dispatch

def _check_dispatch(sm, cfg, heap, idx, w, x_dev, sample_rows=None):
    """Layout bit-exact against the oracle; rows checked fully (small) or by
    property + samples (large)."""
    W, E, k = cfg["world"], cfg["num_experts"], cfg["topk"]
    e_loc = E // W
    T = cfg["tokens_per_slot"]
    # the oracle's own routing of the same logits; the launch's must equal it
    idx_h, w_h = checked_oracle_routing(cfg, idx, w)
    w_gpu = w.cpu().numpy().reshape(-1)
    cnt, off, tot = oracle.count_experts(idx_h, E, W)
    pos, rp, rw = oracle.place_pairs(idx_h, w_h, E, W)
    g_cnt = np.concatenate([heap.cnt(d).cpu().numpy() for d in range(W)])
    g_off = np.concatenate([heap.recv_off(d).cpu().numpy() for d in range(W)])
    g_tot = np.array([int(heap.total_recv(d).item()) for d in range(W)])
    assert np.array_equal(g_cnt, cnt)
    assert np.array_equal(g_off, off)
    assert np.array_equal(g_tot, tot)
    g_pos = np.concatenate([heap.pos(d).cpu().numpy() for d in range(W)])
    assert np.array_equal(g_pos, pos)
    for d in range(W):
        t = int(tot[d])
        assert np.array_equal(heap.recv_pair(d)[:t].cpu().numpy(), rp[d])
        # each row's weight is a bit copy of its pair's routing weight
        assert np.array_equal(heap.recv_w(d)[:t].cpu().numpy(), w_gpu[rp[d]])
        assert np.abs(heap.recv_w(d)[:t].cpu().numpy().astype(np.float64) - rw[d]).max(initial=0.0) <= W_TOL
        # every received row is a bit copy of its source token (any size)
        src = torch.from_numpy(rp[d] // k).to(DEV)
        assert torch.equal(heap.recv_x(d)[:t].view(torch.int16), x_dev[src].view(torch.int16))
        # ready counters: rows landed per 128-row block
        rd = heap.ready(d).cpu().numpy()
        nb = (t + 127) // 128
        exp = np.array([min(128, t - 128 * b) for b in range(nb)])
        assert np.array_equal(rd[:nb], exp)
    if sample_rows is not None:  # rows against host-generated x
        rng = np.random.default_rng(1)
        for d in rng.choice(W, size=min(W, 3), replace=False):
            t = int(tot[d])
            if t == 0:
                continue
            ps = rng.choice(t, size=min(t, sample_rows), replace=False)
            gsrc = rp[d][ps] // k
            assert np.array_equal(bits(heap.recv_x(int(d))[torch.from_numpy(ps).to(DEV)]),
                                  ms.x_np(cfg, rows=gsrc))
    return cnt, off, tot, pos, rp


@pytest.mark.parametrize("name", list(SMALL))
def test_dispatch_small(sm, name):
    cfg = SMALL[name]
    logits, x, wg, wu, wd = device_inputs(cfg, DEV)
    heap, idx, w, out = run_gpu_stages(sm, cfg, logits, x, wg, wu, wd)
    assert heap.status() == 0
    _check_dispatch(sm, cfg, heap, idx, w, x, sample_rows=16)


@pytest.mark.parametrize("name", ["mixtral", "deepseek", "skewed", "decode"])
def test_dispatch_full_size(sm, name):
    cfg = ms.CONFIGS[name]
    n, k = cfg["world"] * cfg["tokens_per_slot"], cfg["topk"]
    small = dict(cfg)
    heap = sm.SymHeap(small, DEV)
    logits = ms.logits_torch(cfg, DEV)
    x = ms.x_torch(cfg, DEV)
    idx = torch.empty((n, k), dtype=torch.int32, device=DEV)
    w = torch.empty((n, k), dtype=torch.float32, device=DEV)
    heap.route_topk(logits, idx, w)
    heap.dispatch(x, idx, w)
    torch.cuda.synchronize()
    assert heap.status() == 0
    _check_dispatch(sm, cfg, heap, idx, w, x, sample_rows=8)


def test_dispatch_bad_indices_flag_overflow(sm):
    cfg = SMALL["tiny"]
    n, k = 128, 2
    heap = sm.SymHeap(cfg, DEV)
    x = ms.x_torch(cfg, DEV)
    idx = torch.tensor([[0, 1]] * n, dtype=torch.int32, device=DEV)
    idx[5, 1] = 99                     # expert out of range
    idx[7] = torch.tensor([2, 2])      # duplicate expert in one token
    w = torch.full((n, k), 0.5, dtype=torch.float32, device=DEV)
    heap.dispatch(x, idx, w)
    torch.cuda.synchronize()
    assert heap.status(clear=True) & sm.SYM_STATUS_OVERFLOW
    assert heap.status() == 0
    assert int(heap.pos(0)[5, 1].item()) == -1


# ----------------------------------------------------------------- a4/a5 expert FFN

@pytest.mark.parametrize("name", list(SMALL))
def test_expert_ffn_small(sm, name):
    cfg = SMALL[name]
    W, E = cfg["world"], cfg["num_experts"]
    logits, x, wg, wu, wd = device_inputs(cfg, DEV)
    heap, idx, w, out = run_gpu_stages(sm, cfg, logits, x, wg, wu, wd)
    assert heap.status() == 0
    ref = oracle.pipeline(ms.logits_np(cfg), ms.x_np(cfg), cfg, host_weight_fn(cfg))
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    for d in range(W):
        t = int(ref["total_recv"][d])
        if t == 0:
            continue
        assert_close(bits(heap.h(d)[:t]), bf16_f64(ref["h"][d]), f"{name} h slot {d}")
        assert_close(bits(heap.y(d)[:t]), ref["y_exact"][d], f"{name} y slot {d}")
    assert_close(bits(out), bf16_f64(ref["out"]), f"{name} out")


def _integer_case(world, tokens, hidden, inter, experts, k):
    """One-hot tokens and small-integer weights: every product and sum is an
    exact small integer, so h, y and out have closed forms (bit-exact)."""
    n = world * tokens
    x = np.zeros((n, hidden), dtype=np.float32)
    col = [(5 * g + 3) % hidden for g in range(n)]
    for g in range(n):
        x[g, col[g]] = 1.0
    wg = np.zeros((experts, inter, hidden), dtype=np.float32)
    wu = np.zeros_like(wg)
    wd = np.zeros((experts, hidden, inter), dtype=np.float32)
    ii, cc = np.meshgrid(np.arange(inter), np.arange(hidden), indexing="ij")
    for e in range(experts):
        wg[e] = 32 + (ii + 2 * cc + e) % 5
        wu[e] = ((ii * 7 + cc + 3 * e) % 5) - 2
        for o in range(hidden):
            wd[e, o, (5 * o + 3 + e) % inter] = 1.0 if (o + e) % 3 else -1.0
    rng = np.random.default_rng(11)
    idx = np.stack([rng.choice(experts, size=k, replace=False) for _ in range(n)]).astype(np.int32)
    w = np.full((n, k), 1.0 / k, dtype=np.float32)
    # closed forms
    y_tok = np.zeros((n, k, hidden))
    for g in range(n):
        c = col[g]
        for j in range(k):
            e = idx[g, j]
            hvec = wg[e][:, c] * wu[e][:, c]          # silu(gate) == gate for gate >= 32
            y_tok[g, j] = wd[e] @ hvec
    out = (y_tok * (1.0 / k)).sum(1)
    return x, wg, wu, wd, idx, w, y_tok, out


@pytest.mark.parametrize("shape", [(2, 64, 128, 256, 4, 2), (2, 150, 256, 128, 8, 2),
                                   (1, 700, 128, 128, 2, 2)])
def test_expert_ffn_integer_bit_exact(sm, shape):
    world, tokens, hidden, inter, experts, k = shape
    cfg = dict(world=world, tokens_per_slot=tokens, hidden=hidden, inter=inter,
               num_experts=experts, topk=k)
    x, wg, wu, wd, idx, w, y_tok, out_ref = _integer_case(*shape)
    tb = lambda a: torch.from_numpy(a).to(DEV).to(torch.bfloat16).contiguous()
    heap, _, _, out = run_gpu_stages(sm, cfg, None, tb(x), tb(wg), tb(wu), tb(wd),
                                     idx=torch.from_numpy(idx).to(DEV), w=torch.from_numpy(w).to(DEV))
    assert heap.status() == 0
    e_loc = experts // world
    for g in range(world * tokens):
        for j in range(k):
            d = int(idx[g, j]) // e_loc
            p = int(heap.pos(g // tokens)[g % tokens, j].item())
            assert np.array_equal(bf16_f64(bits(heap.y(d)[p])), y_tok[g, j]), (g, j)
    assert np.array_equal(bf16_f64(bits(out)), out_ref)


def test_expert_ffn_zero_up_is_zero(sm):
    cfg = SMALL["ragged"]
    logits, x, wg, wu, wd = device_inputs(cfg, DEV)
    heap, idx, w, out = run_gpu_stages(sm, cfg, logits, x, wg, torch.zeros_like(wu), wd)
    for d in range(cfg["world"]):
        t = int(heap.total_recv(d).item())
        assert torch.count_nonzero(heap.y(d)[:t].float()) == 0
    assert torch.count_nonzero(out.float()) == 0


# ----------------------------------------------------------------- a6 combine

def test_combine_zero_copy_and_fallback(sm):
    cfg = SMALL["ragged"]
    logits, x, wg, wu, wd = device_inputs(cfg, DEV)
    heap, idx, w, out = run_gpu_stages(sm, cfg, logits, x, wg, wu, wd)
    before = sm.moe_combine_fallback_copies()
    out_view = torch.empty_like(out)
    heap.combine(idx, w, out_view, expert_out=heap.combine_in_view())   # data_ptr match
    torch.cuda.synchronize()
    assert sm.moe_combine_fallback_copies() == before
    assert torch.equal(out_view.view(torch.int16), out.view(torch.int16))
    # a caller-allocated expert output: silent staging copy, identical result
    mine = torch.stack([heap.y(d).clone() for d in range(cfg["world"])])
    for d in range(cfg["world"]):
        heap.y(d).zero_()
    out_copy = torch.empty_like(out)
    heap.combine(idx, w, out_copy, expert_out=mine)
    torch.cuda.synchronize()
    assert sm.moe_combine_fallback_copies() == before + 1
    assert torch.equal(out_copy.view(torch.int16), out.view(torch.int16))


def test_combine_of_oracle_y(sm):
    cfg = SMALL["many"]
    ref = oracle.pipeline(ms.logits_np(cfg), ms.x_np(cfg), cfg, host_weight_fn(cfg))
    logits, x, wg, wu, wd = device_inputs(cfg, DEV)
    heap, idx, w, _ = run_gpu_stages(sm, cfg, logits, x, wg, wu, wd)
    for d in range(cfg["world"]):
        t = int(ref["total_recv"][d])
        heap.y(d)[:t].view(torch.int16).copy_(torch.from_numpy(ref["y"][d].view(np.int16)))
    out = torch.empty((cfg["world"] * cfg["tokens_per_slot"], cfg["hidden"]), dtype=torch.bfloat16,
                      device=DEV)
    heap.combine(idx, w, out)
    torch.cuda.synchronize()
    got = bf16_f64(bits(out))
    exp = bf16_f64(ref["out"])
    ulp = np.maximum(np.abs(exp), 1e-30)
    ulp = 2.0 ** (np.floor(np.log2(ulp)) - 7)
    assert np.all(np.abs(got - exp) <= ulp)


# ----------------------------------------------------------------- whole path

@pytest.mark.parametrize("name", list(SMALL))
def test_pipeline_call_matches_oracle_and_repeats(sm, name):
    cfg = SMALL[name]
    n, k = cfg["world"] * cfg["tokens_per_slot"], cfg["topk"]
    logits, x, wg, wu, wd = device_inputs(cfg, DEV)
    heap = sm.SymHeap(cfg, DEV)
    idx = torch.empty((n, k), dtype=torch.int32, device=DEV)
    w = torch.empty((n, k), dtype=torch.float32, device=DEV)
    outs = []
    for _ in range(2):
        out = torch.empty((n, cfg["hidden"]), dtype=torch.bfloat16, device=DEV)
        heap.pipeline(logits, x, wg, wu, wd, idx, w, out, fused=0)
        outs.append(out)
    torch.cuda.synchronize()
    assert heap.status() == 0 and heap.desc.epoch == 2
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    ref = oracle.pipeline(ms.logits_np(cfg), ms.x_np(cfg), cfg, host_weight_fn(cfg))
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    assert_close(bits(outs[0]), bf16_f64(ref["out"]), f"{name} pipeline out")


def _sample_tokens(idx_h, n_tok, max_experts, rng):
    """Tokens whose experts together stay within max_experts (bounds oracle cost)."""
    chosen, experts = [], set()
    for g in rng.permutation(idx_h.shape[0]):
        es = set(idx_h[g].tolist())
        if len(experts | es) <= max_experts:
            chosen.append(int(g))
            experts |= es
        if len(chosen) == n_tok:
            break
    return chosen


@pytest.mark.slow
@pytest.mark.parametrize("name,ntok,maxe", [("mixtral", 8, 4), ("deepseek", 4, 24),
                                            ("skewed", 6, 24), ("decode", 4, 24)])
def test_pipeline_full_size_sampled(sm, name, ntok, maxe):
    """The benchmark's workload and launch sequence; sampled tokens recomputed
    one by one by the oracle from host-generated inputs."""
    cfg = ms.CONFIGS[name]
    n, k = cfg["world"] * cfg["tokens_per_slot"], cfg["topk"]
    logits, x, wg, wu, wd = device_inputs(cfg, DEV)
    heap = sm.SymHeap(cfg, DEV)
    idx = torch.empty((n, k), dtype=torch.int32, device=DEV)
    w = torch.empty((n, k), dtype=torch.float32, device=DEV)
    out = torch.empty((n, cfg["hidden"]), dtype=torch.bfloat16, device=DEV)
    heap.pipeline(logits, x, wg, wu, wd, idx, w, out, fused=0)
    torch.cuda.synchronize()
    assert heap.status() == 0
    del wg, wu, wd
    torch.cuda.empty_cache()
    lg_h = ms.logits_np(cfg)
    ridx, rw = oracle.route_topk(lg_h, k)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    toks = _sample_tokens(ridx, ntok, maxe, np.random.default_rng(5))
    assert toks
    wfn = fresh_weight_fn(cfg, DEV)
    xs = ms.x_np(cfg, rows=np.array(toks))
    for i, g in enumerate(toks):
        acc = np.zeros(cfg["hidden"])
        for j in range(k):
            _, yb, _ = oracle.expert_ffn_rows(xs[i:i + 1], *wfn(int(ridx[g, j])))
            acc += float(rw[g, j]) * bf16_f64(yb[0])
        ref_out = oracle.round_f64_to_bf16_bits(acc)
        assert_close(bits(out[g]), bf16_f64(ref_out), f"{name} token {g}")


def _full_size_run(sm, name):
    """The full workload through the staged pipeline; returns the heap and the
    oracle's routing of the same logits (bit-exact against the launch's)."""
    cfg = ms.CONFIGS[name]
    n, k = cfg["world"] * cfg["tokens_per_slot"], cfg["topk"]
    logits, x, wg, wu, wd = device_inputs(cfg, DEV)
    heap = sm.SymHeap(cfg, DEV)
    idx = torch.empty((n, k), dtype=torch.int32, device=DEV)
    w = torch.empty((n, k), dtype=torch.float32, device=DEV)
    out = torch.empty((n, cfg["hidden"]), dtype=torch.bfloat16, device=DEV)
    heap.pipeline(logits, x, wg, wu, wd, idx, w, out, fused=0)
    torch.cuda.synchronize()
    assert heap.status() == 0
    del wg, wu, wd, x
    torch.cuda.empty_cache()
    ridx, _ = oracle.route_topk(ms.logits_np(cfg), k)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    return cfg, heap, ridx


def _expert_every_element(cfg, heap, ridx, e, what):
    """Every h and y element of expert e against the oracle, its received
    rows bit-exact."""
    E, W = cfg["num_experts"], cfg["world"]
    cnt, off, _ = oracle.count_experts(ridx, E, W)
    d, o, c = e // (E // W), int(off[e]), int(cnt[e])
    tokens = np.nonzero((ridx == e).any(axis=1))[0]   # its rows, in receive order
    assert len(tokens) == c
    rows = bits(ms.x_torch(cfg, DEV)[torch.from_numpy(tokens).to(DEV)])
    assert np.array_equal(bits(heap.recv_x(d)[o:o + c]), rows)
    h_bits, _, y_exact = oracle.expert_ffn_rows(rows, *fresh_weight_fn(cfg, DEV)(e))
    assert_close(bits(heap.h(d)[o:o + c]), bf16_f64(h_bits), f"{what}: expert {e} h ({c} rows)")
    assert_close(bits(heap.y(d)[o:o + c]), y_exact, f"{what}: expert {e} y ({c} rows)")
    return c


@pytest.mark.slow
def test_skewed_heaviest_expert_every_element(sm):
    """The full Skewed workload (Zipf-biased routing): every h and y element of
    its heaviest expert (thousands of rows: many token tiles, gate/up token
    groups, a ragged last tile) against the oracle, and its received rows
    bit-exact."""
    cfg, heap, ridx = _full_size_run(sm, "skewed")
    cnt, _, _ = oracle.count_experts(ridx, cfg["num_experts"], cfg["world"])
    assert _expert_every_element(cfg, heap, ridx, int(np.argmax(cnt)), "skewed") > 8 * 256


@pytest.mark.slow
@pytest.mark.parametrize("name", ["mixtral", "deepseek", "decode"])
def test_full_size_experts_every_element(sm, name):
    """Every h and y element of chosen experts of the full workloads against the
    oracle: Mixtral-like's last expert (~4096 rows: 16 token tiles, the down
    tiles in two groups); DeepSeek-like's largest expert with 257..288 rows (the
    remainder on its one tile as a second MMA) and its largest with at most 256;
    Decode's largest expert (a few dozen rows, one short tile)."""
    cfg, heap, ridx = _full_size_run(sm, name)
    E = cfg["num_experts"]
    cnt, _, _ = oracle.count_experts(ridx, E, cfg["world"])
    if name == "mixtral":
        chosen = [E - 1]
    elif name == "deepseek":
        fold = [e for e in range(E) if 256 < cnt[e] <= 288]
        plain = [e for e in range(E) if 0 < cnt[e] <= 256]
        assert fold and plain
        chosen = [max(fold, key=lambda e: cnt[e]), max(plain, key=lambda e: cnt[e])]
    else:
        chosen = [int(np.argmax(cnt))]
    for e in chosen:
        _expert_every_element(cfg, heap, ridx, e, name)


# ----------------------------------------------------------------- bounded waits

def test_ready_counter_timeout_returns_with_status(sm):
    """A ready counter that no producer will complete: the expert kernel gives
    up after the heap's wait limit, flags SYM_STATUS_TIMEOUT and returns; the
    context stays usable."""
    cfg = SMALL["ragged"]
    logits, x, wg, wu, wd = device_inputs(cfg, DEV)
    heap, idx, w, out_ok = run_gpu_stages(sm, cfg, logits, x, wg, wu, wd)
    assert heap.status() == 0
    heap.dispatch(x, idx, w)
    torch.cuda.synchronize()
    heap.ready(0)[0] = 0                       # row block 0 of slot 0 never lands
    heap.desc.wait_timeout_us = 20000          # 20 ms
    heap.expert_ffn(wg, wu, wd)
    torch.cuda.synchronize()
    assert heap.status(clear=True) & sm.SYM_STATUS_TIMEOUT
    heap.desc.wait_timeout_us = 2_000_000
    _, _, _, out = run_gpu_stages(sm, cfg, logits, x, wg, wu, wd, heap=heap, idx=idx, w=w)
    assert heap.status() == 0
    assert torch.equal(out.view(torch.int16), out_ok.view(torch.int16))


@pytest.mark.parametrize("name", ["tiny", "ragged", "allk", "multi"])
def test_weights_in_ffn_variant(sm, name):
    """Routing weights applied in the down epilogue (recv_w) and an unweighted
    combine, staged and fused, against the oracle variant; staged and fused
    agree bit for bit."""
    cfg = SMALL[name]
    logits, x, wg, wu, wd = device_inputs(cfg, DEV)
    n, k, H = cfg["world"] * cfg["tokens_per_slot"], cfg["topk"], cfg["hidden"]
    ref = oracle.pipeline(ms.logits_np(cfg), ms.x_np(cfg), cfg, fresh_weight_fn(cfg, DEV), weights_in_ffn=True)
    runs = []
    for fused in (0, 1):
        heap = sm.SymHeap(cfg, DEV)
        idx = torch.empty((n, k), dtype=torch.int32, device=DEV)
        w = torch.empty((n, k), dtype=torch.float32, device=DEV)
        out = torch.full((n, H), float("nan"), dtype=torch.bfloat16, device=DEV)
        heap.pipeline(logits, x, wg, wu, wd, idx, w, out, fused=fused, weights_in_ffn=True)
        torch.cuda.synchronize()
        assert heap.status() == 0
        for d in range(cfg["world"]):
            t = int(ref["total_recv"][d])
            assert_close(bits(heap.y(d)[:t]), bf16_f64(ref["y"][d]), f"{name} weighted y slot {d}")
        assert_close(bits(out), bf16_f64(ref["out"]), f"{name} fused={fused} out")
        runs.append((heap, out))
    (hs, os_), (hf, of) = runs
    assert torch.equal(os_.view(torch.int16), of.view(torch.int16))
    for d in range(cfg["world"]):
        t = int(ref["total_recv"][d])
        assert torch.equal(hs.y(d)[:t].view(torch.int16), hf.y(d)[:t].view(torch.int16))


def test_weights_in_ffn_staged_calls(sm):
    """The _ex calls one by one equal the pipeline mode, and an unweighted
    combine of unweighted rows is the plain sum of the expert rows."""
    cfg = SMALL["ragged"]
    logits, x, wg, wu, wd = device_inputs(cfg, DEV)
    n, k, H = cfg["world"] * cfg["tokens_per_slot"], cfg["topk"], cfg["hidden"]
    heap = sm.SymHeap(cfg, DEV)
    idx = torch.empty((n, k), dtype=torch.int32, device=DEV)
    w = torch.empty((n, k), dtype=torch.float32, device=DEV)
    a = torch.empty((n, H), dtype=torch.bfloat16, device=DEV)
    b = torch.empty_like(a)
    heap.pipeline(logits, x, wg, wu, wd, idx, w, a, weights_in_ffn=True)
    heap.route_topk(logits, idx, w)
    heap.dispatch(x, idx, w)
    heap.expert_ffn(wg, wu, wd, weighted_rows=True)
    heap.combine(idx, None, b, unweighted=True)        # w not read
    torch.cuda.synchronize()
    assert heap.status() == 0
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    ref = oracle.pipeline(ms.logits_np(cfg), ms.x_np(cfg), cfg, fresh_weight_fn(cfg, DEV))
    heap.expert_ffn(wg, wu, wd)                          # plain rows again
    heap.combine(idx, None, b, unweighted=True)
    torch.cuda.synchronize()
    plain = oracle.combine_sum(ref["y"], ref["idx"], ref["pos"], cfg["num_experts"], cfg["world"])
    assert_close(bits(b), bf16_f64(plain), "unweighted combine of plain rows")
