"""Pins of the CPU oracle against things other than itself: brute force on tiny
inputs, closed forms, invariants, a hand-worked example (tests/golden/) and
an independent library implementation (torch CPU) of the expert FFN."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import moe_synth as ms

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------- bf16 helpers

def test_bf16_round_trip_and_ties():
    assert oracle.bf16_bits_to_f64(np.array([0x3F80]))[0] == 1.0
    assert oracle.bf16_bits_to_f64(np.array([0x4049]))[0] == 3.140625
    assert oracle.bf16_bits_to_f64(np.array([0xC000]))[0] == -2.0
    v = np.array([1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, -2.0, 3.390625, 1 + 2 ** -8 + 2 ** -20,
                  1 + 2 ** -8 + 2 ** -30])
    got = oracle.round_f64_to_bf16_bits(v).tolist()
    # 1+2^-8 is half-way between 0x3F80 and 0x3F81: ties to even -> 0x3F80;
    # 1+3*2^-8 is half-way between 0x3F81 and 0x3F82 -> 0x3F82; just above the
    # first tie (by an fp32-representable 2^-20) it rounds up -> 0x3F81.  The
    # stated rounding goes through fp32 (as an fp32 accumulator does), so an
    # excess of 2^-30, below half an fp32 ulp, is lost first and the tie rule
    # applies -> 0x3F80.
    assert got == [0x3F80, 0x3F80, 0x3F82, 0xC000, 0x4059, 0x3F81, 0x3F80]


# --------------------------------------------------------------- address

def test_peer_address_golden():
    g = _golden("peer_address.json")
    for c in g["cases"]:
        stride = c["stride4G"] << 32
        got = oracle.slot_address(int(c["win_base"], 16), c["peer"], stride, int(c["offset"], 16))
        assert got == int(c["expect"], 16)


# --------------------------------------------------------------- routing

def _brute_topk(lg, k):
    n, e = lg.shape
    out = np.zeros((n, k), dtype=np.int64)
    for g in range(n):
        for a in range(e):
            rank = sum(1 for b in range(e) if lg[g, b] > lg[g, a] or (lg[g, b] == lg[g, a] and b < a))
            if rank < k:
                out[g, rank] = a
    return out


@pytest.mark.parametrize("e,k", [(4, 2), (8, 2), (16, 8), (16, 1), (9, 3)])
def test_route_brute_force_with_ties(e, k):
    rng = np.random.default_rng(e * 10 + k)
    # coarse quantisation makes ties frequent
    lg = (np.round(rng.standard_normal((64, e)) * 2) / 2).astype(np.float32)
    idx, w = oracle.route_topk(lg, k)
    assert np.array_equal(idx, _brute_topk(lg, k))
    for g in range(64):
        sel = [float(lg[g, i]) for i in idx[g]]
        for j in range(k):
            ref = 1.0 / sum(math.exp(s - sel[j]) for s in sel)
            assert abs(float(w[g, j]) - ref) <= 1e-6 * max(1.0, ref)
    assert np.all(np.abs(w.astype(np.float64).sum(1) - 1.0) <= 1e-6)
    assert all(len(set(r)) == k for r in idx.tolist())


@pytest.mark.parametrize("k", [1, 2, 4, 8])
def test_route_all_equal(k):
    lg = np.full((5, 16), 0.25, dtype=np.float32)
    idx, w = oracle.route_topk(lg, k)
    assert np.array_equal(idx, np.tile(np.arange(k), (5, 1)))
    assert np.all(w == np.float32(1.0 / k))


def test_route_k1_weight_is_one():
    lg = ms.logits_np(ms.CONFIGS["tiny"])
    idx, w = oracle.route_topk(lg, 1)
    assert np.all(w == 1.0)
    assert np.array_equal(idx[:, 0], np.argmax(lg, axis=1))


def test_route_hand_golden():
    g = _golden("dispatch_hand.json")
    idx, w = oracle.route_topk(np.array(g["logits"], dtype=np.float32), g["topk"])
    assert idx.tolist() == g["idx"]
    assert np.allclose(w, np.array(g["w"]), rtol=0, atol=1e-7)


# --------------------------------------------------------------- count / place

def test_place_hand_golden():
    g = _golden("dispatch_hand.json")
    idx = np.array(g["idx"])
    w = np.array(g["w"], dtype=np.float32)
    cnt, off, tot = oracle.count_experts(idx, g["num_experts"], g["world"])
    assert cnt.tolist() == g["cnt"] and off.tolist() == g["recv_off"] and tot.tolist() == g["total_recv"]
    pos, rp, rw = oracle.place_pairs(idx, w, g["num_experts"], g["world"])
    assert pos.tolist() == g["pos"]
    assert [r.tolist() for r in rp] == g["recv_pair"]
    assert rw[1][0] == w[0, 1] and rw[0][0] == w[1, 0]


def _random_routing(n, e, k, seed):
    rng = np.random.default_rng(seed)
    lg = rng.standard_normal((n, e)).astype(np.float32)
    return oracle.route_topk(lg, k)


@pytest.mark.parametrize("n,e,w,k", [(40, 8, 2, 2), (33, 16, 4, 3), (24, 4, 4, 1), (30, 12, 3, 4)])
def test_place_brute_force_and_invariants(n, e, w, k):
    idx, wt = _random_routing(n, e, k, n + e)
    cnt, off, tot = oracle.count_experts(idx, e, w)
    e_loc = e // w
    assert cnt.sum() == n * k
    for d in range(w):
        local = cnt[d * e_loc:(d + 1) * e_loc]
        assert np.array_equal(off[d * e_loc:(d + 1) * e_loc], np.concatenate([[0], np.cumsum(local)[:-1]]))
        assert tot[d] == local.sum()
    pos, rp, _ = oracle.place_pairs(idx, wt, e, w)
    flat = idx.reshape(-1)
    for p in range(n * k):
        ex = int(flat[p])
        before = int(np.sum(flat[:p] == ex))        # O(P^2) independent count
        assert pos.reshape(-1)[p] == off[ex] + before
    # bijection: every row [0, total_recv[d]) of every slot is hit exactly once
    seen = [np.zeros(int(tot[d]), dtype=np.int64) for d in range(w)]
    for g in range(n):
        for j in range(k):
            d = int(idx[g, j]) // e_loc
            seen[d][pos[g, j]] += 1
            assert rp[d][pos[g, j]] == g * k + j
    assert all(np.all(s == 1) for s in seen)


def test_place_receive_order_is_slot_token_k():
    # tokens 0..T-1 live on slot 0, T..2T-1 on slot 1; inside one expert the
    # received rows must be ordered by (source slot, token, k)
    idx, wt = _random_routing(64, 4, 2, 7)
    pos, rp, _ = oracle.place_pairs(idx, wt, 4, 2)
    cnt, off, _ = oracle.count_experts(idx, 4, 2)
    for e in range(4):
        d = e // 2
        pairs = rp[d][off[e]:off[e] + cnt[e]]
        assert np.all(np.diff(pairs) > 0)


def test_dispatch_rows_are_bit_copies():
    cfg = ms.CONFIGS["tiny"]
    x = ms.x_np(cfg)
    idx, w = oracle.route_topk(ms.logits_np(cfg), cfg["topk"])
    pos, rp, _ = oracle.place_pairs(idx, w, cfg["num_experts"], cfg["world"])
    rx = oracle.dispatch_rows(x, rp, cfg["topk"])
    e_loc = cfg["num_experts"] // cfg["world"]
    for g in range(x.shape[0]):
        for j in range(cfg["topk"]):
            assert np.array_equal(rx[int(idx[g, j]) // e_loc][pos[g, j]], x[g])


# --------------------------------------------------------------- FFN

def _bits(a):
    return ms.f32_to_bf16_bits_np(np.asarray(a, dtype=np.float32))


def test_ffn_zero_up_gives_zero():
    rng = np.random.default_rng(1)
    a = _bits(rng.standard_normal((5, 16)))
    wg = _bits(rng.standard_normal((8, 16)) * 0.1)
    wu = np.zeros((8, 16), dtype=np.uint16)
    wd = _bits(rng.standard_normal((16, 8)) * 0.1)
    h, y, ye = oracle.expert_ffn_rows(a, wg, wu, wd)
    assert np.all(oracle.bf16_bits_to_f64(h) == 0) and np.all(oracle.bf16_bits_to_f64(y) == 0)


def integer_ffn_case(rows, hidden, inter):
    """One-hot rows, small-integer weights with gate >= 32 so that silu(gate)
    equals gate after rounding to fp32; every product and sum is an exact
    small integer, so h and y have closed forms."""
    a = np.zeros((rows, hidden), dtype=np.float32)
    col = [(3 * r + 1) % hidden for r in range(rows)]
    for r in range(rows):
        a[r, col[r]] = 1.0
    wg = np.zeros((inter, hidden), dtype=np.float32)
    wu = np.zeros((inter, hidden), dtype=np.float32)
    for i in range(inter):
        for c in range(hidden):
            wg[i, c] = 32 + (i + 2 * c) % 5
            wu[i, c] = ((i * 7 + c) % 5) - 2
    wd = np.zeros((hidden, inter), dtype=np.float32)
    for o in range(hidden):
        wd[o, (5 * o + 3) % inter] = 1.0
        wd[o, (o + 1) % inter] = -1.0 if (o + 1) % inter != (5 * o + 3) % inter else 0.0
    h = np.zeros((rows, inter))
    for r in range(rows):
        c = col[r]
        for i in range(inter):
            h[r, i] = (32 + (i + 2 * c) % 5) * (((i * 7 + c) % 5) - 2)
    y = np.zeros((rows, hidden))
    for r in range(rows):
        for o in range(hidden):
            y[r, o] = sum(h[r, i] * wd[o, i] for i in range(inter) if wd[o, i] != 0)
    return _bits(a), _bits(wg), _bits(wu), _bits(wd), h, y


def test_ffn_integer_closed_form():
    a, wg, wu, wd, h_ref, y_ref = integer_ffn_case(6, 24, 40)
    h, y, ye = oracle.expert_ffn_rows(a, wg, wu, wd)
    assert np.array_equal(oracle.bf16_bits_to_f64(h), h_ref)
    assert np.array_equal(oracle.bf16_bits_to_f64(y), y_ref)


def test_ffn_matches_torch_cpu_fp32():
    cfg = ms.CONFIGS["tiny"]
    x = ms.x_np(cfg)[:40]
    wg, wu, wd = (ms.weight_np(cfg, n, 1) for n in ("gate", "up", "down"))
    h, y, ye = oracle.expert_ffn_rows(x, wg, wu, wd)
    t = lambda b: torch.from_numpy(oracle.bf16_bits_to_f64(b).astype(np.float32))
    ht = torch.nn.functional.silu(t(x) @ t(wg).T) * (t(x) @ t(wu).T)
    yt = ht @ t(wd).T
    assert torch.allclose(torch.from_numpy(oracle.bf16_bits_to_f64(h)).float(), ht, rtol=1e-2, atol=1e-3)
    rel = np.linalg.norm(ye - yt.double().numpy()) / np.linalg.norm(yt.double().numpy())
    assert rel < 1e-2
    # a transposed or swapped operand would be far off
    bad = (torch.nn.functional.silu(t(x) @ t(wu).T) * (t(x) @ t(wg).T)) @ t(wd).T
    assert np.linalg.norm(ye - bad.double().numpy()) / np.linalg.norm(bad.double().numpy()) > 0.1


# --------------------------------------------------------------- combine

def test_combine_hand_golden():
    g = _golden("dispatch_hand.json")
    y = [_bits(np.array(v, dtype=np.float32)) for v in g["y"]]
    out = oracle.combine(y, np.array(g["idx"]), np.array(g["w"], dtype=np.float32),
                         np.array(g["pos"]), g["num_experts"], g["world"])
    assert oracle.bf16_bits_to_f64(out).tolist() == g["out"]


def test_combine_k1_is_the_row():
    rng = np.random.default_rng(3)
    idx, w = _random_routing(20, 4, 1, 5)
    pos, rp, _ = oracle.place_pairs(idx, w, 4, 2)
    _, _, tot = oracle.count_experts(idx, 4, 2)
    y = [_bits(rng.standard_normal((int(tot[d]), 8))) for d in range(2)]
    out = oracle.combine(y, idx, w, pos, 4, 2)
    for g in range(20):
        assert np.array_equal(out[g], y[int(idx[g, 0]) // 2][pos[g, 0]])


# --------------------------------------------------------------- whole path

def test_pipeline_tiny_consistency():
    cfg = ms.CONFIGS["tiny"]
    res = oracle.pipeline(ms.logits_np(cfg), ms.x_np(cfg), cfg,
                          lambda e: tuple(ms.weight_np(cfg, n, e) for n in ("gate", "up", "down")))
    n, k = cfg["world"] * cfg["tokens_per_slot"], cfg["topk"]
    assert res["cnt"].sum() == n * k
    assert res["out"].shape == (n, cfg["hidden"])
    # out equals the weighted sum of per-token FFN rows computed token by token
    for g in (0, 17, 127):
        acc = np.zeros(cfg["hidden"])
        for j in range(k):
            e = int(res["idx"][g, j])
            wts = tuple(ms.weight_np(cfg, nm, e) for nm in ("gate", "up", "down"))
            _, yb, _ = oracle.expert_ffn_rows(ms.x_np(cfg, rows=[g]), *wts)
            acc += float(res["w"][g, j]) * oracle.bf16_bits_to_f64(yb[0])
        assert np.array_equal(res["out"][g], oracle.round_f64_to_bf16_bits(acc))


# ------------------------------------------ variant: weights in the expert epilogue

def test_scale_rows_rounds_once():
    # 3 * (1 + 3*2^-9) = 3.017578125 -> bf16 3.015625.  Weighting the already
    # rounded y (1.0078125) instead would give 3.0234375 -> 3.03125 (tie to even).
    ye = [np.array([[1.0 + 3 * 2.0 ** -9, -2.0]])]
    yw = oracle.scale_rows(ye, [np.array([3.0], dtype=np.float32)])
    assert oracle.bf16_bits_to_f64(yw[0]).tolist() == [[3.015625, -6.0]]
    late = oracle.round_f64_to_bf16_bits(3.0 * oracle.bf16_bits_to_f64(oracle.round_f64_to_bf16_bits(ye[0])))
    assert oracle.bf16_bits_to_f64(late)[0, 0] == 3.03125   # the mistake the pin excludes


def test_combine_sum_is_combine_with_unit_weights():
    rng = np.random.default_rng(11)
    idx, w = _random_routing(30, 6, 3, 4)
    pos, _, _ = oracle.place_pairs(idx, w, 6, 3)
    _, _, tot = oracle.count_experts(idx, 6, 3)
    y = [_bits(rng.standard_normal((int(tot[d]), 8))) for d in range(3)]
    a = oracle.combine_sum(y, idx, pos, 6, 3)
    b = oracle.combine(y, idx, np.ones_like(w), pos, 6, 3)
    assert np.array_equal(a, b)
    # brute force for one token
    g = 7
    acc = sum(oracle.bf16_bits_to_f64(y[int(idx[g, j]) // 2][pos[g, j]]) for j in range(3))
    assert np.array_equal(a[g], oracle.round_f64_to_bf16_bits(acc))


def test_weights_in_ffn_k1_equals_baseline():
    # k = 1: every weight is exactly 1, so scaling and the plain sum change nothing
    cfg = dict(ms.CONFIGS["tiny"], topk=1)
    wfn = lambda e: tuple(ms.weight_np(cfg, n, e) for n in ("gate", "up", "down"))
    a = oracle.pipeline(ms.logits_np(cfg), ms.x_np(cfg), cfg, wfn)
    b = oracle.pipeline(ms.logits_np(cfg), ms.x_np(cfg), cfg, wfn, weights_in_ffn=True)
    assert np.all(a["w"] == 1.0)
    assert np.array_equal(a["out"], b["out"])
    for d in range(cfg["world"]):
        assert np.array_equal(a["y"][d], b["y"][d])


def test_weights_in_ffn_exact_on_integer_ffn():
    # integer expert outputs and power-of-two weights: w*y is exact in bf16, so
    # weighting before or after the rounding and summing in the combine agree
    a, wg, wu, wd, h_ref, y_ref = integer_ffn_case(6, 24, 40)
    _, y, ye = oracle.expert_ffn_rows(a, wg, wu, wd)
    w = np.array([0.5, 0.25, 2.0, 1.0, 0.125, 4.0], dtype=np.float32)
    yw = oracle.scale_rows([ye], [w])[0]
    assert np.array_equal(oracle.bf16_bits_to_f64(yw), y_ref * w[:, None])


# ------------------------------------------------------- router (gate) GEMM

def test_router_logits_one_hot_rows_pick_columns():
    rng = np.random.default_rng(5)
    wr = _bits(rng.standard_normal((6, 32)))
    x = np.zeros((4, 32), dtype=np.float32)
    cols = [0, 7, 31, 12]
    for r, c in enumerate(cols):
        x[r, c] = 1.0
    lg = oracle.router_logits(_bits(x), wr)
    assert lg.dtype == np.float32 and lg.shape == (4, 6)
    for r, c in enumerate(cols):
        assert np.array_equal(lg[r], oracle.bf16_bits_to_f64(wr)[:, c].astype(np.float32))


def test_router_logits_integer_exact_and_orientation():
    # small integers: every product and sum is exact; E = H so a transposed
    # operand would still have the right shape and must be caught by value
    x = np.array([[1, 2, 0, -1], [3, 0, 1, 1]], dtype=np.float32)
    wr = np.array([[1, 0, 0, 0], [0, 1, 0, 2], [1, 1, 1, 1], [-2, 0, 3, 0]], dtype=np.float32)
    lg = oracle.router_logits(_bits(x), _bits(wr))
    assert lg.tolist() == [[1, 0, 2, -2], [3, 2, 5, -3]]   # worked by hand
    assert not np.array_equal(lg, (x @ wr).astype(np.float32))


def test_router_logits_matches_torch_cpu_fp32():
    cfg = ms.CONFIGS["tiny"]
    x = ms.x_np(cfg)
    wr = ms.router_weight_np(cfg)
    lg = oracle.router_logits(x, wr)
    t = lambda b: torch.from_numpy(oracle.bf16_bits_to_f64(b).astype(np.float32))
    ref = (t(x) @ t(wr).T).numpy()
    assert np.allclose(lg, ref, rtol=1e-5, atol=1e-6)


# ------------------------------------------- GEMM + all-to-all (second workload)

def _bf16_bits_of_ints(a):
    """Exact bf16 bit patterns of small integers (|v| < 256)."""
    return oracle.round_f64_to_bf16_bits(np.asarray(a, dtype=np.float64))


def test_linear_a2a_hand_example():
    g = _golden("linear_a2a_hand.json")
    W, T = g["world"], g["tokens_per_slot"]
    wb = _bf16_bits_of_ints(g["weight"])
    r, _ = oracle.gemm_a2a(_bf16_bits_of_ints(g["x"]), wb, W, T)
    assert [oracle.bf16_bits_to_f64(rj).tolist() for rj in r] == g["gemm_a2a"]
    c, _ = oracle.a2a_gemm(_bf16_bits_of_ints(g["z"]), wb, W, T)
    assert [oracle.bf16_bits_to_f64(cj).tolist() for cj in c] == g["a2a_gemm"]


@pytest.mark.parametrize("W,T", [(1, 3), (2, 4), (4, 8), (3, 9)])
def test_a2a_blocks_brute_force(W, T):
    """Every (source slot, row) lands exactly once, at the place an independent
    per-row formula gives; applying the exchange twice is the identity."""
    B = T // W
    labels = [np.array([[s * 1000 + r] for r in range(T)]) for s in range(W)]
    out = oracle.a2a_blocks(labels, W)
    seen = set()
    for s in range(W):
        for r in range(T):
            j, rr = r // B, r % B               # destination slot, row inside the block
            assert out[j][s * B + rr, 0] == s * 1000 + r
            seen.add((j, s * B + rr))
    assert len(seen) == W * T
    back = oracle.a2a_blocks(out, W)
    assert all(np.array_equal(b, l) for b, l in zip(back, labels))


@pytest.mark.parametrize("W,T,Hs", [(1, 2, 3), (2, 3, 2), (4, 2, 1)])
def test_shard_gather_brute_force(W, T, Hs):
    N = W * T
    z = np.array([[[s * 10000 + g * 10 + c for c in range(Hs)] for g in range(N)] for s in range(W)])
    u = oracle.shard_gather(z, W, T)
    for j in range(W):
        assert u[j].shape == (T, W * Hs)
        for r in range(T):
            for col in range(W * Hs):
                s, c = col // Hs, col % Hs      # feature col comes from slot s's shard
                assert u[j][r, col] == s * 10000 + (j * T + r) * 10 + c


def test_linear_integer_closed_form():
    """Small integers: every product and sum is exact, so bf16(a W^T) equals the
    int64 matrix product wherever it fits bf16's 8-bit significand."""
    rng = np.random.default_rng(3)
    a = rng.integers(-3, 4, size=(5, 16))
    w = rng.integers(-2, 3, size=(6, 16))
    ref = a.astype(np.int64) @ w.astype(np.int64).T
    assert np.abs(ref).max() < 256
    got = oracle.bf16_bits_to_f64(oracle.linear(_bf16_bits_of_ints(a), _bf16_bits_of_ints(w)))
    assert np.array_equal(got, ref.astype(np.float64))


def test_identity_weight_reduces_to_the_exchange():
    """W = I: GEMM -> A2A is the row exchange of x and A2A -> GEMM is the shard
    gather, bit for bit."""
    cfg = dict(world=4, tokens_per_slot=8, hidden=16, num_experts=4, topk=1, inter=128)
    W, T, H = cfg["world"], cfg["tokens_per_slot"], cfg["hidden"]
    x = ms.x_np(cfg)
    eye = _bf16_bits_of_ints(np.eye(H))
    r, _ = oracle.gemm_a2a(x, eye, W, T)
    ex = oracle.a2a_blocks([x[s * T:(s + 1) * T] for s in range(W)], W)
    assert all(np.array_equal(a, b) for a, b in zip(r, ex))
    z = np.stack([x[:, s * (H // W):(s + 1) * (H // W)] for s in range(W)])
    c, _ = oracle.a2a_gemm(z, eye, W, T)
    assert all(np.array_equal(a, x[j * T:(j + 1) * T]) for j, a in enumerate(c))


def test_linear_against_torch():
    """An independent library routine (torch CPU, fp32) on random bf16 data."""
    cfg = dict(world=2, tokens_per_slot=16, hidden=64, num_experts=2, topk=1, inter=128)
    x = ms.x_np(cfg)
    w = ms.router_weight_np(dict(cfg, num_experts=64))
    ref = (torch.from_numpy(oracle.bf16_bits_to_f64(x)).float()
           @ torch.from_numpy(oracle.bf16_bits_to_f64(w)).float().T).double().numpy()
    got = oracle.linear_exact(x, w)
    assert np.allclose(got, ref, rtol=1e-5, atol=1e-5)


# ------------------------------------------------ rank-deduplicated dispatch

@pytest.mark.parametrize("n,E,W,k", [(6, 4, 2, 2), (9, 8, 4, 3), (5, 6, 3, 6), (7, 4, 4, 1)])
def test_dedup_tokens_brute_force(n, E, W, k):
    """Token g appears in slot d's staging iff one of its k experts lives on d,
    exactly once, in ascending g; the counts equal an independent per-slot
    set count."""
    rng = np.random.default_rng(n * 100 + E)
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(n)])
    toks = oracle.dedup_tokens(idx, E, W)
    e_loc = E // W
    for d in range(W):
        expect = [g for g in range(n) if any(int(e) // e_loc == d for e in idx[g])]
        assert toks[d].tolist() == expect
    # fewer rows cross than pairs, unless every token's experts sit on distinct slots
    assert sum(len(t) for t in toks) <= n * k


def test_dedup_expansion_reproduces_the_pair_layout():
    """Expanding each slot's staging rows through the row sources gives the
    expert-expanded receive rows of the plain dispatch, bit for bit."""
    cfg = dict(ms.CONFIGS["tiny"], tokens_per_slot=16)
    E, W, k = cfg["num_experts"], cfg["world"], cfg["topk"]
    lg = ms.logits_np(cfg)
    idx, w = oracle.route_topk(lg, k)
    pos, rp, rw = oracle.place_pairs(idx, w, E, W)
    x = ms.x_np(cfg)
    plain = oracle.dispatch_rows(x, rp, k)
    toks = oracle.dedup_tokens(idx, E, W)
    src = oracle.dedup_row_source(idx, E, W, pos)
    for d in range(W):
        staging = x[toks[d]]
        assert np.array_equal(staging[src[d]], plain[d])


def test_dedup_hand_example():
    """E = 4 on W = 2 slots (experts 0-1 on slot 0, 2-3 on slot 1), k = 2.
    Token 0 -> experts (1, 0): twice on slot 0, so it crosses to slot 0 once;
    token 1 -> (2, 1): once to each slot; token 2 -> (3, 2): twice on slot 1.
    Staging: slot 0 holds tokens [0, 1], slot 1 holds [1, 2].  Pair rows of
    slot 0 (expert 0 then 1, ascending token): e0: t0; e1: t0, t1 -> staging
    rows [0, 0, 1]; slot 1: e2: t1, t2; e3: t2 -> staging rows [0, 1, 1]."""
    idx = np.array([[1, 0], [2, 1], [3, 2]])
    w = np.ones((3, 2), dtype=np.float32)
    toks = oracle.dedup_tokens(idx, 4, 2)
    assert [t.tolist() for t in toks] == [[0, 1], [1, 2]]
    pos, _, _ = oracle.place_pairs(idx, w, 4, 2)
    src = oracle.dedup_row_source(idx, 4, 2, pos)
    assert [s.tolist() for s in src] == [[0, 0, 1], [0, 1, 1]]


# ------------------------------------------------------------- FP8 dispatch

def test_e4m3_table():
    """The format's landmarks: 1.0, the largest finite 448, the smallest normal
    2^-6 and subnormal 2^-9, -0, NaN; positive values increase with the code."""
    d = oracle.e4m3_decode
    assert d(0x38) == 1.0 and d(0x7E) == 448.0 and d(0x08) == 2.0 ** -6 and d(0x01) == 2.0 ** -9
    assert d(0x00) == 0.0 and np.signbit(d(0x80)) and math.isnan(d(0x7F)) and math.isnan(d(0xFF))
    assert d(0x77) == 240.0 and d(0x07) == 7 * 2.0 ** -9 and d(0xB8) == -1.0
    vals = [d(c) for c in range(0x7F)]
    assert all(a < b for a, b in zip(vals, vals[1:]))


def test_e4m3_encode_round_trip_ties_and_saturation():
    for c in list(range(0x7F)) + list(range(0x80, 0xFF)):
        assert oracle.e4m3_encode(oracle.e4m3_decode(c)) == c
    # halfway between 1.0 (0x38) and 1.125 (0x39) -> even 0x38; between 1.125 and 1.25 -> 0x3A
    assert oracle.e4m3_encode(1.0625) == 0x38 and oracle.e4m3_encode(1.1875) == 0x3A
    # halfway between the two smallest subnormals (2^-9, 2^-8) -> even 0x02; below half of 2^-9 -> 0
    assert oracle.e4m3_encode(1.5 * 2.0 ** -9) == 0x02 and oracle.e4m3_encode(0.4 * 2.0 ** -9) == 0
    assert oracle.e4m3_encode(1000.0) == 0x7E and oracle.e4m3_encode(-1000.0) == 0xFE
    # the array form is the scalar definition
    rng = np.random.default_rng(4)
    v = np.concatenate([rng.normal(0, 50, 4000), rng.normal(0, 0.01, 1000), [0.0, -0.0, 448.0, 464.0]])
    assert np.array_equal(oracle.e4m3_encode_array(v), [oracle.e4m3_encode(t) for t in v])


def test_token_scale_is_the_smallest_power_of_two():
    for amax, e in [(448.0, 0), (449.0, 1), (896.0, 1), (1.0, -8), (0.875, -9), (0.0, 0)]:
        assert oracle.token_scale_exp(np.array([0.5 * amax, -amax])) == e
    rng = np.random.default_rng(5)
    for _ in range(50):
        row = rng.normal(0, 10.0 ** rng.uniform(-3, 3), 64)
        e = oracle.token_scale_exp(row)
        m = np.max(np.abs(row)) * 2.0 ** -e
        assert 224.0 < m <= 448.0


def test_quantize_dequantize_exact_and_bounded():
    """Rows already of the form code * 2^e come back bit for bit; random rows
    within half an E4M3 step (2^-4 relative for normal codes, 2^-10 * 2^e below)."""
    table = np.array([oracle.e4m3_decode(c) for c in range(0x7F)])
    rng = np.random.default_rng(6)
    exact = rng.choice(table, size=(3, 32)) * np.array([[2.0 ** 5], [2.0 ** -3], [1.0]])
    exact[:, 0] = 448.0 * np.array([2.0 ** 5, 2.0 ** -3, 1.0])      # pins e
    xb = oracle.round_f64_to_bf16_bits(exact)
    codes, exps = oracle.quantize_rows_e4m3(xb)
    assert exps.tolist() == [5, -3, 0]
    assert np.array_equal(oracle.dequantize_rows(codes, exps), xb)
    cfg = dict(world=2, tokens_per_slot=8, hidden=256, num_experts=2, topk=1, inter=128)
    xb = ms.x_np(cfg)
    codes, exps = oracle.quantize_rows_e4m3(xb)
    x = oracle.bf16_bits_to_f64(xb)
    back = oracle.bf16_bits_to_f64(oracle.dequantize_rows(codes, exps))
    bound = np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * np.exp2(exps)[:, None])
    assert np.all(np.abs(back - x) <= bound)
