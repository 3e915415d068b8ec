"""GEMM + all-to-all on the heap's slots (GEMM -> A2A and A2A -> GEMM), fused
and split, against the oracle: bf16 results within the path's tolerance, the
fused and split forms bit-identical (same tiles, same fp32 sums), the
exchanged rows landing exactly where the oracle puts them."""
import numpy as np
import pytest
import torch

import moe_synth as ms
import oracle
from _cases import assert_close, bits, bf16_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def sm():
    import combine_symmetric_heap_gb300 as m
    return m


# W, T, H and the expert shape that sizes the heap (cap = N*min(k, E/W) rows,
# so that a slot's ready window holds the fused A2A -> GEMM counters)
CASES = {
    # one token tile per slot
    "tiny": dict(world=2, tokens_per_slot=64, hidden=256, num_experts=4, topk=2, inter=128),
    # ragged token tile (200 rows), two output feature tiles, 50-row blocks
    "ragged": dict(world=4, tokens_per_slot=200, hidden=512, num_experts=8, topk=2, inter=128),
    # 256 + 16 rows: the remainder rides on the full tile; 68-row blocks
    "folded": dict(world=4, tokens_per_slot=272, hidden=512, num_experts=4, topk=1, inter=128),
    # 2 full tiles + 8 rows (a tile of its own), 8 slots, 65-row blocks
    "wide": dict(world=8, tokens_per_slot=520, hidden=1024, num_experts=8, topk=1, inter=128),
    # H = 384: the last feature tile is half empty; shards of 3 K blocks
    "odd_h": dict(world=2, tokens_per_slot=130, hidden=384, num_experts=2, topk=1, inter=128),
}


def _token_tiles(T):
    """256-row tiles of T rows; a remainder of up to 32 rows behind a single
    full tile rides on it."""
    full, rem = divmod(T, 256)
    return full + (1 if rem and not (full == 1 and rem <= 32) else 0)


def _y_rows(heap, cfg):
    T = cfg["tokens_per_slot"]
    return [bits(heap.y(d)[:T]) for d in range(cfg["world"])]


def _run_gemm_a2a(sm, cfg, fused):
    heap = sm.SymHeap(cfg, DEV)
    x = ms.x_torch(cfg, DEV)
    w = ms.linear_weight_torch(cfg, DEV)
    heap.gemm_a2a(x, w, fused=fused)
    torch.cuda.synchronize()
    assert heap.status() == 0
    return heap


def _run_a2a_gemm(sm, cfg, mode):
    """mode: "split", "fused" (shards read in place) or "engines" (copy engines)."""
    heap = sm.SymHeap(cfg, DEV)
    z = ms.shards_torch(cfg, DEV)
    w = ms.linear_weight_torch(cfg, DEV)
    heap.a2a_gemm(z, w, fused=mode != "split", copy_engines=mode == "engines")
    torch.cuda.synchronize()
    assert heap.status() == 0
    return heap


@pytest.mark.parametrize("name", list(CASES))
def test_gemm_a2a_small(sm, name):
    cfg = CASES[name]
    W, T = cfg["world"], cfg["tokens_per_slot"]
    ref_bits, ref_exact = oracle.gemm_a2a(ms.x_np(cfg), ms.linear_weight_np(cfg), W, T)
    outs = {}
    for fused in (False, True):
        heap = _run_gemm_a2a(sm, cfg, fused)
        got = _y_rows(heap, cfg)
        for j in range(W):
            assert_close(got[j], ref_exact[j], f"{name} fused={fused} slot {j}")
        outs[fused] = got
    assert all(np.array_equal(a, b) for a, b in zip(outs[False], outs[True]))


@pytest.mark.parametrize("name", list(CASES))
def test_a2a_gemm_small(sm, name):
    cfg = CASES[name]
    W, T, H = cfg["world"], cfg["tokens_per_slot"], cfg["hidden"]
    z = ms.shards_np(cfg)
    ref_bits, ref_exact = oracle.a2a_gemm(z, ms.linear_weight_np(cfg), W, T)
    gathered = oracle.shard_gather(z, W, T)
    outs = {}
    for mode in ("split", "fused", "engines"):
        heap = _run_a2a_gemm(sm, cfg, mode)
        if mode == "engines":   # every shard of every slot counted once
            for j in range(W):
                assert torch.all(heap.ready(j)[:W] == 1)
        if mode != "fused":     # the gathered shards, bit-exact, shard major in the window
            for j in range(W):
                blocks = bits(heap.recv_x(j).view(-1)[:T * H].view(W, T, H // W))
                assert np.array_equal(np.concatenate(list(blocks), axis=1), gathered[j])
        got = _y_rows(heap, cfg)
        for j in range(W):
            assert_close(got[j], ref_exact[j], f"{name} {mode} slot {j}")
        outs[mode] = got
    for mode in ("fused", "engines"):
        assert all(np.array_equal(a, b) for a, b in zip(outs["split"], outs[mode])), mode


def test_identity_weight_is_a_pure_exchange(sm):
    """W = I: every result is a copy of an input row, so the GPU must match the
    oracle's exchange bit for bit (this pins the row routing of the epilogue)."""
    cfg = CASES["wide"]
    W, T, H = cfg["world"], cfg["tokens_per_slot"], cfg["hidden"]
    eye = torch.eye(H, dtype=torch.bfloat16, device=DEV)
    x = ms.x_torch(cfg, DEV)
    expect = oracle.a2a_blocks([ms.x_np(cfg)[s * T:(s + 1) * T] for s in range(W)], W)
    for fused in (False, True):
        heap = sm.SymHeap(cfg, DEV)
        heap.gemm_a2a(x, eye, fused=fused)
        torch.cuda.synchronize()
        got = _y_rows(heap, cfg)
        assert all(np.array_equal(g, e) for g, e in zip(got, expect))


# full-size workloads: sampled rows recomputed one by one by the oracle
FULL = {
    "mixtral": dict(ms.CONFIGS["mixtral"]),
    "deepseek": dict(ms.CONFIGS["deepseek"]),
}


def _fresh_linear_weight(cfg):
    """The oracle's weight, generated afresh on the device by the input module
    (never a buffer the CUDA path touched), as host bits."""
    return bits(ms.linear_weight_torch(cfg, DEV))


@pytest.mark.parametrize("name", list(FULL))
def test_gemm_a2a_full_size_sampled(sm, name):
    cfg = FULL[name]
    W, T = cfg["world"], cfg["tokens_per_slot"]
    B = T // W
    heap = _run_gemm_a2a(sm, cfg, True)
    wb = _fresh_linear_weight(cfg)
    rng = np.random.default_rng(9)
    for j in range(W):
        rows = np.sort(rng.choice(T, size=6, replace=False))   # destination rows of slot j
        src = np.array([(r // B) * T + j * B + r % B for r in rows])  # source token of each
        ref = oracle.linear_exact(ms.x_np(cfg, rows=src), wb)
        assert_close(bits(heap.y(j)[torch.from_numpy(rows).to(DEV)]), ref, f"{name} slot {j}")


@pytest.mark.parametrize("mode", ["fused", "engines"])
@pytest.mark.parametrize("name", list(FULL))
def test_a2a_gemm_full_size_sampled(sm, name, mode):
    cfg = FULL[name]
    W, T = cfg["world"], cfg["tokens_per_slot"]
    heap = _run_a2a_gemm(sm, cfg, mode)
    wb = _fresh_linear_weight(cfg)
    rng = np.random.default_rng(10)
    for j in range(W):
        rows = np.sort(rng.choice(T, size=6, replace=False))
        zs = ms.shards_np(cfg, tokens=j * T + rows)                 # [W][6][H/W]
        u = np.concatenate([zs[s] for s in range(W)], axis=1)      # the gathered rows
        ref = oracle.linear_exact(u, wb)
        assert_close(bits(heap.y(j)[torch.from_numpy(rows).to(DEV)]), ref, f"{name} slot {j}")
