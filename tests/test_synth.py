"""The seeded input generator: host (numpy) and torch implementations agree to
the bit, slices are addressable by element index, and the moments are those
of the stated distributions."""
import numpy as np
import pytest
import torch

import moe_synth as ms


def test_splitmix64_known_vector():
    # splitmix64 seeded with state 0: first output is 0xE220A8397B1DCDAF
    # (published reference sequence of the algorithm).
    assert ms._mix64_int(ms.GOLDEN) == 0xE220A8397B1DCDAF
    z = ms._mix64_np(np.array([ms.GOLDEN], dtype=np.uint64))
    assert int(z[0]) == 0xE220A8397B1DCDAF


@pytest.mark.parametrize("stream,sigma", [(1, 1.0), (2, 1.0), (3, 0.02), (5, 0.02)])
def test_numpy_torch_bit_identical(stream, sigma):
    start, count = 12345, 50000
    a = ms.normal_f32_np(0, stream, np.arange(start, start + count), sigma)
    b = ms.normal_f32_torch(0, stream, start, count, sigma, "cpu").numpy()
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    ab = ms.f32_to_bf16_bits_np(a)
    bb = ms.f32_to_bf16_torch(torch.from_numpy(b)).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ab, bb)


def test_bf16_rounding_matches_torch_cast():
    v = ms.normal_f32_np(0, 9, np.arange(100000), 3.0)
    mine = ms.f32_to_bf16_bits_np(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mine, ref)


def test_slices_are_addressable():
    cfg = ms.CONFIGS["tiny"]
    x = ms.x_np(cfg)
    rows = np.array([3, 77, 127])
    assert np.array_equal(ms.x_np(cfg, rows=rows), x[rows])
    lg = ms.logits_np(cfg)
    assert np.array_equal(ms.logits_np(cfg, rows=rows), lg[rows])
    wg = ms.weight_np(cfg, "gate", 2)
    wg_t = ms.weights_torch(cfg, "cpu")[0][2].view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(wg, wg_t)


def test_whole_tensors_numpy_vs_torch_tiny_and_skew():
    cfg = ms.CONFIGS["tiny"]
    xt = ms.x_torch(cfg, "cpu").view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ms.x_np(cfg), xt)
    sk = dict(ms.CONFIGS["skewed"], tokens_per_slot=8)
    assert np.array_equal(ms.logits_np(sk), ms.logits_torch(sk, "cpu").numpy())


def test_linear_workload_inputs_numpy_vs_torch_and_slices():
    cfg = dict(world=4, tokens_per_slot=6, hidden=256, num_experts=4, topk=1, inter=128)
    u16 = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    w = ms.linear_weight_np(cfg)
    assert np.array_equal(w, u16(ms.linear_weight_torch(cfg, "cpu")))
    assert np.array_equal(ms.linear_weight_np(cfg, rows=np.array([5, 200])), w[[5, 200]])
    z = ms.shards_np(cfg)
    assert z.shape == (4, 24, 64)
    assert np.array_equal(z, u16(ms.shards_torch(cfg, "cpu")))
    assert np.array_equal(ms.shards_np(cfg, tokens=np.array([0, 17])), z[:, [0, 17]])


def test_moments():
    v = ms.normal_f32_np(0, 2, np.arange(400000), 1.0).astype(np.float64)
    assert abs(v.mean()) < 0.01
    assert abs(v.std() - 1.0) < 0.01
    w = ms.normal_f32_np(0, 3, np.arange(400000), 0.02).astype(np.float64)
    assert abs(w.std() - 0.02) < 0.0003


def test_zipf_bias():
    perm = ms.zipf_permutation(0, 256)
    assert sorted(perm.tolist()) == list(range(1, 257))
    b = ms.zipf_bias_f32(0, 256)
    top = int(np.argmax(b))
    assert perm[top] == 1 and b[top] == 0.0
    assert np.isclose(b[int(np.argmin(b))], -1.2 * np.log(256), rtol=1e-6)
