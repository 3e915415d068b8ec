"""Plain fp64 numpy definition of GEMM -> all-to-all and all-to-all -> GEMM
on the W slots of the symmetric heap.

TEST INFRASTRUCTURE ONLY (see the package docstring): never imported by the
product path.

Source: the AMD technical blog "MORI CCO: Next-Generation Collective
Communication Object for GPUs", section "Examples", "GEMM + all-to-all
fusion": a GEMM whose epilogue puts output tiles straight into the peers'
windows (GEMM -> A2A), and a GEMM that consumes remote K-shards as they
arrive, polling ready counters (A2A -> GEMM); both are compared with split
pipelines (GEMM, then a separate all-to-all, or the reverse).  The pages give
no shapes or layouts.  The readings taken here:

* the GEMM is one linear layer shared by every slot: out = bf16(a W^T) with
  W [H][H] (K-major, like nn.Linear), fp64 accumulation here;
* GEMM -> A2A: slot s computes Y_s = X_s W^T for its T token rows and the rows
  are exchanged all-to-all in W equal blocks of B = T/W rows: slot j receives
  block j of every slot, stacked by source slot,
      R_j[s*B + r] = Y_s[j*B + r]        (0 <= r < B);
* A2A -> GEMM: slot s holds the K-shard s (features [s*H/W, (s+1)*H/W)) of all
  N = W*T tokens; the all-to-all gives slot j its own T tokens with every
  feature, shard s from slot s,
      U_j[r][s*H/W + c] = Z_s[j*T + r][c],
  and slot j computes C_j = U_j W^T.

Values stored as bf16 are rounded fp64 -> fp32 -> bf16, each to nearest even
(the rounding of a kernel that accumulates in fp32), with the helpers of
``oracle.moe``.
"""
from __future__ import annotations

import numpy as np

from .moe import bf16_bits_to_f64, round_f64_to_bf16_bits


def linear_exact(a_bits: np.ndarray, w_bits: np.ndarray) -> np.ndarray:
    """a W^T in fp64 (a: [n][H] bf16 bits, W: [H_out][H] bf16 bits)."""
    return bf16_bits_to_f64(a_bits) @ bf16_bits_to_f64(w_bits).T


def linear(a_bits: np.ndarray, w_bits: np.ndarray) -> np.ndarray:
    """bf16(a W^T) as uint16 bits."""
    return round_f64_to_bf16_bits(linear_exact(a_bits, w_bits))


def a2a_blocks(y_slots: list, world: int) -> list:
    """Row all-to-all in W equal blocks: R_j[s*B + r] = Y_s[j*B + r].

    y_slots[s] is slot s's [T][C] array (any dtype); T must be a multiple of W.
    """
    T = y_slots[0].shape[0]
    assert T % world == 0
    B = T // world
    out = []
    for j in range(world):
        out.append(np.concatenate([y_slots[s][j * B:(j + 1) * B] for s in range(world)], axis=0))
    return out


def gemm_a2a(x_bits: np.ndarray, w_bits: np.ndarray, world: int, tokens_per_slot: int):
    """GEMM -> A2A: slot s's rows x[s*T:(s+1)*T] through the linear layer, then
    the row all-to-all.  Returns (R bits per slot [T][H], exact values per slot)."""
    T = tokens_per_slot
    exact = [linear_exact(x_bits[s * T:(s + 1) * T], w_bits) for s in range(world)]
    y = [round_f64_to_bf16_bits(e) for e in exact]
    return a2a_blocks(y, world), a2a_blocks(exact, world)


def shard_gather(z_bits: np.ndarray, world: int, tokens_per_slot: int) -> list:
    """The all-to-all of K-shards: U_j[r][s*Hs + c] = Z_s[j*T + r][c].

    z_bits: [W][N][Hs] (slot s's feature shard of every token)."""
    T = tokens_per_slot
    return [np.concatenate([z_bits[s][j * T:(j + 1) * T] for s in range(world)], axis=1)
            for j in range(world)]


def a2a_gemm(z_bits: np.ndarray, w_bits: np.ndarray, world: int, tokens_per_slot: int):
    """A2A -> GEMM: gather slot j's K-shards, then the linear layer.  Returns
    (C bits per slot [T][H], exact values per slot)."""
    u = shard_gather(z_bits, world, tokens_per_slot)
    exact = [linear_exact(uj, w_bits) for uj in u]
    return [round_f64_to_bf16_bits(e) for e in exact], exact
