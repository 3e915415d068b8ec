"""Seeded synthetic inputs for the zero-copy MoE dispatch -> expert -> combine path.

This module is shared by the oracle's tests, the CUDA path's tests and the
benchmark. It holds no arithmetic of the MoE method (no routing, placement,
expert FFN or combine): only the workload presets and one counter-based random
generator, implemented twice with bit-identical results:

* ``*_np``    numpy on the host (used to feed the oracle and small cases);
* ``*_torch`` torch on any device (used to fill multi-GB device tensors fast).

Generator definition (every value is addressable by its element index, so a
slice of a tensor can be generated without the rest):

* ``base(seed, stream) = mix64((seed << 8) ^ stream)``
* raw draw ``n`` of a stream: ``z_n = mix64(base + (n + 1) * GOLDEN mod 2^64)``,
  i.e. output ``n`` of the splitmix64 sequence started at ``base``;
  ``mix64`` is the splitmix64 finaliser (Steele, Lea, Flood, "Fast splittable
  pseudorandom number generators", OOPSLA 2014).
* element ``i`` of a normal tensor sums the twelve 16-bit fields of the raw
  draws ``3i, 3i+1, 3i+2`` (the classic sum-of-twelve-uniforms approximation
  of a unit normal) and centres and scales it exactly:
  ``v = fp32(S - 393210) / 65536 * fp32(sigma)``, one IEEE fp32 multiply, so
  host and device agree to the bit.  bf16 tensors take ``v`` rounded to
  nearest-even on the upper 16 bits.

Streams: logits 1, x 2, W_gate 3, W_up 4, W_down 5, skew permutation 6.
"""
from __future__ import annotations

import math

import numpy as np

GOLDEN = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB
MASK64 = (1 << 64) - 1

STREAM_LOGITS = 1
STREAM_X = 2
STREAM_WG = 3
STREAM_WU = 4
STREAM_WD = 5
STREAM_PERM = 6
STREAM_WR = 7  # router (gate) weights [E, H]
STREAM_WL = 8  # linear layer of the GEMM + all-to-all workload [H, H]
STREAM_Z = 9   # its K-shards [W, N, H/W]

LOGIT_SIGMA = 1.0
X_SIGMA = 1.0
W_SIGMA = 0.02
ZIPF_S = 1.2

# Workload presets: W slots, T tokens per slot, H hidden, E experts, k top-k,
# I expert intermediate size.  N = W*T global tokens, E/W experts per slot.
CONFIGS = {
    "tiny": dict(world=2, tokens_per_slot=64, hidden=128, num_experts=4, topk=2,
                 inter=256, skew=False, fused=False),
    "mixtral": dict(world=8, tokens_per_slot=2048, hidden=4096, num_experts=8,
                    topk=2, inter=14336, skew=False, fused=False),
    "deepseek": dict(world=8, tokens_per_slot=1024, hidden=7168, num_experts=256,
                     topk=8, inter=2048, skew=False, fused=False),
    "skewed": dict(world=8, tokens_per_slot=1024, hidden=7168, num_experts=256,
                   topk=8, inter=2048, skew=True, fused=False),
    "decode": dict(world=8, tokens_per_slot=128, hidden=7168, num_experts=256,
                   topk=8, inter=2048, skew=False, fused=True),
}

CONFIG_TITLES = {
    "tiny": "Tiny (W=2,T=64,H=128,E=4,k=2,I=256)",
    "mixtral": "Mixtral-like (W=8,T=2048,H=4096,E=8,k=2,I=14336)",
    "deepseek": "DeepSeek-V3-like prefill (W=8,T=1024,H=7168,E=256,k=8,I=2048)",
    "skewed": "Skewed Zipf(1.2) routing, DeepSeek-V3-like shapes",
    "decode": "Decode (W=8,T=128,H=7168,E=256,k=8,I=2048)",
}


def shape_of(cfg: dict) -> dict:
    return {k: cfg[k] for k in ("world", "tokens_per_slot", "hidden", "inter",
                                "num_experts", "topk")}


# --------------------------------------------------------------------------
# numpy implementation
# --------------------------------------------------------------------------

def _mix64_int(z: int) -> int:
    z &= MASK64
    z = ((z ^ (z >> 30)) * MIX1) & MASK64
    z = ((z ^ (z >> 27)) * MIX2) & MASK64
    return z ^ (z >> 31)


def stream_base(seed: int, stream: int) -> int:
    return _mix64_int(((seed << 8) ^ stream) & MASK64)


def _mix64_np(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * np.uint64(MIX1)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(MIX2)
    return z ^ (z >> np.uint64(31))


def raw_np(seed: int, stream: int, n: np.ndarray) -> np.ndarray:
    """Raw 64-bit draws number ``n`` (uint64 array) of stream (seed, stream)."""
    base = np.uint64(stream_base(seed, stream))
    with np.errstate(over="ignore"):
        state = base + (n.astype(np.uint64) + np.uint64(1)) * np.uint64(GOLDEN)
        return _mix64_np(state)


def _sum16_np(z: np.ndarray) -> np.ndarray:
    m = np.uint64(0xFFFF)
    return ((z & m) + ((z >> np.uint64(16)) & m) + ((z >> np.uint64(32)) & m)
            + (z >> np.uint64(48))).astype(np.int64)


def normal_f32_np(seed: int, stream: int, index: np.ndarray, sigma: float) -> np.ndarray:
    """fp32 values of elements ``index`` (int array) of a normal tensor."""
    i = index.astype(np.uint64)
    with np.errstate(over="ignore"):
        s = (_sum16_np(raw_np(seed, stream, i * np.uint64(3)))
             + _sum16_np(raw_np(seed, stream, i * np.uint64(3) + np.uint64(1)))
             + _sum16_np(raw_np(seed, stream, i * np.uint64(3) + np.uint64(2))))
    v = (s - 393210).astype(np.float32) / np.float32(65536.0)
    return v * np.float32(sigma)


def f32_to_bf16_bits_np(v: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest-even), returned as uint16 bit patterns."""
    u = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def normal_bf16_np(seed: int, stream: int, index: np.ndarray, sigma: float) -> np.ndarray:
    return f32_to_bf16_bits_np(normal_f32_np(seed, stream, index, sigma))


def _chunked(fn, start: int, count: int, chunk: int = 1 << 22) -> np.ndarray:
    parts = []
    for s in range(start, start + count, chunk):
        n = min(chunk, start + count - s)
        parts.append(fn(np.arange(s, s + n, dtype=np.int64)))
    if not parts:
        return fn(np.zeros(0, dtype=np.int64))
    return np.concatenate(parts)


def zipf_permutation(seed: int, num_experts: int) -> np.ndarray:
    """Seeded permutation pi of 1..E (Fisher-Yates on stream 6)."""
    perm = np.arange(1, num_experts + 1, dtype=np.int64)
    z = raw_np(seed, STREAM_PERM, np.arange(num_experts, dtype=np.int64))
    for i in range(num_experts - 1, 0, -1):
        j = int(z[i] % np.uint64(i + 1))
        perm[i], perm[j] = perm[j], perm[i]
    return perm


def zipf_bias_f32(seed: int, num_experts: int, s: float = ZIPF_S) -> np.ndarray:
    """Per-expert logit bias -s*ln(pi(e)): expert popularity ~ Zipf(s)."""
    perm = zipf_permutation(seed, num_experts)
    return np.array([-s * math.log(float(p)) for p in perm], dtype=np.float32)


def logits_np(cfg: dict, seed: int = 0, rows: np.ndarray | None = None) -> np.ndarray:
    """fp32 router logits [N, E] (or the given global token rows)."""
    n = cfg["world"] * cfg["tokens_per_slot"]
    e = cfg["num_experts"]
    rows = np.arange(n) if rows is None else np.asarray(rows, dtype=np.int64)
    idx = (rows[:, None] * e + np.arange(e)[None, :]).reshape(-1)
    out = normal_f32_np(seed, STREAM_LOGITS, idx, LOGIT_SIGMA).reshape(len(rows), e)
    if cfg.get("skew"):
        out = out + zipf_bias_f32(seed, e)[None, :]
    return out


def x_np(cfg: dict, seed: int = 0, rows: np.ndarray | None = None) -> np.ndarray:
    """bf16 bit patterns (uint16) of the tokens x [N, H] (or the given rows)."""
    n = cfg["world"] * cfg["tokens_per_slot"]
    h = cfg["hidden"]
    if rows is None:
        return _chunked(lambda i: normal_bf16_np(seed, STREAM_X, i, X_SIGMA), 0, n * h).reshape(n, h)
    rows = np.asarray(rows, dtype=np.int64)
    idx = (rows[:, None] * h + np.arange(h)[None, :]).reshape(-1)
    return normal_bf16_np(seed, STREAM_X, idx, X_SIGMA).reshape(len(rows), h)


def weight_np(cfg: dict, which: str, expert: int, seed: int = 0) -> np.ndarray:
    """bf16 bit patterns of one expert's weight: 'gate'/'up' [I,H], 'down' [H,I]."""
    h, i = cfg["hidden"], cfg["inter"]
    stream = {"gate": STREAM_WG, "up": STREAM_WU, "down": STREAM_WD}[which]
    rows, cols = (i, h) if which in ("gate", "up") else (h, i)
    per = rows * cols
    return _chunked(lambda ix: normal_bf16_np(seed, stream, ix, W_SIGMA),
                    expert * per, per).reshape(rows, cols)


def router_weight_np(cfg: dict, seed: int = 0) -> np.ndarray:
    """bf16 bit patterns of the router weight Wr [E, H] (logits = x Wr^T)."""
    e, h = cfg["num_experts"], cfg["hidden"]
    return _chunked(lambda ix: normal_bf16_np(seed, STREAM_WR, ix, W_SIGMA), 0, e * h).reshape(e, h)


def linear_weight_np(cfg: dict, seed: int = 0, rows: np.ndarray | None = None) -> np.ndarray:
    """bf16 bit patterns of the linear layer W [H, H] ([out][in]), or of its
    rows ``rows``."""
    h = cfg["hidden"]
    if rows is None:
        return _chunked(lambda ix: normal_bf16_np(seed, STREAM_WL, ix, W_SIGMA), 0, h * h).reshape(h, h)
    ix = (np.asarray(rows, dtype=np.int64)[:, None] * h + np.arange(h, dtype=np.int64)[None, :]).ravel()
    return normal_bf16_np(seed, STREAM_WL, ix, W_SIGMA).reshape(len(rows), h)


def shards_np(cfg: dict, seed: int = 0, tokens: np.ndarray | None = None) -> np.ndarray:
    """bf16 bit patterns of the K-shards Z [W, N, H/W] (slot s holds features
    [s*H/W, (s+1)*H/W) of every token), or [W, len(tokens), H/W] for the given
    tokens only."""
    W, T, h = cfg["world"], cfg["tokens_per_slot"], cfg["hidden"]
    n, hs = W * T, h // W
    tok = np.arange(n, dtype=np.int64) if tokens is None else np.asarray(tokens, dtype=np.int64)
    ix = ((np.arange(W, dtype=np.int64)[:, None, None] * n + tok[None, :, None]) * hs
          + np.arange(hs, dtype=np.int64)[None, None, :]).ravel()
    return normal_bf16_np(seed, STREAM_Z, ix, X_SIGMA).reshape(W, len(tok), hs)


def bf16_bits_to_f32_np(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# --------------------------------------------------------------------------
# torch implementation (bit-identical; int64 arithmetic wraps mod 2^64)
# --------------------------------------------------------------------------

def _s64(c: int) -> int:
    c &= MASK64
    return c - (1 << 64) if c >= (1 << 63) else c


def _lsr(t, s: int):
    import torch  # noqa: F401
    return (t >> s) & ((1 << (64 - s)) - 1)


def _mix64_torch(z):
    z = (z ^ _lsr(z, 30)) * _s64(MIX1)
    z = (z ^ _lsr(z, 27)) * _s64(MIX2)
    return z ^ _lsr(z, 31)


def _sum16_torch(z):
    return (z & 0xFFFF) + (_lsr(z, 16) & 0xFFFF) + (_lsr(z, 32) & 0xFFFF) + _lsr(z, 48)


def normal_f32_torch(seed: int, stream: int, start: int, count: int, sigma: float, device):
    """fp32 values of elements [start, start+count) of a normal tensor."""
    import torch
    base = _s64(stream_base(seed, stream))
    i = torch.arange(start, start + count, dtype=torch.int64, device=device)
    s = torch.zeros_like(i)
    for r in range(3):
        n = i * 3 + (r + 1)              # (n + 1) for raw draw 3i + r
        s += _sum16_torch(_mix64_torch(n * _s64(GOLDEN) + base))
    v = (s - 393210).to(torch.float32) / 65536.0
    return v * torch.tensor(sigma, dtype=torch.float32, device=device)


def f32_to_bf16_torch(v):
    import torch
    u = v.contiguous().view(torch.int32).to(torch.int64) & 0xFFFFFFFF
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    r = torch.where(r >= 32768, r - 65536, r).to(torch.int16)
    return r.view(torch.bfloat16)


def fill_normal_bf16_torch(out, seed: int, stream: int, start: int, sigma: float,
                           chunk: int = 1 << 26):
    """Fill the contiguous bf16 tensor ``out`` with elements [start, start+numel)."""
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk):
        c = min(chunk, n - s)
        flat[s:s + c] = f32_to_bf16_torch(
            normal_f32_torch(seed, stream, start + s, c, sigma, out.device))
    return out


def logits_torch(cfg: dict, device, seed: int = 0):
    import torch
    n = cfg["world"] * cfg["tokens_per_slot"]
    e = cfg["num_experts"]
    out = normal_f32_torch(seed, STREAM_LOGITS, 0, n * e, LOGIT_SIGMA, device).view(n, e)
    if cfg.get("skew"):
        out = out + torch.from_numpy(zipf_bias_f32(seed, e)).to(device)[None, :]
    return out


def x_torch(cfg: dict, device, seed: int = 0):
    import torch
    n = cfg["world"] * cfg["tokens_per_slot"]
    out = torch.empty((n, cfg["hidden"]), dtype=torch.bfloat16, device=device)
    return fill_normal_bf16_torch(out, seed, STREAM_X, 0, X_SIGMA)


def weight_expert_torch(cfg: dict, which: str, expert: int, device, seed: int = 0):
    """One expert's weight, generated afresh by the torch implementation:
    'gate'/'up' [I,H], 'down' [H,I] bf16 (the same bits as ``weight_np``)."""
    import torch
    h, i = cfg["hidden"], cfg["inter"]
    stream = {"gate": STREAM_WG, "up": STREAM_WU, "down": STREAM_WD}[which]
    rows, cols = (i, h) if which in ("gate", "up") else (h, i)
    out = torch.empty((rows, cols), dtype=torch.bfloat16, device=device)
    return fill_normal_bf16_torch(out, seed, stream, expert * rows * cols, W_SIGMA)


def router_weight_torch(cfg: dict, device, seed: int = 0):
    """Router weight Wr [E, H] bf16 on ``device`` (the bits of ``router_weight_np``)."""
    import torch
    out = torch.empty((cfg["num_experts"], cfg["hidden"]), dtype=torch.bfloat16, device=device)
    return fill_normal_bf16_torch(out, seed, STREAM_WR, 0, W_SIGMA)


def linear_weight_torch(cfg: dict, device, seed: int = 0):
    """Linear layer W [H, H] bf16 on ``device`` (the bits of ``linear_weight_np``)."""
    import torch
    out = torch.empty((cfg["hidden"], cfg["hidden"]), dtype=torch.bfloat16, device=device)
    return fill_normal_bf16_torch(out, seed, STREAM_WL, 0, W_SIGMA)


def shards_torch(cfg: dict, device, seed: int = 0):
    """K-shards Z [W, N, H/W] bf16 on ``device`` (the bits of ``shards_np``)."""
    import torch
    W, T, h = cfg["world"], cfg["tokens_per_slot"], cfg["hidden"]
    out = torch.empty((W, W * T, h // W), dtype=torch.bfloat16, device=device)
    return fill_normal_bf16_torch(out, seed, STREAM_Z, 0, X_SIGMA)


def weights_torch(cfg: dict, device, seed: int = 0):
    """(W_gate [E,I,H], W_up [E,I,H], W_down [E,H,I]) bf16 on ``device``."""
    import torch
    e, h, i = cfg["num_experts"], cfg["hidden"], cfg["inter"]
    wg = torch.empty((e, i, h), dtype=torch.bfloat16, device=device)
    wu = torch.empty((e, i, h), dtype=torch.bfloat16, device=device)
    wd = torch.empty((e, h, i), dtype=torch.bfloat16, device=device)
    fill_normal_bf16_torch(wg, seed, STREAM_WG, 0, W_SIGMA)
    fill_normal_bf16_torch(wu, seed, STREAM_WU, 0, W_SIGMA)
    fill_normal_bf16_torch(wd, seed, STREAM_WD, 0, W_SIGMA)
    return wg, wu, wd
