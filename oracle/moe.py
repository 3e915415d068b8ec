"""Plain fp64 numpy definition of the zero-copy MoE dispatch -> expert -> combine.

TEST INFRASTRUCTURE ONLY (see the package docstring): never imported by the
product path.

Source: the AMD technical blog "MORI CCO: Next-Generation Collective
Communication Object for GPUs", sections "What is MORI CCO?" (the flat
symmetric address of a peer window) and "Zero-copy MoE dispatch -> expert ->
combine" (the EPv2 dispatch / expert_gemm / combine pipeline).  The pages
leave routing, the expert function and the receive order to the caller; the
readings taken here are:

* routing: top-k of the E fp32 logits per token, ties to the lower expert
  index, the k selected in descending order, weights = softmax over the
  selected k;
* expert e lives on slot e // (E/W) (contiguous placement);
* one received row per (token, k) pair, grouped by expert inside the slot
  (experts ascending), and inside one expert in (source slot, token, k)
  order -- with global token g = s*T + t that is simply ascending g;
* expert = SwiGLU FFN: h = bf16(silu(a Wg^T) * (a Wu^T)), y = bf16(h Wd^T);
* combine: out[g] = bf16(sum_j w[g,j] * y[row of pair (g,j)]), j ascending,
  weights applied on the source side as the combine call takes them.

Floating point: fp64 everywhere; values that the path stores as bf16 (h, y,
out) are rounded from fp64 to fp32 and then to bf16, each round-to-nearest-
even, which is what a kernel that accumulates in fp32 stores.
"""
from __future__ import annotations

import numpy as np


# ---------------------------------------------------------------------------
# bf16 helpers (own implementation; bf16 = upper 16 bits of an fp32)
# ---------------------------------------------------------------------------

def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16) as float64."""
    u = np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def round_f64_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """fp64 -> fp32 (nearest-even) -> bf16 (nearest-even), as uint16 bits."""
    f = np.asarray(v, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    keep = u >> np.uint64(16)
    rest = u & np.uint64(0xFFFF)
    up = (rest > np.uint64(0x8000)) | ((rest == np.uint64(0x8000)) & ((keep & np.uint64(1)) == np.uint64(1)))
    return (keep + up.astype(np.uint64)).astype(np.uint16)


# ---------------------------------------------------------------------------
# symmetric heap address (blog, "What is MORI CCO?": peer address formula)
# ---------------------------------------------------------------------------

def slot_address(win_base: int, peer: int, per_rank_size: int, offset: int) -> int:
    """Address of ``offset`` inside the window copy that slot ``peer`` owns.

    Every window sits at the same offset in every slot, so the peer address is
    the window base plus ``peer`` slot strides plus the offset.
    """
    return win_base + peer * per_rank_size + offset


# ---------------------------------------------------------------------------
# next: the router (gate) GEMM that produces the logits
# ---------------------------------------------------------------------------

def router_logits(x_bits: np.ndarray, wr_bits: np.ndarray) -> np.ndarray:
    """logits[g, e] = fp32( sum_h x[g, h] * Wr[e, h] ), the products and the
    sum in fp64 (x: [N, H] bf16 bits, Wr: [E, H] bf16 bits)."""
    return (bf16_bits_to_f64(x_bits) @ bf16_bits_to_f64(wr_bits).T).astype(np.float32)


# ---------------------------------------------------------------------------
# a1: routing (the pages take indices/weights as dispatch inputs)
# ---------------------------------------------------------------------------

def route_topk(logits: np.ndarray, k: int):
    """Top-k experts per token and their softmax-over-the-k weights.

    logits: [N, E] fp32.  Returns idx [N, k] int32 (descending logit, ties to
    the lower expert index) and w [N, k] fp32 with
    w_j = exp(l_j - l_0) / sum_i exp(l_i - l_0) evaluated in fp64.
    """
    logits = np.asarray(logits, dtype=np.float32)
    # a stable ascending sort of -logit gives descending logit, equal logits
    # keeping ascending expert index
    order = np.argsort(-logits, axis=1, kind="stable")[:, :k]
    sel = np.take_along_axis(logits, order, axis=1).astype(np.float64)
    z = np.exp(sel - sel[:, :1])
    w = z / z.sum(axis=1, keepdims=True)
    return order.astype(np.int32), w.astype(np.float32)


# ---------------------------------------------------------------------------
# a2: counts, per-slot receive offsets
# ---------------------------------------------------------------------------

def count_experts(idx: np.ndarray, num_experts: int, world: int):
    """Per-expert pair counts, each expert's first row inside its slot, and
    the number of rows every slot receives.

    cnt[e]        = #{(g, j) : idx[g, j] == e}
    recv_off[e]   = sum of cnt[e'] over the experts e' < e of the same slot
    total_recv[d] = sum of cnt[e] over the experts of slot d
    """
    e_loc = num_experts // world
    cnt = np.zeros(num_experts, dtype=np.int64)
    for e in np.asarray(idx).reshape(-1):
        cnt[int(e)] += 1
    recv_off = np.zeros(num_experts, dtype=np.int64)
    total_recv = np.zeros(world, dtype=np.int64)
    for e in range(num_experts):
        d = e // e_loc
        recv_off[e] = total_recv[d]
        total_recv[d] += cnt[e]
    return cnt, recv_off, total_recv


# ---------------------------------------------------------------------------
# a3: placement of every (token, k) pair (the dispatch scatter's layout)
# ---------------------------------------------------------------------------

def place_pairs(idx: np.ndarray, w: np.ndarray, num_experts: int, world: int):
    """Receive row of every pair, in (source slot, token, k) order per expert.

    Returns pos [N, k] (row inside the destination slot), and per slot the
    lists recv_pair[d] (g*k + j of the pair in each received row) and
    recv_w[d] (its routing weight), each of length total_recv[d].
    """
    idx = np.asarray(idx)
    n, k = idx.shape
    e_loc = num_experts // world
    cnt, recv_off, total_recv = count_experts(idx, num_experts, world)
    fill = np.zeros(num_experts, dtype=np.int64)
    pos = np.zeros((n, k), dtype=np.int64)
    recv_pair = [np.full(int(total_recv[d]), -1, dtype=np.int64) for d in range(world)]
    recv_w = [np.zeros(int(total_recv[d]), dtype=np.float32) for d in range(world)]
    for g in range(n):
        for j in range(k):
            e = int(idx[g, j])
            d = e // e_loc
            p = int(recv_off[e] + fill[e])
            fill[e] += 1
            pos[g, j] = p
            recv_pair[d][p] = g * k + j
            recv_w[d][p] = w[g, j]
    return pos, recv_pair, recv_w


def dispatch_rows(x_bits: np.ndarray, recv_pair: list, topk: int):
    """Received token rows of every slot: row p of slot d is x[g] of its pair
    (a bit copy of the bf16 row)."""
    return [np.asarray(x_bits)[rp // topk] for rp in recv_pair]


# ---------------------------------------------------------------------------
# rank-deduplicated dispatch: each token crosses to a slot once, then the
# receiving slot expands it to its expert rows
# ---------------------------------------------------------------------------

def dedup_tokens(idx: np.ndarray, num_experts: int, world: int) -> list:
    """Per slot d, the tokens that have at least one expert on d, in ascending
    token order (source slot, then token): row q of slot d's staging holds
    token dedup_tokens(...)[d][q].  The pages leave the receive layout open;
    this is the deduplicated reading of the dispatch (one row per destination
    slot and token instead of one per (token, k) pair)."""
    idx = np.asarray(idx)
    e_loc = num_experts // world
    out = [[] for _ in range(world)]
    for g in range(idx.shape[0]):
        slots = sorted({int(e) // e_loc for e in idx[g]})
        for d in slots:
            out[d].append(g)
    return [np.array(t, dtype=np.int64) for t in out]


def dedup_row_source(idx: np.ndarray, num_experts: int, world: int, pos: np.ndarray) -> list:
    """Per slot d and received row p (the expert-expanded layout of
    place_pairs), the staging row q whose token the row copies."""
    idx = np.asarray(idx)
    n, k = idx.shape
    e_loc = num_experts // world
    toks = dedup_tokens(idx, num_experts, world)
    q_of = [{int(g): q for q, g in enumerate(t)} for t in toks]
    total = [0] * world
    for g in range(n):
        for j in range(k):
            d = int(idx[g, j]) // e_loc
            total[d] = max(total[d], int(pos[g, j]) + 1)
    src = [np.full(total[d], -1, dtype=np.int64) for d in range(world)]
    for g in range(n):
        for j in range(k):
            d = int(idx[g, j]) // e_loc
            src[d][int(pos[g, j])] = q_of[d][g]
    return src


# ---------------------------------------------------------------------------
# FP8 dispatch with per-token scales (the blog's dispatch carries scales,
# recv_s): each row crosses as e4m3 codes and one scale 2^e, and the receiving
# slot multiplies back to bf16.  Readings: OCP FP8 E4M3 (bias 7, 3 mantissa
# bits, subnormals, largest finite 448, no infinities); the per-token scale is
# the smallest power of two 2^e with max|x| <= 448 * 2^e (so scaling is exact
# and only the e4m3 rounding loses bits); rounding to nearest, ties to even;
# the dequantized value code * 2^e is exact in bf16.
# ---------------------------------------------------------------------------

E4M3_MAX = 448.0


def e4m3_decode(code: int) -> float:
    """Value of an E4M3 code (NaN for the two NaN codes)."""
    c = int(code) & 0xFF
    sign = -1.0 if c & 0x80 else 1.0
    ex, man = (c >> 3) & 0xF, c & 0x7
    if ex == 0xF and man == 0x7:
        return float("nan")
    if ex == 0:
        return sign * man * 2.0 ** -9           # subnormal: man/8 * 2^(1-7)
    return sign * (1.0 + man / 8.0) * 2.0 ** (ex - 7)


def e4m3_encode(v: float) -> int:
    """Nearest E4M3 code to v (ties to the even code), saturating at +-448."""
    v = float(v)
    sign = 0x80 if (v < 0 or (v == 0 and np.signbit(v))) else 0
    a = abs(v)
    if a >= E4M3_MAX:
        return sign | 0x7E
    best, best_d = 0, None
    for c in range(0x7F):                      # the 127 finite non-negative codes
        d = abs(e4m3_decode(c) - a)
        if best_d is None or d < best_d or (d == best_d and (c & 1) == 0 and (best & 1) == 1):
            best, best_d = c, d
    return sign | best


def token_scale_exp(row_f64: np.ndarray) -> int:
    """Smallest e with max|x| <= 448 * 2^e (0 for an all-zero row)."""
    amax = float(np.max(np.abs(row_f64))) if row_f64.size else 0.0
    if amax == 0.0:
        return 0
    e = int(np.floor(np.log2(amax / E4M3_MAX))) - 1
    while amax > E4M3_MAX * 2.0 ** e:
        e += 1
    return e


def e4m3_encode_array(v: np.ndarray) -> np.ndarray:
    """e4m3_encode over an array: the nearest of the 127 non-negative finite
    values (increasing with the code) by a sorted search, ties to the even
    code, saturating at 448, sign from the input."""
    v = np.asarray(v, dtype=np.float64)
    table = np.array([e4m3_decode(c) for c in range(0x7F)])
    a = np.minimum(np.abs(v), E4M3_MAX)
    hi = np.clip(np.searchsorted(table, a, side="left"), 0, 0x7E)
    lo = np.maximum(hi - 1, 0)
    d_lo, d_hi = a - table[lo], table[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    return code | np.where(np.signbit(v), 0x80, 0).astype(np.uint8)


def quantize_rows_e4m3(x_bits: np.ndarray):
    """Per row: the scale exponent e and the codes of x / 2^e."""
    x = bf16_bits_to_f64(x_bits)
    n, h = x.shape
    exps = np.array([token_scale_exp(x[g]) for g in range(n)], dtype=np.int64)
    codes = e4m3_encode_array(x * np.exp2(-exps.astype(np.float64))[:, None])
    return codes, exps


def dequantize_rows(codes: np.ndarray, exps: np.ndarray) -> np.ndarray:
    """bf16 bits of code * 2^e (exact)."""
    table = np.array([e4m3_decode(c) for c in range(256)])
    vals = table[np.asarray(codes, dtype=np.int64)] * np.exp2(np.asarray(exps, dtype=np.float64))[:, None]
    return round_f64_to_bf16_bits(vals)


# ---------------------------------------------------------------------------
# a4 + a5: SwiGLU expert on a block of received rows
# ---------------------------------------------------------------------------

def expert_ffn_rows(a_bits: np.ndarray, wg_bits: np.ndarray, wu_bits: np.ndarray,
                    wd_bits: np.ndarray):
    """One expert on rows a [M, H] (bf16 bits) with Wg, Wu [I, H], Wd [H, I].

    gate = a Wg^T, up = a Wu^T (fp64), h = bf16(silu(gate) * up) with
    silu(z) = z / (1 + exp(-z)); y = bf16(h Wd^T).  Returns (h bits, y bits,
    y before its bf16 rounding as fp64).
    """
    a = bf16_bits_to_f64(a_bits)
    gate = a @ bf16_bits_to_f64(wg_bits).T
    up = a @ bf16_bits_to_f64(wu_bits).T
    with np.errstate(over="ignore"):
        silu = gate / (1.0 + np.exp(-gate))
    h_bits = round_f64_to_bf16_bits(silu * up)
    y_exact = bf16_bits_to_f64(h_bits) @ bf16_bits_to_f64(wd_bits).T
    return h_bits, round_f64_to_bf16_bits(y_exact), y_exact


def expert_ffn(recv_x: list, cnt, recv_off, num_experts: int, world: int, weight_fn):
    """All experts over all slots.  ``weight_fn(e)`` returns (Wg, Wu, Wd) bits
    of expert e.  Returns per slot (h bits, y bits, y fp64), rows [0,total)."""
    e_loc = num_experts // world
    hidden = recv_x[0].shape[1] if len(recv_x) and recv_x[0].ndim == 2 else None
    out_h, out_y, out_ye = [], [], []
    for d in range(world):
        rows = recv_x[d].shape[0]
        out_h.append(None)
        out_y.append(np.zeros((rows, hidden), dtype=np.uint16))
        out_ye.append(np.zeros((rows, hidden), dtype=np.float64))
    for e in range(num_experts):
        c = int(cnt[e])
        if c == 0:
            continue
        d, o = e // e_loc, int(recv_off[e])
        wg, wu, wd = weight_fn(e)
        h, y, ye = expert_ffn_rows(recv_x[d][o:o + c], wg, wu, wd)
        if out_h[d] is None:
            out_h[d] = np.zeros((recv_x[d].shape[0], h.shape[1]), dtype=np.uint16)
        out_h[d][o:o + c] = h
        out_y[d][o:o + c] = y
        out_ye[d][o:o + c] = ye
    return out_h, out_y, out_ye


# ---------------------------------------------------------------------------
# a6: weighted combine
# ---------------------------------------------------------------------------

def combine(y_bits: list, idx: np.ndarray, w: np.ndarray, pos: np.ndarray,
            num_experts: int, world: int) -> np.ndarray:
    """out[g] = bf16(sum_j w[g, j] * y[slot of idx[g, j]][pos[g, j]]), j ascending."""
    idx = np.asarray(idx)
    n, k = idx.shape
    e_loc = num_experts // world
    hidden = y_bits[0].shape[1]
    acc = np.zeros((n, hidden), dtype=np.float64)
    for j in range(k):
        for g in range(n):
            d = int(idx[g, j]) // e_loc
            acc[g] += float(w[g, j]) * bf16_bits_to_f64(y_bits[d][int(pos[g, j])])
    return round_f64_to_bf16_bits(acc)


# ---------------------------------------------------------------------------
# variant: routing weights applied in the expert epilogue
# ---------------------------------------------------------------------------
# The pages apply the weights where combine takes them.  The variant moves
# them to the receiving side: each received row's expert output is scaled by
# the weight of its (token, k) pair (recv_w, written by the dispatch) before
# the output is rounded, and the combine only sums.

def scale_rows(y_exact: list, recv_w: list) -> list:
    """y_w[d][p] = bf16(recv_w[d][p] * y[d][p]) with y before its rounding:
    one rounding of the weighted expert output."""
    return [round_f64_to_bf16_bits(np.asarray(ye, dtype=np.float64) *
                                   np.asarray(rw, dtype=np.float64)[:, None])
            for ye, rw in zip(y_exact, recv_w)]


def combine_sum(y_bits: list, idx: np.ndarray, pos: np.ndarray, num_experts: int,
                world: int) -> np.ndarray:
    """out[g] = bf16(sum_j y[slot of idx[g, j]][pos[g, j]]), j ascending: the
    combine of rows that already carry their weights."""
    idx = np.asarray(idx)
    n, k = idx.shape
    e_loc = num_experts // world
    acc = np.zeros((n, y_bits[0].shape[1]), dtype=np.float64)
    for j in range(k):
        for g in range(n):
            d = int(idx[g, j]) // e_loc
            acc[g] += bf16_bits_to_f64(y_bits[d][int(pos[g, j])])
    return round_f64_to_bf16_bits(acc)


# ---------------------------------------------------------------------------
# whole path
# ---------------------------------------------------------------------------

def pipeline(logits, x_bits, shape: dict, weight_fn, weights_in_ffn: bool = False):
    """route -> count/place -> dispatch rows -> expert FFN -> combine.

    ``shape`` has world, num_experts, topk; ``weight_fn(e)`` gives expert e's
    (Wg, Wu, Wd) bf16 bits.  ``weights_in_ffn``: the variant above (y holds
    the weighted rows, the combine sums).  Returns a dict with every
    intermediate.
    """
    world, num_experts, k = shape["world"], shape["num_experts"], shape["topk"]
    idx, w = route_topk(logits, k)
    cnt, recv_off, total_recv = count_experts(idx, num_experts, world)
    pos, recv_pair, recv_w = place_pairs(idx, w, num_experts, world)
    recv_x = dispatch_rows(x_bits, recv_pair, k)
    h, y, y_exact = expert_ffn(recv_x, cnt, recv_off, num_experts, world, weight_fn)
    if weights_in_ffn:
        y = scale_rows(y_exact, recv_w)
        out = combine_sum(y, idx, pos, num_experts, world)
    else:
        out = combine(y, idx, w, pos, num_experts, world)
    return dict(idx=idx, w=w, cnt=cnt, recv_off=recv_off, total_recv=total_recv,
                pos=pos, recv_pair=recv_pair, recv_w=recv_w, recv_x=recv_x,
                h=h, y=y, y_exact=y_exact, out=out)
