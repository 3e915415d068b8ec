"""Host-side checks of the C-ABI library (no GPU needed): it loads, exports
every function include/symmoe.h declares, its structs match the binding, the
heap arithmetic follows the symmetric-heap rule, and bad arguments are
rejected before any device work."""
import ctypes
import os
import re
import subprocess

import pytest

import combine_symmetric_heap_gb300 as sm
import moe_synth as ms

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "symmoe.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b([a-z_][a-z0-9_]*)\s*\([^;{]*\)\s*;", text, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol():
    names = _declared_functions()
    assert {"sym_heap_init", "moe_route_topk", "moe_dispatch", "moe_expert_ffn", "moe_combine",
            "moe_pipeline"} <= set(names)
    lib = sm.lib()
    for n in names:
        assert hasattr(lib, n), f"{n} declared in symmoe.h but not exported"


def test_struct_layout_matches_header(tmp_path):
    fields = [f[0] for f in sm.SymHeapDesc._fields_]
    src = tmp_path / "probe.c"
    lines = ['#include <stdio.h>', '#include <stddef.h>', f'#include "{HEADER}"', "int main(void){",
             'printf("size %zu\\n", sizeof(sym_heap));',
             'printf("shape %zu\\n", sizeof(moe_shape));']
    for f in fields:
        lines.append(f'printf("{f} %zu\\n", offsetof(sym_heap, {f}));')
    lines.append("return 0;}")
    src.write_text("\n".join(lines))
    exe = tmp_path / "probe"
    subprocess.run(["gcc", "-std=c99", "-o", str(exe), str(src)], check=True)
    out = dict(l.split() for l in subprocess.run([str(exe)], capture_output=True, text=True,
                                                 check=True).stdout.splitlines())
    assert int(out["size"]) == ctypes.sizeof(sm.SymHeapDesc)
    assert int(out["shape"]) == ctypes.sizeof(sm.MoeShape)
    for f in fields:
        assert int(out[f]) == getattr(sm.SymHeapDesc, f).offset, f


@pytest.mark.parametrize("name", list(ms.CONFIGS))
def test_heap_layout(name):
    cfg = ms.CONFIGS[name]
    prs, total = sm.sym_heap_bytes(cfg)
    assert prs % (2 << 20) == 0 and total == prs * cfg["world"]
    fake = 1 << 40
    d = sm.sym_heap_init(cfg, fake, total)
    n = cfg["world"] * cfg["tokens_per_slot"]
    e_loc = cfg["num_experts"] // cfg["world"]
    assert d.cap == n * min(cfg["topk"], e_loc)
    H, I, T, k = cfg["hidden"], cfg["inter"], cfg["tokens_per_slot"], cfg["topk"]
    wins = [(d.off_recv_x, d.cap * H * 2), (d.off_y, d.cap * H * 2), (d.off_h, d.cap * I * 2),
            (d.off_recv_pair, d.cap * 4), (d.off_recv_w, d.cap * 4), (d.off_pos, T * k * 4),
            (d.off_cnt, e_loc * 4), (d.off_recv_off, e_loc * 4), (d.off_total, 4),
            (d.off_status, 4), (d.off_ready, d.num_ready * 4),
            (d.off_hist, cfg["num_experts"] * ((n + 31) // 32) * 4),
            # control words + one h and one y readiness counter per 256-row token
            # tile + a route-task counter per 32-token chunk
            (d.off_ctrl, 4 * (64 + 2 * (n * k // 256 + cfg["num_experts"] + 1) + (n + 31) // 32))]
    for (o, b), (o2, _) in zip(wins, wins[1:]):
        assert o % 1024 == 0 and o + b + sm.SYM_GUARD_BYTES <= o2   # a guard band after every window
    assert wins[-1][0] + wins[-1][1] + sm.SYM_GUARD_BYTES <= prs
    # the library's own account of the windows is the same layout
    assert sm.sym_heap_windows(d) == [(int(o), int(b)) for o, b in wins]
    assert d.num_ready == (d.cap + 127) // 128
    assert d.wait_timeout_us == 2_000_000 and d.epoch == 0


def test_slot_ptr_is_the_peer_address():
    cfg = ms.CONFIGS["tiny"]
    prs, total = sm.sym_heap_bytes(cfg, align=1 << 32)
    assert prs == 1 << 32                      # the CCO kernel's 4 GiB stride
    base = 0x7F0000000000
    d = sm.sym_heap_init(cfg, base, total, align=1 << 32)
    assert sm.sym_heap_slot_ptr(d, 1, 0x100) == 0x7F0100000100
    assert sm.sym_heap_slot_ptr(d, 0, 0) == base
    assert sm.sym_heap_slot_ptr(d, 2, 0) is None
    assert sm.sym_heap_slot_ptr(d, 1, prs) is None


@pytest.mark.parametrize("bad", [
    dict(num_experts=5),            # E % W != 0
    dict(topk=5),                   # k > E
    dict(hidden=100),               # H % 128 != 0
    dict(inter=64),                 # I < 128
    dict(world=0),
    dict(num_experts=2048, world=2),  # E > 1024
])
def test_bad_shapes_rejected(bad):
    cfg = dict(ms.CONFIGS["tiny"], **bad)
    with pytest.raises(sm.SymmoeError) as ei:
        sm.sym_heap_bytes(cfg)
    assert ei.value.code == sm.SYM_EINVAL


def test_init_errors():
    cfg = ms.CONFIGS["tiny"]
    prs, total = sm.sym_heap_bytes(cfg)
    with pytest.raises(sm.SymmoeError) as ei:
        sm.sym_heap_init(cfg, 1 << 40, total - 1)
    assert ei.value.code == sm.SYM_ENOSPACE
    with pytest.raises(sm.SymmoeError) as ei:
        sm.sym_heap_init(cfg, (1 << 40) + 16, total)       # base not 256-aligned
    assert ei.value.code == sm.SYM_EINVAL
    with pytest.raises(sm.SymmoeError) as ei:
        sm.sym_heap_bytes(cfg, align=3000)
    assert ei.value.code == sm.SYM_EINVAL


def test_calls_reject_bad_pointers_without_device_work():
    cfg = ms.CONFIGS["tiny"]
    prs, total = sm.sym_heap_bytes(cfg)
    d = sm.sym_heap_init(cfg, 1 << 40, total)
    A = 1 << 41  # aligned fake address, never dereferenced on these paths
    cases = [
        lambda: sm.moe_route_topk(d, None, A, A, 0),
        lambda: sm.moe_dispatch(d, A + 8, A, A, 0),          # x not 16-byte aligned
        lambda: sm.moe_expert_ffn(d, A, None, A, 0),
        lambda: sm.moe_combine(d, None, A, A, A + 2, 0),     # out misaligned
        lambda: sm.moe_pipeline(d, A, A, A, A, A, A, A, A, 16, 0),  # unknown mode bit
        lambda: sm.moe_pipeline(d, A, A, A, A, A, A, A, A, 5, 0),  # dedup only staged
        lambda: sm.moe_expert_ffn_ex(d, A, A, A, 2, 0),      # unknown flag
        lambda: sm.moe_combine_ex(d, None, A, A, A, 2, 0),   # unknown flag
        lambda: sm.moe_combine_ex(d, None, A, None, A, 0, 0),  # weighted combine needs w
        lambda: sm.moe_router_logits(d, A + 8, A, A, 0),     # x not 16-byte aligned
        lambda: sm.moe_router_logits(d, A, A, A + 2, 0),     # logits not 4-byte aligned
        lambda: sm.sym_gemm_a2a(d, A + 8, A, 0, 0),          # x not 16-byte aligned
        lambda: sm.sym_gemm_a2a(d, A, A, 2, 0),              # unknown mode bit
        lambda: sm.sym_a2a_gemm(d, A, None, 1, 0),           # no weight
        lambda: sm.sym_a2a_gemm(d, A, A, 4, 0),              # unknown mode bit
        lambda: sm.sym_a2a_gemm(d, A, A, 2, 0),              # copy engines without the fused bit
        lambda: sm.sym_gemm_a2a(d, A, A, 3, 0),              # copy engines: A2A -> GEMM only
        lambda: sm.moe_dispatch_ex(d, A, A, A, 4, 0),        # unknown flag
        lambda: sm.moe_dispatch_ex(d, A, A, A, 3, 0),        # deduplicated and FP8 together
        lambda: sm.moe_pipeline(d, A, A, A, A, A, A, A, A, 9, 0),   # FP8 only staged
        lambda: sm.moe_pipeline(d, A, A, A, A, A, A, A, A, 12, 0),  # deduplicated and FP8 together
    ]
    for c in cases:
        with pytest.raises(sm.SymmoeError) as ei:
            c()
        assert ei.value.code == sm.SYM_EINVAL
    bad = sm.SymHeapDesc.from_buffer_copy(d)
    bad.cap += 1                                              # inconsistent descriptor
    with pytest.raises(sm.SymmoeError):
        sm.moe_route_topk(bad, A, A, A, 0)
    with pytest.raises(sm.SymmoeError) as ei:
        sm.moe_router_splits(bad)
    assert ei.value.code == sm.SYM_EINVAL
    assert d.epoch == 0                                       # rejected calls change nothing


def test_strerror():
    assert sm.sym_strerror(0) == "success"
    assert "wait" in sm.sym_strerror(sm.SYM_ETIMEOUT)
    assert sm.sym_strerror(-99).startswith("unknown")


def test_linear_a2a_shape_rules():
    """GEMM -> A2A needs T % W == 0; A2A -> GEMM needs whole K blocks per
    shard (H % (64*W) == 0), and its copy-engine form W counters in a slot's
    ready window."""
    A = 1 << 41
    def desc(cfg):
        prs, total = sm.sym_heap_bytes(cfg)
        return sm.sym_heap_init(cfg, 1 << 40, total)
    odd_t = desc(dict(world=4, tokens_per_slot=6, hidden=256, num_experts=4, topk=1, inter=128))
    with pytest.raises(sm.SymmoeError) as ei:
        sm.sym_gemm_a2a(odd_t, A, A, 1, 0)
    assert ei.value.code == sm.SYM_EINVAL
    narrow = desc(dict(world=4, tokens_per_slot=8, hidden=128, num_experts=4, topk=1, inter=128))
    with pytest.raises(sm.SymmoeError) as ei:
        sm.sym_a2a_gemm(narrow, A, A, 0, 0)
    assert ei.value.code == sm.SYM_EINVAL
    # 2 slots x 64 tokens, k = 1: cap = 128 rows, one ready word per slot, 2 needed
    few = desc(dict(world=2, tokens_per_slot=64, hidden=128, num_experts=2, topk=1, inter=128))
    assert few.num_ready == 1
    with pytest.raises(sm.SymmoeError) as ei:
        sm.sym_a2a_gemm(few, A, A, 3, 0)
    assert ei.value.code == sm.SYM_ENOSPACE


def test_dedup_dispatch_needs_at_most_32_slots():
    A = 1 << 41
    cfg = dict(world=64, tokens_per_slot=2, hidden=128, num_experts=64, topk=2, inter=128)
    prs, total = sm.sym_heap_bytes(cfg)
    d = sm.sym_heap_init(cfg, 1 << 40, total)
    with pytest.raises(sm.SymmoeError) as ei:
        sm.moe_dispatch_ex(d, A, A, A, sm.SYM_DISPATCH_DEDUP, 0)
    assert ei.value.code == sm.SYM_EINVAL
    assert d.epoch == 0

