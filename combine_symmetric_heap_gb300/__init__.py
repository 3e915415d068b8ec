"""Zero-copy MoE dispatch -> expert -> combine over a flat symmetric heap, GB300.

Thin Python binding of the C-ABI library ``libsymmoe.so`` (declared in
``include/symmoe.h``).  Functions keep the C names and only marshal
arguments: torch tensors or raw device addresses in, ``SymmoeError`` on a
non-zero return.  Every step of the path runs in the library's CUDA kernels;
torch is used for device memory and streams only.  There is no CPU fallback:
importing the package fails loudly if the library has not been built
(``python combine_symmetric_heap_gb300/build.py``).

``SymHeap`` is a convenience owner of one heap allocation (a torch uint8
tensor) with zero-copy tensor views of its windows, e.g.
``heap.combine_in_view()`` -- the expert-output window whose ``data_ptr``
``moe_combine`` recognises (MORI CCO blog, "Zero-copy MoE dispatch -> expert
-> combine": combine skips its staging copy when the expert wrote into the
view it handed out).
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libsymmoe.so")

SYM_OK = 0
SYM_EINVAL = -1
SYM_ENOSPACE = -2
SYM_ECUDA = -3
SYM_ETIMEOUT = -4
SYM_EOVERFLOW = -5
SYM_ENOTSUP = -6
SYM_STATUS_TIMEOUT = 0x1
SYM_STATUS_OVERFLOW = 0x2
SYM_ROWS_PER_FLAG = 128
SYM_COUNT_CHUNK = 128
SYM_GUARD_BYTES = 1024
SYM_HEAP_WINDOWS = 13

_u64 = ctypes.c_uint64
_u32 = ctypes.c_uint32
_i32 = ctypes.c_int32
_vp = ctypes.c_void_p


class MoeShape(ctypes.Structure):
    _fields_ = [("world", _i32), ("tokens_per_slot", _i32), ("hidden", _i32),
                ("inter", _i32), ("num_experts", _i32), ("topk", _i32)]


class SymHeapDesc(ctypes.Structure):
    _fields_ = [("base", _u64), ("per_rank_size", _u64), ("bytes", _u64), ("cap", _u64),
                ("off_recv_x", _u64), ("off_y", _u64), ("off_h", _u64),
                ("off_recv_pair", _u64), ("off_recv_w", _u64), ("off_pos", _u64),
                ("off_cnt", _u64), ("off_recv_off", _u64), ("off_total", _u64),
                ("off_status", _u64), ("off_ready", _u64), ("off_hist", _u64),
                ("off_ctrl", _u64), ("num_ready", _u32), ("epoch", _u32),
                ("wait_timeout_us", _u32), ("reserved", _u32), ("s", MoeShape)]


class SymmoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {sym_strerror(code)} ({code})")


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libsymmoe.so not built ({LIB_PATH}); run "
                               "python combine_symmetric_heap_gb300/build.py")
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.POINTER
        L.sym_heap_bytes.argtypes = [P(MoeShape), _u64, P(_u64), P(_u64)]
        L.sym_heap_init.argtypes = [P(MoeShape), _vp, _u64, _u64, P(SymHeapDesc)]
        L.sym_heap_slot_ptr.argtypes = [P(SymHeapDesc), ctypes.c_int, _u64]
        L.sym_heap_slot_ptr.restype = _vp
        L.sym_heap_windows.argtypes = [P(SymHeapDesc), P(_u64), P(_u64), ctypes.c_int]
        L.moe_route_topk.argtypes = [P(SymHeapDesc), _vp, _vp, _vp, _vp]
        L.moe_router_logits.argtypes = [P(SymHeapDesc), _vp, _vp, _vp, _vp]
        L.moe_router_splits.argtypes = [P(SymHeapDesc), P(ctypes.c_int)]
        L.moe_dispatch.argtypes = [P(SymHeapDesc), _vp, _vp, _vp, _vp]
        L.moe_dispatch_ex.argtypes = [P(SymHeapDesc), _vp, _vp, _vp, ctypes.c_int, _vp]
        L.moe_expert_ffn.argtypes = [P(SymHeapDesc), _vp, _vp, _vp, _vp]
        L.moe_expert_ffn_ex.argtypes = [P(SymHeapDesc), _vp, _vp, _vp, ctypes.c_int, _vp]
        L.moe_combine.argtypes = [P(SymHeapDesc), _vp, _vp, _vp, _vp, _vp]
        L.moe_combine_ex.argtypes = [P(SymHeapDesc), _vp, _vp, _vp, _vp, ctypes.c_int, _vp]
        L.moe_combine_fallback_copies.restype = _u64
        L.moe_pipeline.argtypes = [P(SymHeapDesc), _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                   ctypes.c_int, _vp]
        L.sym_heap_status.argtypes = [P(SymHeapDesc), P(_i32), ctypes.c_int, _vp]
        L.sym_gemm_a2a.argtypes = [P(SymHeapDesc), _vp, _vp, ctypes.c_int, _vp]
        L.sym_a2a_gemm.argtypes = [P(SymHeapDesc), _vp, _vp, ctypes.c_int, _vp]
        L.moe_dispatch_layout_noalloc.argtypes = [P(MoeShape), _vp, _vp, _vp, _vp, _vp, _vp]
        L.sym_strerror.argtypes = [ctypes.c_int]
        L.sym_strerror.restype = ctypes.c_char_p
        _lib = L
    return _lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        return x.data_ptr()
    return int(x)


def _stream(s) -> int | None:
    if s is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(s, torch.cuda.Stream):
        return s.cuda_stream
    return int(s)


def _check(rc: int, where: str) -> None:
    if rc != SYM_OK:
        raise SymmoeError(rc, where)


def _shape(shape) -> MoeShape:
    if isinstance(shape, MoeShape):
        return shape
    return MoeShape(shape["world"], shape["tokens_per_slot"], shape["hidden"], shape["inter"],
                    shape["num_experts"], shape["topk"])


# ------------------------------------------------------------------ C calls

def sym_strerror(code: int) -> str:
    return lib().sym_strerror(code).decode()


def sym_heap_bytes(shape, align: int = 0):
    prs, tot = _u64(), _u64()
    s = _shape(shape)
    _check(lib().sym_heap_bytes(ctypes.byref(s), align, ctypes.byref(prs), ctypes.byref(tot)),
           "sym_heap_bytes")
    return prs.value, tot.value


def sym_heap_init(shape, dev_base, nbytes: int, align: int = 0) -> SymHeapDesc:
    out = SymHeapDesc()
    s = _shape(shape)
    _check(lib().sym_heap_init(ctypes.byref(s), _ptr(dev_base), nbytes, align, ctypes.byref(out)),
           "sym_heap_init")
    return out


def sym_heap_slot_ptr(heap: SymHeapDesc, slot: int, offset: int) -> int | None:
    return lib().sym_heap_slot_ptr(ctypes.byref(heap), slot, offset)


def moe_route_topk(heap: SymHeapDesc, logits, idx, w, stream=None) -> None:
    _check(lib().moe_route_topk(ctypes.byref(heap), _ptr(logits), _ptr(idx), _ptr(w),
                                _stream(stream)), "moe_route_topk")


def moe_router_logits(heap: SymHeapDesc, x, w_router, logits, stream=None) -> None:
    _check(lib().moe_router_logits(ctypes.byref(heap), _ptr(x), _ptr(w_router), _ptr(logits),
                                   _stream(stream)), "moe_router_logits")


def moe_router_splits(heap: SymHeapDesc) -> int:
    out = ctypes.c_int(0)
    _check(lib().moe_router_splits(ctypes.byref(heap), ctypes.byref(out)), "moe_router_splits")
    return out.value


def moe_dispatch(heap: SymHeapDesc, x, idx, w, stream=None) -> None:
    _check(lib().moe_dispatch(ctypes.byref(heap), _ptr(x), _ptr(idx), _ptr(w), _stream(stream)),
           "moe_dispatch")


def moe_expert_ffn(heap: SymHeapDesc, w_gate, w_up, w_down, stream=None) -> None:
    _check(lib().moe_expert_ffn(ctypes.byref(heap), _ptr(w_gate), _ptr(w_up), _ptr(w_down),
                                _stream(stream)), "moe_expert_ffn")


def moe_combine(heap: SymHeapDesc, expert_out, idx, w, out, stream=None) -> None:
    _check(lib().moe_combine(ctypes.byref(heap), _ptr(expert_out), _ptr(idx), _ptr(w), _ptr(out),
                             _stream(stream)), "moe_combine")


# flags of the _ex calls and pipeline modes (include/symmoe.h)
SYM_FFN_WEIGHTED_ROWS = 1
SYM_COMBINE_UNWEIGHTED = 1
SYM_PIPE_FUSED = 1
SYM_PIPE_WEIGHTS_IN_FFN = 2
SYM_PIPE_DEDUP = 4
SYM_PIPE_FP8 = 8
SYM_LA_FUSED = 1
SYM_DISPATCH_DEDUP = 1
SYM_DISPATCH_FP8 = 2
SYM_LA_COPY_ENGINES = 2


def sym_gemm_a2a(heap: SymHeapDesc, x, w, mode: int = 0, stream=None) -> None:
    """GEMM -> all-to-all: slot s's rows of x through w, exchanged in W row
    blocks into the y windows (mode SYM_LA_FUSED: the epilogue stores at the
    destination; 0: GEMM, then a copy kernel)."""
    _check(lib().sym_gemm_a2a(ctypes.byref(heap), _ptr(x), _ptr(w), int(mode), _stream(stream)),
           "sym_gemm_a2a")


def sym_a2a_gemm(heap: SymHeapDesc, z, w, mode: int = 0, stream=None) -> None:
    """All-to-all -> GEMM: K-shards z [W][N][H/W] gathered per slot, then w;
    results in the y windows (mode SYM_LA_FUSED: the GEMM reads each shard in
    place; SYM_LA_FUSED | SYM_LA_COPY_ENGINES: copy-engine copies consumed as
    they land; 0: a copy kernel, then the GEMM)."""
    _check(lib().sym_a2a_gemm(ctypes.byref(heap), _ptr(z), _ptr(w), int(mode), _stream(stream)),
           "sym_a2a_gemm")


def moe_dispatch_ex(heap: SymHeapDesc, x, idx, w, flags: int = 0, stream=None) -> None:
    """flags: SYM_DISPATCH_DEDUP for the rank-deduplicated dispatch (same windows),
    SYM_DISPATCH_FP8 for the FP8 dispatch with per-token scales."""
    _check(lib().moe_dispatch_ex(ctypes.byref(heap), _ptr(x), _ptr(idx), _ptr(w), int(flags),
                                 _stream(stream)), "moe_dispatch_ex")


def moe_expert_ffn_ex(heap: SymHeapDesc, w_gate, w_up, w_down, flags: int = 0, stream=None) -> None:
    _check(lib().moe_expert_ffn_ex(ctypes.byref(heap), _ptr(w_gate), _ptr(w_up), _ptr(w_down),
                                   int(flags), _stream(stream)), "moe_expert_ffn_ex")


def moe_combine_ex(heap: SymHeapDesc, expert_out, idx, w, out, flags: int = 0, stream=None) -> None:
    _check(lib().moe_combine_ex(ctypes.byref(heap), _ptr(expert_out), _ptr(idx), _ptr(w), _ptr(out),
                                int(flags), _stream(stream)), "moe_combine_ex")


def moe_combine_fallback_copies() -> int:
    return int(lib().moe_combine_fallback_copies())


def moe_pipeline(heap: SymHeapDesc, logits, x, w_gate, w_up, w_down, idx, w, out,
                 mode: int = 0, stream=None) -> None:
    """mode: SYM_PIPE_FUSED, SYM_PIPE_WEIGHTS_IN_FFN, SYM_PIPE_DEDUP bits (0: staged)."""
    _check(lib().moe_pipeline(ctypes.byref(heap), _ptr(logits), _ptr(x), _ptr(w_gate),
                              _ptr(w_up), _ptr(w_down), _ptr(idx), _ptr(w), _ptr(out),
                              int(mode), _stream(stream)), "moe_pipeline")


def moe_dispatch_layout_noalloc(shape, idx, cnt, recv_off, total_recv, pos, stream=None) -> None:
    """Dispatch layout from the routing indices alone, for callers that cannot
    allocate device memory (its scratch is a library-owned device array)."""
    s = _shape(dict(shape, hidden=shape.get("hidden", 128), inter=shape.get("inter", 128)))
    _check(lib().moe_dispatch_layout_noalloc(ctypes.byref(s), _ptr(idx), _ptr(cnt), _ptr(recv_off),
                                             _ptr(total_recv), _ptr(pos), _stream(stream)),
           "moe_dispatch_layout_noalloc")


def sym_heap_windows(heap: SymHeapDesc) -> list:
    """(offset, bytes) of every window inside a slot, in layout order."""
    n = SYM_HEAP_WINDOWS
    offs, sizes = (_u64 * n)(), (_u64 * n)()
    rc = lib().sym_heap_windows(ctypes.byref(heap), offs, sizes, n)
    if rc < 0:
        raise SymmoeError(rc, "sym_heap_windows")
    return [(int(offs[i]), int(sizes[i])) for i in range(rc)]


def sym_heap_status(heap: SymHeapDesc, clear: bool = False, stream=None) -> int:
    st = _i32()
    _check(lib().sym_heap_status(ctypes.byref(heap), ctypes.byref(st), int(clear), _stream(stream)),
           "sym_heap_status")
    return st.value


# ------------------------------------------------------------------ heap owner

class SymHeap:
    """One symmetric heap in a torch-owned device allocation, with views.

    Every view is a slice of ``self.buf`` (no copy); slot ``d``'s copy of a
    window starts at ``d * per_rank_size + off``.
    """

    def __init__(self, shape: dict, device="cuda", align: int = 0):
        self.shape = dict(shape)
        prs, total = sym_heap_bytes(shape, align)
        # zeroed once: the status word and the fused-kernel counters start at 0
        self.buf = torch.zeros(total + 256, dtype=torch.uint8, device=device)
        pad = (-self.buf.data_ptr()) % 256
        self.buf = self.buf[pad:pad + total]
        self.desc = sym_heap_init(shape, self.buf.data_ptr(), total, align)

    # raw window views --------------------------------------------------
    def _win(self, slot: int, off: int, nbytes: int, dtype) -> torch.Tensor:
        base = slot * self.desc.per_rank_size + off
        return self.buf[base:base + nbytes].view(dtype)

    @property
    def cap(self) -> int:
        return self.desc.cap

    def recv_x(self, d: int) -> torch.Tensor:
        H = self.shape["hidden"]
        return self._win(d, self.desc.off_recv_x, self.cap * H * 2, torch.bfloat16).view(self.cap, H)

    def y(self, d: int) -> torch.Tensor:
        H = self.shape["hidden"]
        return self._win(d, self.desc.off_y, self.cap * H * 2, torch.bfloat16).view(self.cap, H)

    def h(self, d: int) -> torch.Tensor:
        I = self.shape["inter"]
        return self._win(d, self.desc.off_h, self.cap * I * 2, torch.bfloat16).view(self.cap, I)

    def recv_pair(self, d: int) -> torch.Tensor:
        return self._win(d, self.desc.off_recv_pair, self.cap * 4, torch.int32)

    def recv_w(self, d: int) -> torch.Tensor:
        return self._win(d, self.desc.off_recv_w, self.cap * 4, torch.float32)

    def pos(self, d: int) -> torch.Tensor:
        T, k = self.shape["tokens_per_slot"], self.shape["topk"]
        return self._win(d, self.desc.off_pos, T * k * 4, torch.int32).view(T, k)

    def cnt(self, d: int) -> torch.Tensor:
        el = self.shape["num_experts"] // self.shape["world"]
        return self._win(d, self.desc.off_cnt, el * 4, torch.int32)

    def recv_off(self, d: int) -> torch.Tensor:
        el = self.shape["num_experts"] // self.shape["world"]
        return self._win(d, self.desc.off_recv_off, el * 4, torch.int32)

    def total_recv(self, d: int) -> torch.Tensor:
        return self._win(d, self.desc.off_total, 4, torch.int32)

    def ready(self, d: int) -> torch.Tensor:
        return self._win(d, self.desc.off_ready, self.desc.num_ready * 4, torch.int32)

    def combine_in_view(self) -> torch.Tensor:
        """Expert-output window as [W, cap, H] (strided by the slot size);
        its data_ptr is the one moe_combine treats as zero-copy."""
        H = self.shape["hidden"]
        W = self.shape["world"]
        base = self.buf[self.desc.off_y:].view(torch.bfloat16)
        return base.as_strided((W, self.cap, H), (self.desc.per_rank_size // 2, H, 1))

    def status(self, clear: bool = False, stream=None) -> int:
        return sym_heap_status(self.desc, clear, stream)

    def guard_bands(self) -> list:
        """(start, length) byte ranges of ``self.buf`` that no call touches:
        the bands after every window of every slot."""
        wins = sym_heap_windows(self.desc)
        prs = self.desc.per_rank_size
        ends = [o + b for o, b in wins]
        starts = [o for o, _ in wins[1:]] + [prs]
        return [(d * prs + e, s - e) for d in range(self.shape["world"]) for e, s in zip(ends, starts)]

    # calls -----------------------------------------------------------------
    def route_topk(self, logits, idx, w, stream=None):
        moe_route_topk(self.desc, logits, idx, w, stream)

    def router_logits(self, x, w_router, logits, stream=None):
        moe_router_logits(self.desc, x, w_router, logits, stream)

    def router_splits(self) -> int:
        return moe_router_splits(self.desc)

    def dispatch(self, x, idx, w, dedup=False, fp8=False, stream=None):
        moe_dispatch_ex(self.desc, x, idx, w,
                        (SYM_DISPATCH_DEDUP if dedup else 0) | (SYM_DISPATCH_FP8 if fp8 else 0), stream)

    def expert_ffn(self, wg, wu, wd, weighted_rows=False, stream=None):
        moe_expert_ffn_ex(self.desc, wg, wu, wd, SYM_FFN_WEIGHTED_ROWS if weighted_rows else 0, stream)

    def combine(self, idx, w, out, expert_out=None, unweighted=False, stream=None):
        moe_combine_ex(self.desc, expert_out, idx, w, out, SYM_COMBINE_UNWEIGHTED if unweighted else 0,
                       stream)

    def pipeline(self, logits, x, wg, wu, wd, idx, w, out, fused=0, weights_in_ffn=False, dedup=False,
                 fp8=False, stream=None):
        mode = ((SYM_PIPE_FUSED if fused else 0) | (SYM_PIPE_WEIGHTS_IN_FFN if weights_in_ffn else 0)
                | (SYM_PIPE_DEDUP if dedup else 0) | (SYM_PIPE_FP8 if fp8 else 0))
        moe_pipeline(self.desc, logits, x, wg, wu, wd, idx, w, out, mode, stream)

    def gemm_a2a(self, x, w, fused=False, stream=None):
        sym_gemm_a2a(self.desc, x, w, SYM_LA_FUSED if fused else 0, stream)

    def a2a_gemm(self, z, w, fused=False, copy_engines=False, stream=None):
        mode = (SYM_LA_FUSED | (SYM_LA_COPY_ENGINES if copy_engines else 0)) if fused else 0
        sym_a2a_gemm(self.desc, z, w, mode, stream)


lib()  # fail loudly at import if the CUDA library is missing
