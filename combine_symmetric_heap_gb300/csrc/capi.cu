// capi.cu -- the extern "C" boundary of libsymmoe: argument validation, the
// symmetric heap layout, and the launch sequence of every call.
//
// Heap layout (MORI CCO guide, "3. Memory and Windows": windows are registered
// collectively, in the same order and with the same size on every rank, so
// each sits at the same offset in every slot).  Windows of one slot, in this
// order, each 1024-byte aligned and followed by a guard band of at least
// SYM_GUARD_BYTES: recv_x, y, h, recv_pair, recv_w, pos, cnt, recv_off, total,
// status, ready, hist, ctrl.  per_rank_size is the sum rounded up to the
// caller's alignment.
#include <atomic>
#include <cstring>

#include "symmoe_dev.cuh"

namespace symmoe {
cudaError_t launch_route_topk(const sym_heap &h, const float *logits, int32_t *idx, float *w,
                              cudaStream_t st);
cudaError_t launch_dispatch(const sym_heap &h, const uint16_t *x, const int32_t *idx,
                            const float *w, int mode, cudaStream_t st);
cudaError_t launch_expert_ffn(const sym_heap &h, const uint16_t *wg, const uint16_t *wu,
                              const uint16_t *wd, int num_sms, int wait_ready, int scale_rows,
                              cudaStream_t st);
cudaError_t launch_combine(const sym_heap &h, const uint16_t *expert_out, const int32_t *idx,
                           const float *w, uint16_t *out, int unit_weights, int num_sms, cudaStream_t st);
cudaError_t launch_router(const sym_heap &h, const uint16_t *x, const uint16_t *wr, float *logits,
                          int num_sms, cudaStream_t st);
cudaError_t router_plan(const sym_heap &h, int num_sms, int *grid, int *splits, int *kb_per_split);
cudaError_t launch_gemm_a2a(const sym_heap &h, const uint16_t *x, const uint16_t *w, int fused, int num_sms,
                            cudaStream_t st);
cudaError_t launch_a2a_gemm(const sym_heap &h, const uint16_t *z, const uint16_t *w, int mode, int num_sms,
                            cudaStream_t st);
int a2a_gemm_counters(const sym_heap &h);
size_t fused_ctrl_bytes(const moe_shape &s);
cudaError_t launch_fused(const sym_heap &h, const float *logits, const uint16_t *x,
                         const uint16_t *wg, const uint16_t *wu, const uint16_t *wd,
                         int32_t *idx, float *w, uint16_t *out, int weights_in_ffn, int num_sms,
                         cudaStream_t st);
}  // namespace symmoe

using namespace symmoe;

namespace {

constexpr uint64_t kWinAlign = 1024;
constexpr uint64_t kDefaultAlign = 2ull << 20;
constexpr uint32_t kDefaultTimeoutUs = 2000000u;

std::atomic<uint64_t> g_fallback_copies{0};

uint64_t round_up(uint64_t v, uint64_t a) { return (v + a - 1) / a * a; }

bool shape_ok(const moe_shape *s) {
  if (!s) return false;
  const int64_t W = s->world, T = s->tokens_per_slot, H = s->hidden, I = s->inter,
                E = s->num_experts, k = s->topk;
  if (W < 1 || T < 1 || E < 1 || k < 1) return false;
  if (E % W != 0 || E > 1024) return false;
  if (k > E || k > 32) return false;
  if (H < 128 || H % 128 != 0 || H > 65536) return false;
  if (I < 128 || I % 128 != 0 || I > 65536) return false;
  const int64_t N = W * T;
  if (N * k >= (int64_t(1) << 31) || N >= (int64_t(1) << 31)) return false;
  return true;
}

struct Layout {
  uint64_t cap, off_recv_x, off_y, off_h, off_recv_pair, off_recv_w, off_pos, off_cnt,
      off_recv_off, off_total, off_status, off_ready, off_hist, off_ctrl, used;
  uint32_t num_ready;
  uint64_t win_off[SYM_HEAP_WINDOWS], win_bytes[SYM_HEAP_WINDOWS];  // in slot order
};

Layout layout_of(const moe_shape *s) {
  Layout L{};
  const uint64_t W = s->world, T = s->tokens_per_slot, H = s->hidden, I = s->inter,
                 E = s->num_experts, k = s->topk;
  const uint64_t N = W * T, E_loc = E / W;
  L.cap = N * (k < E_loc ? k : E_loc);
  L.num_ready = (uint32_t)((L.cap + SYM_ROWS_PER_FLAG - 1) / SYM_ROWS_PER_FLAG);
  uint64_t o = 0;
  int nwin = 0;
  // every window is followed by at least SYM_GUARD_BYTES that no call reads
  // or writes (a guard band: a store past a window's end lands there first)
  auto take = [&](uint64_t bytes) {
    const uint64_t at = o;
    L.win_off[nwin] = at;
    L.win_bytes[nwin++] = bytes;
    o = round_up(o + bytes + SYM_GUARD_BYTES, kWinAlign);
    return at;
  };
  L.off_recv_x = take(L.cap * H * 2);
  L.off_y = take(L.cap * H * 2);
  L.off_h = take(L.cap * I * 2);
  L.off_recv_pair = take(L.cap * 4);
  L.off_recv_w = take(L.cap * 4);
  L.off_pos = take(T * k * 4);
  L.off_cnt = take(E_loc * 4);
  L.off_recv_off = take(E_loc * 4);
  L.off_total = take(4);
  L.off_status = take(4);
  L.off_ready = take((uint64_t)L.num_ready * 4);
  // chunk histograms: 128-token chunks for the stand-alone dispatch, 32-token
  // chunks for the fused pipeline (the larger of the two)
  L.off_hist = take(E * ((N + 31) / 32) * 4);
  L.off_ctrl = take(fused_ctrl_bytes(*s));
  L.used = o;
  return L;
}

bool heap_ok(const sym_heap *h) {
  if (!h || !shape_ok(&h->s) || h->base == 0 || (h->base & 255u)) return false;
  const Layout L = layout_of(&h->s);
  return h->cap == L.cap && h->per_rank_size >= L.used && h->off_ctrl == L.off_ctrl &&
         h->num_ready == L.num_ready;
}

bool aligned16(const void *p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return p && (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

int num_sms_of_current_device() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  if (dev < 64 && cache[dev]) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev < 64) cache[dev] = n;
  return n;
}

int from_cuda(cudaError_t e) { return e == cudaSuccess ? SYM_OK : SYM_ECUDA; }

}  // namespace

extern "C" {

int sym_heap_bytes(const moe_shape *s, uint64_t align, uint64_t *per_rank_size,
                   uint64_t *total_bytes) {
  if (!shape_ok(s)) return SYM_EINVAL;
  if (align == 0) align = kDefaultAlign;
  if (align < 256 || (align & (align - 1))) return SYM_EINVAL;
  const Layout L = layout_of(s);
  const uint64_t prs = round_up(L.used, align);
  if (per_rank_size) *per_rank_size = prs;
  if (total_bytes) *total_bytes = prs * (uint64_t)s->world;
  return SYM_OK;
}

int sym_heap_init(const moe_shape *s, void *dev_base, uint64_t bytes, uint64_t align,
                  sym_heap *out) {
  if (!out || !dev_base || (reinterpret_cast<uintptr_t>(dev_base) & 255u)) return SYM_EINVAL;
  uint64_t prs = 0, total = 0;
  const int rc = sym_heap_bytes(s, align, &prs, &total);
  if (rc != SYM_OK) return rc;
  if (bytes < total) return SYM_ENOSPACE;
  const Layout L = layout_of(s);
  sym_heap h;
  std::memset(&h, 0, sizeof(h));
  h.base = reinterpret_cast<uint64_t>(dev_base);
  h.per_rank_size = prs;
  h.bytes = total;
  h.cap = L.cap;
  h.off_recv_x = L.off_recv_x;
  h.off_y = L.off_y;
  h.off_h = L.off_h;
  h.off_recv_pair = L.off_recv_pair;
  h.off_recv_w = L.off_recv_w;
  h.off_pos = L.off_pos;
  h.off_cnt = L.off_cnt;
  h.off_recv_off = L.off_recv_off;
  h.off_total = L.off_total;
  h.off_status = L.off_status;
  h.off_ready = L.off_ready;
  h.off_hist = L.off_hist;
  h.off_ctrl = L.off_ctrl;
  h.num_ready = L.num_ready;
  h.epoch = 0;
  h.wait_timeout_us = kDefaultTimeoutUs;
  h.s = *s;
  *out = h;
  return SYM_OK;
}

int sym_heap_windows(const sym_heap *h, uint64_t *offsets, uint64_t *bytes, int max_windows) {
  if (!heap_ok(h) || max_windows < 0 || (max_windows > 0 && (!offsets || !bytes))) return SYM_EINVAL;
  const Layout L = layout_of(&h->s);
  for (int i = 0; i < SYM_HEAP_WINDOWS && i < max_windows; ++i) {
    offsets[i] = L.win_off[i];
    bytes[i] = L.win_bytes[i];
  }
  return SYM_HEAP_WINDOWS;
}

void *sym_heap_slot_ptr(const sym_heap *h, int slot, uint64_t offset) {
  if (!h || slot < 0 || slot >= h->s.world || offset >= h->per_rank_size) return nullptr;
  return reinterpret_cast<void *>(h->base + (uint64_t)slot * h->per_rank_size + offset);
}

int moe_route_topk(const sym_heap *h, const float *logits, int32_t *idx, float *w,
                   symmoe_stream_t stream) {
  if (!heap_ok(h) || !aligned4(logits) || !aligned4(idx) || !aligned4(w)) return SYM_EINVAL;
  return from_cuda(launch_route_topk(*h, logits, idx, w, (cudaStream_t)stream));
}

int moe_router_logits(const sym_heap *h, const uint16_t *x, const uint16_t *w_router, float *logits,
                      symmoe_stream_t stream) {
  if (!heap_ok(h) || !aligned16(x) || !aligned16(w_router) || !aligned4(logits)) return SYM_EINVAL;
  const int sms = num_sms_of_current_device();
  if (sms <= 0) return SYM_ECUDA;
  return from_cuda(launch_router(*h, x, w_router, logits, sms, (cudaStream_t)stream));
}

int moe_router_splits(const sym_heap *h, int *splits) {
  if (!heap_ok(h) || !splits) return SYM_EINVAL;
  const int sms = num_sms_of_current_device();
  if (sms <= 0) return SYM_ECUDA;
  int grid, kb;
  return from_cuda(router_plan(*h, sms, &grid, splits, &kb));
}

int sym_gemm_a2a(const sym_heap *h, const uint16_t *x, const uint16_t *w, int mode, symmoe_stream_t stream) {
  if (!heap_ok(h) || !aligned16(x) || !aligned16(w) || (mode & ~SYM_LA_FUSED) ||
      h->s.tokens_per_slot % h->s.world != 0)
    return SYM_EINVAL;
  const int sms = num_sms_of_current_device();
  if (sms <= 0) return SYM_ECUDA;
  return from_cuda(launch_gemm_a2a(*h, x, w, mode & SYM_LA_FUSED, sms, (cudaStream_t)stream));
}

int sym_a2a_gemm(const sym_heap *h, const uint16_t *z, const uint16_t *w, int mode, symmoe_stream_t stream) {
  if (!heap_ok(h) || !aligned16(z) || !aligned16(w) || (mode & ~(SYM_LA_FUSED | SYM_LA_COPY_ENGINES)) ||
      mode == SYM_LA_COPY_ENGINES || h->s.hidden % (64 * h->s.world) != 0)
    return SYM_EINVAL;
  const bool engines = (mode & SYM_LA_COPY_ENGINES) != 0;
  if (engines && (uint32_t)a2a_gemm_counters(*h) > h->num_ready) return SYM_ENOSPACE;
  const int sms = num_sms_of_current_device();
  if (sms <= 0) return SYM_ECUDA;
  return from_cuda(launch_a2a_gemm(*h, z, w, engines ? 2 : (mode & SYM_LA_FUSED), sms, (cudaStream_t)stream));
}

int moe_dispatch(sym_heap *h, const uint16_t *x, const int32_t *idx, const float *w,
                 symmoe_stream_t stream) {
  return moe_dispatch_ex(h, x, idx, w, 0, stream);
}

// The deduplicated dispatch keeps its scratch in the h windows: per slot the
// row sources [cap], and in slot 0 also the chunk counts [W][N/32] and the
// pair ranks [N][k] (int32).
static bool dedup_fits(const sym_heap *h) {
  const uint64_t W = h->s.world, N = W * h->s.tokens_per_slot, k = h->s.topk;
  const uint64_t need = 4 * (h->cap + W * ((N + 31) / 32) + N * k);
  return W <= 32 && need <= h->cap * (uint64_t)h->s.inter * 2;
}

int moe_dispatch_ex(sym_heap *h, const uint16_t *x, const int32_t *idx, const float *w, int flags,
                    symmoe_stream_t stream) {
  if (!heap_ok(h) || !aligned16(x) || !aligned4(idx) || !aligned4(w) ||
      (flags & ~(SYM_DISPATCH_DEDUP | SYM_DISPATCH_FP8)) || flags == (SYM_DISPATCH_DEDUP | SYM_DISPATCH_FP8))
    return SYM_EINVAL;
  const int mode = (flags & SYM_DISPATCH_FP8) ? 2 : (flags & SYM_DISPATCH_DEDUP) ? 1 : 0;
  if (mode == 1 && !dedup_fits(h)) return SYM_EINVAL;
  h->epoch += 1;
  return from_cuda(launch_dispatch(*h, x, idx, w, mode, (cudaStream_t)stream));
}

int moe_expert_ffn_ex(const sym_heap *h, const uint16_t *w_gate, const uint16_t *w_up,
                      const uint16_t *w_down, int flags, symmoe_stream_t stream) {
  if (!heap_ok(h) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down) ||
      (flags & ~SYM_FFN_WEIGHTED_ROWS))
    return SYM_EINVAL;
  const int sms = num_sms_of_current_device();
  if (sms <= 0) return SYM_ECUDA;
  return from_cuda(launch_expert_ffn(*h, w_gate, w_up, w_down, sms, 1, (flags & SYM_FFN_WEIGHTED_ROWS) ? 1 : 0,
                                     (cudaStream_t)stream));
}

int moe_expert_ffn(const sym_heap *h, const uint16_t *w_gate, const uint16_t *w_up,
                   const uint16_t *w_down, symmoe_stream_t stream) {
  return moe_expert_ffn_ex(h, w_gate, w_up, w_down, 0, stream);
}

int moe_combine_ex(const sym_heap *h, const uint16_t *expert_out, const int32_t *idx,
                   const float *w, uint16_t *out, int flags, symmoe_stream_t stream) {
  const bool unit = (flags & SYM_COMBINE_UNWEIGHTED) != 0;
  if (!heap_ok(h) || !aligned4(idx) || (!unit && !aligned4(w)) || !aligned16(out) ||
      (flags & ~SYM_COMBINE_UNWEIGHTED))
    return SYM_EINVAL;
  const uint16_t *view = reinterpret_cast<const uint16_t *>(h->base + h->off_y);
  const uint16_t *stage = nullptr;
  if (expert_out && expert_out != view) {
    if (!aligned16(expert_out)) return SYM_EINVAL;
    stage = expert_out;
    g_fallback_copies.fetch_add(1);
  }
  const int sms = num_sms_of_current_device();
  if (sms <= 0) return SYM_ECUDA;
  return from_cuda(launch_combine(*h, stage, idx, w, out, unit ? 1 : 0, sms, (cudaStream_t)stream));
}

int moe_combine(const sym_heap *h, const uint16_t *expert_out, const int32_t *idx,
                const float *w, uint16_t *out, symmoe_stream_t stream) {
  return moe_combine_ex(h, expert_out, idx, w, out, 0, stream);
}

uint64_t moe_combine_fallback_copies(void) { return g_fallback_copies.load(); }

int moe_pipeline(sym_heap *h, const float *logits, const uint16_t *x, const uint16_t *w_gate,
                 const uint16_t *w_up, const uint16_t *w_down, int32_t *idx, float *w,
                 uint16_t *out, int mode, symmoe_stream_t stream) {
  if (!heap_ok(h) || !aligned4(logits) || !aligned16(x) || !aligned16(w_gate) ||
      !aligned16(w_up) || !aligned16(w_down) || !aligned4(idx) || !aligned4(w) ||
      !aligned16(out) || (mode & ~(SYM_PIPE_FUSED | SYM_PIPE_WEIGHTS_IN_FFN | SYM_PIPE_DEDUP | SYM_PIPE_FP8)))
    return SYM_EINVAL;
  const int dmode = (mode & SYM_PIPE_FP8) ? 2 : (mode & SYM_PIPE_DEDUP) ? 1 : 0;
  if (dmode && ((mode & SYM_PIPE_FUSED) || ((mode & SYM_PIPE_DEDUP) && (mode & SYM_PIPE_FP8)) ||
                (dmode == 1 && !dedup_fits(h))))
    return SYM_EINVAL;
  const cudaStream_t st = (cudaStream_t)stream;
  const int sms = num_sms_of_current_device();
  if (sms <= 0) return SYM_ECUDA;
  const int weighted = (mode & SYM_PIPE_WEIGHTS_IN_FFN) ? 1 : 0;
  h->epoch += 1;
  if (mode & SYM_PIPE_FUSED)
    return from_cuda(launch_fused(*h, logits, x, w_gate, w_up, w_down, idx, w, out, weighted, sms, st));
  cudaError_t e = launch_route_topk(*h, logits, idx, w, st);
  if (e == cudaSuccess) e = launch_dispatch(*h, x, idx, w, dmode, st);
  if (e == cudaSuccess) e = launch_expert_ffn(*h, w_gate, w_up, w_down, sms, 1, weighted, st);
  if (e == cudaSuccess) e = launch_combine(*h, nullptr, idx, w, out, weighted, sms, st);
  return from_cuda(e);
}

int sym_heap_status(const sym_heap *h, int32_t *status, int clear, symmoe_stream_t stream) {
  if (!h || !status || h->base == 0) return SYM_EINVAL;
  const cudaStream_t st = (cudaStream_t)stream;
  int32_t *dev = reinterpret_cast<int32_t *>(h->base + h->off_status);
  if (cudaStreamSynchronize(st) != cudaSuccess) return SYM_ECUDA;
  if (cudaMemcpy(status, dev, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return SYM_ECUDA;
  if (clear && cudaMemset(dev, 0, sizeof(int32_t)) != cudaSuccess) return SYM_ECUDA;
  return SYM_OK;
}

const char *sym_strerror(int code) {
  switch (code) {
    case SYM_OK: return "success";
    case SYM_EINVAL: return "invalid shape, pointer, alignment or argument";
    case SYM_ENOSPACE: return "heap (or a window of it) too small for the call";
    case SYM_ECUDA: return "CUDA runtime call or kernel launch failed";
    case SYM_ETIMEOUT: return "a bounded device wait expired";
    case SYM_EOVERFLOW: return "a row or expert index out of range";
    case SYM_ENOTSUP: return "not supported on this device";
    default: return "unknown symmoe status code";
  }
}

}  // extern "C"
