// dispatch_noalloc.cu -- the dispatch layout (per-expert counts, receive
// offsets and every pair's receive row) for callers that cannot allocate
// device memory.
//
// The regular dispatch keeps its chunk histograms in the heap's scratch area,
// so a caller must first allocate a heap.  Some callers cannot: a plug-in
// whose host framework hands it only its input and output buffers and owns
// every allocation, or a process that fixes its device-memory footprint at
// start-up and makes no device allocation afterwards.  This file gives them a
// layout call whose only scratch is a file-scope __device__ array, so the
// call itself allocates nothing.
//
// Scratch: `g_noalloc_hist`, SYM_NOALLOC_HIST_MAX int32 (1 MiB) per device
// that loads the library, held until the process exits.  Every call on a
// device shares it and it keeps the last call's contents; nothing in it needs
// to start at zero (the count kernel writes every histogram entry that the
// scan and the position pass later read).  Calls that overlap on the GPU
// (different streams without ordering) race on it.  Its address is looked up
// on the first call on a device (and again after that device's context was
// reset), which therefore must not run under stream capture.
#include <mutex>

#include "symmoe_dev.cuh"

namespace symmoe {

constexpr int NA_CHUNK = SYM_COUNT_CHUNK;  // 128 tokens per chunk

static __device__ __align__(256) int32_t g_noalloc_hist[SYM_NOALLOC_HIST_MAX];

// per chunk: bitmask of the chunk's tokens per expert -> rank of each pair
// inside the chunk (written to pos) and the chunk histogram (hist[e][chunk])
__global__ void __launch_bounds__(NA_CHUNK)
    noalloc_count_kernel(const int32_t *__restrict__ idx, int32_t *__restrict__ pos,
                         int32_t *__restrict__ hist, int n, int E, int k, int nchunks) {
  extern __shared__ uint32_t mask[];  // [E][NA_CHUNK/32]
  const int chunk = blockIdx.x, t = threadIdx.x, g = chunk * NA_CHUNK + t;
  for (int i = t; i < E * (NA_CHUNK / 32); i += NA_CHUNK) mask[i] = 0;
  __syncthreads();
  const uint32_t bit = 1u << (t & 31);
  const int word = t >> 5;
  // a token that lists an expert twice sets its bit once: the later copies
  // (dup, one bit per j) are not placed and get pos -1, so every placed pair
  // has its own row and the counts add up to the placed pairs
  uint32_t dup = 0;
  if (g < n) {
    for (int j = 0; j < k; ++j) {
      const int e = idx[(size_t)g * k + j];
      if (e >= 0 && e < E && (atomicOr(&mask[e * (NA_CHUNK / 32) + word], bit) & bit)) dup |= 1u << j;
    }
  }
  __syncthreads();
  if (g < n) {
    for (int j = 0; j < k; ++j) {
      const int e = idx[(size_t)g * k + j];
      int r = -1;
      if (e >= 0 && e < E && !((dup >> j) & 1u)) {
        const uint32_t *m = mask + e * (NA_CHUNK / 32);
        r = __popc(m[word] & (bit - 1u));
        for (int w = 0; w < word; ++w) r += __popc(m[w]);
      }
      pos[(size_t)g * k + j] = r;
    }
  }
  for (int e = t; e < E; e += NA_CHUNK) {
    const uint32_t *m = mask + e * (NA_CHUNK / 32);
    int c = 0;
#pragma unroll
    for (int w = 0; w < NA_CHUNK / 32; ++w) c += __popc(m[w]);
    hist[(size_t)e * nchunks + chunk] = c;
  }
}

// one CTA: exclusive scan of the chunk histograms per expert (in place), then
// counts, receive offsets inside each slot, and rows per slot
__global__ void __launch_bounds__(1024)
    noalloc_scan_kernel(int32_t *__restrict__ hist, int32_t *__restrict__ cnt,
                        int32_t *__restrict__ recv_off, int32_t *__restrict__ total_recv, int E,
                        int W, int nchunks) {
  __shared__ int32_t cnt_s[1024];
  const int E_loc = E / W;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int e = wid; e < E; e += nw) {
    int32_t *row = hist + (size_t)e * nchunks;
    int carry = 0;
    for (int c0 = 0; c0 < nchunks; c0 += 32) {
      const int c = c0 + lane;
      const int v = c < nchunks ? row[c] : 0;
      int incl = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      if (c < nchunks) row[c] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) cnt_s[e] = carry;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int d = e / E_loc, l = e % E_loc;
    int off = 0;
    for (int i = 0; i < l; ++i) off += cnt_s[d * E_loc + i];
    cnt[e] = cnt_s[e];
    recv_off[e] = off;
    if (l == E_loc - 1) total_recv[d] = off + cnt_s[e];
  }
}

// pos = recv_off[e] + chunk base of e + rank inside the chunk
__global__ void __launch_bounds__(256)
    noalloc_pos_kernel(const int32_t *__restrict__ idx, const int32_t *__restrict__ hist,
                       const int32_t *__restrict__ recv_off, int32_t *__restrict__ pos, int n,
                       int E, int k, int nchunks) {
  const int p = blockIdx.x * blockDim.x + threadIdx.x;
  if (p >= n * k) return;
  const int g = p / k;
  const int e = idx[p];
  const int r = pos[p];
  if (e < 0 || e >= E || r < 0) {
    pos[p] = -1;
    return;
  }
  pos[p] = recv_off[e] + hist[(size_t)e * nchunks + g / NA_CHUNK] + r;
}

namespace {
std::mutex g_setup_mu;
int32_t *g_hist_ptr[64] = {nullptr};
void *g_hist_ctx[64] = {nullptr};  // the context each address was taken in

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  }
  return fn;
}
}  // namespace

// Device address of the scratch array on the current device.  Looked up once
// per device with that device current, and again only if the device's
// context has changed since (cudaDeviceReset tears the old one down and the
// array may then sit elsewhere).  A look-up cannot run while `st` is being
// captured: that case returns SYM_EINVAL.
static int noalloc_scratch(int32_t **out, cudaStream_t st) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SYM_ECUDA;
  if (dev < 0 || dev >= 64) return SYM_ECUDA;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  CUcontext ctx = nullptr;
  CtxGetCurrentFn getctx = ctx_get_current();
  if (getctx && getctx(&ctx) != CUDA_SUCCESS) ctx = nullptr;
  if (!g_hist_ptr[dev] || (ctx && ctx != g_hist_ctx[dev])) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) return SYM_ECUDA;
    if (cap != cudaStreamCaptureStatusNone) return SYM_EINVAL;
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_hist) != cudaSuccess) return SYM_ECUDA;
    g_hist_ptr[dev] = static_cast<int32_t *>(p);
    g_hist_ctx[dev] = ctx;
  }
  *out = g_hist_ptr[dev];
  return SYM_OK;
}

}  // namespace symmoe

extern "C" int moe_dispatch_layout_noalloc(const moe_shape *s, const int32_t *idx, int32_t *cnt,
                                           int32_t *recv_off, int32_t *total_recv, int32_t *pos,
                                           symmoe_stream_t stream) {
  using namespace symmoe;
  if (!s || !idx || !cnt || !recv_off || !total_recv || !pos) return SYM_EINVAL;
  const int64_t W = s->world, T = s->tokens_per_slot, E = s->num_experts, k = s->topk;
  if (W < 1 || T < 1 || E < 1 || k < 1 || E % W != 0 || E > 1024 || k > E || k > 32)
    return SYM_EINVAL;
  const int64_t n = W * T;
  if (n * k >= (int64_t(1) << 31)) return SYM_EINVAL;
  const int64_t nchunks = (n + NA_CHUNK - 1) / NA_CHUNK;
  if (E * nchunks > SYM_NOALLOC_HIST_MAX) return SYM_ENOSPACE;
  const cudaStream_t st = (cudaStream_t)stream;
  int32_t *hist = nullptr;
  const int rc = noalloc_scratch(&hist, st);
  if (rc != SYM_OK) return rc;
  // cudaLaunchKernel reports each launch's own error: an error that an
  // earlier, unrelated launch left behind is neither blamed on this call nor
  // cleared by it
  int ni = (int)n, Ei = (int)E, ki = (int)k, Wi = (int)W, nc = (int)nchunks;
  const size_t mask_bytes = (size_t)E * (NA_CHUNK / 32) * sizeof(uint32_t);
  void *a_count[] = {(void *)&idx, (void *)&pos, (void *)&hist, &ni, &Ei, &ki, &nc};
  if (cudaLaunchKernel(noalloc_count_kernel, dim3((unsigned)nchunks), dim3(NA_CHUNK), a_count, mask_bytes, st) !=
      cudaSuccess)
    return SYM_ECUDA;
  void *a_scan[] = {(void *)&hist, (void *)&cnt, (void *)&recv_off, (void *)&total_recv, &Ei, &Wi, &nc};
  if (cudaLaunchKernel(noalloc_scan_kernel, dim3(1), dim3(1024), a_scan, 0, st) != cudaSuccess) return SYM_ECUDA;
  void *a_pos[] = {(void *)&idx, (void *)&hist, (void *)&recv_off, (void *)&pos, &ni, &Ei, &ki, &nc};
  if (cudaLaunchKernel(noalloc_pos_kernel, dim3((unsigned)((n * k + 255) / 256)), dim3(256), a_pos, 0, st) !=
      cudaSuccess)
    return SYM_ECUDA;
  return SYM_OK;
}
