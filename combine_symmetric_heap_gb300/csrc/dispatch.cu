// dispatch.cu -- the all-to-all scatter of the zero-copy MoE pipeline.
//
// MORI CCO blog, "Zero-copy MoE dispatch -> expert -> combine": each rank
// writes its tokens directly into the receive window ("disp_out") of the rank
// that owns each selected expert, with no staging copy.  Here every rank is a
// slot of one heap and the "peer store" is a 16-byte vector store to
// base + slot * per_rank_size + off_recv_x + row * H * 2.
//
// Receive order (the pages leave it open): rows grouped by expert, experts
// ascending inside a slot; inside one expert by (source slot, token, k),
// i.e. by global token g because the k experts of a token are distinct.
//
// Three launches, all with programmatic dependent launch (each is scheduled
// while its predecessor drains and waits for that kernel's results on the device):
//   count   one CTA per 128-token chunk: per-expert bitmask of the chunk's
//           tokens in shared memory -> each pair's rank inside the chunk
//           (popcount of the lower bits) and the chunk histogram.
//   scan    one CTA per slot: exclusive scan of the chunk histograms of the
//           slot's experts (a warp per expert), expert counts, receive
//           offsets, total rows; clears the slot's ready counters.
//   scatter one 64-thread CTA per token: x[g] is read once and stored k times
//           (one per destination), then recv_pair / recv_w / pos are written
//           and the ready counter of each destination row block is raised.
#include <cuda_fp16.h>

#include <algorithm>

#include "symmoe_dev.cuh"

namespace symmoe {

constexpr int CHUNK = SYM_COUNT_CHUNK;  // 128 tokens: 4 mask words per expert

__global__ void __launch_bounds__(CHUNK) dispatch_count_kernel(sym_heap h,
                                                               const int32_t *__restrict__ idx) {
  extern __shared__ uint32_t mask[];  // [E][CHUNK/32]
  const int E = h.s.num_experts, k = h.s.topk, T = h.s.tokens_per_slot;
  const int N = h.s.world * T;
  const int nchunks = (N + CHUNK - 1) / CHUNK;
  const int chunk = blockIdx.x;
  const int t = threadIdx.x;
  const int g = chunk * CHUNK + t;
  pdl_launch_dependents();  // the scan may be scheduled now; it waits for this grid
  pdl_wait();               // idx from the routing (or any earlier kernel)
  for (int i = t; i < E * (CHUNK / 32); i += CHUNK) mask[i] = 0;
  __syncthreads();
  const uint32_t bit = 1u << (t & 31);
  const int word = t >> 5;
  if (g < N) {
    for (int j = 0; j < k; ++j) {
      const int e = idx[(size_t)g * k + j];
      if (e < 0 || e >= E) {
        raise_status(h, SYM_STATUS_OVERFLOW);
        continue;
      }
      const uint32_t old = atomicOr(&mask[e * (CHUNK / 32) + word], bit);
      if (old & bit) raise_status(h, SYM_STATUS_OVERFLOW);  // duplicate expert in a token
    }
  }
  __syncthreads();
  if (g < N) {
    int32_t *pos = win<int32_t>(h, g / T, h.off_pos) + (size_t)(g % T) * k;
    for (int j = 0; j < k; ++j) {
      const int e = idx[(size_t)g * k + j];
      int r = -1;
      if (e >= 0 && e < E) {
        const uint32_t *m = mask + e * (CHUNK / 32);
        r = __popc(m[word] & (bit - 1u));
        for (int w = 0; w < word; ++w) r += __popc(m[w]);
      }
      pos[j] = r;  // rank inside the chunk; the scatter adds the bases
    }
  }
  int32_t *hist = win<int32_t>(h, 0, h.off_hist);  // [E][nchunks]
  for (int e = t; e < E; e += CHUNK) {
    const uint32_t *m = mask + e * (CHUNK / 32);
    int c = 0;
#pragma unroll
    for (int w = 0; w < CHUNK / 32; ++w) c += __popc(m[w]);
    hist[(size_t)e * nchunks + chunk] = c;
  }
}

// One CTA per slot: a slot's receive offsets depend only on its own experts.
// A warp per expert scans the expert's chunk histogram row (warp scans, 32
// chunks at a time), then the slot's counts, offsets and total are written
// and its ready counters cleared for this call.
__global__ void __launch_bounds__(1024) dispatch_scan_kernel(sym_heap h) {
  __shared__ int32_t cnt_s[1024];
  const int E = h.s.num_experts, W = h.s.world;
  const int E_loc = E / W;
  const int d = blockIdx.x;
  const int N = W * h.s.tokens_per_slot;
  const int nchunks = (N + CHUNK - 1) / CHUNK;
  int32_t *hist = win<int32_t>(h, 0, h.off_hist);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  pdl_launch_dependents();
  pdl_wait();  // the count kernel's histogram
  for (int l = wid; l < E_loc; l += nw) {
    int32_t *row = hist + (size_t)(d * E_loc + l) * nchunks;
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
    if (lane == 0) cnt_s[l] = carry;
  }
  __syncthreads();
  for (int l = threadIdx.x; l < E_loc; l += blockDim.x) {
    int off = 0;
    for (int i = 0; i < l; ++i) off += cnt_s[i];
    win<int32_t>(h, d, h.off_cnt)[l] = cnt_s[l];
    win<int32_t>(h, d, h.off_recv_off)[l] = off;
    if (l == E_loc - 1) *win<int32_t>(h, d, h.off_total) = off + cnt_s[l];
  }
  for (int i = threadIdx.x; i < (int)h.num_ready; i += blockDim.x) win<uint32_t>(h, d, h.off_ready)[i] = 0u;
}

// Scatter: a CTA of 64 threads per token, each thread holding VEC 16-byte
// vectors of the row in registers between its load and its k stores.  Few
// threads with many vectors keep more rows in flight per SM than many threads
// with few (the register file, not the thread count, is the limit).
constexpr int SCATTER_THREADS = 64;

template <int VEC>
__global__ void __launch_bounds__(SCATTER_THREADS)
    dispatch_scatter_kernel(sym_heap h, const uint4 *__restrict__ x,
                            const int32_t *__restrict__ idx, const float *__restrict__ w) {
  __shared__ uint4 *dst_s[32];
  __shared__ int32_t slot_s[32], row_s[32];
  const int E = h.s.num_experts, k = h.s.topk, T = h.s.tokens_per_slot, H = h.s.hidden;
  const int E_loc = E / h.s.world;
  const int N = h.s.world * T;
  const int nchunks = (N + CHUNK - 1) / CHUNK;
  const int g = blockIdx.x;
  const int tid = threadIdx.x;
  const int nvec = H / 8;  // 16-byte vectors per row
  const uint4 *src = x + (size_t)g * nvec;
  pdl_wait();  // offsets from the scan; nothing is touched before it

  // start the first pass's row loads before resolving the destinations
  uint4 v[VEC];
#pragma unroll
  for (int i = 0; i < VEC; ++i) {
    const int c = tid + i * SCATTER_THREADS;
    if (c < nvec) v[i] = __ldg(src + c);
  }
  if (tid < k) {
    const int j = tid;
    const int e = idx[(size_t)g * k + j];
    int32_t *pos = win<int32_t>(h, g / T, h.off_pos) + (size_t)(g % T) * k;
    uint4 *dst = nullptr;
    int d = -1, p = -1;
    if (e >= 0 && e < E) {
      d = e / E_loc;
      const int l = e % E_loc;
      const int rank = pos[j];
      p = win<int32_t>(h, d, h.off_recv_off)[l] +
          win<int32_t>(h, 0, h.off_hist)[(size_t)e * nchunks + g / CHUNK] + rank;
      if (rank < 0 || p < 0 || (uint64_t)p >= h.cap) {
        raise_status(h, SYM_STATUS_OVERFLOW);
        p = -1;
      } else {
        dst = win<uint4>(h, d, h.off_recv_x) + (size_t)p * nvec;
      }
    }
    pos[j] = p;
    dst_s[j] = dst;
    slot_s[j] = d;
    row_s[j] = p;
  }
  __syncthreads();
  for (int base = 0;;) {
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
      const int c = base + tid + i * SCATTER_THREADS;
      if (c < nvec)
        for (int j = 0; j < k; ++j)
          if (dst_s[j]) dst_s[j][c] = v[i];
    }
    base += VEC * SCATTER_THREADS;
    if (base >= nvec) break;
    // rows wider than one pass
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
      const int c = base + tid + i * SCATTER_THREADS;
      if (c < nvec) v[i] = __ldg(src + c);
    }
  }
  if (tid < k && row_s[tid] >= 0) {
    const int d = slot_s[tid], p = row_s[tid];
    win<int32_t>(h, d, h.off_recv_pair)[p] = g * k + tid;
    win<float>(h, d, h.off_recv_w)[p] = w[(size_t)g * k + tid];
  }
  // every thread's stores precede the barrier; the fence of each signalling
  // thread is cumulative over them (release of the row block)
  __syncthreads();
  if (tid < k && row_s[tid] >= 0) {
    __threadfence();
    atomicAdd(win<uint32_t>(h, slot_s[tid], h.off_ready) + row_s[tid] / SYM_ROWS_PER_FLAG, 1u);
  }
}

// ---------------------------------------------------------------------------
// Rank-deduplicated dispatch: a token crosses to each destination slot once,
// into that slot's staging rows (its y window, idle until the down GEMM), and
// the slot expands the staged rows to its expert rows locally.  The staging
// order is ascending token g per slot; the windows the expert FFN and the
// combine read come out bit-identical to the plain dispatch's.  Scratch in
// the h windows (idle until the gate/up GEMM): per slot d its row sources
// [cap] at the start of its h window; slot 0's h window also holds, after
// that, the per-slot 32-token chunk counts [W][nch] and each pair's rank
// among its chunk's tokens bound for the pair's slot [N][k].
//   dedup_count    one warp per 32 tokens: per slot a ballot of the tokens
//                  with an expert there -> counts and ranks
//   dedup_scan     exclusive scan of each slot's chunk counts
//   dedup_scatter  per token: x[g] read once, stored once per distinct slot
//                  (row base + rank); every pair's receive row (the plain
//                  layout), its metadata and its staging row
//   dedup_expand   per slot and received row: copy the staged row, raise the
//                  row block's ready counter
// ---------------------------------------------------------------------------
constexpr int DEDUP_MAX_WORLD = 32;

__device__ __forceinline__ int32_t *dedup_hist(const sym_heap &h) {
  return reinterpret_cast<int32_t *>(win<uint8_t>(h, 0, h.off_h) + h.cap * 4);
}
__device__ __forceinline__ int32_t *dedup_rank(const sym_heap &h, int nch) {
  return dedup_hist(h) + (size_t)h.s.world * nch;
}

__global__ void __launch_bounds__(256) dedup_count_kernel(sym_heap h, const int32_t *__restrict__ idx) {
  const int W = h.s.world, E_loc = h.s.num_experts / W, k = h.s.topk;
  const int N = W * h.s.tokens_per_slot, nch = (N + 31) / 32;
  const int lane = threadIdx.x & 31, chunk = (int)(blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5));
  pdl_launch_dependents();
  pdl_wait();  // the plain count and scan (and the routing) are done
  if (chunk >= nch) return;
  const int g = chunk * 32 + lane;
  uint32_t mask = 0;
  if (g < N)
    for (int j = 0; j < k; ++j) {
      const int e = idx[(size_t)g * k + j];
      if (e >= 0 && e < h.s.num_experts) mask |= 1u << (e / E_loc);
    }
  int32_t *hist = dedup_hist(h), *rank = dedup_rank(h, nch);
  for (int d = 0; d < W; ++d) {
    const uint32_t b = __ballot_sync(0xffffffffu, (mask >> d) & 1u);
    if (lane == 0) hist[(size_t)d * nch + chunk] = __popc(b);
    if (g < N)
      for (int j = 0; j < k; ++j) {
        const int e = idx[(size_t)g * k + j];
        if (e >= 0 && e < h.s.num_experts && e / E_loc == d)
          rank[(size_t)g * k + j] = __popc(b & ((1u << lane) - 1u));
      }
  }
}

__global__ void __launch_bounds__(1024) dedup_scan_kernel(sym_heap h) {
  const int W = h.s.world, N = W * h.s.tokens_per_slot, nch = (N + 31) / 32;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  pdl_launch_dependents();
  pdl_wait();
  int32_t *hist = dedup_hist(h);
  for (int d = wid; d < W; d += nw) {
    int32_t *row = hist + (size_t)d * nch;
    int carry = 0;
    for (int c0 = 0; c0 < nch; c0 += 32) {
      const int c = c0 + lane;
      const int v = c < nch ? row[c] : 0;
      int incl = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      if (c < nch) row[c] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
}

template <int VEC>
__global__ void __launch_bounds__(SCATTER_THREADS)
    dedup_scatter_kernel(sym_heap h, const uint4 *__restrict__ x, const int32_t *__restrict__ idx,
                         const float *__restrict__ w) {
  __shared__ uint4 *dst_s[32];  // staging row of pair j, or null when an earlier pair has its slot
  const int E = h.s.num_experts, k = h.s.topk, T = h.s.tokens_per_slot, H = h.s.hidden;
  const int E_loc = E / h.s.world;
  const int N = h.s.world * T;
  const int nchunks = (N + CHUNK - 1) / CHUNK, nch = (N + 31) / 32;
  const int g = blockIdx.x;
  const int tid = threadIdx.x;
  const int nvec = H / 8;
  const uint4 *src = x + (size_t)g * nvec;
  pdl_launch_dependents();
  pdl_wait();  // offsets, chunk bases and ranks
  uint4 v[VEC];
#pragma unroll
  for (int i = 0; i < VEC; ++i) {
    const int c = tid + i * SCATTER_THREADS;
    if (c < nvec) v[i] = __ldg(src + c);
  }
  if (tid < k) {
    const int j = tid;
    const int e = idx[(size_t)g * k + j];
    int32_t *pos = win<int32_t>(h, g / T, h.off_pos) + (size_t)(g % T) * k;
    uint4 *dst = nullptr;
    int p = -1;
    if (e >= 0 && e < E) {
      const int d = e / E_loc, l = e % E_loc;
      const int q = dedup_hist(h)[(size_t)d * nch + g / 32] + dedup_rank(h, nch)[(size_t)g * k + j];
      const int rank = pos[j];
      p = win<int32_t>(h, d, h.off_recv_off)[l] +
          win<int32_t>(h, 0, h.off_hist)[(size_t)e * nchunks + g / CHUNK] + rank;
      if (rank < 0 || p < 0 || (uint64_t)p >= h.cap || q < 0 || q >= N) {
        raise_status(h, SYM_STATUS_OVERFLOW);
        p = -1;
      } else {
        bool first = true;  // the first of the token's pairs on slot d carries the row
        for (int i = 0; i < j; ++i) {
          const int ei = idx[(size_t)g * k + i];
          if (ei >= 0 && ei < E && ei / E_loc == d) first = false;
        }
        if (first) dst = win<uint4>(h, d, h.off_y) + (size_t)q * nvec;
        win<int32_t>(h, d, h.off_h)[p] = q;  // row source for the expansion
        win<int32_t>(h, d, h.off_recv_pair)[p] = g * k + j;
        win<float>(h, d, h.off_recv_w)[p] = w[(size_t)g * k + j];
      }
    }
    pos[j] = p;
    dst_s[j] = dst;
  }
  __syncthreads();
  for (int base = 0;;) {
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
      const int c = base + tid + i * SCATTER_THREADS;
      if (c < nvec)
        for (int j = 0; j < k; ++j)
          if (dst_s[j]) dst_s[j][c] = v[i];
    }
    base += VEC * SCATTER_THREADS;
    if (base >= nvec) break;
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
      const int c = base + tid + i * SCATTER_THREADS;
      if (c < nvec) v[i] = __ldg(src + c);
    }
  }
}

// grid (blocks, W): the blocks of slot blockIdx.y stride over its received
// rows (the total is only known on the device).  Each of the 64 threads holds
// VEC 16-byte vectors of a row between load and store (as the scatter does),
// so a row is one round trip to memory; a staged row is read once per pair of
// its token on the slot, so its loads stay cacheable.
constexpr int EXPAND_BLOCKS = 4096;  // over all slots
template <int VEC>
__global__ void __launch_bounds__(SCATTER_THREADS) dedup_expand_kernel(sym_heap h) {
  const int d = (int)blockIdx.y;
  const int nvec = h.s.hidden / 8, N = h.s.world * h.s.tokens_per_slot;
  const int tid = threadIdx.x;
  pdl_launch_dependents();
  pdl_wait();  // the staged rows and the row sources
  const int total = checked_total(h, d, blockIdx.x == 0 && tid == 0);
  for (int p = (int)blockIdx.x; p < total; p += (int)gridDim.x) {
    const int q = win<const int32_t>(h, d, h.off_h)[p];
    if (q < 0 || q >= N) {
      if (tid == 0) raise_status(h, SYM_STATUS_OVERFLOW);
      continue;
    }
    const uint4 *src = win<const uint4>(h, d, h.off_y) + (size_t)q * nvec;
    uint4 *dst = win<uint4>(h, d, h.off_recv_x) + (size_t)p * nvec;
    for (int base = 0; base < nvec; base += VEC * SCATTER_THREADS) {
      uint4 v[VEC];
#pragma unroll
      for (int i = 0; i < VEC; ++i) {
        const int c = base + tid + i * SCATTER_THREADS;
        if (c < nvec) v[i] = __ldg(src + c);
      }
#pragma unroll
      for (int i = 0; i < VEC; ++i) {
        const int c = base + tid + i * SCATTER_THREADS;
        if (c < nvec) dst[c] = v[i];
      }
    }
    // every thread's stores precede the barrier; thread 0's fence is cumulative
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      atomicAdd(win<uint32_t>(h, d, h.off_ready) + p / SYM_ROWS_PER_FLAG, 1u);
    }
  }
}

// ---------------------------------------------------------------------------
// FP8 dispatch with per-token scales: each row crosses as E4M3 codes (H bytes
// instead of 2H) and one scale 2^e, the smallest power of two with
// max|x| <= 448 * 2^e, so that x / 2^e is exact and only the E4M3 rounding
// (to nearest, ties to even) loses bits.  The codes of pair row p go to row p
// of the destination slot's staging (its y window, H bytes a row), the scale
// to word p of its h window; the slot then multiplies back to bf16 (exact:
// a code has 4 significant bits) into recv_x and raises the ready counters.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint16_t e4m3x2_rn(float lo, float hi) {
  uint16_t r;  // upper byte from the first operand
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t c) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(c));
  return r;
}
__device__ __forceinline__ float bf16_bits_to_float(uint32_t b16) { return __uint_as_float(b16 << 16); }

template <int VEC>
__global__ void __launch_bounds__(SCATTER_THREADS)
    fp8_scatter_kernel(sym_heap h, const uint4 *__restrict__ x, const int32_t *__restrict__ idx,
                       const float *__restrict__ w) {
  __shared__ uint2 *dst_s[32];
  __shared__ int32_t slot_s[32], row_s[32];
  __shared__ uint32_t amax_s[SCATTER_THREADS / 32];
  const int E = h.s.num_experts, k = h.s.topk, T = h.s.tokens_per_slot, H = h.s.hidden;
  const int E_loc = E / h.s.world;
  const int N = h.s.world * T;
  const int nchunks = (N + CHUNK - 1) / CHUNK;
  const int g = blockIdx.x;
  const int tid = threadIdx.x;
  const int nvec = H / 8;  // 16-byte bf16 vectors; each becomes 8 code bytes
  const uint4 *src = x + (size_t)g * nvec;
  pdl_launch_dependents();
  pdl_wait();
  // pass 1: the row's largest magnitude (bf16 magnitudes order as integers)
  uint32_t am = 0;
  for (int c = tid; c < nvec; c += SCATTER_THREADS) {
    const uint4 v = __ldg(src + c);
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) am = max(am, max(u[i] & 0x7FFFu, (u[i] >> 16) & 0x7FFFu));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) am = max(am, __shfl_xor_sync(0xffffffffu, am, off));
  if ((tid & 31) == 0) amax_s[tid >> 5] = am;
  if (tid < k) {
    const int j = tid;
    const int e = idx[(size_t)g * k + j];
    int32_t *pos = win<int32_t>(h, g / T, h.off_pos) + (size_t)(g % T) * k;
    uint2 *dst = nullptr;
    int p = -1;
    if (e >= 0 && e < E) {
      const int d = e / E_loc, l = e % E_loc;
      const int rank = pos[j];
      p = win<int32_t>(h, d, h.off_recv_off)[l] +
          win<int32_t>(h, 0, h.off_hist)[(size_t)e * nchunks + g / CHUNK] + rank;
      if (rank < 0 || p < 0 || (uint64_t)p >= h.cap) {
        raise_status(h, SYM_STATUS_OVERFLOW);
        p = -1;
      } else {
        dst = reinterpret_cast<uint2 *>(win<uint8_t>(h, d, h.off_y) + (size_t)p * H);
        win<int32_t>(h, d, h.off_recv_pair)[p] = g * k + j;
        win<float>(h, d, h.off_recv_w)[p] = w[(size_t)g * k + j];
      }
    }
    pos[j] = p;
    dst_s[j] = dst;
    slot_s[j] = e >= 0 && e < E ? e / E_loc : -1;
    row_s[j] = p;
  }
  __syncthreads();
  // the scale: amax = m * 2^ex with m in [0.5, 1); 448 = 0.875 * 2^9
  int ex = 0;
  const float amax = bf16_bits_to_float(max(amax_s[0], amax_s[1]));
  const float m = frexpf(amax, &ex);
  const int es = amax == 0.f ? 0 : (m <= 0.875f ? ex - 9 : ex - 8);
  if (tid < k && dst_s[tid]) win<float>(h, slot_s[tid], h.off_h)[row_s[tid]] = ldexpf(1.f, es);
  // pass 2: codes of x / 2^es, 8 bytes per 16-byte vector, to every destination
  for (int base = 0; base < nvec; base += VEC * SCATTER_THREADS) {
    uint2 q[VEC];
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
      const int c = base + tid + i * SCATTER_THREADS;
      if (c < nvec) {
        const uint4 v = __ldg(src + c);
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
        uint16_t r[4];
#pragma unroll
        for (int t = 0; t < 4; ++t)
          r[t] = e4m3x2_rn(ldexpf(bf16_bits_to_float(u[t] & 0xFFFFu), -es),
                           ldexpf(bf16_bits_to_float(u[t] >> 16), -es));
        q[i] = make_uint2((uint32_t)r[0] | ((uint32_t)r[1] << 16), (uint32_t)r[2] | ((uint32_t)r[3] << 16));
      }
    }
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
      const int c = base + tid + i * SCATTER_THREADS;
      if (c < nvec)
        for (int j = 0; j < k; ++j)
          if (dst_s[j]) dst_s[j][c] = q[i];
    }
  }
}

// grid (blocks, W): the blocks of slot blockIdx.y stride over its received
// rows: bf16 row p = codes of staging row p times its scale (exact), then the
// row block's ready counter
template <int VEC>
__global__ void __launch_bounds__(SCATTER_THREADS) fp8_dequant_kernel(sym_heap h) {
  const int d = (int)blockIdx.y;
  const int H = h.s.hidden, nvec = H / 8;
  const int tid = threadIdx.x;
  pdl_launch_dependents();
  pdl_wait();  // the codes and the scales
  const int total = checked_total(h, d, blockIdx.x == 0 && tid == 0);
  for (int p = (int)blockIdx.x; p < total; p += (int)gridDim.x) {
    const float sc = win<const float>(h, d, h.off_h)[p];
    const uint2 *src = reinterpret_cast<const uint2 *>(win<const uint8_t>(h, d, h.off_y) + (size_t)p * H);
    uint4 *dst = win<uint4>(h, d, h.off_recv_x) + (size_t)p * nvec;
    for (int base = 0; base < nvec; base += VEC * SCATTER_THREADS) {
      uint2 q[VEC];
#pragma unroll
      for (int i = 0; i < VEC; ++i) {
        const int c = base + tid + i * SCATTER_THREADS;
        if (c < nvec) q[i] = src[c];
      }
#pragma unroll
      for (int i = 0; i < VEC; ++i) {
        const int c = base + tid + i * SCATTER_THREADS;
        if (c < nvec) {
          const uint32_t words[2] = {q[i].x, q[i].y};
          uint32_t o[4];
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const uint32_t f2 = e4m3x2_to_f16x2((uint16_t)(words[t >> 1] >> ((t & 1) * 16)));
            const float lo = __half2float(__ushort_as_half((unsigned short)(f2 & 0xFFFFu))) * sc;
            const float hi = __half2float(__ushort_as_half((unsigned short)(f2 >> 16))) * sc;
            // exact in bf16: the upper 16 bits of the fp32 value
            o[t] = (__float_as_uint(lo) >> 16) | (__float_as_uint(hi) & 0xFFFF0000u);
          }
          dst[c] = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
    }
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      atomicAdd(win<uint32_t>(h, d, h.off_ready) + p / SYM_ROWS_PER_FLAG, 1u);
    }
  }
}

cudaError_t launch_dispatch(const sym_heap &h, const uint16_t *x, const int32_t *idx,
                            const float *w, int mode, cudaStream_t st) {
  const int N = h.s.world * h.s.tokens_per_slot;
  const int nchunks = (N + CHUNK - 1) / CHUNK;
  const size_t mask_bytes = (size_t)h.s.num_experts * (CHUNK / 32) * sizeof(uint32_t);
  cudaError_t err = launch_pdl(dispatch_count_kernel, dim3(nchunks), dim3(CHUNK), mask_bytes, st, h, idx);
  if (err != cudaSuccess) return err;
  // scan and scatter are scheduled while their predecessor drains (they wait
  // for its results on the device)
  const int scan_threads = std::min(1024, 32 * (h.s.num_experts / h.s.world));
  if ((err = launch_pdl(dispatch_scan_kernel, dim3(h.s.world), dim3(scan_threads), 0, st, h)) != cudaSuccess)
    return err;
  // vectors per thread: the whole row in one pass up to H = 8192
  const int nvec = h.s.hidden / 8;
  if (mode == 2) {
    auto fk = nvec <= 4 * SCATTER_THREADS   ? fp8_scatter_kernel<4>
              : nvec <= 8 * SCATTER_THREADS ? fp8_scatter_kernel<8>
                                            : fp8_scatter_kernel<16>;
    if ((err = launch_pdl(fk, dim3(N), dim3(SCATTER_THREADS), 0, st, h, reinterpret_cast<const uint4 *>(x), idx,
                          w)) != cudaSuccess)
      return err;
    auto qk = nvec <= 4 * SCATTER_THREADS   ? fp8_dequant_kernel<4>
              : nvec <= 8 * SCATTER_THREADS ? fp8_dequant_kernel<8>
                                            : fp8_dequant_kernel<16>;
    const unsigned per_slot =
        (unsigned)std::max<long long>(1, std::min<long long>(EXPAND_BLOCKS / h.s.world, (long long)h.cap));
    return launch_pdl(qk, dim3(per_slot, h.s.world), dim3(SCATTER_THREADS), 0, st, h);
  }
  if (mode == 1) {
    const int nch = (N + 31) / 32;
    if ((err = launch_pdl(dedup_count_kernel, dim3((nch + 7) / 8), dim3(256), 0, st, h, idx)) != cudaSuccess)
      return err;
    if ((err = launch_pdl(dedup_scan_kernel, dim3(1), dim3(1024), 0, st, h)) != cudaSuccess) return err;
    auto dk = nvec <= 4 * SCATTER_THREADS   ? dedup_scatter_kernel<4>
              : nvec <= 8 * SCATTER_THREADS ? dedup_scatter_kernel<8>
                                            : dedup_scatter_kernel<16>;
    if ((err = launch_pdl(dk, dim3(N), dim3(SCATTER_THREADS), 0, st, h, reinterpret_cast<const uint4 *>(x), idx,
                          w)) != cudaSuccess)
      return err;
    auto ek = nvec <= 4 * SCATTER_THREADS   ? dedup_expand_kernel<4>
              : nvec <= 8 * SCATTER_THREADS ? dedup_expand_kernel<8>
                                            : dedup_expand_kernel<16>;
    const unsigned per_slot =
        (unsigned)std::max<long long>(1, std::min<long long>(EXPAND_BLOCKS / h.s.world, (long long)h.cap));
    return launch_pdl(ek, dim3(per_slot, h.s.world), dim3(SCATTER_THREADS), 0, st, h);
  }
  auto kern = nvec <= 4 * SCATTER_THREADS   ? dispatch_scatter_kernel<4>
              : nvec <= 8 * SCATTER_THREADS ? dispatch_scatter_kernel<8>
                                            : dispatch_scatter_kernel<16>;
  return launch_pdl(kern, dim3(N), dim3(SCATTER_THREADS), 0, st, h, reinterpret_cast<const uint4 *>(x), idx, w);
}

}  // namespace symmoe
