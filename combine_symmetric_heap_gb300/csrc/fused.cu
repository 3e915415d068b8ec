// fused.cu -- the whole MoE pipeline in one persistent launch.
//
// MORI CCO blog, "Mega-MoE: mega-kernel co-design with FlyDSL": dispatch,
// expert GEMM and combine fused into a single kernel, removing the
// synchronisation between kernels; and "In-kernel compute-communication
// fusion": compute and data movement overlap at tile granularity inside one
// launch.  Here the four stages run in one launch (CTAs in clusters of two,
// one per SM, all resident) and overlap per tile:
//
//   phase 1  route + count, one task per 32-token chunk: route the chunk
//            (logits rows staged in shared memory), then per-expert bitmasks
//            give every pair its rank in the chunk and the chunk histogram.
//            The CTA that completes the last chunk runs the scan (counts,
//            receive offsets, totals) and clears the readiness counters, then
//            publishes scan_done = epoch.
//   phase 2  scatter, one warp per token: rows go straight into the
//            destination slot's recv_x window; each row raises the ready
//            counter of its 128-row block (release).
//   phase 3  expert GEMM tiles on CTA pairs (the tcgen05 cta_group::2 tiles of
//            the stand-alone GEMM): each pair takes its gate/up tiles, then its
//            down tiles, round-robin.  A gate/up tile starts once the ready
//            counters of its token rows are complete; a down tile once every
//            gate/up feature tile of its 256 token rows is stored (h_ready);
//            each epilogue warp of both CTAs bumps h_ready / y_ready of the
//            tile's token block after storing its share.
//   phase 4  combine, one warp per token, each pair gated on y_ready.
//
// Forward progress: phases 1, 2 and 4 claim work from per-phase counters and
// a CTA moves on only after finding the previous phase's counter exhausted, so
// a task only waits for work already claimed by a running CTA; phase 3's tiles
// are assigned statically to pairs, which is safe because the grid holds only
// as many pairs as can be resident at once and a pair finishes its gate/up
// tiles before its down tiles.  Every wait is also bounded by the heap's
// wait_timeout_us (on expiry: SYM_STATUS_TIMEOUT, a global abort flag, and
// every CTA skips the rest of its work).  The last CTA to exit resets the
// counters, so the next launch on the stream starts clean.
#include <type_traits>

#include "gemm2sm.cuh"

namespace symmoe {

constexpr int FUSED_THREADS = 256;  // warps 0-5 run the GEMM roles, all 8 the memory phases
constexpr int EPI_WARPS_PER_TILE = 8;  // 4 epilogue warps in each CTA of a pair
constexpr int FUSED_CHUNK = 32;  // tokens per route+count task (one bitmask word per expert)
constexpr int SCATTER_TOKENS = 8;  // tokens per scatter task (one warp each)
constexpr int COMBINE_TOKENS = 8;  // tokens per combine task
constexpr int FUSED_CTRL_SMEM = 512;

// control words in slot 0's ctrl window
enum Ctl : int {
  C_ROUTE_NEXT = 0,
  C_ROUTE_DONE = 1,
  C_SCAN_DONE = 2,  // epoch of the last completed scan
  C_SCATTER_NEXT = 3,
  C_COMB_NEXT = 6,
  C_EXIT = 7,
  C_ABORT = 8,
  C_WORDS = 64
};

// readiness counters: one per 256-row token tile of every expert
__host__ __device__ inline int fused_h_blocks(const moe_shape &s) {
  return s.world * s.tokens_per_slot * s.topk / gemm2::BN + s.num_experts + 1;
}
__host__ __device__ inline int fused_y_blocks(const moe_shape &s) { return fused_h_blocks(s); }

struct FusedArgs {
  const float *logits;
  const uint16_t *x;
  int32_t *idx;
  float *w;
  uint16_t *out;
};

__device__ __forceinline__ uint32_t *ctl(const sym_heap &h) { return win<uint32_t>(h, 0, h.off_ctrl); }
__device__ __forceinline__ uint32_t *h_ready(const sym_heap &h) { return ctl(h) + C_WORDS; }
__device__ __forceinline__ uint32_t *y_ready(const sym_heap &h) {
  return ctl(h) + C_WORDS + fused_h_blocks(h.s);
}
__device__ __forceinline__ bool global_abort(const sym_heap &h) {
  return *reinterpret_cast<volatile uint32_t *>(ctl(h) + C_ABORT) != 0;
}
__device__ __forceinline__ void set_abort(const sym_heap &h) {
  raise_status(h, SYM_STATUS_TIMEOUT);
  atomicExch(ctl(h) + C_ABORT, 1u);
}

// Bounded acquire-wait until *p >= target; gives up on timeout (setting the
// global abort) or when another CTA aborted.
__device__ inline bool wait_geq(const sym_heap &h, const uint32_t *p, uint32_t target) {
  if (ld_acquire_u32(p) >= target) return true;
  const uint64_t t0 = globaltimer_ns();
  const uint64_t limit = (uint64_t)h.wait_timeout_us * 1000ull;
  for (uint32_t it = 0;; ++it) {
    if (ld_acquire_u32(p) >= target) return true;
    if (global_abort(h)) return false;
    if ((it & 63u) == 63u && globaltimer_ns() - t0 > limit) {
      set_abort(h);
      return false;
    }
    __nanosleep(128);
  }
}

// Claim the next task of a phase (thread 0), broadcast to the CTA.
__device__ inline int claim(const sym_heap &h, int counter, int *bcast) {
  __syncthreads();
  if (threadIdx.x == 0) *bcast = global_abort(h) ? 0x7fffffff : (int)atomicAdd(ctl(h) + counter, 1u);
  __syncthreads();
  return *bcast;
}

// ---------------------------------------------------------------- phase 1
// Top-k of one token by one warp over its logits row staged in shared memory
// (row[] is consumed: selected entries become -inf).
__device__ inline void route_token(float *row, int E, int k, int32_t *idx_out, float *w_out,
                                   int lane) {
  float my_val = -INFINITY;  // lane j keeps the j-th selected logit
  int my_idx = -1;
  for (int r = 0; r < k; ++r) {
    float bv = -INFINITY;
    int be = 0x7fffffff;
    for (int e = lane; e < E; e += 32) {  // ascending index: '>' keeps the lower one on ties
      const float v = row[e];
      if (v > bv || be == 0x7fffffff) {
        bv = v;
        be = e;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oe = __shfl_xor_sync(0xffffffffu, be, off);
      if (ov > bv || (ov == bv && oe < be)) {
        bv = ov;
        be = oe;
      }
    }
    if (lane == (be & 31)) row[be] = -INFINITY;  // logits are finite: never picked again
    __syncwarp();
    if (lane == r) {
      my_val = bv;
      my_idx = be;
    }
  }
  const float top = __shfl_sync(0xffffffffu, my_val, 0);
  const float z = lane < k ? expf(my_val - top) : 0.f;
  float s = z;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane < k) {
    idx_out[lane] = my_idx;
    w_out[lane] = z / s;
  }
}

// Route the 32 tokens of a chunk (4 per warp), then rank each pair inside the
// chunk by the per-expert bitmask and write the chunk histogram.
// smem: 8 logits rows of E floats, then the E mask words.
__device__ inline void route_count_chunk(const sym_heap &h, const FusedArgs &a, int chunk,
                                         float *smem) {
  const int E = h.s.num_experts, k = h.s.topk, T = h.s.tokens_per_slot;
  const int N = h.s.world * T;
  const int nchunks = (N + FUSED_CHUNK - 1) / FUSED_CHUNK;
  const int wid = warp_id(), lane = lane_id(), nw = blockDim.x >> 5;
  float *row = smem + (size_t)wid * E;
  uint32_t *mask = reinterpret_cast<uint32_t *>(smem + (size_t)nw * E);
  for (int t = wid; t < FUSED_CHUNK; t += nw) {
    const int g = chunk * FUSED_CHUNK + t;
    if (g >= N) break;
    const float *src = a.logits + (size_t)g * E;
    for (int e = lane; e < E; e += 32) row[e] = __ldg(src + e);
    __syncwarp();
    route_token(row, E, k, a.idx + (size_t)g * k, a.w + (size_t)g * k, lane);
    __syncwarp();
  }
  for (int i = threadIdx.x; i < E; i += blockDim.x) mask[i] = 0;
  __syncthreads();
  const int t = threadIdx.x;
  const int g = chunk * FUSED_CHUNK + t;
  const uint32_t bit = 1u << t;
  if (t < FUSED_CHUNK && g < N)
    for (int j = 0; j < k; ++j)
      if (atomicOr(&mask[a.idx[(size_t)g * k + j]], bit) & bit) raise_status(h, SYM_STATUS_OVERFLOW);
  __syncthreads();
  if (t < FUSED_CHUNK && g < N) {
    int32_t *pos = win<int32_t>(h, g / T, h.off_pos) + (size_t)(g % T) * k;
    for (int j = 0; j < k; ++j) pos[j] = __popc(mask[a.idx[(size_t)g * k + j]] & (bit - 1u));
  }
  int32_t *hist = win<int32_t>(h, 0, h.off_hist);
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(size_t)e * nchunks + chunk] = __popc(mask[e]);
}

// The scan, run by the CTA that completed the last chunk.
__device__ inline void scan_and_publish(const sym_heap &h, int32_t *cnt_s) {
  const int E = h.s.num_experts, W = h.s.world, E_loc = E / W;
  const int N = W * h.s.tokens_per_slot;
  const int nchunks = (N + FUSED_CHUNK - 1) / FUSED_CHUNK;
  int32_t *hist = win<int32_t>(h, 0, h.off_hist);
  const int lane = lane_id(), wid = warp_id(), nw = blockDim.x >> 5;
  __threadfence();
  for (int e = wid; e < E; e += nw) {
    int32_t *row = hist + (size_t)e * nchunks;
    int carry = 0;
    for (int c0 = 0; c0 < nchunks; c0 += 32) {
      const int c = c0 + lane;
      const int v = c < nchunks ? __ldcg(row + c) : 0;
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
    win<int32_t>(h, d, h.off_cnt)[l] = cnt_s[e];
    win<int32_t>(h, d, h.off_recv_off)[l] = off;
    if (l == E_loc - 1) *win<int32_t>(h, d, h.off_total) = off + cnt_s[e];
  }
  for (int i = threadIdx.x; i < W * (int)h.num_ready; i += blockDim.x)
    win<uint32_t>(h, i / h.num_ready, h.off_ready)[i % h.num_ready] = 0u;
  const int nh = fused_h_blocks(h.s), ny = fused_y_blocks(h.s);
  for (int i = threadIdx.x; i < nh; i += blockDim.x) h_ready(h)[i] = 0u;
  for (int i = threadIdx.x; i < ny; i += blockDim.x) y_ready(h)[i] = 0u;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicExch(ctl(h) + C_SCAN_DONE, h.epoch);
  }
}

// ---------------------------------------------------------------- phase 2
// One warp per token; dst_s is this warp's 32-entry destination table.
__device__ inline void scatter_token(const sym_heap &h, const FusedArgs &a, int g, int lane,
                                     uint4 **dst_s) {
  const int E = h.s.num_experts, k = h.s.topk, T = h.s.tokens_per_slot, H = h.s.hidden;
  const int E_loc = E / h.s.world;
  const int N = h.s.world * T;
  const int nchunks = (N + FUSED_CHUNK - 1) / FUSED_CHUNK;
  int32_t *pos = win<int32_t>(h, g / T, h.off_pos) + (size_t)(g % T) * k;
  int d = 0, p = -1;
  if (lane < k) {
    const int e = __ldcg(a.idx + (size_t)g * k + lane);
    d = e / E_loc;
    p = __ldcg(win<int32_t>(h, d, h.off_recv_off) + e % E_loc) +
        __ldcg(win<int32_t>(h, 0, h.off_hist) + (size_t)e * nchunks + g / FUSED_CHUNK) +
        __ldcg(pos + lane);
    uint4 *dst = nullptr;
    if (p < 0 || (uint64_t)p >= h.cap) {
      raise_status(h, SYM_STATUS_OVERFLOW);
      p = -1;
    } else {
      dst = win<uint4>(h, d, h.off_recv_x) + (size_t)p * (H / 8);
    }
    pos[lane] = p;
    dst_s[lane] = dst;
  }
  __syncwarp();
  const uint4 *src = reinterpret_cast<const uint4 *>(a.x) + (size_t)g * (H / 8);
  for (int c = lane; c < H / 8; c += 32) {
    const uint4 v = __ldg(src + c);
    for (int j = 0; j < k; ++j)
      if (dst_s[j]) dst_s[j][c] = v;
  }
  if (lane < k && p >= 0) {
    win<int32_t>(h, d, h.off_recv_pair)[p] = g * k + lane;
    win<float>(h, d, h.off_recv_w)[p] = __ldcg(a.w + (size_t)g * k + lane);
  }
  // the rows are read next by TMA (async proxy) in other CTAs
  asm volatile("fence.proxy.async.global;" ::: "memory");
  __threadfence();
  __syncwarp();
  if (lane < k && p >= 0) atomicAdd(win<uint32_t>(h, d, h.off_ready) + p / SYM_ROWS_PER_FLAG, 1u);
  __syncwarp();
}

// ---------------------------------------------------------------- phase 4
// One warp per token; src_s / w_s are this warp's 32-entry tables.
__device__ inline void combine_token(const sym_heap &h, const FusedArgs &a, const gemm2::TokTables &tb,
                                     int g, int lane, const uint4 **src_s, float *w_s) {
  const int E = h.s.num_experts, k = h.s.topk, T = h.s.tokens_per_slot, H = h.s.hidden;
  const int E_loc = E / h.s.world;
  const uint32_t target = EPI_WARPS_PER_TILE * (uint32_t)gemm2::nf_of(h, gemm2::DOWN);
  bool ok = true;
  if (lane < k) {
    const int e = __ldcg(a.idx + (size_t)g * k + lane);
    const int p = __ldcg(win<const int32_t>(h, g / T, h.off_pos) + (size_t)(g % T) * k + lane);
    const uint4 *src = nullptr;
    if (p >= 0) {
      // the 256-row down tile holding this row: every epilogue warp of every
      // feature tile has stored its share
      ok = wait_geq(h, y_ready(h) + tb.tokprefix[e] + (p - tb.roff[e]) / gemm2::BN, target);
      src = win<const uint4>(h, e / E_loc, h.off_y) + (size_t)p * (H / 8);
    }
    src_s[lane] = src;
    w_s[lane] = __ldcg(a.w + (size_t)g * k + lane);
  }
  if (!__all_sync(0xffffffffu, ok)) return;
  uint4 *dst = reinterpret_cast<uint4 *>(a.out) + (size_t)g * (H / 8);
  for (int c = lane; c < H / 8; c += 32) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    for (int j = 0; j < k; ++j) {
      const uint4 *sj = src_s[j];
      if (!sj) continue;
      const float ww = w_s[j];
      const uint4 v = __ldcg(sj + c);
      acc[0] = fmaf(ww, bf16lo(v.x), acc[0]);
      acc[1] = fmaf(ww, bf16hi(v.x), acc[1]);
      acc[2] = fmaf(ww, bf16lo(v.y), acc[2]);
      acc[3] = fmaf(ww, bf16hi(v.y), acc[3]);
      acc[4] = fmaf(ww, bf16lo(v.z), acc[4]);
      acc[5] = fmaf(ww, bf16hi(v.z), acc[5]);
      acc[6] = fmaf(ww, bf16lo(v.w), acc[6]);
      acc[7] = fmaf(ww, bf16hi(v.w), acc[7]);
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    dst[c] = o;
  }
  __syncwarp();
}

// ---------------------------------------------------------------- kernel
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(FUSED_THREADS, 1)
    moe_fused_kernel(const sym_heap h, const FusedArgs a, const __grid_constant__ CUtensorMap tm_g,
                     const __grid_constant__ CUtensorMap tm_u,
                     const __grid_constant__ gemm2::BMaps tm_rx,
                     const __grid_constant__ CUtensorMap tm_d,
                     const __grid_constant__ gemm2::BMaps tm_h) {
  using namespace gemm2;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *ring = smem;
  float *xch = reinterpret_cast<float *>(smem + (size_t)STAGES * STAGE_BYTES);
  uint8_t *ctrl_s = smem + (size_t)STAGES * STAGE_BYTES + XCH_BYTES;
  uint64_t *full = reinterpret_cast<uint64_t *>(ctrl_s);
  uint64_t *empty = full + STAGES;
  uint64_t *acc_full = empty + STAGES;
  uint64_t *acc_empty = acc_full + 2;
  uint64_t *drained = acc_empty + 2;  // every MMA of this launch has completed
  uint32_t *tmem_base_s = reinterpret_cast<uint32_t *>(drained + 1);
  volatile int *abort_s = reinterpret_cast<volatile int *>(tmem_base_s + 1);
  volatile int *never_s = abort_s + 1;  // "stop before tile" bound: never
  int *bcast = const_cast<int *>(never_s + 1);
  const int E = h.s.num_experts;
  int *tab = reinterpret_cast<int *>(ctrl_s + FUSED_CTRL_SMEM);
  const TokTables tb{tab, tab + E, tab + 2 * E};
  const int wid = warp_id(), lane = lane_id();
  // per-warp destination / source pointer and weight tables (32 entries each)
  uint8_t *warp_tab = ctrl_s + FUSED_CTRL_SMEM + ((tok_tables_bytes(E) + 15) & ~size_t(15));
  void **ptr_s = reinterpret_cast<void **>(warp_tab) + wid * 32;
  float *wgt_s = reinterpret_cast<float *>(warp_tab + FUSED_THREADS / 32 * 32 * sizeof(void *)) + wid * 32;
  const uint32_t tmo = h.wait_timeout_us;
  const int N = h.s.world * h.s.tokens_per_slot;
  const int nchunks = (N + FUSED_CHUNK - 1) / FUSED_CHUNK;
  const uint32_t rank = cta_rank();
  const int pair_id = (int)cluster_id_x(), npairs = (int)num_clusters_x();

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);  // used on the leader: one arrive (with both CTAs' bytes)
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 8);  // leader: 4 epilogue warps of each CTA
    }
    mbar_init(drained, 1);
    *abort_s = 0;
    *never_s = 0x7fffffff;
    fence_mbar_init();
    tma_prefetch_desc(&tm_g);
    tma_prefetch_desc(&tm_u);
    tma_prefetch_desc(&tm_d);
    for (int i = 0; i < NBOX; ++i) {
      tma_prefetch_desc(&tm_rx.m[i]);
      tma_prefetch_desc(&tm_h.m[i]);
    }
  }
  if (wid == 1) {
    tmem_alloc2(tmem_base_s, TMEM_COLS);
    tmem_relinquish2();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // barriers of both CTAs initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem_base = *tmem_base_s;

  // ---------------- phase 1: route + count (the last finisher scans)
  for (;;) {
    const int c = claim(h, C_ROUTE_NEXT, bcast);
    if (c >= nchunks) break;
    route_count_chunk(h, a, c, reinterpret_cast<float *>(ring));
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) *bcast = (int)atomicAdd(ctl(h) + C_ROUTE_DONE, 1u);
    __syncthreads();
    if (*bcast == nchunks - 1) scan_and_publish(h, reinterpret_cast<int32_t *>(ring));
  }

  // ---------------- phase 2: scatter
  if (threadIdx.x == 0) *bcast = wait_geq(h, ctl(h) + C_SCAN_DONE, h.epoch) ? 1 : 0;
  __syncthreads();
  const bool scanned = *bcast != 0 && ld_acquire_u32(ctl(h) + C_SCAN_DONE) == h.epoch;
  if (scanned) {
    const int ntask = (N + SCATTER_TOKENS - 1) / SCATTER_TOKENS;
    for (;;) {
      const int t = claim(h, C_SCATTER_NEXT, bcast);
      if (t >= ntask) break;
      for (int i = wid; i < SCATTER_TOKENS; i += FUSED_THREADS / 32) {
        const int g = t * SCATTER_TOKENS + i;
        if (g < N) scatter_token(h, a, g, lane, reinterpret_cast<uint4 **>(ptr_s));
      }
    }
  }

  // ---------------- phase 3: expert GEMM tiles on the CTA pair
  if (scanned) build_tok_tables(h, tb);
  // the ring held phase 1's logits rows (generic stores); TMA writes it next
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncthreads();
  if (scanned) {
    const int nf1 = nf_of(h, GATE_UP), nf2 = nf_of(h, DOWN);
    const int total1 = tb.tokprefix[E] * nf1, total2 = tb.tokprefix[E] * nf2;
    const uint32_t h_target = EPI_WARPS_PER_TILE * (uint32_t)nf1;
    using GU = std::integral_constant<int, GATE_UP>;
    using DN = std::integral_constant<int, DOWN>;
    // this CTA's token rows of a tile: the MMA takes n_mma rows, half per CTA
    auto my_rows = [&](const TileInfo &ti, int &r0, int &cnt) {
      const int half = n_mma(ti.valid) / 2;
      r0 = ti.row0 + (int)rank * half;
      cnt = max(0, min(half, ti.valid - (int)rank * half));
    };
    // inputs of a tile in place: the dispatched rows (gate/up) or every
    // gate/up feature tile of the token tile (down)
    auto inputs_ready = [&](int kind, const TileInfo &ti, bool block) -> bool {
      if (kind == DOWN) {
        const uint32_t *c = h_ready(h) + tb.tokprefix[ti.e] + ti.n;
        return block ? wait_geq(h, c, h_target) : ld_acquire_u32(c) >= h_target;
      }
      int r0, cnt;
      my_rows(ti, r0, cnt);
      if (cnt == 0) return true;
      const int total = __ldcg(win<const int32_t>(h, ti.d, h.off_total));
      const uint32_t *ready = win<const uint32_t>(h, ti.d, h.off_ready);
      for (int b = r0 / SYM_ROWS_PER_FLAG; b <= (r0 + cnt - 1) / SYM_ROWS_PER_FLAG; ++b) {
        const uint32_t target = (uint32_t)min(SYM_ROWS_PER_FLAG, total - b * SYM_ROWS_PER_FLAG);
        if (block ? !wait_geq(h, ready + b, target) : ld_acquire_u32(ready + b) < target) return false;
      }
      return true;
    };
    // the pair's tile after (kind, t): its gate/up tiles, then its down tiles
    auto next_of = [&](int &kind, int &t) {
      t += npairs;
      if (kind == GATE_UP && t >= total1) {
        kind = DOWN;
        t = pair_id;
      }
    };
    auto total_of = [&](int kind) { return kind == GATE_UP ? total1 : total2; };
    auto nf_k = [&](int kind) { return kind == GATE_UP ? nf1 : nf2; };

    if (wid == 0) {
      if (lane == 0) {
        // ------------------------------------------------------------ producer
        int stage = 0;
        uint32_t phase = 0;
        const uint32_t full_leader = map_to(&full[0], 0);
        auto produce = [&](auto kd, const TileInfo &ti, int kind_n, int t_n, bool &next_ok) -> bool {
          constexpr int KIND = decltype(kd)::value;
          int r0, cnt;
          my_rows(ti, r0, cnt);
          const CUtensorMap *ma = KIND == GATE_UP ? &tm_g : &tm_d;
          const int box = box_index(n_mma(ti.valid) / 2);
          const uint32_t tx = stage_tx(box);
          const CUtensorMap *mb = KIND == GATE_UP ? &tm_rx.m[box] : &tm_h.m[box];
          const int arow = KIND == GATE_UP ? ti.e * h.s.inter + ti.f * 128 + (int)rank * 64
                                           : ti.e * h.s.hidden + ti.f * 256 + (int)rank * 128;
          const int nk = nk_of(h, KIND);
          for (int kb = 0; kb < nk; ++kb) {
            if (!next_ok && kb == nk / 2)
              next_ok = inputs_ready(kind_n, decode_tok(h, tb, nf_k(kind_n), t_n), false);
            if (!wait_or_stop(&empty[stage], phase ^ 1u, -1, never_s, abort_s, tmo, h)) return false;
            uint8_t *sb = ring + (size_t)stage * STAGE_BYTES;
            const uint32_t bar = full_leader + (uint32_t)(stage * sizeof(uint64_t));
            if (rank == 0) mbar_arrive_expect_tx(&full[stage], tx);  // both halves
            if (KIND == GATE_UP) {
              tma_load_2d_pair(sb, ma, bar, kb * BK, arow);               // 64 gate rows
              tma_load_2d_pair(sb + A_BYTES / 2, &tm_u, bar, kb * BK, arow);  // 64 up rows
            } else {
              tma_load_2d_pair(sb, ma, bar, kb * BK, arow);               // 128 down rows
            }
            tma_load_3d_pair(sb + A_BYTES, mb, bar, kb * BK, r0, ti.d);   // this CTA's tokens
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          return true;
        };
        int kind = GATE_UP, t = pair_id;
        if (t >= total1) {
          kind = DOWN;
          t = pair_id;
        }
        bool ok = t < total_of(kind) ? inputs_ready(kind, decode_tok(h, tb, nf_k(kind), t), true) : true;
        while (ok && t < total_of(kind) && !*abort_s) {
          fence_proxy_async();  // the inputs were written by generic stores in this launch
          const TileInfo ti = decode_tok(h, tb, nf_k(kind), t);
          int kind_n = kind, t_n = t;
          next_of(kind_n, t_n);
          const bool has_next = t_n < total_of(kind_n);
          bool next_ok = !has_next;
          ok = kind == GATE_UP ? produce(GU{}, ti, kind_n, t_n, next_ok)
                               : produce(DN{}, ti, kind_n, t_n, next_ok);
          if (!ok) break;
          if (has_next && !next_ok) ok = inputs_ready(kind_n, decode_tok(h, tb, nf_k(kind_n), t_n), true);
          kind = kind_n;
          t = t_n;
        }
        if (!ok) *abort_s = 1;
      }
    } else if (wid == 1) {
      if (lane == 0 && rank == 0) {
        // ------------------------------------------------------ MMA issuer (leader)
        int stage = 0, abuf = 0;
        uint32_t phase = 0, aphase = 0;
        auto mma_tile = [&](auto kd, const TileInfo &ti) -> bool {
          constexpr int KIND = decltype(kd)::value;
          const uint32_t idesc = idesc_bf16_f32(256, n_mma(ti.valid));
          if (!wait_or_stop(&acc_empty[abuf], aphase ^ 1u, -1, never_s, abort_s, tmo, h)) return false;
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + (uint32_t)(abuf * ACC_COLS);
          const int nk = nk_of(h, KIND);
          for (int kb = 0; kb < nk; ++kb) {
            if (!wait_or_stop(&full[stage], phase, -1, never_s, abort_s, tmo, h)) return false;
            tc_fence_after();
            uint8_t *sb = ring + (size_t)stage * STAGE_BYTES;
            const uint64_t da = smem_desc_sw128(sb), db = smem_desc_sw128(sb + A_BYTES);
#pragma unroll
            for (int kk = 0; kk < BK / UK; ++kk) {
              const uint64_t adv = (uint64_t)(kk * UK * 2 / 16);
              mma2(d_tmem, da + adv, db + adv, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
            }
            commit2_both(&empty[stage]);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          commit2_both(&acc_full[abuf]);
          if (++abuf == 2) {
            abuf = 0;
            aphase ^= 1u;
          }
          return true;
        };
        for (int kind = GATE_UP, t = pair_id; kind <= DOWN;) {
          if (t >= total_of(kind)) {
            if (kind == DOWN) break;
            kind = DOWN;
            t = pair_id;
            continue;
          }
          const TileInfo ti = decode_tok(h, tb, nf_k(kind), t);
          if (!(kind == GATE_UP ? mma_tile(GU{}, ti) : mma_tile(DN{}, ti))) break;
          t += npairs;
        }
        // after an abort the epilogue may stop before the last accumulator:
        // wait for the MMAs still in flight before TMEM is released
        commit2_both(drained);
        mbar_wait(drained, 0, tmo, nullptr);
      }
    } else if (wid < 6) {
      // -------------------------------------------------------------- epilogue
      const int q = wid & 3;  // TMEM lane quarter this warp may access
      int abuf = 0;
      uint32_t aphase = 0;
      uint32_t chunk_ctr = 0;
      const uint32_t leader_acc_empty0 = map_to(&acc_empty[0], 0);
      auto epi_tile = [&](auto kd, const TileInfo &ti) -> bool {
        constexpr int KIND = decltype(kd)::value;
        bool ok = wait_or_stop(&acc_full[abuf], aphase, -1, never_s, abort_s, tmo, h);
        // warp-collective TMEM loads and the gate/up exchange follow: decide together
        ok = KIND == GATE_UP ? xch_vote(q & 1, ok) : __all_sync(0xffffffffu, ok);
        if (!ok) return false;
        tc_fence_after();
        const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(abuf * ACC_COLS);
        if (KIND == GATE_UP) {
          const int pair = q & 1;  // gate lanes 32*pair.., up lanes 64 + 32*pair..
          const bool is_gate = q < 2;
          const int ld = h.s.inter;
          const int feature = ti.f * 128 + (int)rank * 64 + pair * 32 + lane;
          uint16_t *out = win<uint16_t>(h, ti.d, h.off_h) + (size_t)ti.row0 * ld + feature;
          for (int c0 = 0; c0 < ti.valid; c0 += 32, ++chunk_ctr) {
            uint32_t v[32];
            tmem_ld32(tbase + c0, v);
            tmem_ld_wait();
            float *xb = xch + ((size_t)(pair * 2 + (chunk_ctr & 1)) * 2) * 16 * 32;
            float *to_partner = xb + (is_gate ? 1 : 0) * 16 * 32;
            const float *from_partner = xb + (is_gate ? 0 : 1) * 16 * 32;
#pragma unroll
            for (int c = 0; c < 16; ++c)
              to_partner[c * 32 + lane] = __uint_as_float(is_gate ? v[16 + c] : v[c]);
            xch_barrier(pair);
            const int keep = is_gate ? 0 : 16;
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const int col = c0 + keep + c;
              const float other = from_partner[c * 32 + lane];
              const float mine = __uint_as_float(is_gate ? v[c] : v[16 + c]);
              const float gt = is_gate ? mine : other;
              const float up = is_gate ? other : mine;
              if (col < ti.valid) out[(size_t)col * ld] = to_bf16(gt / (1.0f + __expf(-gt)) * up);
            }
          }
        } else {
          const int ld = h.s.hidden;
          const int feature = ti.f * 256 + (int)rank * 128 + q * 32 + lane;
          uint16_t *out = win<uint16_t>(h, ti.d, h.off_y) + (size_t)ti.row0 * ld + feature;
          const bool live = feature < ld;
          for (int c0 = 0; c0 < ti.valid; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(tbase + c0, v);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 32; ++c)
              if (live && c0 + c < ti.valid) out[(size_t)(c0 + c) * ld] = to_bf16(__uint_as_float(v[c]));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (rank == 0) mbar_arrive(&acc_empty[abuf]);
          else mbar_arrive_remote(leader_acc_empty0 + (uint32_t)(abuf * sizeof(uint64_t)));
        }
        if (++abuf == 2) {
          abuf = 0;
          aphase ^= 1u;
        }
        // publish this warp's share of the tile (read next by TMA or by the
        // combine's generic loads in other CTAs)
        __threadfence();
        asm volatile("fence.proxy.async.global;" ::: "memory");
        __syncwarp();
        if (lane == 0)
          atomicAdd((KIND == GATE_UP ? h_ready(h) : y_ready(h)) + tb.tokprefix[ti.e] + ti.n, 1u);
        return true;
      };
      for (int kind = GATE_UP, t = pair_id; kind <= DOWN;) {
        if (t >= total_of(kind)) {
          if (kind == DOWN) break;
          kind = DOWN;
          t = pair_id;
          continue;
        }
        const TileInfo ti = decode_tok(h, tb, nf_k(kind), t);
        if (!(kind == GATE_UP ? epi_tile(GU{}, ti) : epi_tile(DN{}, ti))) break;
        t += npairs;
      }
    }
    if (*abort_s) set_abort(h);
  }
  __syncthreads();

  // ---------------- phase 4: combine
  if (scanned) {
    const int ntask = (N + COMBINE_TOKENS - 1) / COMBINE_TOKENS;
    for (;;) {
      const int t = claim(h, C_COMB_NEXT, bcast);
      if (t >= ntask) break;
      for (int i = wid; i < COMBINE_TOKENS; i += FUSED_THREADS / 32) {
        const int g = t * COMBINE_TOKENS + i;
        if (g < N)
          combine_token(h, a, tb, g, lane, reinterpret_cast<const uint4 **>(const_cast<const void **>(ptr_s)),
                        wgt_s);
      }
    }
  }

  // ---------------- teardown
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no remote arrive or MMA of the pair is still in flight
  tc_fence_after();
  if (wid == 1) tmem_dealloc2(tmem_base, TMEM_COLS);
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(ctl(h) + C_EXIT, 1u) == gridDim.x - 1) {
      // last CTA out: reset the counters for the next launch
      uint32_t *c = ctl(h);
      c[C_ROUTE_NEXT] = 0;
      c[C_ROUTE_DONE] = 0;
      c[C_SCATTER_NEXT] = 0;
      c[C_COMB_NEXT] = 0;
      c[C_ABORT] = 0;
      __threadfence();
      c[C_EXIT] = 0;
    }
  }
}

size_t fused_ctrl_bytes(const moe_shape &s) {
  return (size_t)(C_WORDS + fused_h_blocks(s) + fused_y_blocks(s)) * 4;
}

cudaError_t launch_fused(const sym_heap &h, const float *logits, const uint16_t *x,
                         const uint16_t *wg, const uint16_t *wu, const uint16_t *wd, int32_t *idx,
                         float *w, uint16_t *out, int num_sms, cudaStream_t st) {
  using namespace gemm2;
  const int E = h.s.num_experts, H = h.s.hidden, I = h.s.inter;
  CUtensorMap tg, tu, td;
  BMaps trx, th;
  if (!encode_2d(&tg, wg, (uint64_t)E * I, H, 64) || !encode_2d(&tu, wu, (uint64_t)E * I, H, 64) ||
      !encode_heap_boxes(&trx, h, h.off_recv_x, H) ||
      !encode_2d(&td, wd, (uint64_t)E * H, I, 128) || !encode_heap_boxes(&th, h, h.off_h, I))
    return cudaErrorInvalidValue;
  const size_t smem = 1024 + (size_t)STAGES * STAGE_BYTES + XCH_BYTES + FUSED_CTRL_SMEM +
                      ((tok_tables_bytes(E) + 15) & ~size_t(15)) +
                      FUSED_THREADS / 32 * 32 * (sizeof(void *) + sizeof(float));
  cudaError_t err = cudaFuncSetAttribute(moe_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
  if (err != cudaSuccess) return err;
  // every pair resident at once: phase 3 assigns tiles to pairs statically
  const int grid = 2 * max_resident_pairs((const void *)moe_fused_kernel, FUSED_THREADS, smem, num_sms);
  if (grid <= 0) return cudaErrorInvalidConfiguration;
  const FusedArgs a{logits, x, idx, w, out};
  moe_fused_kernel<<<grid, FUSED_THREADS, smem, st>>>(h, a, tg, tu, trx, td, th);
  return cudaGetLastError();
}

}  // namespace symmoe
