// fused.cu -- the whole MoE pipeline in one persistent launch.
//
// MORI CCO blog, "Mega-MoE: mega-kernel co-design with FlyDSL": dispatch,
// expert GEMM and combine fused into a single kernel, removing the
// synchronisation between kernels; and "In-kernel compute-communication
// fusion": compute and data movement overlap at tile granularity inside one
// launch.  Here the four stages run in one launch (CTAs in clusters of two,
// one per SM, all resident) and overlap per tile:
//
//   phase 1  route + count: route tasks of a 32-token chunk, or of one token
//            per warp when there are fewer chunks than CTAs (logits rows
//            staged in shared memory); the CTA that finishes the last route
//            task of a 32-token chunk counts the chunk (per-expert bitmasks give
//            every pair its rank in the chunk and the chunk histogram).  Once
//            every chunk is counted, CTAs take per-expert scan tasks (prefix
//            over the chunks, expert counts); the CTA completing the last one
//            computes receive offsets and totals, clears the readiness
//            counters and publishes scan_done = epoch.
//   phase 2  scatter, one warp per token: rows go straight into the
//            destination slot's recv_x window; each row raises the ready
//            counter of its 128-row block (release).
//   phase 3  expert GEMM tiles on CTA pairs (the tcgen05 cta_group::2 tiles of
//            the stand-alone GEMM): pairs claim tiles from one counter, every
//            gate/up tile before any down tile (the pair engine's dynamic
//            schedule).  A gate/up tile starts once the ready
//            counters of its token rows are complete; a down tile once every
//            gate/up feature tile of its 256 token rows is stored (h_ready);
//            each epilogue warp of both CTAs bumps h_ready / y_ready of the
//            tile's token block after storing its share.
//   phase 4  combine, one warp per token, each pair gated on y_ready.
//
// Forward progress: phases 1, 2 and 4 claim work from per-phase counters and
// a CTA moves on only after finding the previous phase's counter exhausted, so
// a task only waits for work already claimed by a running CTA; in phase 3 a
// down tile waits only on gate/up tiles, all of which were claimed before it
// by resident pairs that stream them without waiting on any down tile.  Every wait is also bounded by the heap's
// wait_timeout_us (on expiry: SYM_STATUS_TIMEOUT, a global abort flag, and
// every CTA skips the rest of its work).  The last CTA to exit resets the
// counters, so the next launch on the stream starts clean.
#include <type_traits>

#include "gemm2sm.cuh"

namespace symmoe {

constexpr int FUSED_THREADS = 256;  // warps 0-5 run the GEMM roles, all 8 the memory phases
constexpr int EPI_WARPS_PER_TILE = 8;  // 4 epilogue warps in each CTA of a pair
constexpr int FUSED_CHUNK = 32;  // tokens per count chunk (one bitmask word per expert)
constexpr int ROUTE_TOKENS = 8;  // tokens per route task with few chunks (one per warp)
constexpr int SCATTER_TOKENS = 8;  // tokens per scatter task (one warp each)
constexpr int COMBINE_TOKENS = 8;  // tokens per combine task
constexpr int SCATTER_SLOTS_MAX = 3;  // rows a warp stages in shared memory at once (scatter)
constexpr int FUSED_CTRL_SMEM = 512;

// control words in slot 0's ctrl window
enum Ctl : int {
  C_ROUTE_NEXT = 0,
  C_ROUTE_DONE = 1,
  C_SCAN_DONE = 2,  // epoch of the last completed scan
  C_SCATTER_NEXT = 3,
  C_SCATTER_DONE = 4,  // scatter tasks completed (pos final for the combine)
  C_SCAN_NEXT = 5,     // per-expert scan tasks claimed
  C_COMB_NEXT = 6,
  C_EXIT = 7,
  C_ABORT = 8,
  C_SCAN_TASKS = 9,  // per-expert scan tasks completed
  C_TILE_NEXT = 10,  // GEMM tiles claimed (gate/up tiles first, then down tiles)
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
  int weights_in_ffn;  // weights applied to y rows in the down epilogue; the combine sums
};

__device__ __forceinline__ uint32_t *ctl(const sym_heap &h) { return win<uint32_t>(h, 0, h.off_ctrl); }
__device__ __forceinline__ uint32_t *h_ready(const sym_heap &h) { return ctl(h) + C_WORDS; }
__device__ __forceinline__ uint32_t *y_ready(const sym_heap &h) {
  return ctl(h) + C_WORDS + fused_h_blocks(h.s);
}
// route tasks finished per count chunk
__device__ __forceinline__ uint32_t *chunk_done(const sym_heap &h) {
  return y_ready(h) + fused_y_blocks(h.s);
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

// Route the rt tokens of a route task, rt / 8 per warp (logits rows staged in
// shared memory).
__device__ inline void route_task(const sym_heap &h, const FusedArgs &a, int task, int rt, float *smem) {
  const int E = h.s.num_experts, k = h.s.topk;
  const int N = h.s.world * h.s.tokens_per_slot;
  const int wid = warp_id(), lane = lane_id(), nw = blockDim.x >> 5;
  float *row = smem + (size_t)wid * E;
  for (int i = wid; i < rt; i += nw) {
    const int g = task * rt + i;
    if (g >= N) break;
    const float *src = a.logits + (size_t)g * E;
    for (int e = lane; e < E; e += 32) row[e] = __ldg(src + e);
    __syncwarp();
    route_token(row, E, k, a.idx + (size_t)g * k, a.w + (size_t)g * k, lane);
    __syncwarp();
  }
}

// Rank each pair of a 32-token chunk inside the chunk by the per-expert
// bitmask and write the chunk histogram.  The routes of the chunk were
// written by other CTAs of this launch (read with __ldcg after an acquire).
// smem: E mask words.
__device__ inline void count_chunk(const sym_heap &h, const FusedArgs &a, int chunk, uint32_t *mask) {
  const int E = h.s.num_experts, k = h.s.topk, T = h.s.tokens_per_slot;
  const int N = h.s.world * T;
  const int nchunks = (N + FUSED_CHUNK - 1) / FUSED_CHUNK;
  for (int i = threadIdx.x; i < E; i += blockDim.x) mask[i] = 0;
  __syncthreads();
  const int t = threadIdx.x;
  const int g = chunk * FUSED_CHUNK + t;
  const uint32_t bit = 1u << t;
  if (t < FUSED_CHUNK && g < N)
    for (int j = 0; j < k; ++j)
      if (atomicOr(&mask[__ldcg(a.idx + (size_t)g * k + j)], bit) & bit) raise_status(h, SYM_STATUS_OVERFLOW);
  __syncthreads();
  if (t < FUSED_CHUNK && g < N) {
    int32_t *pos = win<int32_t>(h, g / T, h.off_pos) + (size_t)(g % T) * k;
    for (int j = 0; j < k; ++j) pos[j] = __popc(mask[__ldcg(a.idx + (size_t)g * k + j)] & (bit - 1u));
  }
  int32_t *hist = win<int32_t>(h, 0, h.off_hist);
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(size_t)e * nchunks + chunk] = __popc(mask[e]);
}

// Scan task: one expert's chunk histogram row, split into 8 contiguous
// segments (one per warp): exclusive prefix over the chunks in place and the
// expert's row count into its slot's cnt window.  seg_s: 8 ints.
__device__ inline void scan_expert(const sym_heap &h, int e, int *seg_s) {
  const int E = h.s.num_experts, W = h.s.world, E_loc = E / W;
  const int N = W * h.s.tokens_per_slot;
  const int nchunks = (N + FUSED_CHUNK - 1) / FUSED_CHUNK;
  const int lane = lane_id(), wid = warp_id(), nw = blockDim.x >> 5;
  int32_t *row = win<int32_t>(h, 0, h.off_hist) + (size_t)e * nchunks;
  const int seg = (nchunks + nw - 1) / nw;
  const int c_begin = min(nchunks, wid * seg), c_end = min(nchunks, c_begin + seg);
  int total = 0;  // pass 1: this segment's sum
  for (int c = c_begin + lane; c < c_end; c += 32) total += __ldcg(row + c);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) total += __shfl_xor_sync(0xffffffffu, total, off);
  if (lane == 0) seg_s[wid] = total;
  __syncthreads();
  int carry = 0;
  for (int w = 0; w < wid; ++w) carry += seg_s[w];
  for (int c0 = c_begin; c0 < c_end; c0 += 32) {  // pass 2: exclusive prefix in place
    const int c = c0 + lane;
    const int v = c < c_end ? __ldcg(row + c) : 0;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    if (c < c_end) row[c] = carry + incl - v;
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (threadIdx.x == 0) {
    int all = 0;
    for (int w = 0; w < nw; ++w) all += seg_s[w];
    win<int32_t>(h, e / E_loc, h.off_cnt)[e % E_loc] = all;
  }
  __syncthreads();  // seg_s is reused by the next task
}

// After the last scan task: receive offsets and totals per slot, clear the
// readiness counters of this launch, publish scan_done = epoch.
__device__ inline void finish_scan(const sym_heap &h) {
  const int E = h.s.num_experts, W = h.s.world, E_loc = E / W;
  const int N = W * h.s.tokens_per_slot;
  const int nchunks = (N + FUSED_CHUNK - 1) / FUSED_CHUNK;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int d = e / E_loc, l = e % E_loc;
    const int32_t *cnt = win<const int32_t>(h, d, h.off_cnt);
    int off = 0;
    for (int i = 0; i < l; ++i) off += __ldcg(cnt + i);
    win<int32_t>(h, d, h.off_recv_off)[l] = off;
    if (l == E_loc - 1) *win<int32_t>(h, d, h.off_total) = off + __ldcg(cnt + l);
  }
  for (int i = threadIdx.x; i < W * (int)h.num_ready; i += blockDim.x)
    win<uint32_t>(h, i / h.num_ready, h.off_ready)[i % h.num_ready] = 0u;
  const int nh = fused_h_blocks(h.s), ny = fused_y_blocks(h.s);
  for (int i = threadIdx.x; i < nh; i += blockDim.x) h_ready(h)[i] = 0u;
  for (int i = threadIdx.x; i < ny; i += blockDim.x) y_ready(h)[i] = 0u;
  for (int i = threadIdx.x; i < nchunks; i += blockDim.x) chunk_done(h)[i] = 0u;  // all counted
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

// Scatter of up to `slots` consecutive tokens by one warp through its share of
// the (idle) GEMM ring: lanes < k resolve each token's destinations; lane 0
// bulk-loads every row into its slot and, as each lands, bulk-stores it to
// the row's k destinations; once all copies are complete it releases the
// ready counters of the destination row blocks.  Rows move by the copy
// engine, so a warp keeps `slots` rows in flight without holding them in
// registers.  Returns false if a row load did not complete in time.
__device__ inline bool scatter_bulk(const sym_heap &h, const FusedArgs &a, int g0, int slots, uint8_t *wring,
                                    uint64_t *sbar, uint32_t &sph, int lane, uint4 **dst_s) {
  const int E = h.s.num_experts, k = h.s.topk, T = h.s.tokens_per_slot, H = h.s.hidden;
  const int E_loc = E / h.s.world;
  const int N = h.s.world * T;
  const int nchunks = (N + FUSED_CHUNK - 1) / FUSED_CHUNK;
  const uint32_t rowbytes = (uint32_t)H * 2;
  int dd[SCATTER_SLOTS_MAX], pp[SCATTER_SLOTS_MAX];
#pragma unroll
  for (int s = 0; s < SCATTER_SLOTS_MAX; ++s) {
    dd[s] = 0;
    pp[s] = -1;
    const int g = g0 + s;
    if (s < slots && g < N && lane < k) {
      int32_t *pos = win<int32_t>(h, g / T, h.off_pos) + (size_t)(g % T) * k;
      const int e = __ldcg(a.idx + (size_t)g * k + lane);
      const int d = e / E_loc;
      int p = __ldcg(win<int32_t>(h, d, h.off_recv_off) + e % E_loc) +
              __ldcg(win<int32_t>(h, 0, h.off_hist) + (size_t)e * nchunks + g / FUSED_CHUNK) + __ldcg(pos + lane);
      uint4 *dst = nullptr;
      if (p < 0 || (uint64_t)p >= h.cap) {
        raise_status(h, SYM_STATUS_OVERFLOW);
        p = -1;
      } else {
        dst = win<uint4>(h, d, h.off_recv_x) + (size_t)p * (H / 8);
        win<int32_t>(h, d, h.off_recv_pair)[p] = g * k + lane;
        win<float>(h, d, h.off_recv_w)[p] = __ldcg(a.w + (size_t)g * k + lane);
      }
      pos[lane] = p;
      dst_s[s * 32 + lane] = dst;
      dd[s] = d;
      pp[s] = p;
    }
  }
  __syncwarp();
  const int nrows = max(0, min(slots, N - g0));
  bool ok = true;
  if (lane == 0) {
    for (int s = 0; s < nrows; ++s) {
      mbar_arrive_expect_tx(&sbar[s], rowbytes);
      bulk_load(wring + (size_t)s * rowbytes, a.x + (size_t)(g0 + s) * H, rowbytes, &sbar[s]);
    }
    for (int s = 0; s < nrows && ok; ++s) {
      ok = mbar_wait(&sbar[s], (sph >> s) & 1u, h.wait_timeout_us, nullptr);
      if (ok)
        for (int j = 0; j < k; ++j)
          if (dst_s[s * 32 + j]) bulk_store(dst_s[s * 32 + j], wring + (size_t)s * rowbytes, rowbytes);
    }
    bulk_commit();
    bulk_wait_all();
    // the rows were written by the async proxy; order them before the release
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __threadfence();
  }
  sph ^= (1u << nrows) - 1u;
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  if (!ok) return false;
#pragma unroll
  for (int s = 0; s < SCATTER_SLOTS_MAX; ++s) {
    if (s >= nrows) break;
    for (int j = 0; j < k; ++j) {
      const int pj = __shfl_sync(0xffffffffu, pp[s], j), dj = __shfl_sync(0xffffffffu, dd[s], j);
      if (lane == 0 && pj >= 0) atomicAdd(win<uint32_t>(h, dj, h.off_ready) + pj / SYM_ROWS_PER_FLAG, 1u);
    }
  }
  __syncwarp();
  return true;
}

// ---------------------------------------------------------------- phase 4
// One warp per token; src_s / w_s are this warp's 32-entry tables.
template <int U, int G>
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
    if (p >= 0 && (p < tb.roff[e] || p >= tb.roff[e] + tb.cnt[e])) {
      raise_status(h, SYM_STATUS_OVERFLOW);  // a row outside its expert's tiles: skipped
    } else if (p >= 0) {
      // the 256-row down tile holding this row: every epilogue warp of every
      // feature tile has stored its share
      ok = wait_geq(h, y_ready(h) + tb.tokprefix[e] + gemm2::tile_of_row(tb.cnt[e], p - tb.roff[e]),
                    target);
      src = win<const uint4>(h, e / E_loc, h.off_y) + (size_t)p * (H / 8);
    }
    src_s[lane] = src;
    w_s[lane] = a.weights_in_ffn ? 1.f : __ldcg(a.w + (size_t)g * k + lane);
  }
  __syncwarp();  // the tables are read by every lane below
  if (!__all_sync(0xffffffffu, ok)) return;
  uint4 *dst = reinterpret_cast<uint4 *>(a.out) + (size_t)g * (H / 8);
  const int nvec = H / 8;
  // U vectors per lane per pass, the loads of G sources issued together, then
  // accumulated in j order (the staged combine's order)
  for (int c0 = lane; c0 < nvec; c0 += 32 * U) {
    float acc[U][8];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[u][i] = 0.f;
    for (int j0 = 0; j0 < k; j0 += G) {
      uint4 v[G][U];
#pragma unroll
      for (int jj = 0; jj < G; ++jj) {
        const uint4 *sp = j0 + jj < k ? src_s[j0 + jj] : nullptr;
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int c = c0 + 32 * u;
          v[jj][u] = (sp && c < nvec) ? __ldcg(sp + c) : make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int jj = 0; jj < G; ++jj) {
        if (j0 + jj >= k || !src_s[j0 + jj]) continue;
        const float ww = w_s[j0 + jj];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const uint4 x = v[jj][u];
          acc[u][0] = fmaf(ww, bf16lo(x.x), acc[u][0]);
          acc[u][1] = fmaf(ww, bf16hi(x.x), acc[u][1]);
          acc[u][2] = fmaf(ww, bf16lo(x.y), acc[u][2]);
          acc[u][3] = fmaf(ww, bf16hi(x.y), acc[u][3]);
          acc[u][4] = fmaf(ww, bf16lo(x.z), acc[u][4]);
          acc[u][5] = fmaf(ww, bf16hi(x.z), acc[u][5]);
          acc[u][6] = fmaf(ww, bf16lo(x.w), acc[u][6]);
          acc[u][7] = fmaf(ww, bf16hi(x.w), acc[u][7]);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + 32 * u;
      if (c < nvec) {
        uint4 o;
        o.x = pack_bf16x2(acc[u][0], acc[u][1]);
        o.y = pack_bf16x2(acc[u][2], acc[u][3]);
        o.z = pack_bf16x2(acc[u][4], acc[u][5]);
        o.w = pack_bf16x2(acc[u][6], acc[u][7]);
        dst[c] = o;
      }
    }
  }
  __syncwarp();
}

// Combine of one token by one warp, its sources streamed through the warp's
// share of the (idle) GEMM ring with cp.async: per pass each lane copies U
// vectors of every source into shared memory, double-buffered, so the next
// pass is in flight while this one is accumulated (in j order).  k <= KMAX.
template <int U, int KMAX>
__device__ inline void combine_token_stream(const sym_heap &h, const FusedArgs &a, const gemm2::TokTables &tb,
                                            int g, int lane, const uint4 **src_s, float *w_s, uint4 *buf) {
  const int E = h.s.num_experts, k = h.s.topk, T = h.s.tokens_per_slot, H = h.s.hidden;
  const int E_loc = E / h.s.world;
  const uint32_t target = EPI_WARPS_PER_TILE * (uint32_t)gemm2::nf_of(h, gemm2::DOWN);
  bool ok = true;
  if (lane < k) {
    const int e = __ldcg(a.idx + (size_t)g * k + lane);
    const int p = __ldcg(win<const int32_t>(h, g / T, h.off_pos) + (size_t)(g % T) * k + lane);
    const uint4 *src = nullptr;
    if (p >= 0 && (p < tb.roff[e] || p >= tb.roff[e] + tb.cnt[e])) {
      raise_status(h, SYM_STATUS_OVERFLOW);  // a row outside its expert's tiles: skipped
    } else if (p >= 0) {
      ok = wait_geq(h, y_ready(h) + tb.tokprefix[e] + gemm2::tile_of_row(tb.cnt[e], p - tb.roff[e]), target);
      src = win<const uint4>(h, e / E_loc, h.off_y) + (size_t)p * (H / 8);
    }
    src_s[lane] = src;
    w_s[lane] = a.weights_in_ffn ? 1.f : __ldcg(a.w + (size_t)g * k + lane);
  }
  __syncwarp();  // the tables are read by every lane below
  if (!__all_sync(0xffffffffu, ok)) return;
  uint4 *dst = reinterpret_cast<uint4 *>(a.out) + (size_t)g * (H / 8);
  const int nvec = H / 8, step = 32 * U;
  const int npass = (nvec + step - 1) / step;
  // buf[b][j][u][lane]
  auto slot = [&](int b, int j, int u) { return buf + (((size_t)b * KMAX + j) * U + u) * 32 + lane; };
  auto issue = [&](int pass, int b) {
    for (int j = 0; j < k; ++j) {
      const uint4 *sp = src_s[j];
      if (!sp) continue;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = pass * step + u * 32 + lane;
        if (c < nvec) cp_async16(slot(b, j, u), sp + c);
      }
    }
    cp_async_commit();
  };
  issue(0, 0);
  for (int pass = 0; pass < npass; ++pass) {
    if (pass + 1 < npass) {
      issue(pass + 1, (pass + 1) & 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    const int b = pass & 1;
    float acc[U][8];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[u][i] = 0.f;
    for (int j = 0; j < k; ++j) {
      if (!src_s[j]) continue;
      const float ww = w_s[j];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = pass * step + u * 32 + lane;
        if (c >= nvec) continue;
        const uint4 x = *slot(b, j, u);
        acc[u][0] = fmaf(ww, bf16lo(x.x), acc[u][0]);
        acc[u][1] = fmaf(ww, bf16hi(x.x), acc[u][1]);
        acc[u][2] = fmaf(ww, bf16lo(x.y), acc[u][2]);
        acc[u][3] = fmaf(ww, bf16hi(x.y), acc[u][3]);
        acc[u][4] = fmaf(ww, bf16lo(x.z), acc[u][4]);
        acc[u][5] = fmaf(ww, bf16hi(x.z), acc[u][5]);
        acc[u][6] = fmaf(ww, bf16lo(x.w), acc[u][6]);
        acc[u][7] = fmaf(ww, bf16hi(x.w), acc[u][7]);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = pass * step + u * 32 + lane;
      if (c < nvec) {
        uint4 o;
        o.x = pack_bf16x2(acc[u][0], acc[u][1]);
        o.y = pack_bf16x2(acc[u][2], acc[u][3]);
        o.z = pack_bf16x2(acc[u][4], acc[u][5]);
        o.w = pack_bf16x2(acc[u][6], acc[u][7]);
        dst[c] = o;
      }
    }
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
  uint8_t *xch_raw = smem + (size_t)STAGES * STAGE_BYTES;
  uint8_t *ctrl_s = xch_raw + XCH_BYTES;
  uint64_t *bars = reinterpret_cast<uint64_t *>(ctrl_s);  // full[6] empty[6] acc_full[2] acc_empty[2] acc_head[2]
  uint64_t *drained = bars + 2 * STAGES + 6;  // every MMA of this launch has completed
  // tile queue of the dynamic schedule at ctrl_s + 168 (barriers) and + 232 (entries)
  const TileQueue tq{reinterpret_cast<volatile int *>(ctrl_s + 232), reinterpret_cast<uint64_t *>(ctrl_s + 168),
                     reinterpret_cast<uint64_t *>(ctrl_s + 168) + TQ};
  uint32_t *tmem_base_s = reinterpret_cast<uint32_t *>(drained + 1);
  volatile int *abort_s = reinterpret_cast<volatile int *>(tmem_base_s + 1);
  volatile int *never_s = abort_s + 1;  // stop bound of the schedule: the entry where this CTA stopped
  int *bcast = const_cast<int *>(never_s + 1);
  // per-warp row-slot barriers of the scatter phase
  uint64_t *sbar = reinterpret_cast<uint64_t *>(ctrl_s + 256) + warp_id() * SCATTER_SLOTS_MAX;
  const int E = h.s.num_experts;
  int *tab = reinterpret_cast<int *>(ctrl_s + FUSED_CTRL_SMEM);
  const TokTables tb{tab, tab + E, tab + 2 * E};
  const int wid = warp_id(), lane = lane_id();
  // per-warp destination / source pointer and weight tables of phases 2 and 4
  // (32 entries each), in the exchange buffer, which only phase 3 uses
  void **ptr_s = reinterpret_cast<void **>(xch_raw) + wid * 32;
  float *wgt_s = reinterpret_cast<float *>(xch_raw + FUSED_THREADS / 32 * 32 * sizeof(void *)) + wid * 32;
  const int N = h.s.world * h.s.tokens_per_slot;
  const int nchunks = (N + FUSED_CHUNK - 1) / FUSED_CHUNK;

  Pipe p;
  p.ring = ring;
  p.xch = reinterpret_cast<float *>(xch_raw);
  p.full = bars;
  p.empty = bars + STAGES;
  p.acc_full = bars + 2 * STAGES;
  p.acc_empty = bars + 2 * STAGES + 2;
  p.acc_head = bars + 2 * STAGES + 4;
  p.rank = cta_rank();
  p.abort = abort_s;
  p.stop = never_s;
  p.tmo = h.wait_timeout_us;
  p.scale_rows = a.weights_in_ffn;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&p.full[s], 1);  // used on the leader: one arrive (with both CTAs' bytes)
      mbar_init(&p.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&p.acc_full[b], 1);
      mbar_init(&p.acc_empty[b], 8);  // leader: 4 epilogue warps of each CTA
      mbar_init(&p.acc_head[b], 8);
    }
    mbar_init(drained, 1);
    tq_init(tq);
    uint64_t *sbar0 = reinterpret_cast<uint64_t *>(ctrl_s + 256);
    for (int i = 0; i < FUSED_THREADS / 32 * SCATTER_SLOTS_MAX; ++i) mbar_init(&sbar0[i], 1);
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
  p.tmem_base = *tmem_base_s;

  // ---------------- phase 1: route, count, scan
  // Route tasks of rt tokens: a whole 32-token chunk when there are chunks
  // for every CTA, else one token per warp (short batches).  The CTA finishing
  // the last route task of a chunk counts that chunk.
  {
    const int rt = nchunks >= (int)gridDim.x ? FUSED_CHUNK : ROUTE_TOKENS;
    const int nroute = (N + rt - 1) / rt;
    const int tasks_per_chunk = FUSED_CHUNK / rt;
    for (;;) {
      const int t = claim(h, C_ROUTE_NEXT, bcast);
      if (t >= nroute) break;
      route_task(h, a, t, rt, reinterpret_cast<float *>(ring));
      const int c = t / tasks_per_chunk;
      const int in_chunk = min(tasks_per_chunk, (min(N, (c + 1) * FUSED_CHUNK) - c * FUSED_CHUNK + rt - 1) / rt);
      __syncthreads();
      if (threadIdx.x == 0) {
        __threadfence();  // release this task's routes
        *bcast = (int)atomicAdd(chunk_done(h) + c, 1u) == in_chunk - 1;
        __threadfence();  // acquire the chunk's other routes
      }
      __syncthreads();
      if (!*bcast) continue;
      count_chunk(h, a, c, reinterpret_cast<uint32_t *>(ring) + (FUSED_THREADS / 32) * h.s.num_experts);
      __threadfence();
      __syncthreads();
      if (threadIdx.x == 0) atomicAdd(ctl(h) + C_ROUTE_DONE, 1u);
    }
  }
  // Scan tasks, one per expert, once every chunk is counted (all route tasks
  // are claimed by running CTAs, so the wait ends); the CTA completing the
  // last scan task finishes the scan.
  if (threadIdx.x == 0) *bcast = wait_geq(h, ctl(h) + C_ROUTE_DONE, (uint32_t)nchunks) ? 1 : 0;
  __syncthreads();
  if (*bcast) {
    int *seg_s = reinterpret_cast<int *>(ring);
    for (;;) {
      const int e = claim(h, C_SCAN_NEXT, bcast);
      if (e >= h.s.num_experts) break;
      scan_expert(h, e, seg_s);
      __threadfence();
      __syncthreads();
      if (threadIdx.x == 0) *bcast = (int)atomicAdd(ctl(h) + C_SCAN_TASKS, 1u);
      __syncthreads();
      if (*bcast == h.s.num_experts - 1) {
        __threadfence();  // acquire every scan task's counts
        finish_scan(h);
      }
    }
  }

  // ---------------- phase 2: scatter
  if (threadIdx.x == 0) *bcast = wait_geq(h, ctl(h) + C_SCAN_DONE, h.epoch) ? 1 : 0;
  __syncthreads();
  const bool scanned = *bcast != 0 && ld_acquire_u32(ctl(h) + C_SCAN_DONE) == h.epoch;
  // rows per warp staged in its share of the ring (0: rows too wide, plain copies)
  const size_t warp_ring = (size_t)STAGES * STAGE_BYTES / (FUSED_THREADS / 32);
  const int slots = min(SCATTER_SLOTS_MAX, (int)(warp_ring / ((size_t)h.s.hidden * 2)));
  const int scatter_tasks = slots > 0 ? (N + FUSED_THREADS / 32 * slots - 1) / (FUSED_THREADS / 32 * slots)
                                      : (N + SCATTER_TOKENS - 1) / SCATTER_TOKENS;
  int tasks_done = 0;
  if (scanned && slots > 0) {
    // the ring held phase 1's logits rows (generic stores); the copy engine writes it next
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    const int per_task = FUSED_THREADS / 32 * slots;
    const int ntask = scatter_tasks;
    uint4 **dst_tab = reinterpret_cast<uint4 **>(xch_raw) + wid * SCATTER_SLOTS_MAX * 32;
    uint32_t sph = 0;
    for (;;) {
      const int t = claim(h, C_SCATTER_NEXT, bcast);
      if (t >= ntask) break;
      if (!scatter_bulk(h, a, t * per_task + wid * slots, slots, ring + wid * warp_ring, sbar, sph, lane,
                        dst_tab))
        set_abort(h);
      ++tasks_done;
    }
  } else if (scanned) {
    for (;;) {
      const int t = claim(h, C_SCATTER_NEXT, bcast);
      if (t >= scatter_tasks) break;
      for (int i = wid; i < SCATTER_TOKENS; i += FUSED_THREADS / 32) {
        const int g = t * SCATTER_TOKENS + i;
        if (g < N) scatter_token(h, a, g, lane, reinterpret_cast<uint4 **>(ptr_s));
      }
      ++tasks_done;
    }
  }
  // publish this CTA's completed scatter tasks (release of its pos / row writes)
  __syncthreads();
  if (threadIdx.x == 0 && tasks_done > 0) {
    __threadfence();
    atomicAdd(ctl(h) + C_SCATTER_DONE, (uint32_t)tasks_done);
  }

  // ---------------- phase 3: expert GEMM tiles on the CTA pair
  if (scanned) build_tok_tables(h, tb);
  // the ring held phase 1's logits rows (generic stores); TMA writes it next
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncthreads();
  if (scanned) {
    const int nf1 = nf_of(h, GATE_UP), nf2 = nf_of(h, DOWN);
    const int g1 = tok_group_of(h, GATE_UP), g2 = tok_group_of(h, DOWN);
    const int total1 = tb.tokprefix[E] * nf1, total2 = tb.tokprefix[E] * nf2;
    const uint32_t h_target = EPI_WARPS_PER_TILE * (uint32_t)nf1;
    auto wait = [&](const uint32_t *c, uint32_t target) { return wait_geq(h, c, target); };
    // inputs of a tile in place: its dispatched rows (gate/up) or every
    // gate/up feature tile of its token tile (down)
    auto inputs_ready = [&](int kind, int t, bool block) -> bool {
      const TileInfo ti = decode_tok(h, tb, kind == GATE_UP ? nf1 : nf2, kind == GATE_UP ? g1 : g2, t);
      if (kind == DOWN) {
        const uint32_t *c = h_ready(h) + tb.tokprefix[ti.e] + ti.n;
        return block ? wait_geq(h, c, h_target) : ld_acquire_u32(c) >= h_target;
      }
      return rows_ready(h, ti.d, ti.row0, ti.valid, block, wait);
    };
    // The pair's tiles, claimed from one counter: claim c < total1 is gate/up
    // tile c, else down tile c - total1.  Every role walks the schedule by
    // entry n (gemm2sm.cuh, TileQueue).
    uint32_t *next = ctl(h) + C_TILE_NEXT;
    auto kind_of = [&](int c) { return c < total1 ? GATE_UP : DOWN; };
    auto tile_of = [&](int c) { return c < total1 ? c : c - total1; };
    auto info_of = [&](int c) {
      return c < total1 ? decode_tok(h, tb, nf1, g1, c) : decode_tok(h, tb, nf2, g2, c - total1);
    };
    if (wid == 0) {
      if (lane == 0) {
        // ------------------------------------------------------------ producer
        ProdState ps;
        auto claim = [&]() {
          const int c = (int)atomicAdd(next, 1u);
          return c < total1 + total2 ? c : -1;
        };
        auto ready = [&](int c, bool block) { return inputs_ready(kind_of(c), tile_of(c), block); };
        auto produce = [&](int c, int n, auto &probe) {
          return kind_of(c) == GATE_UP
                     ? produce_tile<GATE_UP>(h, p, ps, info_of(c), &tm_g, &tm_u, tm_rx, n, probe)
                     : produce_tile<DOWN>(h, p, ps, info_of(c), &tm_d, &tm_d, tm_h, n, probe);
        };
        if (!produce_schedule(h, p, tq, never_s, true, claim, ready, produce)) *abort_s = 1;
      }
    } else if (wid == 1) {
      if (lane == 0 && p.rank == 0) {
        // ------------------------------------------------------ MMA issuer (leader)
        MmaState ms;
        for (int n = 0;; ++n) {
          const int c = tq_pop(h, p, tq, n);
          if (c < 0) break;
          const bool ok = kind_of(c) == GATE_UP ? mma_tile<GATE_UP>(h, p, ms, info_of(c), n)
                                                : mma_tile<DOWN>(h, p, ms, info_of(c), n);
          if (!ok) break;
        }
        // after an abort the epilogue may stop before the last accumulator:
        // wait for the MMAs still in flight before TMEM is released
        commit2_both(drained);
        mbar_wait(drained, 0, p.tmo, nullptr);
      }
    } else if (wid < 6) {
      // -------------------------------------------------------------- epilogue
      const int q = wid & 3;  // TMEM lane quarter this warp may access
      EpiState es;
      for (int n = 0;; ++n) {
        int c = 0;
        if (lane == 0) c = tq_pop(h, p, tq, n);  // lane 0 reads the entry and hands it back
        c = __shfl_sync(0xffffffffu, c, 0);
        // The gate/up epilogue's partner warps meet at named barriers, so they
        // act on an entry only together: they read the same entries, but a
        // failed wait (an abort in this CTA) can end one partner's read early.
        if (!xch_vote(q & 1, c >= 0)) break;
        const TileInfo ti = info_of(c);
        const bool ok = kind_of(c) == GATE_UP ? epi_tile<GATE_UP>(h, p, es, ti, n, q, lane)
                                              : epi_tile<DOWN>(h, p, es, ti, n, q, lane);
        if (!ok) break;
        // publish this warp's share of the tile (read next by TMA or by the
        // combine's generic loads in other CTAs)
        __threadfence();
        asm volatile("fence.proxy.async.global;" ::: "memory");
        __syncwarp();
        if (lane == 0)
          atomicAdd((kind_of(c) == GATE_UP ? h_ready(h) : y_ready(h)) + tb.tokprefix[ti.e] + ti.n, 1u);
      }
    }
    if (*abort_s) set_abort(h);
  }
  __syncthreads();

  // ---------------- phase 4: combine
  // every token's pos is final once all scatter tasks are done (a CTA with no
  // GEMM tiles gets here while other CTAs may still be scattering)
  if (threadIdx.x == 0)
    *bcast = scanned && wait_geq(h, ctl(h) + C_SCATTER_DONE, (uint32_t)scatter_tasks) ? 1 : 0;
  // the ring was last touched by the async proxy (TMA, MMA); cp.async writes it next
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncthreads();
  if (*bcast) {
    const int ntask = (N + COMBINE_TOKENS - 1) / COMBINE_TOKENS;
    for (;;) {
      const int t = claim(h, C_COMB_NEXT, bcast);
      if (t >= ntask) break;
      for (int i = wid; i < COMBINE_TOKENS; i += FUSED_THREADS / 32) {
        const int g = t * COMBINE_TOKENS + i;
        if (g >= N) continue;
        const uint4 **src_tab = reinterpret_cast<const uint4 **>(const_cast<const void **>(ptr_s));
        uint4 *cbuf = reinterpret_cast<uint4 *>(ring + wid * warp_ring);
        if (h.s.topk <= 2)
          combine_token_stream<8, 2>(h, a, tb, g, lane, src_tab, wgt_s, cbuf);
        else if (h.s.topk <= 4)
          combine_token_stream<6, 4>(h, a, tb, g, lane, src_tab, wgt_s, cbuf);
        else if (h.s.topk <= 8)
          combine_token_stream<3, 8>(h, a, tb, g, lane, src_tab, wgt_s, cbuf);
        else
          combine_token<4, 4>(h, a, tb, g, lane, src_tab, wgt_s);
      }
    }
  }

  // ---------------- teardown
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no remote arrive or MMA of the pair is still in flight
  tc_fence_after();
  if (wid == 1) tmem_dealloc2(p.tmem_base, TMEM_COLS);
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(ctl(h) + C_EXIT, 1u) == gridDim.x - 1) {
      // last CTA out: reset the counters for the next launch
      uint32_t *c = ctl(h);
      c[C_ROUTE_NEXT] = 0;
      c[C_ROUTE_DONE] = 0;
      c[C_SCAN_NEXT] = 0;
      c[C_SCAN_TASKS] = 0;
      c[C_SCATTER_NEXT] = 0;
      c[C_SCATTER_DONE] = 0;
      c[C_COMB_NEXT] = 0;
      c[C_TILE_NEXT] = 0;
      c[C_ABORT] = 0;
      __threadfence();
      c[C_EXIT] = 0;
    }
  }
}

size_t fused_ctrl_bytes(const moe_shape &s) {
  const int nchunks = (s.world * s.tokens_per_slot + FUSED_CHUNK - 1) / FUSED_CHUNK;
  return (size_t)(C_WORDS + fused_h_blocks(s) + fused_y_blocks(s) + nchunks) * 4;
}

cudaError_t launch_fused(const sym_heap &h, const float *logits, const uint16_t *x,
                         const uint16_t *wg, const uint16_t *wu, const uint16_t *wd, int32_t *idx,
                         float *w, uint16_t *out, int weights_in_ffn, int num_sms, cudaStream_t st) {
  using namespace gemm2;
  const int E = h.s.num_experts, H = h.s.hidden, I = h.s.inter;
  CUtensorMap tg, tu, td;
  BMaps trx, th;
  if (!encode_2d(&tg, wg, (uint64_t)E * I, H, 64) || !encode_2d(&tu, wu, (uint64_t)E * I, H, 64) ||
      !encode_heap_boxes(&trx, h, h.off_recv_x, H) ||
      !encode_2d(&td, wd, (uint64_t)E * H, I, 128) || !encode_heap_boxes(&th, h, h.off_h, I))
    return cudaErrorInvalidValue;
  static_assert(FUSED_THREADS / 32 * 32 * (sizeof(void *) + sizeof(float)) <= (size_t)XCH_BYTES &&
                    FUSED_THREADS / 32 * SCATTER_SLOTS_MAX * 32 * sizeof(void *) <= (size_t)XCH_BYTES,
                "per-warp tables live in the exchange buffer");
  static_assert(256 + FUSED_THREADS / 32 * SCATTER_SLOTS_MAX * 8 <= FUSED_CTRL_SMEM, "scatter barriers");
  static_assert(2 * 8 * 3 * 32 * 16 <= STAGES * STAGE_BYTES / (FUSED_THREADS / 32) &&
                    2 * 4 * 6 * 32 * 16 <= STAGES * STAGE_BYTES / (FUSED_THREADS / 32) &&
                    2 * 2 * 8 * 32 * 16 <= STAGES * STAGE_BYTES / (FUSED_THREADS / 32),
                "combine stream buffers fit a warp's share of the ring");
  const size_t smem = 1024 + (size_t)STAGES * STAGE_BYTES + XCH_BYTES + FUSED_CTRL_SMEM +
                      tok_tables_bytes(E);
  cudaError_t err = cudaFuncSetAttribute(moe_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
  if (err != cudaSuccess) return err;
  // every pair resident at once: a down tile waits for gate/up tiles that other pairs hold
  const int grid = 2 * max_resident_pairs((const void *)moe_fused_kernel, FUSED_THREADS, smem, num_sms);
  if (grid <= 0) return cudaErrorInvalidConfiguration;
  const FusedArgs a{logits, x, idx, w, out, weights_in_ffn};
  moe_fused_kernel<<<grid, FUSED_THREADS, smem, st>>>(h, a, tg, tu, trx, td, th);
  return cudaGetLastError();
}

}  // namespace symmoe
