// router_gemm.cu -- the router (gate) GEMM that produces the routing logits:
//   logits[g][e] = sum_h x[g][h] * Wr[e][h],  fp32 accumulation and output.
//
// The pages take the routing indices and weights as dispatch inputs (MORI CCO
// blog, "Zero-copy MoE dispatch -> expert -> combine"); this is the step that
// produces them from the token activations, the gate GEMM of an MoE layer.
// It runs on the CTA-pair tile engine of the expert GEMM (gemm2sm.cuh): tokens
// on the MMA's M side (256 per pair tile, rows past N zero-filled by the copy)
// and the E router rows on the N side, as the rows of one pseudo-expert (256
// per tile, the same remainder rule as an expert's rows; the MMA width is the
// row count rounded up to 16), K = H.  With E = 8 the MMA is 256 x 16 rather
// than an M side of 8 rows padded to 256.
//
// With few tiles (small N, E <= 256) most CTA pairs would sit idle, so K is
// split S ways: work item (tile, ks) accumulates K blocks
// [ks*kb_per_split, (ks+1)*kb_per_split) and stores an fp32 partial tile at
// split ks of a scratch array [S][N][E]; router_reduce_kernel then adds the S
// partials in split order, so the result does not depend on the schedule.
// S = 1 writes the logits directly.
#include "gemm2sm.cuh"

namespace symmoe {

constexpr int ROUTER_THREADS = 192;
constexpr int ROUTER_CTRL_BYTES = 256;

static size_t router_smem_bytes() {
  return 1024 + (size_t)gemm2::STAGES * gemm2::STAGE_BYTES + gemm2::XCH_BYTES + ROUTER_CTRL_BYTES;
}

// work item t: split ks = t / tiles of tile t % tiles; a tile is (token tile
// f, router-row tile n), router-row tile minor so that the tiles of one token
// tile run side by side and share its x reads in L2
__device__ inline gemm2::TileInfo decode_router(int E, int tiles, int t) {
  const int nrt = gemm2::ntok_of(E);
  const int tile = t % tiles;
  gemm2::TileInfo ti;
  ti.e = 0;
  ti.d = 0;
  ti.ks = t / tiles;
  ti.f = tile / nrt;
  ti.n = tile % nrt;
  ti.row0 = ti.n * gemm2::BN;
  ti.valid = ti.n == nrt - 1 ? E - ti.n * gemm2::BN : gemm2::BN;
  return ti;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(ROUTER_THREADS, 1)
    router_gemm_kernel(const sym_heap h, const __grid_constant__ CUtensorMap tm_x,
                       const __grid_constant__ gemm2::BMaps tm_wr, float *logits, int splits,
                       int kb_per_split) {
  using namespace gemm2;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *ctrl = smem + (size_t)STAGES * STAGE_BYTES + XCH_BYTES;
  uint64_t *bars = reinterpret_cast<uint64_t *>(ctrl);  // full[6] empty[6] acc_full[2] acc_empty[2] acc_head[2]
  uint32_t *tmem_base_s = reinterpret_cast<uint32_t *>(bars + 2 * STAGES + 6);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_base_s + 1);
  volatile int *stop_tile = abort_flag + 1;
  const int wid = warp_id(), lane = lane_id();
  const int pair_id = (int)cluster_id_x(), npairs = (int)num_clusters_x();
  Pipe p;
  p.ring = smem;
  p.xch = reinterpret_cast<float *>(smem + (size_t)STAGES * STAGE_BYTES);
  p.full = bars;
  p.empty = bars + STAGES;
  p.acc_full = bars + 2 * STAGES;
  p.acc_empty = bars + 2 * STAGES + 2;
  p.acc_head = bars + 2 * STAGES + 4;
  p.rank = cta_rank();
  p.abort = abort_flag;
  p.stop = stop_tile;
  p.tmo = h.wait_timeout_us;
  p.scale_rows = 0;
  p.logits = logits;
  p.kb_per_split = splits > 1 ? kb_per_split : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&p.full[s], 1);
      mbar_init(&p.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&p.acc_full[b], 1);
      mbar_init(&p.acc_empty[b], 8);
      mbar_init(&p.acc_head[b], 8);
    }
    *abort_flag = 0;
    *stop_tile = 0x7fffffff;
    fence_mbar_init();
    tma_prefetch_desc(&tm_x);
    for (int i = 0; i < NBOX; ++i) tma_prefetch_desc(&tm_wr.m[i]);
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
  pdl_launch_dependents();  // the reduction may be scheduled; it waits for this grid to finish
  const int E = h.s.num_experts;
  const int tiles = nf_of(h, ROUTER) * ntok_of(E);
  const int total_tiles = tiles * splits;

  if (wid == 0) {
    if (lane == 0) {
      ProdState ps;
      for (int i = 0, t; (t = pair_tile(i, pair_id, npairs)) < total_tiles; ++i)
        if (!produce_tile<ROUTER>(h, p, ps, decode_router(E, tiles, t), &tm_x, &tm_x, tm_wr, t, []() {})) break;
    }
  } else if (wid == 1) {
    if (lane == 0 && p.rank == 0) {
      MmaState ms;
      for (int i = 0, t; (t = pair_tile(i, pair_id, npairs)) < total_tiles; ++i)
        if (!mma_tile<ROUTER>(h, p, ms, decode_router(E, tiles, t), t)) break;
    }
  } else {
    const int q = wid & 3;
    EpiState es;
    for (int i = 0, t; (t = pair_tile(i, pair_id, npairs)) < total_tiles; ++i)
      if (!epi_tile<ROUTER>(h, p, es, decode_router(E, tiles, t), t, q, lane)) break;
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no remote arrive or MMA of the pair is still in flight
  tc_fence_after();
  if (wid == 1) tmem_dealloc2(p.tmem_base, TMEM_COLS);
}

// logits[i] = sum over ks = 0..S-1, in that order, of part[ks][i]
__global__ void __launch_bounds__(256) router_reduce_kernel(const float *part, float *logits, size_t n, int S) {
  pdl_wait();  // the partials of the router GEMM
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  const size_t i0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if ((reinterpret_cast<uintptr_t>(logits) & 15u) == 0 && (n & 3u) == 0) {
    const size_t n4 = n / 4;
    const float4 *p4 = reinterpret_cast<const float4 *>(part);
    for (size_t i = i0; i < n4; i += stride) {
      float4 a = __ldcs(p4 + i);
      for (int s = 1; s < S; ++s) {
        const float4 b = __ldcs(p4 + (size_t)s * n4 + i);
        a.x += b.x;
        a.y += b.y;
        a.z += b.z;
        a.w += b.w;
      }
      reinterpret_cast<float4 *>(logits)[i] = a;
    }
  } else {
    for (size_t i = i0; i < n; i += stride) {
      float a = __ldcs(part + i);
      for (int s = 1; s < S; ++s) a += __ldcs(part + (size_t)s * n + i);
      logits[i] = a;
    }
  }
}

// Number of K splits S, from a rough time model: the busiest pair runs
// ceil(tiles*S / pairs) items of ceil(nk/S) K blocks plus a fixed cost per
// item (pipeline start, epilogue), about 0.45 us per block; each split adds
// its partial's write and read at about 6 TB/s.  At least 2 K blocks per
// split, and the partials must fit the scratch.
static int router_splits(int tiles, int nk, int npairs, size_t scratch_bytes, size_t part_bytes) {
  constexpr double KB_US = 0.45, ITEM_KB = 3.0, BYTES_PER_US = 6.0e6, REDUCE_US = 2.0;
  int best = 1;
  double best_us = (double)((tiles + npairs - 1) / npairs) * (nk + ITEM_KB) * KB_US;
  for (int S = 2; S <= nk / 2 && (size_t)S * part_bytes <= scratch_bytes; ++S) {
    const double waves = (double)(((long)tiles * S + npairs - 1) / npairs);
    const double us = waves * ((nk + S - 1) / S + ITEM_KB) * KB_US + 2.0 * S * part_bytes / BYTES_PER_US + REDUCE_US;
    if (us < best_us) best = S, best_us = us;
  }
  return best;
}

// bf16 rows [rows][cols] as a 3-D map {cols, rows, 1} with the token-row boxes
static bool encode_rows_boxes(gemm2::BMaps *m, const void *ptr, uint64_t rows, uint64_t cols) {
  sym_heap fake = {};
  fake.base = reinterpret_cast<uint64_t>(ptr);
  fake.cap = rows;
  fake.per_rank_size = rows * cols * 2;
  fake.s.world = 1;
  return encode_heap_boxes(m, fake, 0, cols);
}

// Launch plan of the router on this device: grid (CTAs), K splits and K blocks
// per split.  The partials live in slot 0's y window, which holds nothing
// between a combine and the next expert FFN.
cudaError_t router_plan(const sym_heap &h, int num_sms, int *grid, int *splits, int *kb_per_split) {
  using namespace gemm2;
  const int E = h.s.num_experts, H = h.s.hidden;
  const uint64_t N = (uint64_t)h.s.world * h.s.tokens_per_slot;
  const size_t smem = router_smem_bytes();
  cudaError_t err = cudaFuncSetAttribute(router_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  *grid = 2 * max_resident_pairs((const void *)router_gemm_kernel, ROUTER_THREADS, smem, num_sms);
  if (*grid <= 0) return cudaErrorInvalidConfiguration;
  const int tiles = nf_of(h, ROUTER) * ntok_of(E), nk = nk_of(h, ROUTER);
  const int S0 = router_splits(tiles, nk, *grid / 2, (size_t)h.cap * H * 2, N * (size_t)E * 4);
  *kb_per_split = (nk + S0 - 1) / S0;
  *splits = (nk + *kb_per_split - 1) / *kb_per_split;  // no split is left without K blocks
  return cudaSuccess;
}

cudaError_t launch_router(const sym_heap &h, const uint16_t *x, const uint16_t *wr, float *logits,
                          int num_sms, cudaStream_t st) {
  using namespace gemm2;
  const int E = h.s.num_experts, H = h.s.hidden;
  const uint64_t N = (uint64_t)h.s.world * h.s.tokens_per_slot;
  CUtensorMap tx;
  BMaps twr;
  if (!encode_2d(&tx, x, N, H, 128) || !encode_rows_boxes(&twr, wr, (uint64_t)E, H))
    return cudaErrorInvalidValue;
  int grid, S, kb_per_split;
  cudaError_t err = router_plan(h, num_sms, &grid, &S, &kb_per_split);
  if (err != cudaSuccess) return err;
  float *part = S > 1 ? reinterpret_cast<float *>(h.base + h.off_y) : logits;
  router_gemm_kernel<<<grid, ROUTER_THREADS, router_smem_bytes(), st>>>(h, tx, twr, part, S, kb_per_split);
  if ((err = cudaGetLastError()) != cudaSuccess || S == 1) return err;
  const size_t n = N * (size_t)E;
  const int rgrid = (int)std::min<size_t>((n / 4 + 255) / 256 + 1, (size_t)num_sms * 8);
  return launch_pdl(router_reduce_kernel, dim3(rgrid), dim3(256), 0, st, (const float *)part, logits, n, S);
}

}  // namespace symmoe
