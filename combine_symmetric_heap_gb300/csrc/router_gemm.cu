// router_gemm.cu -- the router (gate) GEMM that produces the routing logits:
//   logits[g][e] = sum_h x[g][h] * Wr[e][h],  fp32 accumulation and output.
//
// The pages take the routing indices and weights as dispatch inputs (MORI CCO
// blog, "Zero-copy MoE dispatch -> expert -> combine"); this is the step that
// produces them from the token activations, the gate GEMM of an MoE layer.
// It runs on the CTA-pair tile engine of the expert GEMM (gemm2sm.cuh) as one
// pseudo-expert over all N tokens: router rows on the MMA's M side (256 per
// pair tile, rows past E zero-filled by the copy), tokens on the N side
// (256 per tile, the same remainder rule as an expert's rows), K = H.
#include "gemm2sm.cuh"

namespace symmoe {

constexpr int ROUTER_THREADS = 192;
constexpr int ROUTER_CTRL_BYTES = 256;

static size_t router_smem_bytes() {
  return 1024 + (size_t)gemm2::STAGES * gemm2::STAGE_BYTES + gemm2::XCH_BYTES + ROUTER_CTRL_BYTES;
}

// tile t of the token list (one pseudo-expert with N rows), feature tile major
__device__ inline gemm2::TileInfo decode_router(int N, int nf, int t) {
  const int ntok = gemm2::ntok_of(N);
  gemm2::TileInfo ti;
  ti.e = 0;
  ti.d = 0;
  ti.f = t / ntok;
  ti.n = t % ntok;
  ti.row0 = ti.n * gemm2::BN;
  ti.valid = ti.n == ntok - 1 ? N - ti.n * gemm2::BN : gemm2::BN;
  (void)nf;
  return ti;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(ROUTER_THREADS, 1)
    router_gemm_kernel(const sym_heap h, const __grid_constant__ CUtensorMap tm_wr,
                       const __grid_constant__ gemm2::BMaps tm_x, float *logits) {
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
  const int N = h.s.world * h.s.tokens_per_slot;
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
    tma_prefetch_desc(&tm_wr);
    for (int i = 0; i < NBOX; ++i) tma_prefetch_desc(&tm_x.m[i]);
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
  const int nf = nf_of(h, ROUTER);
  const int total_tiles = ntok_of(N) * nf;

  if (wid == 0) {
    if (lane == 0) {
      ProdState ps;
      for (int i = 0, t; (t = pair_tile(i, pair_id, npairs)) < total_tiles; ++i)
        if (!produce_tile<ROUTER>(h, p, ps, decode_router(N, nf, t), &tm_wr, &tm_wr, tm_x, t, []() {})) break;
    }
  } else if (wid == 1) {
    if (lane == 0 && p.rank == 0) {
      MmaState ms;
      for (int i = 0, t; (t = pair_tile(i, pair_id, npairs)) < total_tiles; ++i)
        if (!mma_tile<ROUTER>(h, p, ms, decode_router(N, nf, t), t)) break;
    }
  } else {
    const int q = wid & 3;
    EpiState es;
    for (int i = 0, t; (t = pair_tile(i, pair_id, npairs)) < total_tiles; ++i)
      if (!epi_tile<ROUTER>(h, p, es, decode_router(N, nf, t), t, q, lane)) break;
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no remote arrive or MMA of the pair is still in flight
  tc_fence_after();
  if (wid == 1) tmem_dealloc2(p.tmem_base, TMEM_COLS);
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

cudaError_t launch_router(const sym_heap &h, const uint16_t *x, const uint16_t *wr, float *logits,
                          int num_sms, cudaStream_t st) {
  using namespace gemm2;
  const int E = h.s.num_experts, H = h.s.hidden;
  const uint64_t N = (uint64_t)h.s.world * h.s.tokens_per_slot;
  CUtensorMap twr;
  BMaps tx;
  if (!encode_2d(&twr, wr, (uint64_t)E, H, 128) || !encode_rows_boxes(&tx, x, N, H))
    return cudaErrorInvalidValue;
  const size_t smem = router_smem_bytes();
  cudaError_t err = cudaFuncSetAttribute(router_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const int grid = 2 * max_resident_pairs((const void *)router_gemm_kernel, ROUTER_THREADS, smem, num_sms);
  if (grid <= 0) return cudaErrorInvalidConfiguration;
  router_gemm_kernel<<<grid, ROUTER_THREADS, smem, st>>>(h, twr, tx, logits);
  return cudaGetLastError();
}

}  // namespace symmoe
