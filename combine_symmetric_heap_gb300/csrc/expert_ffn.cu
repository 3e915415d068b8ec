// expert_ffn.cu -- grouped SwiGLU expert FFN on the 5th-generation tensor
// cores (tcgen05.mma, accumulators in TMEM, operands staged by TMA), run on
// CTA pairs (cta_group::2: one M=256 MMA spans two SMs of a cluster).
//
// MORI CCO blog, "Zero-copy MoE dispatch -> expert -> combine": the expert
// GEMM reads the dispatched rows in place from the receive window and writes
// its output straight into the combine staging window.  Per expert e with
// cnt_e received rows A (a contiguous block of slot e/(E/W)'s recv_x window):
//   GEMM1  h = bf16( silu(A Wg_e^T) * (A Wu_e^T) )    -> h window
//   GEMM2  y = bf16( h Wd_e^T )                         -> y window (out_tok)
// Tile geometry, barriers and the pair protocol are described in gemm2sm.cuh.
//
// One persistent CTA per SM, in clusters of two, warp-specialised:
//   warp 0   TMA producer (one thread): waits for the dispatch ready counters
//            of its token rows (bounded; the next tile's are probed while the
//            current one streams), then streams K blocks of 64 through a
//            6-deep shared-memory ring;
//   warp 1   allocates TMEM (both CTAs) and, in the pair's first CTA, issues
//            the tcgen05.mma; two accumulator buffers let the epilogue of
//            tile i overlap the main loop of tile i+1;
//   warps 2-5 epilogue: tcgen05.ld, SwiGLU / bf16 rounding, stores.
// Pairs claim tiles dynamically (the leader's producer takes the next index
// from a counter in the heap's control window and hands it to the pair's
// other roles, gemm2sm.cuh); row counts come from the dispatch signal area on
// the device (no host sync).
#include <mutex>

#include "gemm2sm.cuh"

namespace symmoe {

constexpr int GEMM_THREADS = 192;

// ---------------------------------------------------------------------------
// CTA-pair (cta_group::2) expert GEMM, used by moe_expert_ffn
// ---------------------------------------------------------------------------
constexpr int G2_CTRL_BYTES = 256;
// words of slot 0's control window used by the staged expert GEMM's dynamic
// schedule: per kind the next tile to claim and the CTAs done (the last CTA
// out resets both, so every launch starts from zero)
constexpr int G2_SCHED_WORD = 32;

static size_t gemm2_smem_bytes(int num_experts) {
  return 1024 + (size_t)gemm2::STAGES * gemm2::STAGE_BYTES + gemm2::XCH_BYTES + G2_CTRL_BYTES +
         gemm2::tok_tables_bytes(num_experts);
}

template <int KIND>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(GEMM_THREADS, 1)
    expert_gemm2_kernel(const sym_heap h, const __grid_constant__ CUtensorMap tm_a0,
                        const __grid_constant__ CUtensorMap tm_a1,
                        const __grid_constant__ gemm2::BMaps tm_b, int wait_ready, int scale_rows) {
  using namespace gemm2;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *ctrl = smem + (size_t)STAGES * STAGE_BYTES + XCH_BYTES;
  uint64_t *bars = reinterpret_cast<uint64_t *>(ctrl);  // full[6] empty[6] acc_full[2] acc_empty[2] acc_head[2]
  // tile queue: full[TQ] empty[TQ] after the ring barriers, then the words
  const TileQueue tq{reinterpret_cast<volatile int *>(bars + 2 * STAGES + 6 + 2 * TQ + 2),
                     bars + 2 * STAGES + 6, bars + 2 * STAGES + 6 + TQ};
  uint32_t *tmem_base_s = reinterpret_cast<uint32_t *>(bars + 2 * STAGES + 6 + 2 * TQ);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_base_s + 1);
  volatile int *stop_tile = abort_flag + 1;
  const int E = h.s.num_experts;
  int *tab = reinterpret_cast<int *>(ctrl + G2_CTRL_BYTES);
  const TokTables tb{tab, tab + E, tab + 2 * E};
  const int wid = warp_id(), lane = lane_id();
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
  p.scale_rows = scale_rows;

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
    tq_init(tq);
    *abort_flag = 0;
    *stop_tile = 0x7fffffff;
    fence_mbar_init();
    tma_prefetch_desc(&tm_a0);
    if (KIND == GATE_UP) tma_prefetch_desc(&tm_a1);
    for (int i = 0; i < NBOX; ++i) tma_prefetch_desc(&tm_b.m[i]);
  }
  if (wid == 1) {
    tmem_alloc2(tmem_base_s, TMEM_COLS);
    tmem_relinquish2();
  }
  build_tok_tables(h, tb);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // barriers of both CTAs initialised before any remote arrive
  tc_fence_after();
  p.tmem_base = *tmem_base_s;
  const int nf = nf_of(h, KIND), grp = tok_group_of(h, KIND);
  const int total_tiles = tb.tokprefix[E] * nf;
  const uint32_t tmo = h.wait_timeout_us;
  auto wait = [&](const uint32_t *c, uint32_t target) { return wait_counter_geq(c, target, tmo, abort_flag); };
  uint32_t *sched = win<uint32_t>(h, 0, h.off_ctrl) + G2_SCHED_WORD + 2 * KIND;  // next tile, CTAs done

  // Every role walks the pair's schedule by entry n; the stop bound and the
  // wait bounds count entries.
  if (wid == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      ProdState ps;
      auto claim = [&]() {
        const int t = (int)atomicAdd(sched, 1u);
        return t < total_tiles ? t : -1;
      };
      // the tile's token rows dispatched (the whole tile, both CTAs' halves)
      auto ready = [&](int t, bool block) {
        if (!wait_ready) return true;
        const TileInfo ti = decode_tok(h, tb, nf, grp, t);
        return rows_ready(h, ti.d, ti.row0, ti.valid, block, wait);
      };
      auto produce = [&](int t, int n, auto &probe) {
        return produce_tile<KIND>(h, p, ps, decode_tok(h, tb, nf, grp, t), &tm_a0, &tm_a1, tm_b, n, probe);
      };
      produce_schedule(h, p, tq, stop_tile, wait_ready != 0, claim, ready, produce);
    }
  } else if (wid == 1) {
    if (lane == 0 && p.rank == 0) {
      // ---------------------------------------------------- MMA issuer (leader)
      MmaState ms;
      for (int n = 0;; ++n) {
        const int t = tq_pop(h, p, tq, n);
        if (t < 0 || !mma_tile<KIND>(h, p, ms, decode_tok(h, tb, nf, grp, t), n)) break;
      }
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int q = wid & 3;  // TMEM lane quarter this warp may access
    EpiState es;
    for (int n = 0;; ++n) {
      int t = 0;
      if (lane == 0) t = tq_pop(h, p, tq, n);  // lane 0 reads the entry and hands it back
      t = __shfl_sync(0xffffffffu, t, 0);
      // The gate/up epilogue's partner warps meet at named barriers, so they
      // act on an entry only together: they read the same entries, but a
      // failed wait (an abort in this CTA) can end one partner's read early.
      if (KIND == GATE_UP ? !xch_vote(q & 1, t >= 0) : t < 0) break;
      if (!epi_tile<KIND>(h, p, es, decode_tok(h, tb, nf, grp, t), n, q, lane)) break;
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no remote arrive or MMA of the pair is still in flight
  tc_fence_after();
  if (wid == 1) tmem_dealloc2(p.tmem_base, TMEM_COLS);
  if (threadIdx.x == 0) {
    // every pair has claimed past the end: the last CTA out resets the schedule
    __threadfence();
    if (atomicAdd(sched + 1, 1u) == gridDim.x - 1) {
      sched[0] = 0u;
      __threadfence();
      sched[1] = 0u;
    }
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// bf16 matrix [rows][cols] (row stride cols), box [box_rows][64], 128B swizzle
bool encode_2d(CUtensorMap *m, const void *ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)gemm2::BK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// per-slot bf16 window [W][cap][cols] with slot stride per_rank_size
bool encode_heap_3d(CUtensorMap *m, const sym_heap &h, uint64_t off, uint64_t cols,
                    uint32_t box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {cols, h.cap, (cuuint64_t)h.s.world};
  cuuint64_t strides[2] = {cols * 2, h.per_rank_size};
  cuuint32_t box[3] = {(cuuint32_t)gemm2::BK, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, reinterpret_cast<void *>(h.base + off), dims,
             strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_heap_boxes(gemm2::BMaps *m, const sym_heap &h, uint64_t off, uint64_t cols) {
  for (int i = 0; i < gemm2::NBOX; ++i)
    if (!encode_heap_3d(&m->m[i], h, off, cols, (uint32_t)(gemm2::BOX_MIN_ROWS << i))) return false;
  return true;
}

int max_resident_pairs(const void *kern, int threads, size_t smem, int num_sms) {
  // A pair needs two SMs of one GPC, so this can be fewer than SMs / 2.
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  struct Entry {
    const void *kern;
    size_t smem;
    int dev, pairs;
  };
  static Entry cache[16] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  for (const Entry &e : cache)
    if (e.kern == kern && e.smem == smem && e.dev == dev && e.pairs > 0) return e.pairs;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms & ~1);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  // no guess on failure: the fused launch relies on every pair being resident
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) return 0;
  for (Entry &e : cache)
    if (e.pairs == 0) {
      e = Entry{kern, smem, dev, n};
      break;
    }
  return n;
}

cudaError_t launch_expert_ffn(const sym_heap &h, const uint16_t *wg, const uint16_t *wu,
                              const uint16_t *wd, int num_sms, int wait_ready, int scale_rows,
                              cudaStream_t st) {
  using namespace gemm2;
  const int E = h.s.num_experts, H = h.s.hidden, I = h.s.inter;
  const size_t smem = gemm2_smem_bytes(E);
  CUtensorMap ta0, ta1;
  BMaps tb;
  // GEMM1: A = 64 gate + 64 up rows of expert e per CTA, B = recv_x token rows
  if (!encode_2d(&ta0, wg, (uint64_t)E * I, H, 64) || !encode_2d(&ta1, wu, (uint64_t)E * I, H, 64) ||
      !encode_heap_boxes(&tb, h, h.off_recv_x, H))
    return cudaErrorInvalidValue;
  {
    auto kern = expert_gemm2_kernel<GATE_UP>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    const int grid = 2 * max_resident_pairs((const void *)kern, GEMM_THREADS, smem, num_sms);
    if (grid <= 0) return cudaErrorInvalidConfiguration;
    kern<<<grid, GEMM_THREADS, smem, st>>>(h, ta0, ta1, tb, wait_ready, 0);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  // GEMM2: A = 128 down rows of expert e per CTA ([E*H][I]), B = h token rows
  if (!encode_2d(&ta0, wd, (uint64_t)E * H, I, 128) || !encode_heap_boxes(&tb, h, h.off_h, I))
    return cudaErrorInvalidValue;
  {
    auto kern = expert_gemm2_kernel<DOWN>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    const int grid = 2 * max_resident_pairs((const void *)kern, GEMM_THREADS, smem, num_sms);
    if (grid <= 0) return cudaErrorInvalidConfiguration;
    kern<<<grid, GEMM_THREADS, smem, st>>>(h, ta0, ta0, tb, 0, scale_rows);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace symmoe
