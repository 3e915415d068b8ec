// expert_ffn.cu -- grouped SwiGLU expert FFN on the 5th-generation tensor
// cores (tcgen05.mma, accumulators in TMEM, operands staged by TMA).
//
// MORI CCO blog, "Zero-copy MoE dispatch -> expert -> combine": the expert
// GEMM reads the dispatched rows in place from the receive window and writes
// its output straight into the combine staging window.  Per expert e with
// cnt_e received rows A (a contiguous block of slot e/(E/W)'s recv_x window):
//   GEMM1  h = bf16( silu(A Wg_e^T) * (A Wu_e^T) )    -> h window
//   GEMM2  y = bf16( h Wd_e^T )                         -> y window (out_tok)
// The tile pieces (loads, MMAs, epilogues) are in gemm_core.cuh.
//
// One persistent CTA per SM per GEMM, warp-specialised:
//   warp 0   TMA producer (one thread): waits for the dispatch ready counters
//            of the token rows (bounded), then streams K blocks of 64 through
//            a 4-deep shared-memory ring;
//   warp 1   allocates TMEM and issues tcgen05.mma (one thread); the two
//            accumulator buffers let the epilogue of tile i overlap the main
//            loop of tile i+1;
//   warps 2-5 epilogue: tcgen05.ld, SwiGLU / bf16 rounding, stores.
// Tiles are taken round-robin (tile = CTA + i * grid); row counts come from
// the dispatch signal area on the device (no host sync).
// (Putting 64 gate + 64 up rows on one M=128 MMA with N=256 and swapping
// halves between warps measured 10-25% slower on GB300 than the two
// accumulators used here.)
#include "gemm_core.cuh"

namespace symmoe {

using gemm::TileInfo;
constexpr int GEMM_THREADS = 192;
constexpr int CTRL_BYTES = 256;

static size_t gemm_smem_bytes(int num_experts) {
  return 1024 + (size_t)gemm::STAGES * gemm::STAGE_BYTES + CTRL_BYTES +
         gemm::tables_bytes(num_experts);
}

template <int KIND>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    expert_gemm_kernel(const sym_heap h, const __grid_constant__ CUtensorMap tm_a0,
                       const __grid_constant__ CUtensorMap tm_a1,
                       const __grid_constant__ CUtensorMap tm_b, int wait_ready) {
  using namespace gemm;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *ring = smem;
  uint8_t *ctrl = smem + (size_t)STAGES * STAGE_BYTES;
  uint64_t *full = reinterpret_cast<uint64_t *>(ctrl);
  uint64_t *empty = full + STAGES;
  uint64_t *acc_full = empty + STAGES;
  uint64_t *acc_empty = acc_full + 2;
  uint32_t *tmem_base_s = reinterpret_cast<uint32_t *>(acc_empty + 2);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_base_s + 1);
  volatile int *stop_tile = abort_flag + 1;
  const int E = h.s.num_experts;
  int *tab = reinterpret_cast<int *>(ctrl + CTRL_BYTES);
  const Tables tb{tab, tab + E, tab + 2 * E, tab + 3 * E + 1};
  const Maps maps{&tm_a0, &tm_a1, &tm_b};
  const int wid = warp_id(), lane = lane_id();

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    *abort_flag = 0;
    *stop_tile = 0x7fffffff;
    fence_mbar_init();
    tma_prefetch_desc(&tm_a0);
    if (KIND == GATE_UP) tma_prefetch_desc(&tm_a1);
    tma_prefetch_desc(&tm_b);
  }
  if (wid == 1) {
    tmem_alloc(tmem_base_s, TMEM_COLS);
    tmem_relinquish();
  }
  build_tables(h, tb);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_base_s;
  const int total_tiles = tb.prefix(KIND)[E];
  const int nk = nk_of(h, KIND);
  const uint32_t tmo = h.wait_timeout_us;

  if (wid == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      // The readiness of tile i+1's rows is probed (without blocking) half way
      // through tile i's K loop, so the acquire round trip hides behind the
      // stages already in flight; only a tile whose rows are not ready yet
      // waits at the tile boundary.
      int stage = 0;
      uint32_t phase = 0;
      int t = blockIdx.x;
      bool ready_ok = true;
      if (wait_ready && t < total_tiles) {
        ready_ok = wait_rows_dispatched(h, decode(h, tb, KIND, t), tmo, abort_flag);
        if (!ready_ok) {
          raise_status(h, SYM_STATUS_TIMEOUT);
          *stop_tile = t;
        }
      }
      while (ready_ok && t < total_tiles && !*abort_flag) {
        if (wait_ready) fence_proxy_async();
        const TileInfo ti = decode(h, tb, KIND, t);
        const int t_next = t + gridDim.x;
        bool next_ok = !wait_ready || t_next >= total_tiles;
        for (int kb = 0; kb < nk; ++kb) {
          if (!next_ok && kb == nk / 2) next_ok = rows_dispatched_now(h, decode(h, tb, KIND, t_next));
          if (!wait_or_stop(&empty[stage], phase ^ 1u, -1, stop_tile, abort_flag, tmo, h)) break;
          issue_loads(h, ti, maps, kb, ring + (size_t)stage * STAGE_BYTES, &full[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!next_ok && !wait_rows_dispatched(h, decode(h, tb, KIND, t_next), tmo, abort_flag)) {
          raise_status(h, SYM_STATUS_TIMEOUT);
          *stop_tile = t_next;  // tiles >= t_next are not loaded; earlier ones finish
          break;
        }
        t = t_next;
      }
    }
  } else if (wid == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      int abuf = 0;
      uint32_t aphase = 0;
      for (int t = blockIdx.x; t < total_tiles; t += gridDim.x) {
        const TileInfo ti = decode(h, tb, KIND, t);
        if (!wait_or_stop(&acc_empty[abuf], aphase ^ 1u, t, stop_tile, abort_flag, tmo, h)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(abuf * ACC_COLS);
        bool stopped = false;
        for (int kb = 0; kb < nk; ++kb) {
          if (!wait_or_stop(&full[stage], phase, t, stop_tile, abort_flag, tmo, h)) {
            stopped = true;
            break;
          }
          tc_fence_after();
          issue_mmas(ti, ring + (size_t)stage * STAGE_BYTES, d_tmem, kb == 0);
          tc_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (stopped) break;
        tc_commit(&acc_full[abuf]);
        if (++abuf == 2) {
          abuf = 0;
          aphase ^= 1u;
        }
      }
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int q = wid & 3;  // TMEM lane quarter this warp may access
    int abuf = 0;
    uint32_t aphase = 0;
    for (int t = blockIdx.x; t < total_tiles; t += gridDim.x) {
      const TileInfo ti = decode(h, tb, KIND, t);
      // every lane waits (tcgen05.ld is warp-collective)
      if (!wait_or_stop(&acc_full[abuf], aphase, t, stop_tile, abort_flag, tmo, h)) break;
      tc_fence_after();
      epilogue(h, ti, tmem_base, (uint32_t)(abuf * ACC_COLS), q, lane);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[abuf]);
      if (++abuf == 2) {
        abuf = 0;
        aphase ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (wid == 1) tmem_dealloc(tmem_base, TMEM_COLS);
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
bool encode_2d(CUtensorMap *m, const void *ptr, uint64_t rows, uint64_t cols,
                      uint32_t box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)gemm::BK, box_rows};
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
  cuuint32_t box[3] = {(cuuint32_t)gemm::BK, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, reinterpret_cast<void *>(h.base + off), dims,
             strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_expert_ffn(const sym_heap &h, const uint16_t *wg, const uint16_t *wu,
                              const uint16_t *wd, int num_sms, int wait_ready, cudaStream_t st) {
  using namespace gemm;
  const int E = h.s.num_experts, H = h.s.hidden, I = h.s.inter;
  const size_t smem = gemm_smem_bytes(E);
  CUtensorMap ta0, ta1, tb;
  // GEMM1: A = gate / up rows of expert e ([E*I][H]), B = recv_x token rows
  if (!encode_2d(&ta0, wg, (uint64_t)E * I, H, BM) || !encode_2d(&ta1, wu, (uint64_t)E * I, H, BM) ||
      !encode_heap_3d(&tb, h, h.off_recv_x, H, K<GATE_UP>::BN))
    return cudaErrorInvalidValue;
  {
    auto kern = expert_gemm_kernel<GATE_UP>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    kern<<<num_sms, GEMM_THREADS, smem, st>>>(h, ta0, ta1, tb, wait_ready);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  // GEMM2: A = down rows of expert e ([E*H][I]), B = h token rows
  if (!encode_2d(&ta0, wd, (uint64_t)E * H, I, BM) ||
      !encode_heap_3d(&tb, h, h.off_h, I, K<DOWN>::BN))
    return cudaErrorInvalidValue;
  {
    auto kern = expert_gemm_kernel<DOWN>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    kern<<<num_sms, GEMM_THREADS, smem, st>>>(h, ta0, ta0, tb, 0);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace symmoe
