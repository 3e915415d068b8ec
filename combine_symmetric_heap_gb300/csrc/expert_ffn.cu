// expert_ffn.cu -- grouped SwiGLU expert FFN on the 5th-generation tensor
// cores (tcgen05.mma, accumulators in TMEM, operands staged by TMA).
//
// MORI CCO blog, "Zero-copy MoE dispatch -> expert -> combine": the expert
// GEMM reads the dispatched rows in place from the receive window and writes
// its output straight into the combine staging window.  Per expert e with
// cnt_e received rows A (a contiguous block of slot e/(E/W)'s recv_x window):
//   GEMM1  h = bf16( silu(A Wg_e^T) * (A Wu_e^T) )    -> h window
//   GEMM2  y = bf16( h Wd_e^T )                         -> y window (out_tok)
//
// Tiling ("swap AB"): the tensor-core M side (128) runs over weight rows
// (output features) and the N side over tokens, so an expert's ragged row
// count only shortens the N of its last tile's MMAs (rounded up to 16).
// GEMM1 issues two MMAs per K step that share the token tile: gate rows and
// up rows into two TMEM accumulators, so silu(gate) * up is a per-thread
// epilogue.  (Putting 64 gate + 64 up rows on one M=128 MMA with N=256 and
// swapping halves between warps measured 10-25% slower on GB300.)
//
// One persistent CTA per SM, warp-specialised:
//   warp 0   TMA producer (one thread): waits for the dispatch ready counters
//            of the token rows (bounded), then streams K blocks of 64 through
//            a STAGES-deep shared-memory ring (128-byte swizzle);
//   warp 1   allocates TMEM and issues tcgen05.mma (one thread); accumulators
//            are double-buffered in TMEM so the epilogue of tile i overlaps
//            the main loop of tile i+1;
//   warps 2-5 epilogue: tcgen05.ld, SwiGLU / bf16 rounding, stores.
// Tiles are enumerated expert-major, then feature tile, then token tile, so
// CTAs running at the same time share a weight tile through L2.  Row counts
// come from the dispatch signal area on the device (no host sync).
#include "symmoe_dev.cuh"

namespace symmoe {

constexpr int BM = 128;  // weight rows per tile (tcgen05 M)
constexpr int BK = 64;   // K per stage: one 128-byte swizzle row of bf16
constexpr int UK = 16;   // K per tcgen05.mma kind::f16
constexpr int GEMM_THREADS = 192;

template <int NUM_A, int BN, int STAGES>
struct GemmCfg {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = NUM_A * A_BYTES + B_BYTES;
  static constexpr int ACC_COLS = NUM_A * BN;  // fp32 TMEM columns of one tile
  static constexpr int TMEM_COLS = 2 * ACC_COLS;
  static_assert(TMEM_COLS <= 512, "two accumulators must fit in TMEM");
  static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "token tile");
  static constexpr int CTRL_BYTES = 256;  // barriers and flags
  static size_t smem_bytes(int num_experts) {
    return 1024 + (size_t)STAGES * STAGE_BYTES + CTRL_BYTES + (size_t)(num_experts + 1) * 4;
  }
};

struct GemmArgs {
  int nk;            // K blocks of 64
  int nf;            // feature tiles of 128
  int a_rows;        // weight rows per expert (I for GEMM1, H for GEMM2)
  uint64_t off_out;  // output window (h or y)
  int out_ld;        // output row length in elements
  int wait_ready;    // wait for the dispatch ready counters before loading B
};

struct TileInfo {
  int e, f, n, d, row0, valid;
};

__device__ __forceinline__ TileInfo decode_tile(const sym_heap &h, const int *prefix,
                                                const int *cnt_s, const int *roff_s, int t,
                                                int nf, int BN) {
  const int E = h.s.num_experts;
  int lo = 0, hi = E;  // largest e with prefix[e] <= t
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= t) lo = mid; else hi = mid;
  }
  TileInfo ti;
  ti.e = lo;
  const int c = cnt_s[lo];
  const int ntok = (c + BN - 1) / BN;
  const int local = t - prefix[lo];
  ti.f = local / ntok;
  ti.n = local % ntok;
  ti.d = lo / (E / h.s.world);
  ti.row0 = roff_s[lo] + ti.n * BN;
  ti.valid = min(BN, c - ti.n * BN);
  (void)nf;
  return ti;
}

// Bounded mbarrier wait that also gives up once the producer has stopped
// before tile t (stop_tile <= t) or any role has aborted.
__device__ __forceinline__ bool wait_or_stop(uint64_t *bar, uint32_t parity, int t,
                                             const volatile int *stop_tile,
                                             volatile int *abort_flag, uint32_t timeout_us,
                                             const sym_heap &h) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  const uint64_t limit = (uint64_t)timeout_us * 1000ull;
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(a, parity)) return true;
    if (*abort_flag || *stop_tile <= t) return false;
    if ((it & 15u) == 15u && globaltimer_ns() - t0 > limit) {
      *abort_flag = 1;
      raise_status(h, SYM_STATUS_TIMEOUT);
      return false;
    }
  }
}

template <int NUM_A, int BN, int STAGES, bool SWIGLU>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    expert_gemm_kernel(const sym_heap h, const __grid_constant__ CUtensorMap tm_a0,
                       const __grid_constant__ CUtensorMap tm_a1,
                       const __grid_constant__ CUtensorMap tm_b, const GemmArgs args) {
  using C = GemmCfg<NUM_A, BN, STAGES>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *ring = smem;
  uint8_t *ctrl = smem + (size_t)STAGES * C::STAGE_BYTES;
  uint64_t *full = reinterpret_cast<uint64_t *>(ctrl);
  uint64_t *empty = full + STAGES;
  uint64_t *acc_full = empty + STAGES;
  uint64_t *acc_empty = acc_full + 2;
  uint32_t *tmem_base_s = reinterpret_cast<uint32_t *>(acc_empty + 2);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_base_s + 1);
  volatile int *stop_tile = abort_flag + 1;
  int *prefix = reinterpret_cast<int *>(ctrl + C::CTRL_BYTES);  // [E+1]
  __shared__ int cnt_s[1024];
  __shared__ int roff_s[1024];

  const int E = h.s.num_experts;
  const int E_loc = E / h.s.world;
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
    if (NUM_A == 2) tma_prefetch_desc(&tm_a1);
    tma_prefetch_desc(&tm_b);
  }
  if (wid == 1) {
    tmem_alloc(tmem_base_s, C::TMEM_COLS);
    tmem_relinquish();
  }
  // tile table: tiles of expert e = ceil(cnt_e / BN) * nf
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int d = e / E_loc, l = e % E_loc;
    cnt_s[e] = win<const int32_t>(h, d, h.off_cnt)[l];
    roff_s[e] = win<const int32_t>(h, d, h.off_recv_off)[l];
  }
  __syncthreads();
  if (wid == 0) {
    int carry = 0;
    if (lane == 0) prefix[0] = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int v = e < E ? ((cnt_s[e] + BN - 1) / BN) * args.nf : 0;
      int incl = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      if (e < E) prefix[e + 1] = carry + incl;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_base_s;
  const int total_tiles = prefix[E];
  const uint32_t tmo = h.wait_timeout_us;

  if (wid == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      int stage = 0;
      uint32_t phase = 0;
      for (int t = blockIdx.x; t < total_tiles && !*abort_flag; t += gridDim.x) {
        const TileInfo ti = decode_tile(h, prefix, cnt_s, roff_s, t, args.nf, BN);
        if (args.wait_ready) {
          const int total = *win<const int32_t>(h, ti.d, h.off_total);
          const uint32_t *ready = win<const uint32_t>(h, ti.d, h.off_ready);
          bool ok = true;
          for (int b = ti.row0 / SYM_ROWS_PER_FLAG;
               ok && b <= (ti.row0 + ti.valid - 1) / SYM_ROWS_PER_FLAG; ++b) {
            const uint32_t target = (uint32_t)min(SYM_ROWS_PER_FLAG, total - b * SYM_ROWS_PER_FLAG);
            ok = wait_counter_geq(ready + b, target, tmo, abort_flag);
          }
          if (!ok) {
            raise_status(h, SYM_STATUS_TIMEOUT);
            *stop_tile = t;  // tiles >= t are not loaded; earlier ones finish
            break;
          }
          fence_proxy_async();
        }
        const int arow = ti.e * args.a_rows + ti.f * BM;
        for (int kb = 0; kb < args.nk; ++kb) {
          if (!wait_or_stop(&empty[stage], phase ^ 1u, -1, stop_tile, abort_flag, tmo, h))
            break;
          uint8_t *sbase = ring + (size_t)stage * C::STAGE_BYTES;
          mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
          tma_load_2d(sbase, &tm_a0, &full[stage], kb * BK, arow);
          if (NUM_A == 2) tma_load_2d(sbase + C::A_BYTES, &tm_a1, &full[stage], kb * BK, arow);
          tma_load_3d(sbase + NUM_A * C::A_BYTES, &tm_b, &full[stage], kb * BK, ti.row0, ti.d);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
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
        // a ragged last token tile runs a narrower MMA (N rounded up to 16)
        const TileInfo ti = decode_tile(h, prefix, cnt_s, roff_s, t, args.nf, BN);
        const uint32_t idesc = idesc_bf16_f32(BM, min(BN, (ti.valid + 15) & ~15));
        if (!wait_or_stop(&acc_empty[abuf], aphase ^ 1u, t, stop_tile, abort_flag, tmo, h)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(abuf * C::ACC_COLS);
        bool stopped = false;
        for (int kb = 0; kb < args.nk; ++kb) {
          if (!wait_or_stop(&full[stage], phase, t, stop_tile, abort_flag, tmo, h)) {
            stopped = true;
            break;
          }
          tc_fence_after();
          uint8_t *sbase = ring + (size_t)stage * C::STAGE_BYTES;
          const uint64_t da0 = smem_desc_sw128(sbase);
          const uint64_t da1 = smem_desc_sw128(sbase + C::A_BYTES);
          const uint64_t db = smem_desc_sw128(sbase + NUM_A * C::A_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / UK; ++kk) {
            // +32 bytes per K step inside the swizzle row (descriptor units of 16 B)
            const uint64_t adv = (uint64_t)(kk * UK * 2 / 16);
            const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
            tc_mma_bf16(d_tmem, da0 + adv, db + adv, idesc, acc);
            if (NUM_A == 2) tc_mma_bf16(d_tmem + BN, da1 + adv, db + adv, idesc, acc);
          }
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
    const int r = q * 32 + lane;
    int abuf = 0;
    uint32_t aphase = 0;
    for (int t = blockIdx.x; t < total_tiles; t += gridDim.x) {
      const TileInfo ti = decode_tile(h, prefix, cnt_s, roff_s, t, args.nf, BN);
      // every lane waits (the tcgen05.ld below is warp-collective)
      if (!wait_or_stop(&acc_full[abuf], aphase, t, stop_tile, abort_flag, tmo, h)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(abuf * C::ACC_COLS);
      const int feature = ti.f * BM + r;
      uint16_t *out = win<uint16_t>(h, ti.d, args.off_out) + (size_t)ti.row0 * args.out_ld + feature;
      for (int c0 = 0; c0 < BN && c0 < ti.valid; c0 += 32) {
        uint32_t a[32];
        tmem_ld32(tbase + c0, a);
        if constexpr (SWIGLU) {
          uint32_t b[32];
          tmem_ld32(tbase + BN + c0, b);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            if (c0 + c < ti.valid) {
              const float gt = __uint_as_float(a[c]);
              const float up = __uint_as_float(b[c]);
              const float act = gt / (1.0f + __expf(-gt)) * up;
              out[(size_t)(c0 + c) * args.out_ld] = to_bf16(act);
            }
          }
        } else {
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (c0 + c < ti.valid)
              out[(size_t)(c0 + c) * args.out_ld] = to_bf16(__uint_as_float(a[c]));
        }
      }
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
  if (wid == 1) tmem_dealloc(tmem_base, C::TMEM_COLS);
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
static bool encode_2d(CUtensorMap *m, const void *ptr, uint64_t rows, uint64_t cols,
                      uint32_t box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// per-slot bf16 window [W][cap][cols] with slot stride per_rank_size
static bool encode_heap_3d(CUtensorMap *m, const sym_heap &h, uint64_t off, uint64_t cols,
                           uint32_t box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {cols, h.cap, (cuuint64_t)h.s.world};
  cuuint64_t strides[2] = {cols * 2, h.per_rank_size};
  cuuint32_t box[3] = {(cuuint32_t)BK, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, reinterpret_cast<void *>(h.base + off), dims,
             strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int G1_BN = 128, G1_STAGES = 4;
constexpr int G2_BN = 256, G2_STAGES = 4;

cudaError_t launch_expert_ffn(const sym_heap &h, const uint16_t *wg, const uint16_t *wu,
                              const uint16_t *wd, int num_sms, int wait_ready, cudaStream_t st) {
  const int E = h.s.num_experts, H = h.s.hidden, I = h.s.inter;
  CUtensorMap ta0, ta1, tb;
  // GEMM1: A = gate / up rows of expert e ([E*I][H]), B = recv_x token rows
  if (!encode_2d(&ta0, wg, (uint64_t)E * I, H, BM) || !encode_2d(&ta1, wu, (uint64_t)E * I, H, BM) ||
      !encode_heap_3d(&tb, h, h.off_recv_x, H, G1_BN))
    return cudaErrorInvalidValue;
  {
    using C = GemmCfg<2, G1_BN, G1_STAGES>;
    auto kern = expert_gemm_kernel<2, G1_BN, G1_STAGES, true>;
    const size_t smem = C::smem_bytes(E);
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    GemmArgs a{H / BK, I / BM, I, h.off_h, I, wait_ready};
    kern<<<num_sms, GEMM_THREADS, smem, st>>>(h, ta0, ta1, tb, a);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  // GEMM2: A = down rows of expert e ([E*H][I]), B = h token rows
  if (!encode_2d(&ta0, wd, (uint64_t)E * H, I, BM) || !encode_heap_3d(&tb, h, h.off_h, I, G2_BN))
    return cudaErrorInvalidValue;
  {
    using C = GemmCfg<1, G2_BN, G2_STAGES>;
    auto kern = expert_gemm_kernel<1, G2_BN, G2_STAGES, false>;
    const size_t smem = C::smem_bytes(E);
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    GemmArgs a{I / BK, H / BM, H, h.off_y, H, 0};
    kern<<<num_sms, GEMM_THREADS, smem, st>>>(h, ta0, ta0, tb, a);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace symmoe
