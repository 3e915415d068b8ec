// linear_a2a.cu -- GEMM + all-to-all fusion on the W slots of the symmetric
// heap, the second workload of the pages.
//
// MORI CCO blog, "Examples", "GEMM + all-to-all fusion": a GEMM whose epilogue
// writes its output tiles straight into the peers' windows (GEMM -> A2A), and
// a GEMM that consumes remote K-shards as they arrive by polling ready
// counters (A2A -> GEMM), each against a split pipeline.  Here one linear
// layer W [H][H] is shared by the slots:
//
//   GEMM -> A2A  slot s: Y_s = X_s W^T (its T rows), exchanged in W blocks of
//                B = T/W rows: slot j's y window row s*B + r <- Y_s[j*B + r].
//                fused: the epilogue stores every row at its destination;
//                split: the GEMM stores Y_s in slot s's recv_x window, then
//                a copy kernel exchanges the blocks.
//   A2A -> GEMM  slot s holds the K-shard s (H/W features) of all N tokens
//                (z [W][N][H/W]); slot j computes C_j = U_j W^T into its y
//                window, U_j = its tokens j*T.. with every feature.
//                fused (the pages' LSA form): the all-to-all is the GEMM's own
//                operand loads; a tile of slot j reads K shard s of its tokens
//                straight from slot s's buffer (a 3-D tensor map over z), so
//                nothing is copied.
//                fused over the copy engines (the pages' SDMA form): slot j's
//                recv_x window receives its shards as [W][T][H/W] (shard
//                major, one contiguous block each) by one cudaMemcpyAsync per
//                (slot, shard) from side streams, each followed by a stream
//                write of 1 into word s of slot j's ready window; the GEMM runs
//                at the same time and its producer waits (bounded) for a
//                shard's word before it loads that K range.
//                split: an SM copy kernel into the same shard-major blocks,
//                then the GEMM.
//
// The GEMM is the CTA-pair tile engine (gemm2sm.cuh) with the LINEAR kind:
// W rows on the MMA's M side (256 output features per pair tile), a slot's
// token rows on the N side (256 per tile, the experts' remainder rule), K = H.
#include <algorithm>
#include <mutex>

#include "gemm2sm.cuh"

namespace symmoe {

constexpr int LA_GEMM_THREADS = 192;
constexpr int LA_CTRL_BYTES = 256;
constexpr int LA_COPY_STREAMS = 2;  // side streams of the fused A2A -> GEMM copies

static size_t la_smem_bytes() {
  return 1024 + (size_t)gemm2::STAGES * gemm2::STAGE_BYTES + gemm2::XCH_BYTES + LA_CTRL_BYTES;
}

// tile t: slot major, then output feature tile, then token tile
__device__ inline gemm2::TileInfo decode_linear(int T, int nf, int t) {
  const int nt = gemm2::ntok_of(T);
  gemm2::TileInfo ti;
  ti.e = 0;
  ti.d = t / (nf * nt);
  const int r = t - ti.d * nf * nt;
  ti.f = r / nt;
  ti.n = r % nt;
  ti.row0 = ti.n * gemm2::BN;
  ti.valid = ti.n == nt - 1 ? T - ti.n * gemm2::BN : gemm2::BN;
  return ti;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(LA_GEMM_THREADS, 1)
    linear_gemm_kernel(const sym_heap h, const __grid_constant__ CUtensorMap tm_w,
                       const __grid_constant__ gemm2::BMaps tm_b, uint64_t out_off, int a2a_block,
                       int shard_kb, int shard_wait, int shard_direct) {
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
  p.logits = nullptr;
  p.out_off = out_off;
  p.a2a_block = a2a_block;
  p.shard_kb = shard_kb;
  p.shard_wait = shard_wait;
  p.shard_direct = shard_direct;

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
    tma_prefetch_desc(&tm_w);
    for (int i = 0; i < NBOX; ++i) tma_prefetch_desc(&tm_b.m[i]);
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
  const int T = h.s.tokens_per_slot;
  const int nf = nf_of(h, LINEAR);
  const int total_tiles = h.s.world * nf * ntok_of(T);

  if (wid == 0) {
    if (lane == 0) {
      ProdState ps;
      for (int i = 0, t; (t = pair_tile(i, pair_id, npairs)) < total_tiles; ++i)
        if (!produce_tile<LINEAR>(h, p, ps, decode_linear(T, nf, t), &tm_w, &tm_w, tm_b, t, []() {})) break;
    }
  } else if (wid == 1) {
    if (lane == 0 && p.rank == 0) {
      MmaState ms;
      for (int i = 0, t; (t = pair_tile(i, pair_id, npairs)) < total_tiles; ++i)
        if (!mma_tile<LINEAR>(h, p, ms, decode_linear(T, nf, t), t)) break;
    }
  } else {
    const int q = wid & 3;
    EpiState es;
    for (int i = 0, t; (t = pair_tile(i, pair_id, npairs)) < total_tiles; ++i)
      if (!epi_tile<LINEAR>(h, p, es, decode_linear(T, nf, t), t, q, lane)) break;
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no remote arrive or MMA of the pair is still in flight
  tc_fence_after();
  if (wid == 1) tmem_dealloc2(p.tmem_base, TMEM_COLS);
}

// split GEMM -> A2A: slot j's y row s*B + r <- slot s's staged row j*B + r
__global__ void __launch_bounds__(128) a2a_exchange_kernel(const sym_heap h) {
  const int W = h.s.world, T = h.s.tokens_per_slot, B = T / W, nv = h.s.hidden / 8;
  const int j = (int)blockIdx.y, dr = (int)blockIdx.x;  // destination slot, row
  const int s = dr / B, r = dr % B;
  const uint4 *src = win<const uint4>(h, s, h.off_recv_x) + (size_t)(j * B + r) * nv;
  uint4 *dst = win<uint4>(h, j, h.off_y) + (size_t)dr * nv;
  for (int c = threadIdx.x; c < nv; c += blockDim.x) dst[c] = __ldcs(src + c);
}

// split A2A -> GEMM: block s of slot j's recv_x window <- z[s][j*T .. (j+1)*T)
// (W*W contiguous blocks of T*H/W bf16; grid (chunks, W*W))
__global__ void __launch_bounds__(256) shard_gather_kernel(const sym_heap h, const uint4 *z) {
  const int W = h.s.world, T = h.s.tokens_per_slot, N = W * T;
  const size_t nb = (size_t)T * (h.s.hidden / W) / 8;  // 16-byte vectors per block
  const int j = (int)blockIdx.y / W, s = (int)blockIdx.y % W;
  const uint4 *src = z + ((size_t)s * N + (size_t)j * T) * (h.s.hidden / W) / 8;
  uint4 *dst = win<uint4>(h, j, h.off_recv_x) + (size_t)s * nb;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nb; i += (size_t)gridDim.x * blockDim.x)
    dst[i] = __ldcs(src + i);
}

// bf16 rows [W][T][cols] of a plain tensor as a 3-D map with the token-row boxes
static bool encode_slot_rows(gemm2::BMaps *m, const void *ptr, int W, int T, int cols) {
  sym_heap fake = {};
  fake.base = reinterpret_cast<uint64_t>(ptr);
  fake.cap = (uint64_t)T;
  fake.per_rank_size = (uint64_t)T * cols * 2;
  fake.s.world = W;
  return encode_heap_boxes(m, fake, 0, (uint64_t)cols);
}

static cudaError_t launch_linear(const sym_heap &h, const CUtensorMap &tw, const gemm2::BMaps &tb, uint64_t out_off,
                                 int a2a_block, int shard_kb, int shard_wait, int shard_direct, int num_sms,
                                 cudaStream_t st) {
  const size_t smem = la_smem_bytes();
  cudaError_t err =
      cudaFuncSetAttribute(linear_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const int grid = 2 * max_resident_pairs((const void *)linear_gemm_kernel, LA_GEMM_THREADS, smem, num_sms);
  if (grid <= 0) return cudaErrorInvalidConfiguration;
  linear_gemm_kernel<<<grid, LA_GEMM_THREADS, smem, st>>>(h, tw, tb, out_off, a2a_block, shard_kb, shard_wait,
                                                          shard_direct);
  return cudaGetLastError();
}

cudaError_t launch_gemm_a2a(const sym_heap &h, const uint16_t *x, const uint16_t *w, int fused, int num_sms,
                            cudaStream_t st) {
  const int W = h.s.world, T = h.s.tokens_per_slot, H = h.s.hidden;
  CUtensorMap tw;
  gemm2::BMaps tb;
  if (!encode_2d(&tw, w, (uint64_t)H, (uint64_t)H, 128) || !encode_slot_rows(&tb, x, W, T, H))
    return cudaErrorInvalidValue;
  if (fused) return launch_linear(h, tw, tb, h.off_y, T / W, 0, 0, 0, num_sms, st);
  cudaError_t err = launch_linear(h, tw, tb, h.off_recv_x, 0, 0, 0, 0, num_sms, st);
  if (err != cudaSuccess) return err;
  a2a_exchange_kernel<<<dim3(T, W), 128, 0, st>>>(h);
  return cudaGetLastError();
}

// fused A2A -> GEMM: one shard counter per (slot, shard)
int a2a_gemm_counters(const sym_heap &h) { return h.s.world; }

__global__ void __launch_bounds__(32) zero_counters_kernel(const sym_heap h, int n) {
  uint32_t *c = win<uint32_t>(h, (int)blockIdx.x, h.off_ready);
  for (int i = threadIdx.x; i < n; i += blockDim.x) c[i] = 0u;
}

// The side streams and events of the fused A2A -> GEMM, one set per device,
// created on first use and kept for the process; and cuStreamWriteValue32
// from the driver.
typedef CUresult (*WriteValue32Fn)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);
struct CopySide {
  cudaStream_t stream[LA_COPY_STREAMS];
  cudaEvent_t start, done[LA_COPY_STREAMS];
  bool ok = false;
};
static std::mutex g_side_mu;
static CopySide g_side[64];
static WriteValue32Fn g_write32 = nullptr;

static cudaError_t copy_side(CopySide **out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_side_mu);
  if (!g_write32) {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuStreamWriteValue32", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return cudaErrorNotSupported;
    g_write32 = reinterpret_cast<WriteValue32Fn>(fn);
  }
  CopySide &c = g_side[dev];
  if (!c.ok) {
    for (int i = 0; i < LA_COPY_STREAMS; ++i) {
      if ((err = cudaStreamCreateWithFlags(&c.stream[i], cudaStreamNonBlocking)) != cudaSuccess) return err;
      if ((err = cudaEventCreateWithFlags(&c.done[i], cudaEventDisableTiming)) != cudaSuccess) return err;
    }
    if ((err = cudaEventCreateWithFlags(&c.start, cudaEventDisableTiming)) != cudaSuccess) return err;
    c.ok = true;
  }
  *out = &c;
  return cudaSuccess;
}

// B maps of the shard-major blocks: rows s*T + r of a slot's window, H/W columns
static bool encode_shard_rows(gemm2::BMaps *m, const sym_heap &h) {
  sym_heap fake = {};
  fake.base = h.base + h.off_recv_x;
  fake.cap = (uint64_t)h.s.world * h.s.tokens_per_slot;
  fake.per_rank_size = h.per_rank_size;
  fake.s.world = h.s.world;
  return encode_heap_boxes(m, fake, 0, (uint64_t)(h.s.hidden / h.s.world));
}

// mode: 0 split, 1 fused (the GEMM reads every shard in its owner's buffer),
// 2 fused over the copy engines
cudaError_t launch_a2a_gemm(const sym_heap &h, const uint16_t *z, const uint16_t *w, int mode, int num_sms,
                            cudaStream_t st) {
  const int W = h.s.world, T = h.s.tokens_per_slot, H = h.s.hidden, hs = H / W;
  CUtensorMap tw;
  gemm2::BMaps tb;
  if (!encode_2d(&tw, w, (uint64_t)H, (uint64_t)H, 128)) return cudaErrorInvalidValue;
  const int shard_kb = hs / gemm2::BK;
  const size_t block = (size_t)T * hs * 2;  // bytes of one (slot, shard) block
  if (mode == 1) {
    // z as [shard][N][H/W]: the owners' buffers
    if (!encode_slot_rows(&tb, z, W, W * T, hs)) return cudaErrorInvalidValue;
    return launch_linear(h, tw, tb, h.off_y, 0, shard_kb, 0, 1, num_sms, st);
  }
  if (!encode_shard_rows(&tb, h)) return cudaErrorInvalidValue;
  if (mode == 0) {
    const int chunks = (int)std::min<size_t>((block / 16 + 255) / 256, (size_t)num_sms);
    shard_gather_kernel<<<dim3(chunks, W * W), 256, 0, st>>>(h, reinterpret_cast<const uint4 *>(z));
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    return launch_linear(h, tw, tb, h.off_y, 0, shard_kb, 0, 0, num_sms, st);  // shards in place: no waits
  }
  CopySide *c = nullptr;
  cudaError_t err = copy_side(&c);
  if (err != cudaSuccess) return err;
  zero_counters_kernel<<<W, 32, 0, st>>>(h, a2a_gemm_counters(h));
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  if ((err = cudaEventRecord(c->start, st)) != cudaSuccess) return err;
  for (int i = 0; i < LA_COPY_STREAMS; ++i)
    if ((err = cudaStreamWaitEvent(c->stream[i], c->start, 0)) != cudaSuccess) return err;
  // slot major, shard minor: the GEMM's tiles go slot major and read K shard by shard
  for (int j = 0; j < W; ++j) {
    cudaStream_t cs = c->stream[j % LA_COPY_STREAMS];
    for (int s = 0; s < W; ++s) {
      const uint8_t *src = reinterpret_cast<const uint8_t *>(z) + ((size_t)s * W * T + (size_t)j * T) * hs * 2;
      uint8_t *dst = reinterpret_cast<uint8_t *>(h.base + (uint64_t)j * h.per_rank_size + h.off_recv_x) + s * block;
      if ((err = cudaMemcpyAsync(dst, src, block, cudaMemcpyDeviceToDevice, cs)) != cudaSuccess) return err;
      const CUdeviceptr ctr = (CUdeviceptr)(h.base + (uint64_t)j * h.per_rank_size + h.off_ready + 4u * s);
      if (g_write32(reinterpret_cast<CUstream>(cs), ctr, 1u, 0) != CUDA_SUCCESS) return cudaErrorUnknown;
    }
  }
  if ((err = launch_linear(h, tw, tb, h.off_y, 0, shard_kb, 1, 0, num_sms, st)) != cudaSuccess) return err;
  // the call completes on the caller's stream
  for (int i = 0; i < LA_COPY_STREAMS; ++i) {
    if ((err = cudaEventRecord(c->done[i], c->stream[i])) != cudaSuccess) return err;
    if ((err = cudaStreamWaitEvent(st, c->done[i], 0)) != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace symmoe
