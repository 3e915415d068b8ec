// gemm2sm.cuh -- the stand-alone expert GEMMs on CTA pairs (tcgen05
// cta_group::2): one M=256 MMA spans the tensor cores of two SMs of a cluster.
//
// Each CTA of the pair stages only its half of both operands: 128 of the 256
// weight rows (A) and N/2 of the N token rows (B); the MMA, issued by the
// pair's first CTA (the leader), reads the four halves from both shared
// memories and leaves output rows 0-127 in the leader's TMEM and rows 128-255
// in the peer's.  Per SM that is 32 KB of operands per 128 x 256 x 64
// multiply-adds instead of 48 KB, so six stages fit and the ring keeps the
// tensor pipe fed.
//
//   GATE_UP: the pair computes 128 features x N tokens.  CTA r's A rows are
//            the gate rows and the up rows of features f*128 + r*64 .. +63, so
//            its TMEM holds gate (lanes 0-63) and up (lanes 64-127) of the
//            same 64 features; the epilogue pairs the warp reading the gate
//            lanes with the warp reading the up lanes and swaps half of each
//            32-column chunk through shared memory: h = silu(gate) * up.
//   DOWN:    the pair computes 256 features x N tokens: CTA r holds the down
//            rows f*256 + r*128 .. +127; y is written straight into the
//            combine-in window.
//
// Completion: the copies of both CTAs count their bytes on the leader's full
// barrier (the .cta_group::2 form of the TMA copy), whose expected byte count
// only the leader posts, for both halves; so the leader's MMA starts when both
// halves are in.  The leader's commits arrive on the empty and accumulator
// barriers of both CTAs (multicast), and both CTAs' epilogue warps arrive on
// the leader's accumulator-empty barrier.  Each CTA reaches the final cluster
// barrier only after its own loops end, so the leader's barriers outlive
// every copy the peer issued.
#pragma once

#include "symmoe_dev.cuh"

namespace symmoe {
namespace gemm2 {

constexpr int BK = 64;
constexpr int UK = 16;
constexpr int BN = 256;         // tokens per pair tile (tcgen05 N)
constexpr int STAGES = 6;
constexpr int A_BYTES = 128 * BK * 2;          // 16 KB: this CTA's weight rows
constexpr int B_ROWS = BN / 2;                 // this CTA's token rows at most (largest box)
constexpr int B_BYTES = B_ROWS * BK * 2;       // 16 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES; // 32 KB
constexpr int ACC_COLS = BN;
constexpr int TMEM_COLS = 512;
constexpr int XCH_BYTES = 2 * 2 * 2 * 16 * 32 * 4;  // pairs x buffers x directions x 16 cols x 32 lanes

// Token-row boxes: a tile loads only the token rows its MMA reads (N/2 per
// CTA, a multiple of 8), rounded up to the next of 8, 16, ..., 128 rows, so a
// ragged tile of a few rows does not stream 128 rows of B per K block.
constexpr int NBOX = 5;
constexpr int BOX_MIN_ROWS = 8;
struct BMaps {
  CUtensorMap m[NBOX];  // m[i]: box of BOX_MIN_ROWS << i rows
};
__host__ __device__ inline int box_index(int half_rows) {
  int i = 0;
  while (i < NBOX - 1 && (BOX_MIN_ROWS << i) < half_rows) ++i;
  return i;
}
// bytes both CTAs' copies of one K block deliver to the leader's full barrier
__host__ __device__ inline uint32_t stage_tx(int box) {
  return 2u * (uint32_t)(A_BYTES + (BOX_MIN_ROWS << box) * BK * 2);
}

enum Kind : int { GATE_UP = 0, DOWN = 1 };

// features per pair tile and K blocks per kind
__host__ __device__ inline int feat_of(int kind) { return kind == GATE_UP ? 128 : 256; }
__host__ __device__ inline int nf_of(const sym_heap &h, int kind) {
  const int n = kind == GATE_UP ? h.s.inter : h.s.hidden;
  return (n + feat_of(kind) - 1) / feat_of(kind);
}
__host__ __device__ inline int nk_of(const sym_heap &h, int kind) {
  return (kind == GATE_UP ? h.s.hidden : h.s.inter) / BK;
}

struct TileInfo {
  int e, f, n, d, row0, valid;
};

struct Tables {
  int *cnt, *roff, *prefix;
};
__host__ __device__ constexpr size_t tables_bytes(int num_experts) {
  return (size_t)(3 * num_experts + 1) * sizeof(int);
}

__device__ inline void build_tables(const sym_heap &h, const Tables &tb, int kind) {
  const int E = h.s.num_experts, E_loc = E / h.s.world;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int d = e / E_loc, l = e % E_loc;
    tb.cnt[e] = win<const int32_t>(h, d, h.off_cnt)[l];
    tb.roff[e] = win<const int32_t>(h, d, h.off_recv_off)[l];
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x, nf = nf_of(h, kind);
    int carry = 0;
    if (lane == 0) tb.prefix[0] = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int v = e < E ? ((tb.cnt[e] + BN - 1) / BN) * nf : 0;
      int incl = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      if (e < E) tb.prefix[e + 1] = carry + incl;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
}

__device__ inline TileInfo decode(const sym_heap &h, const Tables &tb, int t) {
  const int E = h.s.num_experts;
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tb.prefix[mid] <= t) lo = mid; else hi = mid;
  }
  TileInfo ti;
  ti.e = lo;
  const int c = tb.cnt[lo];
  const int ntok = (c + BN - 1) / BN;
  const int local = t - tb.prefix[lo];
  ti.f = local / ntok;
  ti.n = local % ntok;
  ti.d = lo / (E / h.s.world);
  ti.row0 = tb.roff[lo] + ti.n * BN;
  ti.valid = min(BN, c - ti.n * BN);
  return ti;
}

__device__ __forceinline__ int n_mma(int valid) { return min(BN, (valid + 15) & ~15); }

// Tables shared by both GEMM kinds (the fused pipeline runs both in one
// launch): token tiles of BN rows per expert, tokprefix = exclusive prefix of
// token tiles.  Kind k enumerates, per expert, f-major then token tile, so
// its tile prefix is tokprefix * nf_k.
struct TokTables {
  int *cnt, *roff, *tokprefix;
};
__host__ __device__ constexpr size_t tok_tables_bytes(int num_experts) {
  return (size_t)(3 * num_experts + 1) * sizeof(int);
}
__device__ inline void build_tok_tables(const sym_heap &h, const TokTables &tb) {
  const int E = h.s.num_experts, E_loc = E / h.s.world;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int d = e / E_loc, l = e % E_loc;
    tb.cnt[e] = __ldcg(win<const int32_t>(h, d, h.off_cnt) + l);
    tb.roff[e] = __ldcg(win<const int32_t>(h, d, h.off_recv_off) + l);
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int carry = 0;
    if (lane == 0) tb.tokprefix[0] = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int v = e < E ? (tb.cnt[e] + BN - 1) / BN : 0;
      int incl = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      if (e < E) tb.tokprefix[e + 1] = carry + incl;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
}
__device__ inline TileInfo decode_tok(const sym_heap &h, const TokTables &tb, int nf, int t) {
  const int E = h.s.num_experts;
  const int key = t / nf;  // expert e owns tiles [tokprefix[e]*nf, tokprefix[e+1]*nf)
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tb.tokprefix[mid] <= key) lo = mid; else hi = mid;
  }
  TileInfo ti;
  ti.e = lo;
  const int c = tb.cnt[lo];
  const int ntok = (c + BN - 1) / BN;
  const int local = t - tb.tokprefix[lo] * nf;
  ti.f = local / ntok;
  ti.n = local % ntok;
  ti.d = lo / (E / h.s.world);
  ti.row0 = tb.roff[lo] + ti.n * BN;
  ti.valid = min(BN, c - ti.n * BN);
  return ti;
}

// Bounded mbarrier wait that also gives up once *stop <= t (the producer
// stopped before tile t) or *abort is set; a timeout sets *abort and the
// heap's SYM_STATUS_TIMEOUT bit.
__device__ __forceinline__ bool wait_or_stop(uint64_t *bar, uint32_t parity, int t,
                                             const volatile int *stop, volatile int *abort,
                                             uint32_t timeout_us, const sym_heap &h) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  const uint64_t limit = (uint64_t)timeout_us * 1000ull;
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(a, parity)) return true;
    if (*abort || *stop <= t) return false;
    if ((it & 15u) == 15u && globaltimer_ns() - t0 > limit) {
      *abort = 1;
      raise_status(h, SYM_STATUS_TIMEOUT);
      return false;
    }
  }
}

// The gate/up epilogue hands half of each 32-column chunk to its partner warp
// (warps 2+pair and 4+pair: 64 threads on named barrier 1 + pair).
__device__ __forceinline__ void xch_barrier(int pair) {
  asm volatile("bar.sync %0, 64;" ::"r"(1 + pair) : "memory");
}
// The same barrier with an AND over `ok` of all 64 threads: both partner warps
// take the same decision, so neither is left waiting on the other.
__device__ __forceinline__ bool xch_vote(int pair, bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, %2, 64, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)ok), "r"(1 + pair)
      : "memory");
  return r != 0;
}

// ---------------------------------------------------------------------------
// cluster helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cta_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t num_clusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// shared::cluster address of the same shared variable in CTA `rank`
__device__ __forceinline__ uint32_t map_to(const void *p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// TMA copy into this CTA's shared memory whose completion is counted on an
// mbarrier of either CTA of the pair (cluster address; .cta_group::2 form)
__device__ __forceinline__ void tma_load_2d_pair(void *dst, const CUtensorMap *m, uint32_t bar_cluster,
                                                 int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(void *dst, const CUtensorMap *m, uint32_t bar_cluster,
                                                 int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05 with cta_group::2 (every tcgen05 op of a kernel uses one group size)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc2(uint32_t *dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish2() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void mma2(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                     uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// arrive once on the barrier at this smem offset in both CTAs of the pair when
// the leader's earlier MMAs have completed
__device__ __forceinline__ void commit2_both(uint64_t *bar) {
  const uint16_t mask = 0x3;
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(mask)
      : "memory");
}

}  // namespace gemm2

// Tensor-map encoders (expert_ffn.cu): a bf16 matrix [rows][cols] with a box
// of [box_rows][64]; a per-slot heap window [W][cap][cols] with the slot
// stride as the outer stride.  Both use the 128-byte swizzle.
bool encode_2d(CUtensorMap *m, const void *ptr, uint64_t rows, uint64_t cols, uint32_t box_rows);
bool encode_heap_3d(CUtensorMap *m, const sym_heap &h, uint64_t off, uint64_t cols,
                    uint32_t box_rows);
// the NBOX token-row maps of one heap window
bool encode_heap_boxes(gemm2::BMaps *m, const sym_heap &h, uint64_t off, uint64_t cols);
// Largest number of CTA pairs of `kern` (192 or 256 threads, `smem` bytes)
// that can be resident at once (cached per device and kernel).
int max_resident_pairs(const void *kern, int threads, size_t smem, int num_sms);
}  // namespace symmoe
