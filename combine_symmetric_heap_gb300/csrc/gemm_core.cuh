// gemm_core.cuh -- tile pieces of the grouped SwiGLU expert GEMMs on tcgen05,
// shared by the stand-alone expert kernels (expert_ffn.cu) and the fused
// single-launch pipeline (fused.cu).
//
// "Swap AB" tiling: the tensor-core M side (128) runs over weight rows
// (output features), the N side over an expert's tokens, so a ragged row count
// only shortens the N of the expert's last token tile (rounded up to 16).
//   GATE_UP (GEMM1): A = 128 gate rows and 128 up rows of expert e (two
//            16 KB tiles), B = 128 token rows of recv_x; two MMAs per K step
//            into two TMEM accumulators; h = bf16(silu(gate) * up).
//   DOWN    (GEMM2): A = 128 down-projection rows, B = 256 token rows of h;
//            y = bf16(h Wd^T) straight into the combine-in window.
// Both kinds use 48 KB stages (K blocks of 64, 128-byte swizzle) and 256 fp32
// TMEM columns per tile, double-buffered in a 512-column allocation.
//
// Tiles are enumerated per kind expert-major, then feature tile, then token
// tile: CTAs that run at the same time share a weight tile through L2.
#pragma once

#include "symmoe_dev.cuh"

namespace symmoe {
namespace gemm {

constexpr int BM = 128;  // tcgen05 M: weight rows per tile
constexpr int BK = 64;   // K per stage (one 128-byte swizzle row of bf16)
constexpr int UK = 16;   // K per tcgen05.mma kind::f16
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
constexpr int STAGE_BYTES = 48 * 1024;
constexpr int ACC_COLS = 256;
constexpr int TMEM_COLS = 512;

enum Kind : int { GATE_UP = 0, DOWN = 1 };

template <int KIND>
struct K;
template <>
struct K<GATE_UP> {
  static constexpr int BN = 128;  // tokens per tile
  static constexpr int NUM_A = 2;
};
template <>
struct K<DOWN> {
  static constexpr int BN = 256;
  static constexpr int NUM_A = 1;
};
__host__ __device__ constexpr int bn_of(int kind) { return kind == GATE_UP ? 128 : 256; }
static_assert(2 * A_BYTES + 128 * BK * 2 == STAGE_BYTES, "gate/up stage");
static_assert(A_BYTES + 256 * BK * 2 == STAGE_BYTES, "down stage");

// Feature tiles of 128 and K blocks of 64 per kind.
__host__ __device__ inline int nf_of(const sym_heap &h, int kind) {
  return (kind == GATE_UP ? h.s.inter : h.s.hidden) / BM;
}
__host__ __device__ inline int nk_of(const sym_heap &h, int kind) {
  return (kind == GATE_UP ? h.s.hidden : h.s.inter) / BK;
}

struct TileInfo {
  int kind, e, f, n, d, row0, valid;
};

// Per-CTA shared tables: cnt[E], roff[E] (receive offset inside the slot),
// prefix[kind][E+1] = exclusive prefix of tiles per expert.
struct Tables {
  int *cnt, *roff, *prefix0, *prefix1;
  __device__ int *prefix(int kind) const { return kind == GATE_UP ? prefix0 : prefix1; }
};
__host__ __device__ constexpr size_t tables_bytes(int num_experts) {
  return (size_t)(4 * num_experts + 2) * sizeof(int);
}

// Fill the tables from the dispatch signal area (all threads call; the
// caller synchronises afterwards).  Uses warp 0 for the scans.
__device__ inline void build_tables(const sym_heap &h, const Tables &tb) {
  const int E = h.s.num_experts, E_loc = E / h.s.world;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int d = e / E_loc, l = e % E_loc;
    tb.cnt[e] = win<const int32_t>(h, d, h.off_cnt)[l];
    tb.roff[e] = win<const int32_t>(h, d, h.off_recv_off)[l];
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    for (int kind = 0; kind < 2; ++kind) {
      int *prefix = tb.prefix(kind);
      const int bn = bn_of(kind), nf = nf_of(h, kind);
      int carry = 0;
      if (lane == 0) prefix[0] = 0;
      for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        const int v = e < E ? ((tb.cnt[e] + bn - 1) / bn) * nf : 0;
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
  }
}

__device__ inline TileInfo decode(const sym_heap &h, const Tables &tb, int kind, int t) {
  const int E = h.s.num_experts;
  const int *prefix = tb.prefix(kind);
  int lo = 0, hi = E;  // largest e with prefix[e] <= t: an expert with tiles
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= t) lo = mid; else hi = mid;
  }
  const int bn = bn_of(kind);
  TileInfo ti;
  ti.kind = kind;
  ti.e = lo;
  const int c = tb.cnt[lo];
  const int ntok = (c + bn - 1) / bn;
  const int local = t - prefix[lo];
  ti.f = local / ntok;
  ti.n = local % ntok;
  ti.d = lo / (E / h.s.world);
  ti.row0 = tb.roff[lo] + ti.n * bn;
  ti.valid = min(bn, c - ti.n * bn);
  return ti;
}

// Index of a tile's token block among all token blocks of its kind (used by
// the fused pipeline's per-token-tile completion counters).
__device__ inline int token_block(const sym_heap &h, const Tables &tb, const TileInfo &ti) {
  return tb.prefix(ti.kind)[ti.e] / nf_of(h, ti.kind) + ti.n;
}

// Tensor maps of one kind: a0/a1 weights (a1 only for GATE_UP), b tokens.
struct Maps {
  const CUtensorMap *a0, *a1, *b;
};

// Issue the TMA loads of K block kb of tile ti into one stage.
__device__ __forceinline__ void issue_loads(const sym_heap &h, const TileInfo &ti, const Maps &m,
                                            int kb, uint8_t *stage, uint64_t *full) {
  mbar_arrive_expect_tx(full, STAGE_BYTES);
  if (ti.kind == GATE_UP) {
    const int arow = ti.e * h.s.inter + ti.f * BM;
    tma_load_2d(stage, m.a0, full, kb * BK, arow);
    tma_load_2d(stage + A_BYTES, m.a1, full, kb * BK, arow);
    tma_load_3d(stage + 2 * A_BYTES, m.b, full, kb * BK, ti.row0, ti.d);
  } else {
    const int arow = ti.e * h.s.hidden + ti.f * BM;
    tma_load_2d(stage, m.a0, full, kb * BK, arow);
    tma_load_3d(stage + A_BYTES, m.b, full, kb * BK, ti.row0, ti.d);
  }
}

// The MMAs of one stage (4 K steps of 16) into the tile's accumulator(s).
__device__ __forceinline__ void issue_mmas(const TileInfo &ti, uint8_t *stage, uint32_t d_tmem,
                                           bool first_kb) {
  const int bn = bn_of(ti.kind);
  const uint32_t idesc = idesc_bf16_f32(BM, min(bn, (ti.valid + 15) & ~15));
  const uint64_t da0 = smem_desc_sw128(stage);
  if (ti.kind == GATE_UP) {
    const uint64_t da1 = smem_desc_sw128(stage + A_BYTES);
    const uint64_t db = smem_desc_sw128(stage + 2 * A_BYTES);
#pragma unroll
    for (int kk = 0; kk < BK / UK; ++kk) {
      const uint64_t adv = (uint64_t)(kk * UK * 2 / 16);  // +32 bytes per K step
      const uint32_t acc = (!first_kb || kk > 0) ? 1u : 0u;
      tc_mma_bf16(d_tmem, da0 + adv, db + adv, idesc, acc);
      tc_mma_bf16(d_tmem + 128, da1 + adv, db + adv, idesc, acc);
    }
  } else {
    const uint64_t db = smem_desc_sw128(stage + A_BYTES);
#pragma unroll
    for (int kk = 0; kk < BK / UK; ++kk) {
      const uint64_t adv = (uint64_t)(kk * UK * 2 / 16);
      tc_mma_bf16(d_tmem, da0 + adv, db + adv, idesc, (!first_kb || kk > 0) ? 1u : 0u);
    }
  }
}

// Epilogue of one tile by one of the four epilogue warps (lane quarter q of
// TMEM = features 32q..32q+31 of the tile).  tacc = accumulator column base.
__device__ __forceinline__ void epilogue(const sym_heap &h, const TileInfo &ti, uint32_t tmem_base,
                                         uint32_t tacc, int q, int lane) {
  const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + tacc;
  if (ti.kind == GATE_UP) {
    const int ld = h.s.inter;
    uint16_t *out = win<uint16_t>(h, ti.d, h.off_h) + (size_t)ti.row0 * ld + ti.f * BM + q * 32 + lane;
    for (int c0 = 0; c0 < ti.valid; c0 += 32) {
      uint32_t a[32], b[32];
      tmem_ld32(tbase + c0, a);
      tmem_ld32(tbase + 128 + c0, b);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        if (c0 + c < ti.valid) {
          const float gt = __uint_as_float(a[c]);
          const float up = __uint_as_float(b[c]);
          out[(size_t)(c0 + c) * ld] = to_bf16(gt / (1.0f + __expf(-gt)) * up);
        }
      }
    }
  } else {
    const int ld = h.s.hidden;
    uint16_t *out = win<uint16_t>(h, ti.d, h.off_y) + (size_t)ti.row0 * ld + ti.f * BM + q * 32 + lane;
    for (int c0 = 0; c0 < ti.valid; c0 += 32) {
      uint32_t a[32];
      tmem_ld32(tbase + c0, a);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 32; ++c)
        if (c0 + c < ti.valid) out[(size_t)(c0 + c) * ld] = to_bf16(__uint_as_float(a[c]));
    }
  }
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

// Wait (bounded, acquire) for the dispatch ready counters of the token rows
// of a GATE_UP tile.
__device__ inline bool wait_rows_dispatched(const sym_heap &h, const TileInfo &ti,
                                            uint32_t timeout_us, const volatile int *abort) {
  const int total = *win<const int32_t>(h, ti.d, h.off_total);
  const uint32_t *ready = win<const uint32_t>(h, ti.d, h.off_ready);
  for (int b = ti.row0 / SYM_ROWS_PER_FLAG; b <= (ti.row0 + ti.valid - 1) / SYM_ROWS_PER_FLAG; ++b) {
    const uint32_t target = (uint32_t)min(SYM_ROWS_PER_FLAG, total - b * SYM_ROWS_PER_FLAG);
    if (!wait_counter_geq(ready + b, target, timeout_us, abort)) return false;
  }
  return true;
}

// Non-blocking probe of the same counters (one acquire load each).
__device__ inline bool rows_dispatched_now(const sym_heap &h, const TileInfo &ti) {
  const int total = *win<const int32_t>(h, ti.d, h.off_total);
  const uint32_t *ready = win<const uint32_t>(h, ti.d, h.off_ready);
  for (int b = ti.row0 / SYM_ROWS_PER_FLAG; b <= (ti.row0 + ti.valid - 1) / SYM_ROWS_PER_FLAG; ++b) {
    const uint32_t target = (uint32_t)min(SYM_ROWS_PER_FLAG, total - b * SYM_ROWS_PER_FLAG);
    if (ld_acquire_u32(ready + b) < target) return false;
  }
  return true;
}

}  // namespace gemm

// Tensor-map encoders (expert_ffn.cu): a bf16 matrix [rows][cols] with a box
// of [box_rows][64]; a per-slot heap window [W][cap][cols] with the slot
// stride as the outer stride.  Both use the 128-byte swizzle.
bool encode_2d(CUtensorMap *m, const void *ptr, uint64_t rows, uint64_t cols, uint32_t box_rows);
bool encode_heap_3d(CUtensorMap *m, const sym_heap &h, uint64_t off, uint64_t cols,
                    uint32_t box_rows);
}  // namespace symmoe
