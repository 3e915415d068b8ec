// gemm2sm.cuh -- the expert GEMM tiles on CTA pairs (tcgen05 cta_group::2):
// one M=256 MMA spans the tensor cores of two SMs of a cluster.  Used by the
// staged expert FFN and by the fused pipeline, and, as two more tile kinds,
// by the router GEMM and the linear layer of the GEMM + all-to-all workload.
//
// Each CTA of the pair stages only its half of both operands: 128 of the 256
// weight rows (A) and N/2 of the N token rows (B); the MMA, issued by the
// pair's first CTA (the leader), reads the four halves from both shared
// memories and leaves output rows 0-127 in the leader's TMEM and rows 128-255
// in the peer's.  Per SM that is 32 KB of operands per 128 x 256 x 64
// multiply-adds, so six stages fit and the ring keeps the tensor pipe fed.
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
// Token tiles hold BN = 256 rows; an expert with 257..288 rows has one tile
// that carries the remainder through a second, narrow MMA on the same weight
// stream, so it streams its weights once.
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
constexpr int REM_MAX = 32;     // rows an expert's last tile may carry beyond BN (second MMA)
constexpr int STAGES = 6;
constexpr int A_BYTES = 128 * BK * 2;          // 16 KB: this CTA's weight rows
constexpr int B_ROWS = BN / 2;                 // this CTA's token rows at most (largest box)
constexpr int B_BYTES = B_ROWS * BK * 2;       // 16 KB
constexpr int B1_BYTES = REM_MAX / 2 * BK * 2; // 2 KB: this CTA's remainder rows
constexpr int STAGE_BYTES = A_BYTES + B_BYTES + B1_BYTES;  // 34 KB
constexpr int ACC_COLS = BN;
constexpr int TMEM_COLS = 512;
constexpr int XCH_BYTES = 2 * 2 * 16 * 32 * 4;  // pairs x directions x 16 cols x 32 lanes

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
// GATE_UP: h = silu(x Wg^T) * x Wu^T;  DOWN: y = h Wd^T;  ROUTER: logits = x Wr^T
// with the roles turned: tokens on the MMA's M side (the "features", 256 per
// pair tile) and the E router rows on the N side (the "rows" of one
// pseudo-expert), so a small E costs a narrow MMA instead of a padded one;
// fp32 output.  LINEAR: out = x W^T with W [H][H] over one slot's token rows
// (the GEMM + all-to-all workload), bf16 output routed by the Pipe.
enum Kind : int { GATE_UP = 0, DOWN = 1, ROUTER = 2, LINEAR = 3 };

// features per pair tile and K blocks per kind
__host__ __device__ inline int feat_of(int kind) { return kind == GATE_UP ? 128 : 256; }
__host__ __device__ inline int nf_of(const sym_heap &h, int kind) {
  const int n = kind == GATE_UP                  ? h.s.inter
                : kind == DOWN || kind == LINEAR ? h.s.hidden
                                                 : h.s.world * h.s.tokens_per_slot;
  return (n + feat_of(kind) - 1) / feat_of(kind);
}
__host__ __device__ inline int nk_of(const sym_heap &h, int kind) {
  return (kind == DOWN ? h.s.inter : h.s.hidden) / BK;
}

struct TileInfo {
  int e, f, n, d, row0, valid;  // valid: token rows of the tile, up to BN + REM_MAX
  int ks = 0;                   // K split of the tile (Pipe::kb_per_split K blocks each)
  int single = 0;               // the expert has one token tile: no other tile reads its weights
};

// Token tiles of an expert with c rows: BN rows each.  An expert with one
// full tile and a remainder of at most REM_MAX rows (BN < c <= BN + REM_MAX)
// streams its weights once: the remainder rides on that tile as a second MMA.
// Such an expert is bound by its weight stream; with more full tiles the
// expert is compute-bound, the narrow second MMA costs more than a separate
// short tile, and the remainder gets a tile of its own.
__host__ __device__ inline int ntok_of(int c) {
  const int full = c / BN, rem = c % BN;
  return full + ((rem > 0 && !(full == 1 && rem <= REM_MAX)) ? 1 : 0);
}
// the token tile of an expert holding its row r (0 <= r < c)
__host__ __device__ inline int tile_of_row(int c, int r) { return min(r / BN, ntok_of(c) - 1); }

// MMA widths of a tile: n0 for its first BN rows, n1 (0: none) for the rest;
// each a multiple of 16 (rows past `valid` are computed and dropped)
struct TileGeom {
  int n0, n1;
};
__device__ __forceinline__ TileGeom geom(int valid) {
  TileGeom g;
  g.n0 = min(BN, (valid + 15) & ~15);
  g.n1 = valid > BN ? ((valid - BN + 15) & ~15) : 0;
  return g;
}

// Per-expert tables for tile decoding, shared by both GEMM kinds (the fused
// pipeline runs both in one launch): tokprefix = exclusive prefix of token
// tiles.  Kind k enumerates, per expert, f-major then token tile, so its tile
// prefix is tokprefix * nf_k.
struct TokTables {
  int *cnt, *roff, *tokprefix;
};
__host__ __device__ constexpr size_t tok_tables_bytes(int num_experts) {
  return (size_t)(3 * num_experts + 1) * sizeof(int);
}
// Reads the dispatch results with __ldcg: in the fused pipeline they were
// written earlier in the same launch.  An expert whose rows [off, off + cnt)
// do not lie inside its slot's windows (a corrupted or stale signal area)
// gets no tiles: the tables say it has no rows, so no tile reads or stores
// past the capacity, and SYM_STATUS_OVERFLOW is raised.
__device__ inline void build_tok_tables(const sym_heap &h, const TokTables &tb) {
  const int E = h.s.num_experts, E_loc = E / h.s.world;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int d = e / E_loc, l = e % E_loc;
    int c = __ldcg(win<const int32_t>(h, d, h.off_cnt) + l);
    int o = __ldcg(win<const int32_t>(h, d, h.off_recv_off) + l);
    if (c < 0 || o < 0 || (uint64_t)o + (uint64_t)c > h.cap) {
      raise_status(h, SYM_STATUS_OVERFLOW);
      c = 0;
      o = 0;
    }
    tb.cnt[e] = c;
    tb.roff[e] = o;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int carry = 0;
    if (lane == 0) tb.tokprefix[0] = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int v = e < E ? ntok_of(tb.cnt[e]) : 0;
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
// Token tiles per group in a kind's tile order.  Inside an expert the tiles
// run feature tile major, so one weight tile serves all the expert's token
// tiles back to back; but each feature tile then sweeps all the expert's token
// rows again, and a heavy expert's rows can outgrow L2 and be re-read from
// DRAM per feature tile.  So the token tiles go in groups: group by group,
// feature tile major inside a group.  Gate/up (K = H): a group's rows fit
// 48 MB.  Down (K = I, the rows are h): a group's rows fit 64 MB, so that a
// wave of tiles touches about as many h tiles as weight tiles (Mixtral-like:
// groups of 8 of an expert's 16 token tiles instead of all 16; the expert FFN
// measured 1.5-2.7% faster at full clock, 1.1% under the power cap).  An
// expert whose rows fit keeps one group (the plain order).
constexpr long long GROUP_B_BYTES = 48ll << 20;
constexpr long long GROUP_H_BYTES = 64ll << 20;
__host__ __device__ inline int tok_group_of(const sym_heap &h, int kind) {
  if (kind != GATE_UP && kind != DOWN) return 1 << 30;
  const long long budget = kind == GATE_UP ? GROUP_B_BYTES : GROUP_H_BYTES;
  const long long tile_b = (long long)BN * (kind == GATE_UP ? h.s.hidden : h.s.inter) * 2;
  return (int)(budget / tile_b) > 1 ? (int)(budget / tile_b) : 1;
}

__device__ inline TileInfo decode_tok(const sym_heap &h, const TokTables &tb, int nf, int group, int t) {
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
  const int ntok = ntok_of(c);
  const int local = t - tb.tokprefix[lo] * nf;
  // group g holds token tiles [g*G, g*G + w), w*nf tiles, feature tile major
  // (G*nf <= ntok*nf: no overflow)
  const int G = min(group, ntok);
  const int g = local / (G * nf);
  const int r = local - g * G * nf;
  const int w = min(G, ntok - g * G);
  ti.f = r / w;
  ti.n = g * G + r % w;
  ti.d = lo / (E / h.s.world);
  ti.row0 = tb.roff[lo] + ti.n * BN;
  ti.valid = ti.n == ntok - 1 ? c - ti.n * BN : BN;
  ti.single = ntok == 1;
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
// The same with an L2 eviction policy (createpolicy): weights that no other
// tile will read are loaded evict-first, so they do not push out the token
// rows and outputs that are read again.
__device__ __forceinline__ void tma_load_2d_pair_hint(void *dst, const CUtensorMap *m, uint32_t bar_cluster,
                                                      int x, int y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster), "r"(x), "r"(y), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
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


// Static pair schedule, for the router and the linear-layer kernels, whose
// tiles all cost about the same (the expert GEMM's tiles differ with their
// row counts and are claimed dynamically, below).  Wave i holds tiles
// [i*npairs, (i+1)*npairs) (consecutive tiles share weight rows, so a wave
// streams each weight block from HBM about once); pair p takes tile
// i*npairs + (p+i) mod npairs of it.  The rotation keeps tiles that recur
// with a period (every expert's last token tile, say) from landing on the
// same few pairs.  Indices grow with i; only the last wave can run past the
// end of the list.
__device__ __forceinline__ int pair_tile(int i, int pair, int npairs) {
  return i * npairs + (pair + i) % npairs;
}

// ---------------------------------------------------------------------------
// The pair tile engine: the three roles of one tile, shared by the staged
// expert GEMM and the fused pipeline.  Shared memory (both CTAs, same offsets):
// a ring of STAGES stages [A 16 KB | B 16 KB | B1 2 KB] and the exchange
// buffer; TMEM: two 256-column fp32 accumulators.  A tile whose rows exceed
// BN (a remainder of <= REM_MAX rows on an expert's last tile) adds a second
// MMA per K step on the remainder rows (B1) into the first columns of the
// other accumulator, which it therefore also holds; its epilogue drains the
// remainder first and hands that accumulator back before the main part.
// ---------------------------------------------------------------------------
struct Pipe {
  uint8_t *ring;
  float *xch;
  uint64_t *full, *empty, *acc_full;
  uint64_t *acc_empty;  // [2] accumulator b drained (main part of its tile)
  uint64_t *acc_head;   // [2] its first 32 columns drained (where a remainder goes)
  uint32_t tmem_base;
  uint32_t rank;              // CTA rank in the pair (0: leader)
  volatile int *abort;        // this CTA gives up (timeout or dependency failure)
  const volatile int *stop;   // roles stop before tile index *stop
  uint32_t tmo;               // wait limit, microseconds
  int scale_rows;             // DOWN: y row p = bf16(recv_w[p] * acc) (weights in the epilogue)
  float *logits;              // ROUTER: the [N][E] fp32 output (split ks: its partial at ks*N*E)
  int kb_per_split = 0;       // K blocks per split of a tile (0: the whole K)
  // LINEAR: output window (offset in a slot) and the all-to-all block (0: the
  // rows stay in the tile's slot; B: source row r of slot d goes to slot r / B,
  // row d*B + r % B).  shard_kb > 0: K arrives in shards of shard_kb blocks,
  // stored shard major ([shard][T rows][H/W] in the B window, the B maps'
  // rows running over shard*T + row); shard_wait: shard s of slot d arrives
  // during the launch and is in place once word s of slot d's ready window
  // is nonzero.  shard_direct: the B maps run over the owners' buffers
  // instead, [shard][N tokens][H/W], and a tile of slot d reads its tokens
  // d*T + row of every shard there (no copy)
  uint64_t out_off = 0;
  int a2a_block = 0;
  int shard_kb = 0;
  int shard_wait = 0;
  int shard_direct = 0;
};

// ---------------------------------------------------------------------------
// Dynamic tile schedule of a CTA pair (expert GEMM kinds).  The leader's
// producer claims the next tile index from a global counter (one atomicAdd per
// tile) just before it streams that tile, so a pair that finishes early takes
// more tiles and the pairs end within about one tile of each other; under a
// static assignment a launch ends with its slowest pair, and tiles differ in
// cost with their row counts.  Consecutive claims are consecutive tiles, so
// the pairs running at one time still share weight rows as a wave does.  The
// index reaches the pair's other roles through a queue of TQ entries held in
// both CTAs' shared memory: full[i] (in each CTA: the leader producer's one
// arrival, after it wrote the entry there) and empty[i] (in the leader: one
// arrival per consumer -- the peer's producer, the leader's MMA thread and the
// 8 epilogue warps -- after it read the entry).  Entry -1 ends the schedule.
// ---------------------------------------------------------------------------
constexpr int TQ = 4;
constexpr int TQ_CONSUMERS = 10;
struct TileQueue {
  volatile int *id;  // [TQ]
  uint64_t *full;    // [TQ]
  uint64_t *empty;   // [TQ] (the leader's are used)
};
// one thread of each CTA, before the cluster barrier that precedes any use
__device__ __forceinline__ void tq_init(const TileQueue &q) {
  for (int i = 0; i < TQ; ++i) {
    mbar_init(&q.full[i], 1);
    mbar_init(&q.empty[i], TQ_CONSUMERS);
  }
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar_addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar_addr), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait with cluster-scope acquire (the entry may come from the other
// CTA of the pair); a timeout raises SYM_STATUS_TIMEOUT.
__device__ inline bool tq_wait(const sym_heap &h, const Pipe &p, uint64_t *bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait_cluster(a, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  const uint64_t limit = (uint64_t)p.tmo * 1000ull;
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait_cluster(a, parity)) return true;
    if (*p.abort) return false;
    if ((it & 15u) == 15u && globaltimer_ns() - t0 > limit) {
      raise_status(h, SYM_STATUS_TIMEOUT);
      return false;
    }
  }
}
// Leader producer: entry n of the pair's schedule is tile `id` (-1: the end).
__device__ inline bool tq_push(const sym_heap &h, const Pipe &p, const TileQueue &q, int n, int id) {
  const int i = n % TQ;
  const uint32_t use = (uint32_t)(n / TQ);
  if (!tq_wait(h, p, &q.empty[i], (use & 1u) ^ 1u)) return false;
  q.id[i] = id;
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(map_to((const void *)&q.id[i], 1)), "r"(id) : "memory");
  mbar_arrive(&q.full[i]);
  mbar_arrive_remote(map_to(&q.full[i], 1));  // release.cluster: orders the store above
  return true;
}
// A consumer's entry n: its tile (-1: the end; -2: the wait failed), the
// entry handed back once read.
__device__ inline int tq_pop(const sym_heap &h, const Pipe &p, const TileQueue &q, int n) {
  const int i = n % TQ;
  const uint32_t use = (uint32_t)(n / TQ);
  if (!tq_wait(h, p, &q.full[i], use & 1u)) return -2;
  const int id = q.id[i];
  if (p.rank == 0) mbar_arrive(&q.empty[i]);
  else mbar_arrive_remote(map_to(&q.empty[i], 0));
  return id;
}

// The producers' walk of the dynamic schedule.  The leader claims one tile
// ahead: while it streams tile c it holds the next claim, checks that tile's
// inputs halfway through c (probe) and publishes it as soon as they are in
// place, so the peer and the MMA learn it early and no check sits between two
// tiles.  A published entry therefore means "inputs ready": the peer streams
// it without checking again (the leader's acquire of the ready counters and
// its cluster-scope release of the entry order the inputs before the peer's
// loads).  claim() gives the next tile or -1; ready(c, block) checks tile c's
// inputs (bounded when blocking); produce(c, n, probe) streams tile c as entry
// n.  fence_inputs: the inputs may have been written by generic stores during
// this launch or one overlapping it (a proxy fence then precedes each tile's
// loads); inputs written by an earlier kernel need none.  On a failure *stop
// = the entry where the pair stopped.  Returns false after a failure.
template <typename Claim, typename Ready, typename Produce>
__device__ bool produce_schedule(const sym_heap &h, const Pipe &p, const TileQueue &q, volatile int *stop,
                                 bool fence_inputs, Claim claim, Ready ready, Produce produce) {
  auto no_probe = []() {};
  if (p.rank != 0) {
    for (int n = 0;; ++n) {
      const int c = tq_pop(h, p, q, n);
      if (c == -2) {
        *stop = n;
        return false;
      }
      if (c < 0) return true;
      if (fence_inputs) fence_proxy_async();  // made visible by the leader's check
      if (!produce(c, n, no_probe)) return false;
    }
  }
  int c = claim();
  if (c >= 0 && !ready(c, true)) {
    raise_status(h, SYM_STATUS_TIMEOUT);
    *stop = 0;
    tq_push(h, p, q, 0, -1);
    return false;
  }
  if (!tq_push(h, p, q, 0, c)) {
    *stop = 0;
    return false;
  }
  for (int n = 0; c >= 0; ++n) {
    const int c_next = claim();
    bool pushed = false, failed = false;
    auto probe = [&]() {
      if (c_next < 0 || ready(c_next, false)) {
        if (tq_push(h, p, q, n + 1, c_next)) pushed = true;
        else failed = true;
      }
    };
    if (fence_inputs) fence_proxy_async();  // inputs written by generic stores
    if (!produce(c, n, probe)) {
      *stop = n;
      if (!pushed && !failed) tq_push(h, p, q, n + 1, -1);
      return false;
    }
    if (failed) {
      *stop = n + 1;
      return false;
    }
    if (!pushed) {
      if (c_next >= 0 && !ready(c_next, true)) {
        raise_status(h, SYM_STATUS_TIMEOUT);
        *stop = n + 1;
        tq_push(h, p, q, n + 1, -1);
        return false;
      }
      if (!tq_push(h, p, q, n + 1, c_next)) {
        *stop = n + 1;
        return false;
      }
    }
    c = c_next;
  }
  return true;
}

// K blocks [kb0, kb1) of tile ti
__device__ __forceinline__ void k_range(const Pipe &p, const TileInfo &ti, int nk, int &kb0, int &kb1) {
  kb0 = p.kb_per_split ? ti.ks * p.kb_per_split : 0;
  kb1 = p.kb_per_split ? min(nk, kb0 + p.kb_per_split) : nk;
}

__device__ __forceinline__ void ring_advance(int &stage, uint32_t &phase) {
  if (++stage == STAGES) {
    stage = 0;
    phase ^= 1u;
  }
}

struct ProdState {
  int stage = 0;
  uint32_t phase = 0;
};

// Producer K loop of one tile; TWO: the tile carries a remainder part (B1);
// ONCE: its weight rows are read by no other tile (loaded evict-first).
// Templated so that no conditional copy sits in the loop.
template <int KIND, bool TWO, bool ONCE, typename Probe>
__device__ __forceinline__ bool produce_k(const sym_heap &h, const Pipe &p, ProdState &s, int d, int arow,
                                          int r0, int r1, const CUtensorMap *ma0, const CUtensorMap *ma1,
                                          const CUtensorMap *mb0, const CUtensorMap *mb1, uint32_t tx, int t,
                                          int kb0, int kb1, const uint32_t *shard_ctr, Probe &probe) {
  const uint32_t full_leader = map_to(&p.full[0], 0);
  const uint64_t pol = ONCE ? l2_evict_first_policy() : 0;
  for (int kb = kb0; kb < kb1; ++kb) {
    if (kb == (kb0 + kb1) / 2) probe();
    int bx = kb * BK, by0 = r0, by1 = r1, bz = d;
    if (KIND == LINEAR && p.shard_kb) {
      const int sh = kb / p.shard_kb;
      if (shard_ctr && kb == sh * p.shard_kb) {
        // this K shard is copied while the GEMM runs: wait until it is counted
        if (!wait_counter_geq(shard_ctr + sh, 1u, p.tmo, p.abort)) {
          *p.abort = 1;
          raise_status(h, SYM_STATUS_TIMEOUT);
          return false;
        }
        fence_proxy_async();
      }
      bx = (kb - sh * p.shard_kb) * BK;
      if (p.shard_direct) {  // shard sh of the tile's tokens, read in the owner's buffer
        by0 += d * h.s.tokens_per_slot;
        by1 += d * h.s.tokens_per_slot;
        bz = sh;
      } else {
        by0 += sh * h.s.tokens_per_slot;
        by1 += sh * h.s.tokens_per_slot;
      }
    }
    if (!wait_or_stop(&p.empty[s.stage], s.phase ^ 1u, t, p.stop, p.abort, p.tmo, h)) return false;
    uint8_t *sb = p.ring + (size_t)s.stage * STAGE_BYTES;
    const uint32_t bar = full_leader + (uint32_t)(s.stage * sizeof(uint64_t));
    if (p.rank == 0) mbar_arrive_expect_tx(&p.full[s.stage], tx);
    if (KIND == GATE_UP && ONCE) {
      tma_load_2d_pair_hint(sb, ma0, bar, kb * BK, arow, pol);               // 64 gate rows
      tma_load_2d_pair_hint(sb + A_BYTES / 2, ma1, bar, kb * BK, arow, pol);  // 64 up rows
    } else if (KIND == GATE_UP) {
      tma_load_2d_pair(sb, ma0, bar, kb * BK, arow);
      tma_load_2d_pair(sb + A_BYTES / 2, ma1, bar, kb * BK, arow);
    } else if (ONCE) {
      tma_load_2d_pair_hint(sb, ma0, bar, kb * BK, arow, pol);  // 128 down rows
    } else {
      tma_load_2d_pair(sb, ma0, bar, kb * BK, arow);
    }
    tma_load_3d_pair(sb + A_BYTES, mb0, bar, bx, by0, bz);
    if (TWO) tma_load_3d_pair(sb + A_BYTES + B_BYTES, mb1, bar, bx, by1, bz);
    ring_advance(s.stage, s.phase);
  }
  return true;
}

// Producer (one thread per CTA): streams tile ti's K blocks into the ring.
// A rows from ma0 (gate or down rows) and ma1 (up rows), this CTA's token
// rows from the box maps.  probe() runs once, halfway through the tile.
template <int KIND, typename Probe>
__device__ bool produce_tile(const sym_heap &h, const Pipe &p, ProdState &s, const TileInfo &ti,
                             const CUtensorMap *ma0, const CUtensorMap *ma1, const BMaps &mb, int t,
                             Probe probe) {
  const TileGeom g = geom(ti.valid);
  const int half0 = g.n0 / 2, half1 = g.n1 / 2;
  const int box0 = box_index(half0), box1 = box_index(max(half1, 1));
  const uint32_t b_rows = (uint32_t)(BOX_MIN_ROWS << box0) + (g.n1 ? (uint32_t)(BOX_MIN_ROWS << box1) : 0u);
  const uint32_t tx = 2u * ((uint32_t)A_BYTES + b_rows * BK * 2);  // both CTAs' bytes
  const int r0 = ti.row0 + (int)p.rank * half0;
  const int r1 = ti.row0 + BN + (int)p.rank * half1;
  const int arow = KIND == GATE_UP ? ti.e * h.s.inter + ti.f * 128 + (int)p.rank * 64
                                   : ti.e * h.s.hidden + ti.f * 256 + (int)p.rank * 128;
  int kb0, kb1;
  k_range(p, ti, nk_of(h, KIND), kb0, kb1);
  // LINEAR with K shards that arrive during the launch: the tile's slot's counters
  const uint32_t *shard_ctr =
      KIND == LINEAR && p.shard_kb && p.shard_wait ? win<const uint32_t>(h, ti.d, h.off_ready) : nullptr;
  // The expert GEMM's weights of an expert with one token tile are read by no
  // other tile: evict-first keeps its token rows and outputs in L2.  Measured
  // on tiles of about 256 rows (DeepSeek-like: 2% faster); tiles of a few
  // rows (Decode-like) have little to protect and ran 1% slower, so they
  // keep the default policy.
  const bool once = (KIND == GATE_UP || KIND == DOWN) && ti.single && ti.valid >= BN / 2;
  if (once)
    return g.n1 ? produce_k<KIND, true, true>(h, p, s, ti.d, arow, r0, r1, ma0, ma1, &mb.m[box0], &mb.m[box1], tx,
                                              t, kb0, kb1, shard_ctr, probe)
                : produce_k<KIND, false, true>(h, p, s, ti.d, arow, r0, r1, ma0, ma1, &mb.m[box0], &mb.m[box1], tx,
                                               t, kb0, kb1, shard_ctr, probe);
  return g.n1 ? produce_k<KIND, true, false>(h, p, s, ti.d, arow, r0, r1, ma0, ma1, &mb.m[box0], &mb.m[box1], tx, t,
                                             kb0, kb1, shard_ctr, probe)
              : produce_k<KIND, false, false>(h, p, s, ti.d, arow, r0, r1, ma0, ma1, &mb.m[box0], &mb.m[box1], tx,
                                              t, kb0, kb1, shard_ctr, probe);
}

struct MmaState {
  int stage = 0;
  uint32_t phase = 0;
  uint32_t e0 = 0, e1 = 0;  // acquisitions of acc_empty[0] / [1] so far (main parts)
  uint32_t h0 = 0, h1 = 0;  // acquisitions of acc_head[0] / [1] (main parts and remainders)
  int abuf = 0;             // accumulator of the next tile's main part
};

// Acquisition n of a barrier waits for its release n-1 (releases never run
// ahead of acquisitions, so the parity is unambiguous).
__device__ __forceinline__ bool acquire(const sym_heap &h, const Pipe &p, uint64_t *bar, uint32_t &n, int t) {
  const bool ok = wait_or_stop(bar, (n & 1u) ^ 1u, t, p.stop, p.abort, p.tmo, h);
  ++n;
  return ok;
}

// MMA K loop of one tile into d0 (and, TWO, the remainder into d1).
template <int KIND, bool TWO>
__device__ __forceinline__ bool mma_k(const sym_heap &h, const Pipe &p, MmaState &s, uint32_t d0, uint32_t d1,
                                      uint32_t idesc0, uint32_t idesc1, int kb0, int kb1, int t) {
  for (int kb = kb0; kb < kb1; ++kb) {
    if (!wait_or_stop(&p.full[s.stage], s.phase, t, p.stop, p.abort, p.tmo, h)) return false;
    tc_fence_after();
    uint8_t *sb = p.ring + (size_t)s.stage * STAGE_BYTES;
    const uint64_t da = smem_desc_sw128(sb), db0 = smem_desc_sw128(sb + A_BYTES);
    const uint64_t db1 = smem_desc_sw128(sb + A_BYTES + B_BYTES);
#pragma unroll
    for (int kk = 0; kk < BK / UK; ++kk) {
      const uint64_t adv = (uint64_t)(kk * UK * 2 / 16);
      const uint32_t acc = (kb > kb0 || kk > 0) ? 1u : 0u;
      mma2(d0, da + adv, db0 + adv, idesc0, acc);
      if (TWO) mma2(d1, da + adv, db1 + adv, idesc1, acc);  // interleaved: issues faster than grouped
    }
    commit2_both(&p.empty[s.stage]);
    ring_advance(s.stage, s.phase);
  }
  return true;
}

// MMA issuer (one thread of the leader CTA).
template <int KIND>
__device__ bool mma_tile(const sym_heap &h, const Pipe &p, MmaState &s, const TileInfo &ti, int t) {
  const TileGeom g = geom(ti.valid);
  const int b = s.abuf;
  // main part: all of accumulator b; remainder: the first columns of the other
  if (!acquire(h, p, &p.acc_empty[b], b ? s.e1 : s.e0, t)) return false;
  if (!acquire(h, p, &p.acc_head[b], b ? s.h1 : s.h0, t)) return false;
  if (g.n1 && !acquire(h, p, &p.acc_head[b ^ 1], b ? s.h0 : s.h1, t)) return false;
  tc_fence_after();
  const uint32_t d0 = p.tmem_base + (uint32_t)(b * ACC_COLS);
  const uint32_t d1 = p.tmem_base + (uint32_t)((b ^ 1) * ACC_COLS);
  const uint32_t idesc0 = idesc_bf16_f32(256, g.n0);
  int kb0, kb1;
  k_range(p, ti, nk_of(h, KIND), kb0, kb1);
  const bool ok = g.n1 ? mma_k<KIND, true>(h, p, s, d0, d1, idesc0, idesc_bf16_f32(256, g.n1), kb0, kb1, t)
                       : mma_k<KIND, false>(h, p, s, d0, d1, idesc0, idesc0, kb0, kb1, t);
  if (!ok) return false;
  commit2_both(&p.acc_full[b]);
  s.abuf = b ^ 1;
  return true;
}

struct EpiState {
  uint32_t used0 = 0, used1 = 0;  // tiles whose main part used each accumulator
  int abuf = 0;
};

// hand (part of) an accumulator back to the leader's MMA: arrive once per
// epilogue warp on the leader's barrier at this offset
__device__ __forceinline__ void release_acc(const Pipe &p, uint64_t *bar, int lane) {
  tc_fence_before();
  __syncwarp();
  if (lane == 0) {
    if (p.rank == 0) mbar_arrive(bar);
    else mbar_arrive_remote(map_to(bar, 0));
  }
}

// Epilogue of token rows [row, row + nrows) whose accumulators start at TMEM
// address tcol (this warp's lane quarter q); head() runs once the first
// 32 columns have been read.
template <int KIND, bool SCALE, typename Head>
__device__ void epi_rows(const sym_heap &h, const Pipe &p, const TileInfo &ti, uint32_t tcol, int row,
                         int nrows, int q, int lane, Head head) {
  if (KIND == GATE_UP) {
    const int pair = q & 1;  // gate lanes 32*pair.., up lanes 64 + 32*pair..
    const bool is_gate = q < 2;
    const int ld = h.s.inter;
    const int feature = ti.f * 128 + (int)p.rank * 64 + pair * 32 + lane;
    uint16_t *out = win<uint16_t>(h, ti.d, h.off_h) + (size_t)row * ld + feature;
    // xch[pair][dir][16][32]: dir 0 carries up columns 0-15 to the gate warp,
    // dir 1 gate columns 16-31 to the up warp
    float *xb = p.xch + (size_t)pair * 2 * 16 * 32;
    float *to_partner = xb + (is_gate ? 1 : 0) * 16 * 32;
    const float *from_partner = xb + (is_gate ? 0 : 1) * 16 * 32;
    for (int c0 = 0; c0 < nrows; c0 += 32) {
      uint32_t v[32];
      tmem_ld32(tcol + c0, v);
      tmem_ld_wait();
      if (c0 == 0) head();
      xch_barrier(pair);  // the partner has read the previous chunk
#pragma unroll
      for (int c = 0; c < 16; ++c) to_partner[c * 32 + lane] = __uint_as_float(is_gate ? v[16 + c] : v[c]);
      xch_barrier(pair);
      const int keep = is_gate ? 0 : 16;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const int col = c0 + keep + c;
        const float other = from_partner[c * 32 + lane];
        const float mine = __uint_as_float(is_gate ? v[c] : v[16 + c]);
        const float gt = is_gate ? mine : other;
        const float up = is_gate ? other : mine;
        if (col < nrows) out[(size_t)col * ld] = to_bf16(__fdividef(gt, 1.0f + __expf(-gt)) * up);
      }
    }
  } else if (KIND == ROUTER) {
    // this lane's token; columns [row, row + nrows) are router rows (experts),
    // stored contiguously in the token's logits row
    const int ld = h.s.num_experts, N = h.s.world * h.s.tokens_per_slot;
    const int token = ti.f * 256 + (int)p.rank * 128 + q * 32 + lane;
    float *out = p.logits + (size_t)ti.ks * N * ld + (size_t)token * ld + row;
    const bool live = token < N;
    const bool vec = (ld & 3) == 0 && (reinterpret_cast<uintptr_t>(p.logits) & 15u) == 0;
    for (int c0 = 0; c0 < nrows; c0 += 32) {
      uint32_t v[32];
      tmem_ld32(tcol + c0, v);
      tmem_ld_wait();
      if (c0 == 0) head();
      if (!live) continue;
      if (vec && c0 + 32 <= nrows) {
#pragma unroll
        for (int c = 0; c < 32; c += 4)
          *reinterpret_cast<float4 *>(out + c0 + c) = make_float4(
              __uint_as_float(v[c]), __uint_as_float(v[c + 1]), __uint_as_float(v[c + 2]), __uint_as_float(v[c + 3]));
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c)
          if (c0 + c < nrows) out[c0 + c] = __uint_as_float(v[c]);
      }
    }
  } else if (KIND == LINEAR) {
    const int ld = h.s.hidden, B = p.a2a_block;
    const int feature = ti.f * 256 + (int)p.rank * 128 + q * 32 + lane;
    const bool live = feature < ld;
    for (int c0 = 0; c0 < nrows; c0 += 32) {
      uint32_t v[32];
      tmem_ld32(tcol + c0, v);
      tmem_ld_wait();
      if (c0 == 0) head();
      // destination (slot j, row rr) of source row row + c0, stepped per row
      int j = ti.d, rr = row + c0;
      if (B) {
        j = rr / B;
        rr -= j * B;
      }
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        if (live && c0 + c < nrows) {
          const size_t drow = B ? (size_t)ti.d * B + rr : (size_t)rr;
          win<uint16_t>(h, j, p.out_off)[drow * ld + feature] = to_bf16(__uint_as_float(v[c]));
        }
        if (++rr == B) {  // never true for B = 0
          rr = 0;
          ++j;
        }
      }
    }
  } else {
    const int ld = h.s.hidden;
    const int feature = ti.f * 256 + (int)p.rank * 128 + q * 32 + lane;
    uint16_t *out = win<uint16_t>(h, ti.d, h.off_y) + (size_t)row * ld + feature;
    const bool live = feature < ld;  // a last feature tile may run past H
    const float *wrow = win<const float>(h, ti.d, h.off_recv_w) + row;  // SCALE: the rows' weights
    for (int c0 = 0; c0 < nrows; c0 += 32) {
      float wl = 1.f;
      if (SCALE && c0 + lane < nrows) wl = __ldcg(wrow + c0 + lane);
      uint32_t v[32];
      tmem_ld32(tcol + c0, v);
      tmem_ld_wait();
      if (c0 == 0) head();
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        float yv = __uint_as_float(v[c]);
        if (SCALE) yv *= __shfl_sync(0xffffffffu, wl, c);
        if (live && c0 + c < nrows) out[(size_t)(c0 + c) * ld] = to_bf16(yv);
      }
    }
  }
}

// Epilogue warp (warps 2-5 of both CTAs; q = TMEM lane quarter).
template <int KIND>
__device__ bool epi_tile(const sym_heap &h, const Pipe &p, EpiState &s, const TileInfo &ti, int t, int q,
                         int lane) {
  const int b = s.abuf;
  bool ok = wait_or_stop(&p.acc_full[b], (b ? s.used1 : s.used0) & 1u, t, p.stop, p.abort, p.tmo, h);
  if (b) ++s.used1; else ++s.used0;
  // warp-collective TMEM loads and the gate/up exchange follow: decide together
  ok = KIND == GATE_UP ? xch_vote(q & 1, ok) : __all_sync(0xffffffffu, ok);
  if (!ok) return false;
  tc_fence_after();
  const uint32_t lanes = p.tmem_base + ((uint32_t)(q * 32) << 16);
  // part 1 (the remainder, in the other accumulator's first columns) first,
  // then part 0; one copy of the drain code for both.  The first 32 columns of
  // an accumulator are handed back as soon as they are read (the next tile's
  // remainder may go there), the whole main accumulator at the end.
  for (int part = ti.valid > BN ? 1 : 0; part >= 0; --part) {
    const int buf = part ? (b ^ 1) : b;
    const uint32_t tcol = lanes + (uint32_t)(buf * ACC_COLS);
    const int row = ti.row0 + part * BN, nrows = part ? ti.valid - BN : min(ti.valid, BN);
    auto head = [&]() { release_acc(p, &p.acc_head[buf], lane); };
    if (KIND == DOWN && p.scale_rows)
      epi_rows<KIND, true>(h, p, ti, tcol, row, nrows, q, lane, head);
    else
      epi_rows<KIND, false>(h, p, ti, tcol, row, nrows, q, lane, head);
    if (part == 0) release_acc(p, &p.acc_empty[buf], lane);
  }
  s.abuf = b ^ 1;
  return true;
}

// Are the dispatched rows [row, row + n) of slot d in place?  (ready counter
// per SYM_ROWS_PER_FLAG-row block; block=false only polls once)
template <typename Wait>
__device__ bool rows_ready(const sym_heap &h, int d, int row, int n, bool block, Wait wait) {
  if (n <= 0) return true;
  const int total = checked_total(h, d, true);
  const uint32_t *ready = win<const uint32_t>(h, d, h.off_ready);
  for (int b = row / SYM_ROWS_PER_FLAG; b <= (row + n - 1) / SYM_ROWS_PER_FLAG; ++b) {
    const uint32_t target = (uint32_t)min(SYM_ROWS_PER_FLAG, total - b * SYM_ROWS_PER_FLAG);
    if (block ? !wait(ready + b, target) : ld_acquire_u32(ready + b) < target) return false;
  }
  return true;
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
