/*
 * symmoe.h -- C ABI of the zero-copy MoE dispatch -> expert -> combine path
 * over a flat symmetric heap, for one GB300 (sm_103a).
 *
 * Source of the operations: the AMD technical blog "MORI CCO: Next-Generation
 * Collective Communication Object for GPUs" --
 *   - section "What is MORI CCO?": every window sits at the same offset in
 *     every rank's slot, so a peer address is window base + peer * per-rank
 *     size + offset;
 *   - section "Zero-copy MoE dispatch -> expert -> combine": dispatch writes
 *     each token straight into the receive window ("disp_out") of the rank
 *     that owns its expert, the expert GEMM reads that window in place and
 *     writes its output into the combine staging window ("out_tok", the
 *     combine_in view), and combine gathers those rows back, weighted;
 *   - section "Mega-MoE: mega-kernel co-design with FlyDSL": dispatch, expert
 *     GEMM and combine fused into one kernel launch;
 *   - section "GEMM + all-to-all fusion": GEMM -> A2A and A2A -> GEMM on the
 *     same windows (sym_gemm_a2a, sym_a2a_gemm);
 * and the "MORI CCO Guide", sections "1. Concepts" (device communicator
 * passed by value into kernels) and "3. Memory and Windows" (collective
 * registration at identical offsets).
 *
 * Here the W "ranks" are W logical slots carved at identical offsets inside
 * ONE device allocation; a cross-slot store is a plain global store to
 * base + slot * per_rank_size + offset.
 *
 * Conventions for every call:
 *   - All pointers named dev_* or documented as device pointers must point to
 *     device memory of the current CUDA device; the library never allocates,
 *     frees or copies to/from host memory except in sym_heap_status (which
 *     reads one status word) -- the caller owns every buffer.  The library's
 *     own resources are a static device array (moe_dispatch_layout_noalloc)
 *     and, for sym_a2a_gemm's copy-engine form, two side streams and three
 *     events per device, created on first use and kept for the process.
 *   - bf16 tensors are passed as uint16_t bit patterns, row-major, contiguous.
 *   - All compute calls are asynchronous on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream) and never synchronise the host.  Calls on
 *     one heap must run one after another on the GPU (one stream, or streams
 *     ordered by events): they share its windows and the work counters in
 *     its control window, which every launch leaves at zero when it ends.
 *   - Return value: SYM_OK (0) or a negative SYM_E* code, detected
 *     synchronously (bad argument, too small a heap, launch failure).
 *     Conditions found on the device while a kernel runs (a bounded wait that
 *     expired, a row beyond capacity) are OR-ed into the heap's status word
 *     and read with sym_heap_status; no kernel traps or aborts.
 *
 * Shapes (moe_shape): W = world slots, T = tokens per slot, N = W*T global
 * tokens (global token g = s*T + t lives on slot s), H = hidden, I = expert
 * intermediate size, E = experts, E/W experts per slot (expert e lives on
 * slot e / (E/W)), k = top-k.  Limits: E % W == 0, 1 <= k <= min(E, 32),
 * E <= 1024, H % 128 == 0, I % 128 == 0, H, I <= 65536.
 *
 * Accuracy: the expert FFN accumulates in fp32 on the tensor cores, whose
 * additions into the accumulator truncate.  Against an exact (fp64)
 * reference, bf16 outputs stay within 2e-2 * max(1, |ref|) per element and
 * 1e-2 relative L2 for K = H or I up to 16384 with weights ~N(0, 0.02).  At
 * K = 65536 with weights that large, |h| reaches ~200 and the truncation
 * over 4096 MMAs moves a few y elements in 10^4 just past that per-element
 * bound (relative L2 stays ~1e-3); the bound holds there for weights scaled
 * like a trained layer (about 1/sqrt(H): gate/up ~N(0, 0.0025) was checked).
 */
#ifndef SYMMOE_H
#define SYMMOE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *symmoe_stream_t; /* == cudaStream_t */

/* ---- status codes -------------------------------------------------------- */
#define SYM_OK 0
#define SYM_EINVAL (-1)    /* bad shape, pointer, alignment or argument        */
#define SYM_ENOSPACE (-2)  /* heap (or a window of it) too small for the call  */
#define SYM_ECUDA (-3)     /* a CUDA runtime call or kernel launch failed      */
#define SYM_ETIMEOUT (-4)  /* (status word) a bounded device wait expired      */
#define SYM_EOVERFLOW (-5) /* (status word) a row index beyond its window      */
#define SYM_ENOTSUP (-6)   /* not supported on this device (needs sm_103a)     */

/* bits of the device status word */
#define SYM_STATUS_TIMEOUT 0x1
#define SYM_STATUS_OVERFLOW 0x2

/* rows covered by one dispatch ready counter (per slot, per row block) */
#define SYM_ROWS_PER_FLAG 128
/* tokens per dispatch counting chunk */
#define SYM_COUNT_CHUNK 128

typedef struct moe_shape {
  int32_t world;           /* W */
  int32_t tokens_per_slot; /* T */
  int32_t hidden;          /* H */
  int32_t inter;           /* I */
  int32_t num_experts;     /* E */
  int32_t topk;            /* k */
} moe_shape;

/*
 * sym_heap: the symmetric heap descriptor.  Plain old data, passed BY VALUE
 * into every kernel (the device-communicator rule of the CCO guide).  Every
 * off_* is a byte offset inside EACH slot; window w of slot d is at
 * base + d * per_rank_size + off_w.  Per-slot windows:
 *   recv_x    [cap][H] bf16  dispatched token rows ("disp_out")
 *   y         [cap][H] bf16  expert outputs ("out_tok", combine_in view)
 *   h         [cap][I] bf16  SwiGLU intermediate of the expert FFN
 *   recv_pair [cap] int32    g*k + j of the pair that filled each row
 *   recv_w    [cap] fp32     routing weight of that pair
 *   pos       [T][k] int32   receive row of each of this slot's own pairs
 *                            (the "routing" handle combine uses)
 *   signal area: cnt [E/W] int32, recv_off [E/W] int32, total_recv int32,
 *                status int32 (slot 0's is the heap status word),
 *                ready [ceil(cap/128)] uint32 (rows landed per 128-row block)
 *   scratch (used in slot 0 only): dispatch chunk histograms, fused-kernel
 *                control block.
 * Every window is followed by a guard band of at least SYM_GUARD_BYTES that
 * no call reads or writes (sym_heap_windows gives each window's extent), so
 * a caller or a test can fill the bands with a pattern and check it after a
 * call.  Counts the kernels read back from the signal area are checked
 * against the window capacity: an expert whose rows [recv_off, recv_off +
 * cnt) or a slot whose total_recv do not fit in [0, cap) is skipped and
 * SYM_STATUS_OVERFLOW is raised (a corrupted or stale signal area never
 * sends a store past a window).
 * Receive rows are grouped by expert (ascending) inside a slot; inside one
 * expert they are in (source slot, token, k) order.
 */
#define SYM_GUARD_BYTES 1024
#define SYM_HEAP_WINDOWS 13
typedef struct sym_heap {
  uint64_t base;          /* device address of slot 0                          */
  uint64_t per_rank_size; /* slot stride in bytes (multiple of align)          */
  uint64_t bytes;         /* W * per_rank_size                                 */
  uint64_t cap;           /* receive rows per slot = N * min(k, E/W)           */
  uint64_t off_recv_x, off_y, off_h, off_recv_pair, off_recv_w, off_pos;
  uint64_t off_cnt, off_recv_off, off_total, off_status, off_ready;
  uint64_t off_hist;      /* chunk histograms, E * ceil(N/32) int32            */
  uint64_t off_ctrl;      /* fused-kernel counters and per-tile readiness      */
  uint32_t num_ready;     /* ready counters per slot = ceil(cap / 128)         */
  uint32_t epoch;         /* bumped by every dispatch / pipeline call          */
  uint32_t wait_timeout_us; /* bound on every device-side wait (default 2 s)   */
  uint32_t reserved;
  moe_shape s;
} sym_heap;

/*
 * sym_heap_bytes: size of the heap a shape needs.
 *   align: slot stride granularity in bytes (power of two >= 256; 0 = 2 MiB).
 *          align = 1<<32 reproduces the CCO kernel's 4 GiB-multiple stride.
 *   per_rank_size (out, may be NULL), total_bytes (out, may be NULL).
 * Host only.  Returns SYM_OK or SYM_EINVAL.
 */
int sym_heap_bytes(const moe_shape *s, uint64_t align, uint64_t *per_rank_size,
                   uint64_t *total_bytes);

/*
 * sym_heap_init: carve the windows into a caller-owned device allocation
 * (collective "alloc + register" of the CCO guide, reduced to arithmetic:
 * same windows, same order, same offsets in every slot).
 *   dev_base: device pointer, 256-byte aligned, owned by the caller, at least
 *             sym_heap_bytes(...) bytes, whose contents are zero before the
 *             first call that uses the heap (e.g. cudaMemsetAsync(dev_base, 0,
 *             bytes)): the status word and the fused-kernel counters start
 *             from zero.  The library keeps no reference other than the copy
 *             in *out.
 *   out:      filled descriptor (epoch 0, wait_timeout_us 2,000,000).
 * Host only, no device access.  SYM_EINVAL on a bad shape or alignment,
 * SYM_ENOSPACE if bytes is too small.
 */
int sym_heap_init(const moe_shape *s, void *dev_base, uint64_t bytes, uint64_t align,
                  sym_heap *out);

/*
 * sym_heap_slot_ptr: base + slot * per_rank_size + offset (the peer address
 * of "What is MORI CCO?").  Returns NULL if slot or offset is out of range.
 */
void *sym_heap_slot_ptr(const sym_heap *h, int slot, uint64_t offset);

/*
 * sym_heap_windows: the extent of every window inside a slot, in layout
 * order (recv_x, y, h, recv_pair, recv_w, pos, cnt, recv_off, total_recv,
 * status, ready, hist, ctrl): offsets[i] and bytes[i] for the first
 * min(max_windows, SYM_HEAP_WINDOWS) windows.  The bytes between the end of
 * window i and the start of window i + 1 (and after the last window, up to
 * per_rank_size) are the guard bands, at least SYM_GUARD_BYTES each.  Not in
 * the pages: a checking aid (a layout with guard bands stands in for a
 * memory checker).  Host only.  Returns SYM_HEAP_WINDOWS, or SYM_EINVAL.
 */
int sym_heap_windows(const sym_heap *h, uint64_t *offsets, uint64_t *bytes, int max_windows);

/*
 * moe_route_topk: per token, the top-k of E fp32 logits (descending, ties to
 * the lower expert index) and softmax weights over the selected k.
 *   logits: device [N][E] fp32;  idx: device [N][k] int32 (out);
 *   w: device [N][k] fp32 (out).  The pages leave routing to the caller; this
 *   is the router that feeds moe_dispatch.
 */
int moe_route_topk(const sym_heap *h, const float *logits, int32_t *idx, float *w,
                   symmoe_stream_t stream);

/*
 * moe_router_logits: the router (gate) GEMM that produces the routing logits
 * from the token activations (the step before moe_route_topk; the pages take
 * the routing as given):
 *   logits[g][e] = sum_h x[g][h] * w_router[e][h],  fp32 accumulation on the
 *   tensor cores, fp32 output.
 *   x: device [N][H] bf16 (16-byte aligned);  w_router: device [E][H] bf16
 *   (16-byte aligned);  logits: device [N][E] fp32.  N, H, E from the heap's
 *   shape.  When there are fewer output tiles than CTA pairs, K is split
 *   across pairs: the fp32 partials go to slot 0's y window (the expert
 *   output, which holds nothing between a combine and the next expert FFN)
 *   and a second kernel adds them in split order, so the logits do not depend
 *   on the schedule.  The call must therefore not overlap an expert FFN or a
 *   combine on the same heap; it writes nothing else of the heap but the
 *   status word.
 * Returns SYM_OK, SYM_EINVAL (pointer/alignment) or SYM_ECUDA; asynchronous.
 */
int moe_router_logits(const sym_heap *h, const uint16_t *x, const uint16_t *w_router, float *logits,
                      symmoe_stream_t stream);

/*
 * moe_router_splits: the number of K splits moe_router_logits uses for this
 * heap's shape on the current device (1: one GEMM launch writing the logits;
 * S > 1: S partials in slot 0's y window and one reduction launch).  No
 * device work; host only apart from reading the device's SM count.
 *   splits: host int (out).
 * Returns SYM_OK, SYM_EINVAL (bad heap or NULL splits) or SYM_ECUDA.
 */
int moe_router_splits(const sym_heap *h, int *splits);

/*
 * moe_dispatch: the all-to-all scatter of "Zero-copy MoE dispatch".
 * Counts pairs per expert, builds receive offsets, and copies every token row
 * x[g] into slot (idx[g][j] / (E/W))'s recv_x window at its receive row
 * (16-byte vector stores), writing recv_pair / recv_w / pos and raising the
 * ready counters (release) of the row blocks it fills.
 *   x: device [N][H] bf16;  idx, w: device [N][k] (from moe_route_topk or the
 *   caller; every idx must be in [0, E) and the k experts of a token distinct).
 *   Bumps h->epoch.  Out-of-range rows are skipped and flagged
 *   SYM_STATUS_OVERFLOW in the status word.
 */
int moe_dispatch(sym_heap *h, const uint16_t *x, const int32_t *idx, const float *w,
                 symmoe_stream_t stream);

/*
 * moe_dispatch_ex: moe_dispatch with flags.  SYM_DISPATCH_DEDUP: the
 * rank-deduplicated dispatch (a reading of "Zero-copy MoE dispatch" in which
 * a token crosses to each destination slot once): every token row is stored
 * once per distinct destination slot, into that slot's staging rows (its y
 * window, rows ordered by token g; the y window holds nothing until the down
 * GEMM), and each slot then expands its staged rows to its expert rows
 * locally.  The windows the expert FFN and the combine read (recv_x,
 * recv_pair, recv_w, pos, counts, offsets, ready counters) come out
 * bit-identical to moe_dispatch's.  Scratch in the h windows (idle until the
 * gate/up GEMM).  Needs W <= 32 and h windows of at least
 * 4*(cap + W*ceil(N/32) + N*k) bytes (cap*I*2; true for I >= 128 and k <= 32
 * but checked): SYM_EINVAL otherwise, or for an unknown flag.
 */
#define SYM_DISPATCH_DEDUP 1
/*
 * SYM_DISPATCH_FP8: the FP8 dispatch with per-token scales (the blog's
 * dispatch carries scales, recv_s).  Each row crosses as OCP E4M3 codes (H
 * bytes instead of 2H) with one scale 2^e per token, the smallest power of
 * two with max|x| <= 448 * 2^e (so x / 2^e is exact; the codes round to
 * nearest, ties to even).  The codes of pair row p land in row p of the
 * destination slot's y window (H bytes a row), the scale in word p of its h
 * window (fp32); the slot multiplies back to bf16 (exact) into recv_x.  The
 * expert FFN then sees the dequantized rows: results differ from the bf16
 * dispatch by the E4M3 rounding of x.  Not with SYM_DISPATCH_DEDUP.
 */
#define SYM_DISPATCH_FP8 2
int moe_dispatch_ex(sym_heap *h, const uint16_t *x, const int32_t *idx, const float *w, int flags,
                    symmoe_stream_t stream);

/*
 * moe_expert_ffn: expert_gemm of "Zero-copy MoE dispatch", here a SwiGLU FFN
 * per expert on its received rows, in place on the heap:
 *   h = bf16(silu(recv_x Wg_e^T) * (recv_x Wu_e^T)),  y = bf16(h Wd_e^T),
 * fp32 accumulation on the tensor cores (tcgen05, TMEM, TMA).  Row counts are
 * read on the device (no host sync); before loading a row block the kernel
 * waits (bounded) for its dispatch ready counter.
 *   w_gate, w_up: device [E][I][H] bf16;  w_down: device [E][H][I] bf16.
 * Writes the h and y windows of every slot.
 */
int moe_expert_ffn(const sym_heap *h, const uint16_t *w_gate, const uint16_t *w_up,
                   const uint16_t *w_down, symmoe_stream_t stream);

/*
 * moe_expert_ffn_ex: moe_expert_ffn with flags (0: identical to it).
 *   SYM_FFN_WEIGHTED_ROWS: the routing weights move from the combine into the
 *     expert epilogue (a variant; the pages apply them where combine takes
 *     them): y[p] = bf16(recv_w[p] * (h Wd_e^T)[p]), the weight of the row's
 *     (token, k) pair, written by moe_dispatch, multiplying the fp32
 *     accumulators before the one rounding.  Pair with moe_combine_ex and
 *     SYM_COMBINE_UNWEIGHTED.
 * Any other flag bit: SYM_EINVAL.
 */
#define SYM_FFN_WEIGHTED_ROWS 1
int moe_expert_ffn_ex(const sym_heap *h, const uint16_t *w_gate, const uint16_t *w_up,
                      const uint16_t *w_down, int flags, symmoe_stream_t stream);

/*
 * moe_combine: the weighted all-to-all gather of "Zero-copy MoE dispatch":
 *   out[g] = bf16( sum_{j<k} w[g][j] * y[slot(idx[g][j])][pos[g][j]] ),
 * fp32 accumulation in j order.
 *   expert_out: NULL or the address of slot 0's y window -> zero copy (the
 *     data_ptr match of the pages).  Any other device pointer is read as a
 *     dense [W][cap][H] bf16 tensor whose rows [0, total_recv[d]) are first
 *     copied into the y windows (the pages' silent fallback copy; counted by
 *     moe_combine_fallback_copies), with the identical result.
 *   idx, w: device [N][k] as given to moe_dispatch;  out: device [N][H] bf16.
 */
int moe_combine(const sym_heap *h, const uint16_t *expert_out, const int32_t *idx,
                const float *w, uint16_t *out, symmoe_stream_t stream);

/*
 * moe_combine_ex: moe_combine with flags (0: identical to it).
 *   SYM_COMBINE_UNWEIGHTED: the rows already carry their weights
 *     (SYM_FFN_WEIGHTED_ROWS): out[g] = bf16(sum_{j<k} y[slot(idx[g][j])][pos[g][j]]),
 *     fp32 sum in j order; w is not read and may be NULL.
 * Any other flag bit: SYM_EINVAL.
 */
#define SYM_COMBINE_UNWEIGHTED 1
int moe_combine_ex(const sym_heap *h, const uint16_t *expert_out, const int32_t *idx,
                   const float *w, uint16_t *out, int flags, symmoe_stream_t stream);

/* Number of fallback copies moe_combine has made in this process. */
uint64_t moe_combine_fallback_copies(void);

/*
 * moe_pipeline: route -> dispatch -> expert FFN -> combine on one stream.
 *   mode bits:
 *   SYM_PIPE_FUSED (1): one persistent launch ("Mega-MoE"): expert tiles start
 *     as soon as the ready counters of their rows land; without it one launch
 *     per stage (7 kernels).
 *   SYM_PIPE_WEIGHTS_IN_FFN (2): routing weights applied in the expert
 *     epilogue and an unweighted combine (SYM_FFN_WEIGHTED_ROWS,
 *     SYM_COMBINE_UNWEIGHTED).
 *   SYM_PIPE_DEDUP (4): the staged pipeline with the rank-deduplicated
 *     dispatch (moe_dispatch_ex, SYM_DISPATCH_DEDUP); not with SYM_PIPE_FUSED.
 *   SYM_PIPE_FP8 (8): the staged pipeline with the FP8 dispatch
 *     (SYM_DISPATCH_FP8); not with SYM_PIPE_FUSED or SYM_PIPE_DEDUP.
 *   Any other bit: SYM_EINVAL.  mode 0 / 1 are the staged / fused pipeline.
 *   idx, w: device [N][k] outputs of the routing step; out: device [N][H].
 *   Bumps h->epoch.
 */
#define SYM_PIPE_FUSED 1
#define SYM_PIPE_WEIGHTS_IN_FFN 2
#define SYM_PIPE_DEDUP 4
#define SYM_PIPE_FP8 8
int moe_pipeline(sym_heap *h, const float *logits, const uint16_t *x, const uint16_t *w_gate,
                 const uint16_t *w_up, const uint16_t *w_down, int32_t *idx, float *w,
                 uint16_t *out, int mode, symmoe_stream_t stream);

/*
 * sym_heap_status: synchronises `stream`, reads the heap status word (slot 0)
 * into *status (SYM_STATUS_* bits) and, if clear != 0, resets it to 0.
 * Returns SYM_OK, SYM_EINVAL or SYM_ECUDA.
 */
int sym_heap_status(const sym_heap *h, int32_t *status, int clear, symmoe_stream_t stream);

/*
 * GEMM + all-to-all fusion, a second workload on the same heap (blog,
 * "Examples", "GEMM + all-to-all fusion": GEMM -> A2A with the epilogue
 * writing output tiles straight into the peers' windows; A2A -> GEMM
 * consuming remote K-shards as they arrive, polling ready counters; each
 * against a split pipeline).  One linear layer w [H][H] (bf16, [out][in],
 * 16-byte aligned) is shared by the W slots; fp32 accumulation on the tensor
 * cores, bf16 results.  mode: SYM_LA_FUSED for the fused form, 0 for the split
 * pipeline (same results, bit for bit).  Neither call may overlap a
 * dispatch, expert FFN or combine on the same heap (they share its windows).
 */
#define SYM_LA_FUSED 1
#define SYM_LA_COPY_ENGINES 2 /* with SYM_LA_FUSED, sym_a2a_gemm only */

/*
 * sym_gemm_a2a: GEMM -> A2A.  Slot s computes Y_s = x_s w^T for its rows
 * x_s = x[s*T, (s+1)*T), and the rows are exchanged all-to-all in W blocks of
 * B = T/W rows: row s*B + r of slot j's y window receives Y_s[j*B + r].
 *   x: device [N][H] bf16, 16-byte aligned.
 *   fused: the GEMM epilogue stores each row at its destination;
 *   split: the GEMM stores Y_s in rows [0, T) of slot s's recv_x window, then
 *   a copy kernel exchanges the blocks.
 * Requires T % W == 0.  Writes rows [0, T) of every y window (split: also of
 * every recv_x window).  Returns SYM_OK, SYM_EINVAL or SYM_ECUDA; async.
 */
int sym_gemm_a2a(const sym_heap *h, const uint16_t *x, const uint16_t *w, int mode,
                 symmoe_stream_t stream);

/*
 * sym_a2a_gemm: A2A -> GEMM.  Slot s holds the K-shard s (features
 * [s*H/W, (s+1)*H/W)) of all N tokens: z [W][N][H/W] bf16, 16-byte aligned
 * (z[s] plays slot s's window).  Slot j computes C_j = U_j w^T into rows
 * [0, T) of its y window, U_j = its tokens j*T + r with every feature (shard s
 * at columns [s*H/W, (s+1)*H/W)).
 *   mode SYM_LA_FUSED: the all-to-all is the GEMM's operand loads: a tile of
 *   slot j reads K shard s of its tokens straight from z[s] (nothing copied).
 *   mode SYM_LA_FUSED | SYM_LA_COPY_ENGINES: slot j's recv_x window receives
 *   its shards shard major, [W][T][H/W], by one cudaMemcpyAsync per (slot,
 *   shard) on the copy engines from the library's side streams, each followed
 *   by a stream write of 1 into word s of slot j's ready window; the GEMM runs
 *   at the same time and its producer waits (bounded) for a shard's word
 *   before it loads that K range.  A wait that expires sets
 *   SYM_STATUS_TIMEOUT.  The call is ordered on `stream` as a whole.  Needs W
 *   words in a ready window (SYM_ENOSPACE if the heap has fewer).
 *   mode 0 (split): an SM copy kernel into the same shard-major blocks, then
 *   the GEMM.
 * Requires H % (64*W) == 0 (whole K blocks per shard).  Returns SYM_OK,
 * SYM_EINVAL, SYM_ENOSPACE or SYM_ECUDA; async.
 */
int sym_a2a_gemm(const sym_heap *h, const uint16_t *z, const uint16_t *w, int mode,
                 symmoe_stream_t stream);

/*
 * moe_dispatch_layout_noalloc: the dispatch layout without a heap, for
 * callers that cannot allocate device memory (a plug-in whose host framework
 * hands it only its input and output buffers and owns every allocation, or a
 * process that fixes its device-memory footprint at start-up).  The pages
 * have no counterpart: their dispatch always runs on a registered window.
 * Computes, from the routing indices alone, what moe_dispatch writes into the
 * heap's signal area and pos windows:
 *   idx:        device [N][k] int32, N = world * tokens_per_slot; every index
 *               in [0, E) and the k of a token distinct (an index outside
 *               [0, E) is not counted and gets pos -1; so does every later
 *               copy of an expert that a token lists twice, which is counted
 *               once);
 *   cnt:        device [E] int32 (out): pairs per expert;
 *   recv_off:   device [E] int32 (out): first receive row of each expert in
 *               its slot;
 *   total_recv: device [W] int32 (out): rows each slot receives;
 *   pos:        device [N][k] int32 (out): receive row of every pair in its
 *               destination slot, in the same order as moe_dispatch.
 * Only s->world, tokens_per_slot, num_experts and topk are used.
 * Scratch: a library-owned __device__ array of SYM_NOALLOC_HIST_MAX int32
 * (1 MiB, on every device that loads the library, until exit) holding the
 * E * ceil(N/128) chunk histograms; larger shapes return SYM_ENOSPACE.  The
 * call makes no device allocation.  Its first call on a device looks up the
 * array's address (cudaGetSymbolAddress) with that device current; make that
 * first call before any stream capture.  The address is kept per device and
 * looked up again on the first call after the device's context changed (after
 * cudaDeviceReset): that call, too, must come before any capture (under
 * capture it returns SYM_EINVAL).  All calls share the array: calls that
 * overlap on the GPU race on it and give wrong results.
 * Asynchronous on `stream`; SYM_OK, SYM_EINVAL, SYM_ENOSPACE or SYM_ECUDA.
 */
#define SYM_NOALLOC_HIST_MAX (1 << 18)
int moe_dispatch_layout_noalloc(const moe_shape *s, const int32_t *idx, int32_t *cnt,
                                int32_t *recv_off, int32_t *total_recv, int32_t *pos,
                                symmoe_stream_t stream);

/* Static description of a SYM_* code (never NULL). */
const char *sym_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* SYMMOE_H */
