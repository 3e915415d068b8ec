// route_topk.cu -- top-k routing with softmax over the selected k.
//
// The MORI CCO blog ("Zero-copy MoE dispatch -> expert -> combine") hands
// dispatch the routing indices and weights; this kernel produces them: per
// token, the k largest of E fp32 logits (descending, equal logits to the lower
// expert index) and w_j = exp(l_j - l_0) / sum_i exp(l_i - l_0).
//
// One warp per token.  Lane l holds logits l, l+32, ...; each of the k rounds
// takes every lane's best remaining candidate and reduces (value, index) over
// the warp with shuffles.  Logits are read once with coalesced 128-byte rows.
#include "symmoe_dev.cuh"

namespace symmoe {

template <int VPL>  // values per lane = ceil(E / 32)
__global__ void __launch_bounds__(256) route_topk_kernel(const float *__restrict__ logits,
                                                         int32_t *__restrict__ idx,
                                                         float *__restrict__ w, int n_tokens,
                                                         int n_experts, int k) {
  pdl_launch_dependents();  // the dispatch count may be scheduled (it waits for idx)
  const int lane = threadIdx.x & 31;
  const int g = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (g >= n_tokens) return;
  const float *row = logits + (size_t)g * n_experts;
  float v[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < n_experts ? __ldg(row + e) : -INFINITY;
  }
  uint32_t taken = 0;
  for (int i = 0; i < VPL; ++i)
    if (lane + 32 * i >= n_experts) taken |= 1u << i;

  float my_val = -INFINITY;  // lane j keeps the j-th selected logit
  int my_idx = -1;
  for (int r = 0; r < k; ++r) {
    // best remaining candidate of this lane (values are visited in ascending
    // expert index, so a strict '>' keeps the lower index on ties)
    float bv = -INFINITY;
    int be = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      if (!(taken & (1u << i)) && (v[i] > bv || be == 0x7fffffff)) {
        bv = v[i];
        be = lane + 32 * i;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oe = __shfl_xor_sync(0xffffffffu, be, off);
      if (ov > bv || (ov == bv && oe < be)) {
        bv = ov;
        be = oe;
      }
    }
    if ((be & 31) == lane && be != 0x7fffffff) taken |= 1u << (be >> 5);
    if (lane == r) {
      my_val = bv;
      my_idx = be;
    }
  }
  const float top = __shfl_sync(0xffffffffu, my_val, 0);
  float z = lane < k ? expf(my_val - top) : 0.f;
  float s = z;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane < k) {
    idx[(size_t)g * k + lane] = my_idx;
    w[(size_t)g * k + lane] = z / s;
  }
}

cudaError_t launch_route_topk(const sym_heap &h, const float *logits, int32_t *idx, float *w,
                              cudaStream_t st) {
  const int n = h.s.world * h.s.tokens_per_slot;
  const int e = h.s.num_experts;
  const int warps = 8;
  dim3 grid((n + warps - 1) / warps), block(32 * warps);
  const int vpl = (e + 31) / 32;
#define SYMMOE_ROUTE(V)                                                                   \
  case V:                                                                                 \
    route_topk_kernel<V><<<grid, block, 0, st>>>(logits, idx, w, n, e, h.s.topk);         \
    break;
  switch (vpl <= 1 ? 1 : vpl <= 2 ? 2 : vpl <= 4 ? 4 : vpl <= 8 ? 8 : vpl <= 16 ? 16 : 32) {
    SYMMOE_ROUTE(1)
    SYMMOE_ROUTE(2)
    SYMMOE_ROUTE(4)
    SYMMOE_ROUTE(8)
    SYMMOE_ROUTE(16)
    SYMMOE_ROUTE(32)
  }
#undef SYMMOE_ROUTE
  return cudaGetLastError();
}

}  // namespace symmoe
