// combine.cu -- the weighted all-to-all gather of the zero-copy MoE pipeline.
//
// MORI CCO blog, "Zero-copy MoE dispatch -> expert -> combine": combine reads
// each token's expert outputs back from the owners' "out_tok" windows and
// applies the routing weights; when the expert already wrote into the
// combine_in view (matching data_ptr) no staging copy is made, otherwise the
// op silently copies first.  Both behaviours are here:
//   combine_kernel        out[g] = bf16(sum_j w[g,j] * y[slot_j][pos[g,j]]),
//                         fp32 fma in j order, 16-byte vector loads/stores,
//                         the loads of up to four sources in flight together;
//   stage_expert_out_kernel  the fallback copy of a caller's [W][cap][H]
//                         expert output into the y windows (rows < total).
#include "symmoe_dev.cuh"

namespace symmoe {

constexpr int COMBINE_THREADS = 128;

// G: sources whose loads are issued together before they are accumulated
template <int G>
__global__ void __launch_bounds__(COMBINE_THREADS)
    combine_kernel(sym_heap h, const int32_t *__restrict__ idx, const float *__restrict__ w,
                   uint4 *__restrict__ out, int unit_weights) {
  __shared__ const uint4 *src_s[32];
  __shared__ float w_s[32];
  const int E = h.s.num_experts, k = h.s.topk, T = h.s.tokens_per_slot, H = h.s.hidden;
  const int E_loc = E / h.s.world;
  const int g = blockIdx.x;
  const int tid = threadIdx.x;
  const int nvec = H / 8;
  if (tid < k) {
    const int e = idx[(size_t)g * k + tid];
    const int p = win<int32_t>(h, g / T, h.off_pos)[(size_t)(g % T) * k + tid];
    const uint4 *src = nullptr;
    if (e >= 0 && e < E && p >= 0 && (uint64_t)p < h.cap)
      src = win<const uint4>(h, e / E_loc, h.off_y) + (size_t)p * nvec;
    src_s[tid] = src;
    w_s[tid] = unit_weights ? 1.f : w[(size_t)g * k + tid];  // 1: rows already weighted
  }
  __syncthreads();
  uint4 *dst = out + (size_t)g * nvec;
  constexpr int U = 2;  // vectors per thread per pass
  for (int c0 = tid; c0 < nvec; c0 += U * COMBINE_THREADS) {
    float acc[U][8];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[u][i] = 0.f;
    for (int j0 = 0; j0 < k; j0 += G) {
      // issue the loads of G sources first, then accumulate in j order
      uint4 v[G][U];
#pragma unroll
      for (int jj = 0; jj < G; ++jj) {
        const uint4 *sp = j0 + jj < k ? src_s[j0 + jj] : nullptr;
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int c = c0 + u * COMBINE_THREADS;
          v[jj][u] = (sp && c < nvec) ? __ldg(sp + c) : make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int jj = 0; jj < G; ++jj) {
        if (j0 + jj >= k || !src_s[j0 + jj]) continue;
        const float wj = w_s[j0 + jj];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const uint4 x = v[jj][u];
          acc[u][0] = fmaf(wj, bf16lo(x.x), acc[u][0]);
          acc[u][1] = fmaf(wj, bf16hi(x.x), acc[u][1]);
          acc[u][2] = fmaf(wj, bf16lo(x.y), acc[u][2]);
          acc[u][3] = fmaf(wj, bf16hi(x.y), acc[u][3]);
          acc[u][4] = fmaf(wj, bf16lo(x.z), acc[u][4]);
          acc[u][5] = fmaf(wj, bf16hi(x.z), acc[u][5]);
          acc[u][6] = fmaf(wj, bf16lo(x.w), acc[u][6]);
          acc[u][7] = fmaf(wj, bf16hi(x.w), acc[u][7]);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + u * COMBINE_THREADS;
      if (c < nvec) {
        uint4 o;
        o.x = pack_bf16x2(acc[u][0], acc[u][1]);
        o.y = pack_bf16x2(acc[u][2], acc[u][3]);
        o.z = pack_bf16x2(acc[u][4], acc[u][5]);
        o.w = pack_bf16x2(acc[u][6], acc[u][7]);
        dst[c] = o;
      }
    }
  }
}

// Fallback: copy rows [0, total_recv[d]) of a dense [W][cap][H] expert output
// into the y windows.  grid = (blocks, W).
__global__ void __launch_bounds__(256)
    stage_expert_out_kernel(sym_heap h, const uint4 *__restrict__ expert_out) {
  const int d = blockIdx.y;
  const int nvec = h.s.hidden / 8;
  const int total = checked_total(h, d, blockIdx.x == 0 && threadIdx.x == 0);
  const uint4 *src = expert_out + (size_t)d * h.cap * nvec;
  uint4 *dst = win<uint4>(h, d, h.off_y);
  const size_t n = (size_t)total * nvec;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    dst[i] = __ldg(src + i);
}

cudaError_t launch_combine(const sym_heap &h, const uint16_t *expert_out, const int32_t *idx,
                           const float *w, uint16_t *out, int unit_weights, int num_sms, cudaStream_t st) {
  const int N = h.s.world * h.s.tokens_per_slot;
  if (expert_out) {
    dim3 grid(num_sms * 2, h.s.world);
    stage_expert_out_kernel<<<grid, 256, 0, st>>>(h, reinterpret_cast<const uint4 *>(expert_out));
  }
  if (h.s.topk <= 2)
    combine_kernel<2><<<N, COMBINE_THREADS, 0, st>>>(h, idx, w, reinterpret_cast<uint4 *>(out), unit_weights);
  else
    combine_kernel<4><<<N, COMBINE_THREADS, 0, st>>>(h, idx, w, reinterpret_cast<uint4 *>(out), unit_weights);
  return cudaGetLastError();
}

}  // namespace symmoe
