// Log-sum-exp merge of split-KV partials.
//
// A row whose key range was cut into chunks (split-KV, or a shared prefix
// read by the cascade plus the request's own suffix) has one normalised
// partial (O_c, LSE_c) per chunk. The exact softmax over the union is
//   O = sum_c exp(LSE_c - LSE*) O_c / sum_c exp(LSE_c - LSE*),
//   LSE = LSE* + log sum_c exp(LSE_c - LSE*),   LSE* = max_c LSE_c,
// the merge that FlashDecoding-style kernels use (named as prior art in the
// "Roadmap" post's list and in "Prefill/Decode disaggregation", section 3).
// Partials carry base-2 LSEs; the final LSE is written in natural log.
//
// One warp per output row; lanes over head dims, so every partial row is
// read with coalesced loads, and the slots' weights computed one per lane.
#include <cuda_runtime.h>
#include <math.h>

#include "../../include/mb.h"
#include "kernels.h"
#include "mb_device.cuh"

namespace mb {
namespace {

constexpr float kLn2 = 0.6931471805599453f;

template <int D>
__global__ void __launch_bounds__(256) combine_kernel(const CombineEntry* __restrict__ ent,
                                                      int32_t n, const float* __restrict__ part_o,
                                                      const float* __restrict__ part_lse,
                                                      int32_t Hq, __nv_bfloat16* __restrict__ out,
                                                      float* __restrict__ lse) {
  constexpr int DL = D / 32;
  // launched to overlap the split-KV kernel's tail: wait here until that grid
  // has finished and its partials are visible (returns at once otherwise)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (w >= n) return;
  const CombineEntry e = ent[w];
  float M = -INFINITY;
  for (int s = lane; s < e.n_slots; s += 32) M = fmaxf(M, part_lse[e.slot_begin + s]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float L = 0.f, O[DL];
#pragma unroll
  for (int k = 0; k < DL; ++k) O[k] = 0.f;
  if (M != -INFINITY) {
    for (int s0 = 0; s0 < e.n_slots; s0 += 32) {
      // the weights of up to 32 slots, one per lane; the rows of four slots
      // are loaded before any is accumulated (the loop is latency-bound)
      const int ns = min(32, e.n_slots - s0);
      const float wl = lane < ns ? dev::fast_exp2(part_lse[e.slot_begin + s0 + lane] - M) : 0.f;
      L += wl;
      const float* base = part_o + (int64_t)(e.slot_begin + s0) * D + lane;
      int s = 0;
      for (; s + 4 <= ns; s += 4) {
        float v[4][DL];
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int k = 0; k < DL; ++k) v[u][k] = base[(int64_t)(s + u) * D + 32 * k];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float f = __shfl_sync(0xffffffffu, wl, s + u);
#pragma unroll
          for (int k = 0; k < DL; ++k) O[k] = fmaf(f, v[u][k], O[k]);
        }
      }
      for (; s < ns; ++s) {
        const float f = __shfl_sync(0xffffffffu, wl, s);
#pragma unroll
        for (int k = 0; k < DL; ++k) O[k] = fmaf(f, base[(int64_t)s * D + 32 * k], O[k]);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  }
  const int64_t orow = (int64_t)e.q_index * Hq + e.q_head;
  const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
  for (int k = 0; k < DL; ++k) out[orow * D + lane + 32 * k] = __float2bfloat16_rn(O[k] * inv);
  if (lane == 0 && lse) lse[orow] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
}

}  // namespace

cudaError_t launch_combine(const CombineEntry* entries, int32_t n, const float* part_o,
                           const float* part_lse, int32_t head_dim, int32_t n_q_heads,
                           void* out, float* lse, cudaStream_t s, bool overlap_previous) {
  if (n <= 0) return cudaSuccess;
  const int warps = 8;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((n + warps - 1) / warps));
  cfg.blockDim = dim3(warps * 32);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap_previous ? 1 : 0;
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out);
  if (head_dim == 128)
    return cudaLaunchKernelEx(&cfg, combine_kernel<128>, entries, n, part_o, part_lse,
                              n_q_heads, o, lse);
  return cudaLaunchKernelEx(&cfg, combine_kernel<64>, entries, n, part_o, part_lse, n_q_heads,
                            o, lse);
}

}  // namespace mb
