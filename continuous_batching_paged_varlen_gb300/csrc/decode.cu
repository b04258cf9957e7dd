// Split-KV attention for rows with few new queries (decode steps, small
// chunks) and for shared-prefix cascade groups.
//
// One CTA owns up to 8 query rows that all read the same KV head -- the g
// query heads of a GQA group ("How To Scale Your Model notes (7-8)",
// section 3: g queries share one KV head, so KV bytes are read once for all
// g of them) and, for a cascade group, the rows of every request that shares
// the prefix pages ("How To Scale Your Model notes (7-8)", section 3: load a
// common KV block once, apply it to all the requests' queries, keep each
// request's own softmax state). The CTA walks the key range [k_begin, k_end)
// of one block-table row and keeps an online softmax (running max m, running
// sum l, accumulator) per row. Each key is masked by the row's own
// visibility bound (S0 + i + 1, "How To Scale Your Model notes (7-8)",
// section 2), so decode rows (m = 1) see everything and multi-row requests
// get the causal diagonal block.
//
// The result is either the final row (bf16 out + LSE) or, when the key
// range was split, a normalised partial (fp32 O, log2-domain LSE) that the
// combine kernel merges.
//
// Work split inside the CTA: 4 warps take interleaved 32-key blocks; in a
// block lane = key for the q.k products (q rows live in shared memory as
// fp32 pre-scaled by scale * log2 e, K rows are read straight from the
// page), then lane = 4 (or 2) consecutive head dims for p.V. The four warps'
// (m, l, acc) are merged through shared memory at the end.
#include <cuda_runtime.h>
#include <math.h>

#include "../../include/mb.h"
#include "kernels.h"
#include "mb_device.cuh"

namespace mb {
namespace {

constexpr int kR = kRowsPerDecodeItem;
constexpr int kWarps = 4;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int D>
__global__ void __launch_bounds__(kWarps * 32) splitkv_kernel(const DecodeArgs a,
                                                              const int ps_shift) {
  constexpr int DL = D / 32;  // head dims per lane in the p.V phase
  __shared__ __align__(16) float q_s[kR][D];
  __shared__ float m_s[kWarps][kR];
  __shared__ float l_s[kWarps][kR];
  __shared__ __align__(16) float acc_s[kWarps][kR][D];
  __shared__ RowDesc rd[kR];

  const DecodeItem it = a.items[blockIdx.x];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nr = it.n_rows;
  if (threadIdx.x < kR) {
    RowDesc d;
    d.q_index = 0;
    d.q_head = 0;
    d.vis_end = 0;  // unused rows see nothing
    d.dst = -1;
    if ((int)threadIdx.x < nr) d = a.rows[it.row_begin + threadIdx.x];
    rd[threadIdx.x] = d;
  }
  __syncthreads();
  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
  for (int i = threadIdx.x; i < kR * D; i += kWarps * 32) {
    const int r = i / D, d = i - r * D;
    float v = 0.f;
    if (r < nr)
      v = __bfloat162float(q[((int64_t)rd[r].q_index * a.n_q_heads + rd[r].q_head) * D + d]) *
          a.scale_log2;
    q_s[r][d] = v;
  }
  int vis[kR];
#pragma unroll
  for (int r = 0; r < kR; ++r) vis[r] = rd[r].vis_end;
  __syncthreads();

  float m[kR], l[kR], acc[kR][DL];
#pragma unroll
  for (int r = 0; r < kR; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int e = 0; e < DL; ++e) acc[r][e] = 0.f;
  }

  const int32_t* btrow = a.block_table + (int64_t)it.bt_row * a.max_blocks;
  const int ps_mask = (1 << ps_shift) - 1;
  const uint4* kc = static_cast<const uint4*>(a.k_cache);
  const __nv_bfloat16* vc = static_cast<const __nv_bfloat16*>(a.v_cache);

  for (int kb = it.k_begin + warp * 32; kb < it.k_end; kb += 32 * kWarps) {
    const int j = kb + lane;
    int valid = j < it.k_end;
    int64_t rowidx = 0;
    if (valid) {
      const int page = __ldg(btrow + (j >> ps_shift));
      if ((unsigned)page >= (unsigned)a.num_pages) {
        dev::set_status(a.status, MB_ERR_DEVICE_INDEX);
        valid = 0;
      } else {
        rowidx = (((int64_t)page * a.n_kv_heads + it.kv_head) << ps_shift) + (j & ps_mask);
      }
    }
    // ---- scores of this lane's key against every row
    float s[kR];
#pragma unroll
    for (int r = 0; r < kR; ++r) s[r] = 0.f;
    if (valid) {
      const uint4* kp = kc + rowidx * (D / 8);
      uint4 kr[D / 8];
#pragma unroll
      for (int c = 0; c < D / 8; ++c) kr[c] = __ldg(kp + c);
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const float k0 = dev::bf16_lo(kr[c].x), k1 = dev::bf16_hi(kr[c].x);
        const float k2 = dev::bf16_lo(kr[c].y), k3 = dev::bf16_hi(kr[c].y);
        const float k4 = dev::bf16_lo(kr[c].z), k5 = dev::bf16_hi(kr[c].z);
        const float k6 = dev::bf16_lo(kr[c].w), k7 = dev::bf16_hi(kr[c].w);
#pragma unroll
        for (int r = 0; r < kR; ++r) {
          const float4 qa = *reinterpret_cast<const float4*>(&q_s[r][c * 8]);
          const float4 qb = *reinterpret_cast<const float4*>(&q_s[r][c * 8 + 4]);
          s[r] = fmaf(qa.x, k0, s[r]);
          s[r] = fmaf(qa.y, k1, s[r]);
          s[r] = fmaf(qa.z, k2, s[r]);
          s[r] = fmaf(qa.w, k3, s[r]);
          s[r] = fmaf(qb.x, k4, s[r]);
          s[r] = fmaf(qb.y, k5, s[r]);
          s[r] = fmaf(qb.z, k6, s[r]);
          s[r] = fmaf(qb.w, k7, s[r]);
        }
      }
    }
    // ---- online softmax update (m is warp-uniform, l is kept per lane)
    float p[kR];
#pragma unroll
    for (int r = 0; r < kR; ++r) {
      const float sr = (valid && j < vis[r]) ? s[r] : -INFINITY;
      const float mn = fmaxf(m[r], warp_max(sr));
      if (mn == -INFINITY) {  // nothing visible to this row yet
        p[r] = 0.f;
        continue;
      }
      const float alpha = dev::fast_exp2(m[r] - mn);
      p[r] = dev::fast_exp2(sr - mn);
      l[r] = l[r] * alpha + p[r];
#pragma unroll
      for (int e = 0; e < DL; ++e) acc[r][e] *= alpha;
      m[r] = mn;
    }
    // ---- p . V, lanes over head dims
    const int nk = min(32, it.k_end - kb);
#pragma unroll 4
    for (int jj = 0; jj < nk; ++jj) {
      const int64_t vr = __shfl_sync(0xffffffffu, rowidx, jj);
      const int vv = __shfl_sync(0xffffffffu, valid, jj);
      float vf[DL];
      if (vv) {
        if constexpr (DL == 4) {
          const uint2 u = __ldg(reinterpret_cast<const uint2*>(vc + vr * D) + lane);
          vf[0] = dev::bf16_lo(u.x);
          vf[1] = dev::bf16_hi(u.x);
          vf[2] = dev::bf16_lo(u.y);
          vf[3] = dev::bf16_hi(u.y);
        } else {
          const uint32_t u = __ldg(reinterpret_cast<const uint32_t*>(vc + vr * D) + lane);
          vf[0] = dev::bf16_lo(u);
          vf[1] = dev::bf16_hi(u);
        }
      } else {
#pragma unroll
        for (int e = 0; e < DL; ++e) vf[e] = 0.f;
      }
#pragma unroll
      for (int r = 0; r < kR; ++r) {
        const float pj = __shfl_sync(0xffffffffu, p[r], jj);
#pragma unroll
        for (int e = 0; e < DL; ++e) acc[r][e] = fmaf(pj, vf[e], acc[r][e]);
      }
    }
  }

  // ---- merge the four warps
#pragma unroll
  for (int r = 0; r < kR; ++r) {
    const float lr = warp_sum(l[r]);
    if (lane == 0) {
      m_s[warp][r] = m[r];
      l_s[warp][r] = lr;
    }
#pragma unroll
    for (int e = 0; e < DL; ++e) acc_s[warp][r][lane * DL + e] = acc[r][e];
  }
  __syncthreads();
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
  for (int i = threadIdx.x; i < nr * D; i += kWarps * 32) {
    const int r = i / D, d = i - r * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, m_s[w][r]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float f = dev::fast_exp2(m_s[w][r] - M);
        L = fmaf(l_s[w][r], f, L);
        O = fmaf(acc_s[w][r][d], f, O);
      }
    }
    const float o = L > 0.f ? O / L : 0.f;
    const float lse2 = L > 0.f ? M + log2f(L) : -INFINITY;
    const RowDesc rw = rd[r];
    if (rw.dst < 0) {
      const int64_t orow = (int64_t)rw.q_index * a.n_q_heads + rw.q_head;
      out[orow * D + d] = __float2bfloat16_rn(o);
      if (d == 0 && a.lse) a.lse[orow] = lse2 * kLn2;
    } else {
      a.part_o[(int64_t)rw.dst * D + d] = o;
      if (d == 0) a.part_lse[rw.dst] = lse2;
    }
  }
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s, bool overlap_previous) {
  if (a.n_items <= 0) return cudaSuccess;
  const int ps_shift = __builtin_ctz((unsigned)a.page_size);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.n_items);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap_previous ? 1 : 0;
  if (a.head_dim == 128) return cudaLaunchKernelEx(&cfg, splitkv_kernel<128>, a, ps_shift);
  return cudaLaunchKernelEx(&cfg, splitkv_kernel<64>, a, ps_shift);
}

}  // namespace mb
