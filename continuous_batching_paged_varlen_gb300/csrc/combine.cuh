// Log-sum-exp merge of split-KV partials, run inside the split-KV kernels.
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
// No separate launch: every CTA that wrote partial rows publishes them
// (each writer fences its stores), then counts one arrival per row on the
// row's counter; the CTA whose arrival completes a row merges it at once,
// from L2, while other CTAs are still streaming keys. The counter goes back
// to zero in the same step, so the next launch of the plan starts clean.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "mb_device.cuh"
#include "mb_internal.h"

namespace mb {
namespace dev {

struct MergeArgs {
  const RowDesc* rows;           // the CTA's rows start at rows[0]
  const MergeRef* refs;          // and their merge references at refs[0]
  int32_t n_rows;
  int32_t* count;                // arrivals per combine entry (zero between launches)
  const float* part_o;           // [n_partials, D], normalised
  const float* part_lse;         // [n_partials], log2 domain
  int32_t n_q_heads;
  __nv_bfloat16* out;
  float* lse;                    // nullable, natural log
};

// Called by all kThreads threads of the CTA after a __syncthreads that
// follows every partial write (and its __threadfence) of this CTA.
// scratch: >= 4 * 129 words of shared memory nobody else uses any more.
template <int D, int kThreads>
__device__ __forceinline__ void merge_completed_rows(const MergeArgs& m, uint32_t* scratch) {
  static_assert(D % 4 == 0, "head dim");
  int* count_n = reinterpret_cast<int*>(scratch + 4 * 128);
  int4* list = reinterpret_cast<int4*>(scratch);  // [128] (out row, slot_begin, n_slots, -)
  const int tid = threadIdx.x;
  if (tid == 0) *count_n = 0;
  __syncthreads();
  if (tid < m.n_rows) {
    const MergeRef ref = m.refs[tid];
    if (ref.entry >= 0) {
      const RowDesc rd = m.rows[tid];
      if (atomicAdd(&m.count[ref.entry], 1) == ref.n_slots - 1) {
        m.count[ref.entry] = 0;  // every arrival of this launch is in: reset for the next
        list[atomicAdd(count_n, 1)] =
            make_int4(rd.q_index * m.n_q_heads + rd.q_head, ref.slot_begin, ref.n_slots, 0);
      }
    }
  }
  __syncthreads();
  const int nl = *count_n;
  if (nl == 0) return;
  // the other CTAs fenced their partials before arriving: order this CTA's
  // reads after the arrivals it observed (and read through L2 below)
  __threadfence();
  // one thread per (row, 4 head dims): every thread of a row derives the same
  // max and sum from the row's LSEs; slots in groups of 16 whose loads are
  // all in flight together, rescaled online between groups
  constexpr int Q4 = D / 4;
  constexpr int G = 16;
  for (int task = tid; task < nl * Q4; task += kThreads) {
    const int i = task / Q4, q4 = task - i * Q4;
    const int4 e = list[i];
    const float* lp = m.part_lse + e.y;
    const float4* op = reinterpret_cast<const float4*>(m.part_o + (int64_t)e.y * D) + q4;
    float M = -INFINITY, L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < e.z; s0 += G) {
      float x[G];
      float4 v[G];
#pragma unroll
      for (int u = 0; u < G; ++u) {
        const bool in = s0 + u < e.z;
        x[u] = in ? __ldcg(lp + s0 + u) : -INFINITY;
        v[u] = in ? __ldcg(op + (int64_t)(s0 + u) * Q4) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      float mc = x[0];
#pragma unroll
      for (int u = 1; u < G; ++u) mc = fmaxf(mc, x[u]);
      if (mc > M) {  // a partial with no visible key has LSE -inf and weight 0
        const float sc = M == -INFINITY ? 0.f : fast_exp2(M - mc);
        L *= sc;
        acc.x *= sc;
        acc.y *= sc;
        acc.z *= sc;
        acc.w *= sc;
        M = mc;
      }
#pragma unroll
      for (int u = 0; u < G; ++u) {
        const float f = x[u] == -INFINITY ? 0.f : fast_exp2(x[u] - M);
        L += f;
        acc.x = fmaf(f, v[u].x, acc.x);
        acc.y = fmaf(f, v[u].y, acc.y);
        acc.z = fmaf(f, v[u].z, acc.z);
        acc.w = fmaf(f, v[u].w, acc.w);
      }
    }
    const float il = L > 0.f ? 1.f / L : 0.f;
    uint2 pk;
    pk.x = pack_bf16x2(acc.x * il, acc.y * il);
    pk.y = pack_bf16x2(acc.z * il, acc.w * il);
    *reinterpret_cast<uint2*>(m.out + (int64_t)e.x * D + 4 * q4) = pk;
    if (q4 == 0 && m.lse) m.lse[e.x] = L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
  }
}

}  // namespace dev
}  // namespace mb
