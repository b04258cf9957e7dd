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

// One arrival on a split row's counter, by a thread whose partial (or
// share of one) is already fenced. `add` of `total` arrivals completes the
// row; the completing thread gets true and puts the counter back to zero
// (every other arrival of this launch is in), so the next launch starts
// clean.
__device__ __forceinline__ bool arrive_partial(int32_t* count, int add, int total) {
  if (atomicAdd(count, add) + add != total) return false;
  *count = 0;
  return true;
}

// Merge the listed rows (x: flat output row q_index * Hq + q_head, y: first
// partial slot, z: partials): all kThreads threads of the CTA, one per
// (row, 4 head dims); every thread of a row derives the same max and sum
// from the row's LSEs; slots in groups of 16 whose loads are all in flight
// together, rescaled online between groups. The caller fences between the
// arrivals it observed and this call; partials are read through L2.
template <int D, int kThreads>
__device__ __forceinline__ void merge_listed_rows(const int4* list, int nl, const float* part_o,
                                                  const float* part_lse, __nv_bfloat16* out,
                                                  float* lse) {
  static_assert(D % 4 == 0, "head dim");
  constexpr int Q4 = D / 4;
  constexpr int G = 16;
  for (int task = threadIdx.x; task < nl * Q4; task += kThreads) {
    const int i = task / Q4, q4 = task - i * Q4;
    const int4 e = list[i];
    const float* lp = part_lse + e.y;
    const float4* op = reinterpret_cast<const float4*>(part_o + (int64_t)e.y * D) + q4;
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
    *reinterpret_cast<uint2*>(out + (int64_t)e.x * D + 4 * q4) = pk;
    if (q4 == 0 && lse) lse[e.x] = L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
  }
}

// The whole step for a kernel whose rows' partials may have several writer
// threads: called by all kThreads threads after a __syncthreads that follows
// every partial write (and its __threadfence) of this CTA; thread r counts
// row r. scratch: >= 4 * 129 words of shared memory nobody else uses.
// With `pre`, thread r < n_rows passes its row's merge reference and flat
// output row (q_index * Hq + q_head), loaded earlier, so that no dependent
// global load sits on the CTA's exit path; without, they are read here.
template <int D, int kThreads>
__device__ __forceinline__ void merge_completed_rows(const MergeArgs& m, uint32_t* scratch,
                                                     bool pre = false, MergeRef my_ref = {},
                                                     int32_t my_out_row = 0) {
  int* count_n = reinterpret_cast<int*>(scratch + 4 * 128);
  int4* list = reinterpret_cast<int4*>(scratch);
  const int tid = threadIdx.x;
  if (tid == 0) *count_n = 0;
  __syncthreads();
  if (tid < m.n_rows) {
    const MergeRef ref = pre ? my_ref : m.refs[tid];
    if (ref.entry >= 0) {
      int32_t orow = my_out_row;
      if (!pre) {
        const RowDesc rd = m.rows[tid];
        orow = rd.q_index * m.n_q_heads + rd.q_head;
      }
      if (arrive_partial(m.count + ref.entry, 1, ref.n_slots))
        list[atomicAdd(count_n, 1)] = make_int4(orow, ref.slot_begin, ref.n_slots, 0);
    }
  }
  __syncthreads();
  const int nl = *count_n;
  if (nl == 0) return;
  // the other CTAs fenced their partials before arriving: order this CTA's
  // reads after the arrivals it observed
  __threadfence();
  merge_listed_rows<D, kThreads>(list, nl, m.part_o, m.part_lse, m.out, m.lse);
}

}  // namespace dev
}  // namespace mb
