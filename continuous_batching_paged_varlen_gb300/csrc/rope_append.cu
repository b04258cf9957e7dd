// Fused rotary embedding + KV append.
//
// "GLM-5.3 e2e token ledger", the per-layer forward and its fusion table: the
// norm, RoPE and the KV write run as one kernel that already holds the layer's
// q and k, so the cache write costs no extra pass over K. The rotation is the
// rotary embedding of the Llama-2 family: the pairs (x_i, x_{i + D/2}) of a
// head vector are rotated by the angle p * theta_i of the token's position p,
// theta_i = base^(-2 i / D). The caller supplies the angle table (cos and sin
// of p * theta_i per position; mb_rope_table builds it). The append itself is
// the one of "ORCA and chunked prefill", section 4 (slot per new row from the
// host, "GLM-5.3 e2e token ledger", stage 4).
//
// One block per token, one warp per head row at a time: lane l owns D/64
// consecutive elements of the first half and the matching elements of the
// second half, computes the rotation in fp32 and rounds once to bf16. Q rows
// are rotated in place; K rows are rotated into their cache slot; V rows are
// copied bit for bit (16-byte chunks).
#include <cuda_runtime.h>
#include <math.h>

#include "../../include/mb.h"
#include "kernels.h"
#include "mb_device.cuh"

namespace mb {
namespace {

template <int D>
__global__ void __launch_bounds__(128) rope_append_kernel(
    __nv_bfloat16* __restrict__ q, __nv_bfloat16* __restrict__ kc, uint4* __restrict__ vc,
    const __nv_bfloat16* __restrict__ kn, const uint4* __restrict__ vn,
    const int32_t* __restrict__ positions, const int32_t* __restrict__ slots, int32_t Hq,
    int32_t Hkv, int32_t ps_shift, int64_t n_slots, const float* __restrict__ cos_sin,
    int32_t max_position, int32_t* status) {
  constexpr int HALF = D / 2;
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t pos = __ldg(positions + t);
  if (pos < 0 || pos >= max_position) {
    if (threadIdx.x == 0) dev::set_status(status, MB_ERR_DEVICE_INDEX);
    return;
  }
  int32_t slot = __ldg(slots + t);
  if ((int64_t)slot >= n_slots) {
    if (threadIdx.x == 0) dev::set_status(status, MB_ERR_DEVICE_INDEX);
    slot = -1;
  }
  // lane l owns elements [E l, E l + E) of each half (E = D / 64: one bf16
  // pair for D = 128, one element for D = 64) and their angles
  constexpr int E = D / 64;
  float c[E], s[E];
  const float* row = cos_sin + (int64_t)pos * D + E * lane;
#pragma unroll
  for (int k = 0; k < E; ++k) {
    c[k] = __ldg(row + k);
    s[k] = __ldg(row + HALF + k);
  }
  auto rotate_row = [&](const __nv_bfloat16* src, __nv_bfloat16* dst) {
    float x[E], y[E];
    if constexpr (E == 2) {
      const uint32_t lo = *reinterpret_cast<const uint32_t*>(src + 2 * lane);
      const uint32_t hi = *reinterpret_cast<const uint32_t*>(src + HALF + 2 * lane);
      x[0] = dev::bf16_lo(lo);
      x[1] = dev::bf16_hi(lo);
      y[0] = dev::bf16_lo(hi);
      y[1] = dev::bf16_hi(hi);
      *reinterpret_cast<uint32_t*>(dst + 2 * lane) =
          dev::pack_bf16x2(fmaf(x[0], c[0], -y[0] * s[0]), fmaf(x[1], c[1], -y[1] * s[1]));
      *reinterpret_cast<uint32_t*>(dst + HALF + 2 * lane) =
          dev::pack_bf16x2(fmaf(y[0], c[0], x[0] * s[0]), fmaf(y[1], c[1], x[1] * s[1]));
    } else {
      x[0] = __bfloat162float(src[lane]);
      y[0] = __bfloat162float(src[HALF + lane]);
      dst[lane] = __float2bfloat16_rn(fmaf(x[0], c[0], -y[0] * s[0]));
      dst[HALF + lane] = __float2bfloat16_rn(fmaf(y[0], c[0], x[0] * s[0]));
    }
  };
  // query rows, in place
  for (int h = warp; h < Hq; h += 4) {
    __nv_bfloat16* r = q + ((int64_t)t * Hq + h) * D;
    rotate_row(r, r);
  }
  if (slot < 0) return;  // padding row (or flagged): no cache write
  const int32_t page = slot >> ps_shift;
  const int32_t off = slot & ((1 << ps_shift) - 1);
  for (int h = warp; h < Hkv; h += 4) {
    const int64_t dst_row = (((int64_t)page * Hkv + h) << ps_shift) + off;
    rotate_row(kn + ((int64_t)t * Hkv + h) * D, kc + dst_row * D);
  }
  // V: plain copy, 16-byte chunks
  constexpr int CH = D / 8;
  for (int i = threadIdx.x; i < Hkv * CH; i += blockDim.x) {
    const int h = i / CH, cidx = i - h * CH;
    const int64_t dst_row = (((int64_t)page * Hkv + h) << ps_shift) + off;
    vc[dst_row * CH + cidx] = __ldg(vn + ((int64_t)t * Hkv + h) * CH + cidx);
  }
}

}  // namespace

cudaError_t launch_rope_append(void* q, void* k_cache, void* v_cache, const void* k_new,
                               const void* v_new, const int32_t* positions,
                               const int32_t* slots, int32_t T, int32_t n_q_heads,
                               int32_t n_kv_heads, int32_t head_dim, int32_t page_size,
                               int32_t num_pages, const float* cos_sin, int32_t max_position,
                               int32_t* status, cudaStream_t s) {
  const int ps_shift = __builtin_ctz((unsigned)page_size);
  const int64_t n_slots = (int64_t)num_pages * page_size;
  if (head_dim == 128)
    rope_append_kernel<128><<<(unsigned)T, 128, 0, s>>>(
        (__nv_bfloat16*)q, (__nv_bfloat16*)k_cache, (uint4*)v_cache,
        (const __nv_bfloat16*)k_new, (const uint4*)v_new, positions, slots, n_q_heads,
        n_kv_heads, ps_shift, n_slots, cos_sin, max_position, status);
  else
    rope_append_kernel<64><<<(unsigned)T, 128, 0, s>>>(
        (__nv_bfloat16*)q, (__nv_bfloat16*)k_cache, (uint4*)v_cache,
        (const __nv_bfloat16*)k_new, (const uint4*)v_new, positions, slots, n_q_heads,
        n_kv_heads, ps_shift, n_slots, cos_sin, max_position, status);
  return cudaGetLastError();
}

}  // namespace mb
