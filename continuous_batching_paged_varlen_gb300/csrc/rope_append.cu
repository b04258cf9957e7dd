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
// One block per token; a thread rotates one 16-byte unit at a time (8
// elements of a row's first half and the matching 8 of its second half, with
// their 8 angles), in fp32, rounded once to bf16. Q rows are rotated in place;
// K rows are rotated into their cache slot; V rows are copied bit for bit
// (16-byte chunks).
#include <cuda_runtime.h>
#include <math.h>

#include "../../include/mb.h"
#include "kernels.h"
#include "mb_device.cuh"

namespace mb {
namespace {

constexpr int kThreads = 128;

// 8 bf16 (one 16-byte chunk) <-> 8 floats
__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    f[2 * k] = dev::bf16_lo(w[k]);
    f[2 * k + 1] = dev::bf16_hi(w[k]);
  }
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  return make_uint4(dev::pack_bf16x2(f[0], f[1]), dev::pack_bf16x2(f[2], f[3]),
                    dev::pack_bf16x2(f[4], f[5]), dev::pack_bf16x2(f[6], f[7]));
}

template <int D>
__global__ void __launch_bounds__(kThreads) rope_append_kernel(
    __nv_bfloat16* __restrict__ q, __nv_bfloat16* __restrict__ kc, uint4* __restrict__ vc,
    const __nv_bfloat16* __restrict__ kn, const uint4* __restrict__ vn,
    const int32_t* __restrict__ positions, const int32_t* __restrict__ slots, int32_t Hq,
    int32_t Hkv, int32_t ps_shift, int64_t n_slots, const float* __restrict__ cos_sin,
    int32_t max_position, int32_t* status) {
  constexpr int HALF = D / 2;
  constexpr int RU = D / 16;  // rotation units per row: 8 elements of each half
  constexpr int CH = D / 8;   // 16-byte chunks per row
  // nothing here runs before the kernel ahead (which may read the cache or
  // q, or write k_new) is done
  dev::pdl_launch_dependents();
  dev::pdl_wait();
  const int t = blockIdx.x;
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
  const bool write_kv = slot >= 0;
  const int32_t page = write_kv ? slot >> ps_shift : 0;
  const int32_t off = write_kv ? slot & ((1 << ps_shift) - 1) : 0;
  const int64_t cache_base = (((int64_t)page * Hkv) << ps_shift) + off;  // head 0's page row
  const float* row = cos_sin + (int64_t)pos * D;
  // query rows (rotated in place), then K rows (rotated into the cache)
  const int n_rot = (Hq + (write_kv ? Hkv : 0)) * RU;
  for (int i = threadIdx.x; i < n_rot; i += kThreads) {
    const int r = i / RU, u = i - r * RU;
    const __nv_bfloat16* src;
    __nv_bfloat16* dst;
    if (r < Hq) {
      src = dst = q + ((int64_t)t * Hq + r) * D;
    } else {
      const int h = r - Hq;
      src = kn + ((int64_t)t * Hkv + h) * D;
      dst = kc + (cache_base + ((int64_t)h << ps_shift)) * D;
    }
    const uint4 lo_v = *reinterpret_cast<const uint4*>(src + 8 * u);
    const uint4 hi_v = *reinterpret_cast<const uint4*>(src + HALF + 8 * u);
    const float4 c0 = __ldg(reinterpret_cast<const float4*>(row + 8 * u));
    const float4 c1 = __ldg(reinterpret_cast<const float4*>(row + 8 * u + 4));
    const float4 s0 = __ldg(reinterpret_cast<const float4*>(row + HALF + 8 * u));
    const float4 s1 = __ldg(reinterpret_cast<const float4*>(row + HALF + 8 * u + 4));
    const float c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    const float sn[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    float x[8], y[8], xo[8], yo[8];
    unpack8(lo_v, x);
    unpack8(hi_v, y);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      xo[e] = fmaf(x[e], c[e], -y[e] * sn[e]);
      yo[e] = fmaf(y[e], c[e], x[e] * sn[e]);
    }
    *reinterpret_cast<uint4*>(dst + 8 * u) = pack8(xo);
    *reinterpret_cast<uint4*>(dst + HALF + 8 * u) = pack8(yo);
  }
  if (!write_kv) return;  // padding row (or flagged): no cache write
  // V: plain copy, 16-byte chunks
  const uint4* vsrc = vn + (int64_t)t * Hkv * CH;
  for (int c = threadIdx.x; c < Hkv * CH; c += kThreads) {
    const int h = c / CH, cc = c - h * CH;
    vc[(cache_base + ((int64_t)h << ps_shift)) * CH + cc] = __ldg(vsrc + c);
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
  return launch_programmatic(head_dim == 128 ? rope_append_kernel<128> : rope_append_kernel<64>,
                             dim3((unsigned)T), dim3(kThreads), 0, s, (__nv_bfloat16*)q,
                             (__nv_bfloat16*)k_cache, (uint4*)v_cache,
                             (const __nv_bfloat16*)k_new, (const uint4*)v_new, positions, slots,
                             n_q_heads, n_kv_heads, ps_shift, n_slots, cos_sin, max_position,
                             status);
}

}  // namespace mb
