// KV append: scatter this iteration's K/V rows into their cache pages.
//
// "ORCA and chunked prefill", section 4: each layer appends its new K and V
// to the request's cache before the attention reads the whole prefix.
// "GLM-5.3 e2e token ledger", stage 4: the host decides, per new token, the
// page and slot it goes to (out_cache_loc); this kernel only moves bytes.
//
// A block takes a group of consecutive tokens (one token when a token's K
// row set is at least kThreads * U chunks, several when rows are short, so a
// block always moves a few KB) and walks the group's 16-byte chunks; K and V
// rows of a token are contiguous in k_new / v_new and land in Hkv page rows
// ps * D elements apart. Blocks stride over the groups, so a long append
// (a whole prompt's history) is not bound by the rate at which blocks can
// be launched. Four chunks of K and four of V are in flight per thread. The
// copy is bit-exact.
#include <cuda_runtime.h>

#include "../../include/mb.h"
#include "kernels.h"
#include "mb_device.cuh"

namespace mb {
namespace {

constexpr int kThreads = 128;
constexpr int kUnroll = 4;
constexpr int kMaxBlocks = 8192;
constexpr int kMinBlocks = 2 * 152;  // two blocks per SM before tokens are grouped

template <int D>
__global__ void __launch_bounds__(kThreads) kv_append_kernel(
    uint4* __restrict__ kc, uint4* __restrict__ vc, const uint4* __restrict__ kn,
    const uint4* __restrict__ vn, const int32_t* __restrict__ slots, int32_t T, int32_t Hkv,
    int32_t ps_shift, int64_t n_slots, int32_t group, int32_t* status) {
  constexpr int CH = D / 8;  // 16-byte chunks per row
  constexpr int U = kUnroll;
  const int n = Hkv * CH;    // chunks of one token's K (and of its V)
  const int32_t off_mask = (1 << ps_shift) - 1;
  // the attention kernel behind may set up meanwhile; nothing here runs
  // before the kernel ahead (which may read the cache or write k_new) is done
  dev::pdl_launch_dependents();
  dev::pdl_wait();
  for (int64_t t0 = (int64_t)blockIdx.x * group; t0 < T; t0 += (int64_t)gridDim.x * group) {
    const int nt = (int)(T - t0 < group ? T - t0 : group);
    const int m = nt * n;  // chunks of this group
    const uint4* ksrc = kn + t0 * n;
    const uint4* vsrc = vn + t0 * n;
    for (int f0 = threadIdx.x; f0 < m; f0 += kThreads * U) {
      uint4 kv[U], vv[U];
      int64_t dst[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int f = f0 + u * kThreads;
        dst[u] = -1;
        if (f < m) {
          const int tl = f / n, c = f - tl * n;
          const int32_t slot = __ldg(slots + t0 + tl);
          if (slot < 0) continue;  // padding row
          if ((int64_t)slot >= n_slots) {
            if (c == 0) dev::set_status(status, MB_ERR_DEVICE_INDEX);
            continue;
          }
          // chunk c (head h, chunk cc of the row) goes to page row
          // ((page * Hkv + h) << ps_shift) + off
          const int h = c / CH, cc = c - h * CH;
          const int64_t row = (((int64_t)(slot >> ps_shift) * Hkv + h) << ps_shift) + (slot & off_mask);
          dst[u] = row * CH + cc;
          kv[u] = __ldg(ksrc + f);
          vv[u] = __ldg(vsrc + f);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (dst[u] >= 0) {
          kc[dst[u]] = kv[u];
          vc[dst[u]] = vv[u];
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_kv_append(void* k_cache, void* v_cache, const void* k_new,
                             const void* v_new, const int32_t* slots, int32_t T,
                             int32_t n_kv_heads, int32_t head_dim, int32_t page_size,
                             int32_t num_pages, int32_t* status, cudaStream_t s) {
  const int ps_shift = __builtin_ctz((unsigned)page_size);
  const int64_t n_slots = (int64_t)num_pages * page_size;
  const int n = n_kv_heads * (head_dim / 8);
  // short appends (a decode step's few hundred rows) keep one token per
  // block so that they still spread over every SM; long ones group tokens
  // until a block moves kThreads * kUnroll chunks
  const int group_max = n >= kThreads * kUnroll ? 1 : (kThreads * kUnroll) / n;
  const int64_t by_size = (int64_t)T / kMinBlocks;
  const int group = by_size < 1 ? 1 : (by_size < group_max ? (int)by_size : group_max);
  const int64_t groups = ((int64_t)T + group - 1) / group;
  const unsigned grid = (unsigned)(groups < kMaxBlocks ? groups : kMaxBlocks);
  return launch_programmatic(head_dim == 128 ? kv_append_kernel<128> : kv_append_kernel<64>,
                             dim3(grid), dim3(kThreads), 0, s, (uint4*)k_cache, (uint4*)v_cache,
                             (const uint4*)k_new, (const uint4*)v_new, slots, T, n_kv_heads,
                             ps_shift, n_slots, group, status);
}

}  // namespace mb

// ---------------------------------------------------------------------------
// fp8 (e4m3) cache: quantize while appending.
//
// "GLM-5.3 e2e token ledger", the KV layout paragraphs: FP8 K/V with FP32
// scales kept next to the data (one per 128 values), read together by the
// attention kernel to dequantize. Here: one fp32 scale per (token, KV head)
// row, scale = amax(|row|) / 448, code = e4m3(x / scale) rounded to nearest
// (ties to even), saturating; a zero row gets scale 0 and zero codes. The
// quotient is one IEEE fp32 division, so the codes are reproducible.
// D/8 lanes per row, 8 consecutive values each (one 16-byte load, one
// 8-byte store of codes), so a warp quantizes 32/(D/8) rows at once and the
// amax reduction and the per-row address work are shared by fewer values'
// worth of instructions (the kernel is issue-bound, not bound by HBM).
namespace mb {
namespace {

template <int D>
__global__ void __launch_bounds__(128) kv_append_fp8_kernel(
    uint8_t* __restrict__ k8, uint8_t* __restrict__ v8, float* __restrict__ ks,
    float* __restrict__ vs, const __nv_bfloat16* __restrict__ kn,
    const __nv_bfloat16* __restrict__ vn, const int32_t* __restrict__ slots, int32_t Hkv,
    int32_t ps_shift, int64_t n_slots, int32_t* status) {
  constexpr int kL = D / 8;       // lanes per row: 8 values (one 16-byte load) each
  constexpr int kRpw = 32 / kL;   // rows a warp handles at once
  dev::pdl_launch_dependents();
  dev::pdl_wait();
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane / kL, l = lane % kL;
  const int32_t slot = __ldg(slots + t);
  if (slot < 0) return;
  if ((int64_t)slot >= n_slots) {
    if (threadIdx.x == 0) dev::set_status(status, MB_ERR_DEVICE_INDEX);
    return;
  }
  const int32_t page = slot >> ps_shift;
  const int32_t off = slot & ((1 << ps_shift) - 1);
  const int n_rows = 2 * Hkv;
  for (int row0 = warp * kRpw; row0 < n_rows; row0 += 4 * kRpw) {
    const int row = row0 + sub;
    const bool valid = row < n_rows;
    const bool is_v = row >= Hkv;
    const int h = is_v ? row - Hkv : row;
    uint4 raw = make_uint4(0u, 0u, 0u, 0u);
    if (valid)
      raw = __ldg(reinterpret_cast<const uint4*>((is_v ? vn : kn) + ((int64_t)t * Hkv + h) * D) + l);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
    float x[8];
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[2 * e] = dev::bf16_lo(w[e]);
      x[2 * e + 1] = dev::bf16_hi(w[e]);
      amax = dev::fmax3(amax, fabsf(x[2 * e]), fabsf(x[2 * e + 1]));
    }
#pragma unroll
    for (int o = kL / 2; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float scale = __fdiv_rn(amax, 448.0f);
    uint32_t code[2] = {0u, 0u};
    if (scale > 0.f) {
      #pragma unroll
      for (int e = 0; e < 8; e += 2) {
        uint16_t pair;
        const float qa = __fdiv_rn(x[e], scale), qb = __fdiv_rn(x[e + 1], scale);
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(qb), "f"(qa));
        code[e >> 2] |= (uint32_t)pair << (8 * (e & 3));
      }
    }
    if (valid) {
      const int64_t drow = (((int64_t)page * Hkv + h) << ps_shift) + off;
      *reinterpret_cast<uint2*>((is_v ? v8 : k8) + drow * D + 8 * l) = make_uint2(code[0], code[1]);
      if (l == 0) (is_v ? vs : ks)[drow] = scale;
    }
  }
}

// Staging for the tensor-core prefill over an fp8 cache: each block turns
// one (staged page, KV head) tile of K or V codes into bf16 values,
// decode(code) * scale in fp32 rounded once to bf16, at the same place of
// the staging region (laid out like the cache, staging page ids). Slots past
// a request's last key are converted too (whatever they hold): the prefill
// kernel masks those keys and zeroes their V rows.
template <int D>
__global__ void __launch_bounds__(128) dequant_pages_kernel(
    const uint4* __restrict__ k8, const uint4* __restrict__ v8, const float* __restrict__ ks,
    const float* __restrict__ vs, const int32_t* __restrict__ stage_pages, int32_t Hkv,
    int32_t ps_shift, int32_t num_pages, uint4* __restrict__ kst, uint4* __restrict__ vst,
    int32_t n_stage, int32_t* status) {
  constexpr int CPR = D / 16;  // 16-code chunks per row
  dev::pdl_launch_dependents();
  dev::pdl_wait();  // the codes may come from the append just ahead
  const int sp = blockIdx.x / (2 * Hkv);
  const int rest = blockIdx.x - sp * 2 * Hkv;
  const bool is_v = rest >= Hkv;
  const int h = is_v ? rest - Hkv : rest;
  const int32_t page = __ldg(stage_pages + sp);
  if ((unsigned)page >= (unsigned)num_pages) {
    if (threadIdx.x == 0) dev::set_status(status, MB_ERR_DEVICE_INDEX);
    return;
  }
  const int ps = 1 << ps_shift;
  const int64_t src_row = ((int64_t)page * Hkv + h) << ps_shift;  // first row of the tile
  const int64_t dst_row = ((int64_t)sp * Hkv + h) << ps_shift;
  const uint4* codes = (is_v ? v8 : k8) + src_row * CPR;
  const float* scales = (is_v ? vs : ks) + src_row;
  uint4* dst = (is_v ? vst : kst) + dst_row * (2 * CPR);
  for (int c = threadIdx.x; c < ps * CPR; c += 128) {
    const float sc = __ldg(scales + c / CPR);
    const uint4 w = __ldg(codes + c);
    const uint32_t words[4] = {w.x, w.y, w.z, w.w};
    uint32_t out[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float a, b, cc, dd;
      dev::f16x2_to_f32x2(dev::e4m3x2_to_f16x2(words[q]), a, b);
      dev::f16x2_to_f32x2(dev::e4m3x2_to_f16x2(words[q] >> 16), cc, dd);
      out[2 * q] = dev::pack_bf16x2(a * sc, b * sc);
      out[2 * q + 1] = dev::pack_bf16x2(cc * sc, dd * sc);
    }
    dst[2 * c] = make_uint4(out[0], out[1], out[2], out[3]);
    dst[2 * c + 1] = make_uint4(out[4], out[5], out[6], out[7]);
  }
}

}  // namespace

cudaError_t launch_dequant_pages(const void* k8, const void* v8, const float* ks,
                                 const float* vs, const int32_t* stage_pages, int32_t n_stage,
                                 int32_t n_kv_heads, int32_t head_dim, int32_t page_size,
                                 int32_t num_pages, void* k_stage, void* v_stage,
                                 int32_t* status, cudaStream_t s) {
  if (n_stage <= 0) return cudaSuccess;
  const int ps_shift = __builtin_ctz((unsigned)page_size);
  const unsigned grid = (unsigned)n_stage * 2u * (unsigned)n_kv_heads;
  return launch_programmatic(
      head_dim == 128 ? dequant_pages_kernel<128> : dequant_pages_kernel<64>, dim3(grid),
      dim3(128), 0, s, (const uint4*)k8, (const uint4*)v8, ks, vs, stage_pages, n_kv_heads,
      ps_shift, num_pages, (uint4*)k_stage, (uint4*)v_stage, n_stage, status);
}

cudaError_t launch_kv_append_fp8(void* k8, void* v8, float* ks, float* vs, const void* k_new,
                                 const void* v_new, const int32_t* slots, int32_t T,
                                 int32_t n_kv_heads, int32_t head_dim, int32_t page_size,
                                 int32_t num_pages, int32_t* status, cudaStream_t s) {
  const int ps_shift = __builtin_ctz((unsigned)page_size);
  const int64_t n_slots = (int64_t)num_pages * page_size;
  return launch_programmatic(
      head_dim == 128 ? kv_append_fp8_kernel<128> : kv_append_fp8_kernel<64>, dim3((unsigned)T),
      dim3(128), 0, s, (uint8_t*)k8, (uint8_t*)v8, ks, vs, (const __nv_bfloat16*)k_new,
      (const __nv_bfloat16*)v_new, slots, n_kv_heads, ps_shift, n_slots, status);
}

}  // namespace mb
