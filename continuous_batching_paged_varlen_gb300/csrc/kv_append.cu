// KV append: scatter this iteration's K/V rows into their cache pages.
//
// "ORCA and chunked prefill", section 4: each layer appends its new K and V
// to the request's cache before the attention reads the whole prefix.
// "GLM-5.3 e2e token ledger", stage 4: the host decides, per new token, the
// page and slot it goes to (out_cache_loc); this kernel only moves bytes.
//
// One block per token: its Hkv rows of K and of V are contiguous in k_new /
// v_new and land in Hkv page rows of ps * D elements apart, so the block's
// threads walk the token's 16-byte chunks with 32-bit index math, four chunks
// of K and four of V in flight per thread. The copy is bit-exact.
#include <cuda_runtime.h>

#include "../../include/mb.h"
#include "kernels.h"
#include "mb_device.cuh"

namespace mb {
namespace {

constexpr int kThreads = 128;

template <int D>
__global__ void __launch_bounds__(kThreads) kv_append_kernel(
    uint4* __restrict__ kc, uint4* __restrict__ vc, const uint4* __restrict__ kn,
    const uint4* __restrict__ vn, const int32_t* __restrict__ slots, int32_t Hkv,
    int32_t ps_shift, int64_t n_slots, int32_t* status) {
  constexpr int CH = D / 8;  // 16-byte chunks per row
  const int t = blockIdx.x;
  const int32_t slot = __ldg(slots + t);
  if (slot < 0) return;  // padding row
  if ((int64_t)slot >= n_slots) {
    if (threadIdx.x == 0) dev::set_status(status, MB_ERR_DEVICE_INDEX);
    return;
  }
  const int32_t page = slot >> ps_shift;
  const int32_t off = slot & ((1 << ps_shift) - 1);
  const int n = Hkv * CH;  // chunks of one token's K (and of its V)
  const uint4* ksrc = kn + (int64_t)t * n;
  const uint4* vsrc = vn + (int64_t)t * n;
  // chunk c of head h goes to page row ((page * Hkv + h) << ps_shift) + off
  const int64_t base = (((int64_t)page * Hkv) << ps_shift) + off;
  constexpr int U = 4;
  for (int c0 = threadIdx.x; c0 < n; c0 += kThreads * U) {
    uint4 kv[U], vv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + u * kThreads;
      if (c < n) {
        kv[u] = __ldg(ksrc + c);
        vv[u] = __ldg(vsrc + c);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + u * kThreads;
      if (c < n) {
        const int h = c / CH, cc = c - h * CH;
        const int64_t dst = (base + ((int64_t)h << ps_shift)) * CH + cc;
        kc[dst] = kv[u];
        vc[dst] = vv[u];
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
  if (head_dim == 128)
    kv_append_kernel<128><<<(unsigned)T, kThreads, 0, s>>>(
        (uint4*)k_cache, (uint4*)v_cache, (const uint4*)k_new, (const uint4*)v_new, slots,
        n_kv_heads, ps_shift, n_slots, status);
  else
    kv_append_kernel<64><<<(unsigned)T, kThreads, 0, s>>>(
        (uint4*)k_cache, (uint4*)v_cache, (const uint4*)k_new, (const uint4*)v_new, slots,
        n_kv_heads, ps_shift, n_slots, status);
  return cudaGetLastError();
}

}  // namespace mb
