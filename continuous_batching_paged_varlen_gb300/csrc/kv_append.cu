// KV append: scatter this iteration's K/V rows into their cache pages.
//
// "ORCA and chunked prefill", section 4: each layer appends its new K and V
// to the request's cache before the attention reads the whole prefix.
// "GLM-5.3 e2e token ledger", stage 4: the host decides, per new token, the
// page and slot it goes to (out_cache_loc); this kernel only moves bytes.
//
// One thread moves one 16-byte chunk of one (token, KV head) row of K and
// the same chunk of V, so a warp covers 2 (D = 128) or 4 (D = 64) rows with
// fully coalesced 16-byte loads and 256-byte (or 128-byte) contiguous stores
// into the page. The copy is bit-exact.
#include <cuda_runtime.h>

#include "../../include/mb.h"
#include "kernels.h"
#include "mb_device.cuh"

namespace mb {
namespace {

template <int D>
__global__ void __launch_bounds__(256) kv_append_kernel(
    uint4* __restrict__ kc, uint4* __restrict__ vc, const uint4* __restrict__ kn,
    const uint4* __restrict__ vn, const int32_t* __restrict__ slots, int32_t T, int32_t Hkv,
    int32_t ps_shift, int64_t n_slots, int32_t* status) {
  constexpr int CH = D / 8;  // 16-byte chunks per row
  const int64_t total = (int64_t)T * Hkv * CH;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    const int64_t row = i / CH;  // (t, h) row of k_new
    const int c = (int)(i - row * CH);
    const int32_t t = (int32_t)(row / Hkv);
    const int32_t h = (int32_t)(row - (int64_t)t * Hkv);
    const int32_t slot = __ldg(slots + t);
    if (slot < 0) continue;  // padding row
    if ((int64_t)slot >= n_slots) {
      if (c == 0 && h == 0) dev::set_status(status, MB_ERR_DEVICE_INDEX);
      continue;
    }
    const int32_t page = slot >> ps_shift;
    const int32_t s = slot & ((1 << ps_shift) - 1);
    const int64_t dst = ((((int64_t)page * Hkv + h) << ps_shift) + s) * CH + c;
    const uint4 kv = __ldg(kn + i);
    const uint4 vv = __ldg(vn + i);
    kc[dst] = kv;
    vc[dst] = vv;
  }
}

}  // namespace

cudaError_t launch_kv_append(void* k_cache, void* v_cache, const void* k_new,
                             const void* v_new, const int32_t* slots, int32_t T,
                             int32_t n_kv_heads, int32_t head_dim, int32_t page_size,
                             int32_t num_pages, int32_t* status, cudaStream_t s) {
  const int64_t chunks = (int64_t)T * n_kv_heads * (head_dim / 8);
  const int threads = 256;
  int64_t blocks = (chunks + threads - 1) / threads;
  const int64_t cap = 152 * 16;  // a few waves of the 152 SMs, then grid-stride
  if (blocks > cap) blocks = cap;
  const int ps_shift = __builtin_ctz((unsigned)page_size);
  const int64_t n_slots = (int64_t)num_pages * page_size;
  if (head_dim == 128)
    kv_append_kernel<128><<<(unsigned)blocks, threads, 0, s>>>(
        (uint4*)k_cache, (uint4*)v_cache, (const uint4*)k_new, (const uint4*)v_new, slots, T,
        n_kv_heads, ps_shift, n_slots, status);
  else
    kv_append_kernel<64><<<(unsigned)blocks, threads, 0, s>>>(
        (uint4*)k_cache, (uint4*)v_cache, (const uint4*)k_new, (const uint4*)v_new, slots, T,
        n_kv_heads, ps_shift, n_slots, status);
  return cudaGetLastError();
}

}  // namespace mb
