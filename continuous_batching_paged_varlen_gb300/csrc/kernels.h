// Launchers of the device kernels (host side; defined next to each kernel).
#pragma once

#include <cuda.h>
#include <cuda_runtime_api.h>
#include <stdint.h>

#include <atomic>

#include "mb_internal.h"

namespace mb {

// Launch attributes a kernel needs once per device (its dynamic shared
// memory size, a device property): `setup` runs on the first launch on each
// of the first 64 devices, and on every launch beyond them.
struct OncePerDevice {
  std::atomic<uint64_t> done{0};
  template <class F>
  cudaError_t run(F&& setup) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = setup(dev);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
    return e;
  }
};

// KV append scatter (kv_append.cu).
cudaError_t launch_kv_append(void* k_cache, void* v_cache, const void* k_new,
                             const void* v_new, const int32_t* slots, int32_t T,
                             int32_t n_kv_heads, int32_t head_dim, int32_t page_size,
                             int32_t num_pages, int32_t* status, cudaStream_t s);

// KV append into an fp8 (e4m3) cache with per-row fp32 scales (kv_append.cu).
cudaError_t launch_kv_append_fp8(void* k8, void* v8, float* ks, float* vs, const void* k_new,
                                 const void* v_new, const int32_t* slots, int32_t T,
                                 int32_t n_kv_heads, int32_t head_dim, int32_t page_size,
                                 int32_t num_pages, int32_t* status, cudaStream_t s);

// Fused rotary embedding + KV append (rope_append.cu).
cudaError_t launch_rope_append(void* q, void* k_cache, void* v_cache, const void* k_new,
                               const void* v_new, const int32_t* positions,
                               const int32_t* slots, int32_t T, int32_t n_q_heads,
                               int32_t n_kv_heads, int32_t head_dim, int32_t page_size,
                               int32_t num_pages, const float* cos_sin, int32_t max_position,
                               int32_t* status, cudaStream_t s);

// Split-KV / cascade kernel (decode.cu): partial or final rows.
struct DecodeArgs {
  const DecodeItem* items;
  const RowDesc* rows;
  int32_t n_items;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_table;
  int32_t max_blocks, n_q_heads, n_kv_heads, head_dim, page_size, num_pages;
  float scale_log2;  // softmax scale * log2(e)
  void* out;
  float* lse;        // nullable
  float* part_o;
  float* part_lse;   // log2 domain
  // split rows: per row its merge reference, and one arrival counter per
  // combine entry (zero between launches); the CTA completing a row merges
  // it (combine.cuh). combine_count null: no split rows.
  const MergeRef* row_merge;
  int32_t* combine_count;
  int32_t* status;
  const CUtensorMap* k_map;  // host copies, passed by value to the kernel
  const CUtensorMap* v_map;
};
// overlap_previous: launch with programmatic stream serialization, so the
// kernel may start while the previous kernel on the stream (which must not
// produce anything it reads) is still running.
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s, bool overlap_previous = false);

// Split-KV / cascade kernel over an fp8 (e4m3) cache with per-row fp32
// scales (decode_fp8.cu). Same work lists and outputs as launch_decode.
struct DecodeFp8Args {
  const DecodeItem* items;
  const RowDesc* rows;
  int32_t n_items;
  const void* q;
  const void* k8;         // e4m3 codes [pages, Hkv, ps, D]
  const void* v8;
  const float* k_scale;   // [pages, Hkv, ps]
  const float* v_scale;
  const int32_t* block_table;
  int32_t max_blocks, n_q_heads, n_kv_heads, head_dim, page_size, num_pages;
  float scale_log2;
  void* out;
  float* lse;
  float* part_o;
  float* part_lse;
  const MergeRef* row_merge;  // as in DecodeArgs
  int32_t* combine_count;
  int32_t* status;
  const CUtensorMap* k_map;  // uint8 codes [rows, D], box D x ps, swizzled (host copy)
};
cudaError_t launch_decode_fp8(const DecodeFp8Args& a, cudaStream_t s);

// tcgen05 prefill kernel (prefill.cu).
struct PrefillArgs {
  const PrefillItem* items;
  int32_t n_items;
  const int32_t* block_table;
  int32_t max_blocks, n_q_heads, n_kv_heads, head_dim, page_size, num_pages;
  float scale_log2;
  void* out;
  float* lse;
  int32_t* status;
  const CUtensorMap* q_map;  // host copies, passed by value to the kernel
  const CUtensorMap* k_map;
  const CUtensorMap* v_map;
};
cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t s);

}  // namespace mb
