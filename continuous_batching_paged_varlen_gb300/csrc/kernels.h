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

// fp8 cache pages -> bf16 staging pages for the prefill kernel (kv_append.cu):
// staged page i (cache page stage_pages[i]) of every KV head, K and V.
cudaError_t launch_dequant_pages(const void* k8, const void* v8, const float* ks,
                                 const float* vs, const int32_t* stage_pages, int32_t n_stage,
                                 int32_t n_kv_heads, int32_t head_dim, int32_t page_size,
                                 int32_t num_pages, void* k_stage, void* v_stage,
                                 int32_t* status, cudaStream_t s);

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
  // 1: the kernel ahead on the stream is the same forward's prefill kernel,
  // which writes nothing this kernel reads: no wait before the work, and the
  // last CTA to finish waits for that kernel (counted in done_counter), so
  // this grid completes after it. 0: the kernel ahead may have written q,
  // this step's K/V rows or the outputs: Q, keys >= an item's k_new and
  // every global write wait for it; history keys stream at once.
  int32_t after_prefill;
  int32_t* done_counter;
  // 1: the build that spreads a row's keys over copies in the softmax warps
  // (CTAs of <= 32 rows with long key ranges); 0: one thread per row
  int32_t copies;
  const CUtensorMap* k_map;  // host copies, passed by value to the kernel
  const CUtensorMap* v_map;
};
// overlap_previous: launch with programmatic stream serialization, so the
// kernel may start while the previous kernel on the stream is running (the
// waits above keep it correct).
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
  int32_t after_prefill;      // as in DecodeArgs (the fp8 kernel is launched
  int32_t* done_counter;      // behind the prefill only, never behind an append)
  const CUtensorMap* k_map;  // uint8 codes [rows, D], box D x ps, swizzled (host copy)
  int32_t max_rows;          // largest n_rows of the items (<= 8 with D = 128: few-row form)
};
cudaError_t launch_decode_fp8(const DecodeFp8Args& a, cudaStream_t s, bool overlap_previous = false);

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
  int32_t max_ctas;          // persistent grid cap (0: one CTA per SM)
  const CUtensorMap* q_map;  // host copies, passed by value to the kernel
  const CUtensorMap* k_map;
  const CUtensorMap* v_map;
};
cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t s);

}  // namespace mb
