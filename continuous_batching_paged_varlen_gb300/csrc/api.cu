// extern "C" entry points that launch work: mb_kv_append and the two forward
// calls. Argument checks happen here on the host; nothing is enqueued when a
// check fails.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>

#include <mutex>

#include "../../include/mb.h"
#include "kernels.h"
#include "mb_device.cuh"
#include "mb_internal.h"
#include "plan_impl.h"

using namespace mb;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// Tiled tensor map; dims/strides innermost first, strides for dims 1.. in
// bytes. Default: 128-byte-swizzled bf16.
bool make_map(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
              const cuuint64_t* strides, const cuuint32_t* box,
              CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  cuuint32_t elem[3] = {1, 1, 1};
  CUresult r = fn(map, dtype, (cuuint32_t)rank, const_cast<void*>(base), dims, strides, box, elem,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

constexpr float kLog2e = 1.4426950408889634f;

// One CTA waits, with the kernels' bounded wait, on an mbarrier that nothing
// completes: the wait gives up after its time limit, flags MB_ERR_TIMEOUT and
// the kernel returns.
__global__ void wait_timeout_kernel(int32_t* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    dev::mbar_init(&bar, 1);
    abort_flag = 0;
    dev::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) dev::mbar_wait(&bar, 0u, &abort_flag, status);
}

}  // namespace

extern "C" {

mb_status_t mb_selftest_wait_timeout(int32_t* status_dev, cudaStream_t stream) {
  if (!status_dev || (reinterpret_cast<uintptr_t>(status_dev) & 3)) return MB_ERR_INVALID_ARG;
  wait_timeout_kernel<<<1, 32, 0, stream>>>(status_dev);
  return cudaGetLastError() == cudaSuccess ? MB_OK : MB_ERR_CUDA;
}

mb_status_t mb_kv_append(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                         const int32_t* slot_mapping, int32_t T, const mb_config_t* cfg,
                         int32_t* status_dev, cudaStream_t stream) {
  mb_status_t st = validate_config(cfg);
  if (st != MB_OK) return st;
  if (T < 0) return MB_ERR_INVALID_ARG;
  if (T == 0) return MB_OK;
  if (!k_cache || !v_cache || !k_new || !v_new || !slot_mapping) return MB_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_new) || !aligned16(v_new) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 3) ||
      (reinterpret_cast<uintptr_t>(status_dev) & 3))
    return MB_ERR_INVALID_ARG;
  cudaError_t e = launch_kv_append(k_cache, v_cache, k_new, v_new, slot_mapping, T,
                                   cfg->n_kv_heads, cfg->head_dim, cfg->page_size,
                                   cfg->num_pages, status_dev, stream);
  return e == cudaSuccess ? MB_OK : MB_ERR_CUDA;
}

mb_status_t mb_kv_append_fp8(void* k_codes, void* v_codes, float* k_scale, float* v_scale,
                             const void* k_new, const void* v_new, const int32_t* slot_mapping,
                             int32_t T, const mb_config_t* cfg, int32_t* status_dev,
                             cudaStream_t stream) {
  mb_status_t st = validate_config(cfg);
  if (st != MB_OK) return st;
  if (T < 0) return MB_ERR_INVALID_ARG;
  if (T == 0) return MB_OK;
  if (!k_codes || !v_codes || !k_scale || !v_scale || !k_new || !v_new || !slot_mapping)
    return MB_ERR_INVALID_ARG;
  if (!aligned16(k_codes) || !aligned16(v_codes) || !aligned16(k_scale) || !aligned16(v_scale) ||
      !aligned16(k_new) || !aligned16(v_new) || (reinterpret_cast<uintptr_t>(slot_mapping) & 3) ||
      (reinterpret_cast<uintptr_t>(status_dev) & 3))
    return MB_ERR_INVALID_ARG;
  cudaError_t e = launch_kv_append_fp8(k_codes, v_codes, k_scale, v_scale, k_new, v_new,
                                       slot_mapping, T, cfg->n_kv_heads, cfg->head_dim,
                                       cfg->page_size, cfg->num_pages, status_dev, stream);
  return e == cudaSuccess ? MB_OK : MB_ERR_CUDA;
}

mb_status_t mb_attn_forward_fp8_timed(const mb_plan_t* plan, const void* q,
                                      const void* k_codes, const void* v_codes,
                                      const float* k_scale, const float* v_scale,
                                      const int32_t* block_table_dev, void* out, float* lse,
                                      cudaStream_t stream, cudaEvent_t* events) {
  if (!plan || !plan->workspace) return MB_ERR_INVALID_ARG;
  const PlanDevice& d = plan->dev;
  // prefill work runs on the tensor-core kernel over bf16 staging pages,
  // which only a plan built with mb_plan_options_t.fp8_cache has
  if (d.n_prefill_items > 0 && d.n_stage_pages == 0) return MB_ERR_UNSUPPORTED;
  if (d.total_q == 0) return MB_OK;
  if (!q || !k_codes || !v_codes || !k_scale || !v_scale || !block_table_dev || !out)
    return MB_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_codes) || !aligned16(v_codes) || !aligned16(k_scale) ||
      !aligned16(v_scale) || !aligned16(out) || (reinterpret_cast<uintptr_t>(lse) & 3) ||
      (reinterpret_cast<uintptr_t>(block_table_dev) & 3))
    return MB_ERR_INVALID_ARG;
  uint8_t* ws = static_cast<uint8_t*>(plan->workspace);
  int32_t* status = reinterpret_cast<int32_t*>(ws);
  const float scale_log2 = d.scale * kLog2e;
  auto rec = [&](int stage, int which) {
    if (events && events[2 * stage + which]) cudaEventRecord(events[2 * stage + which], stream);
  };
  cudaError_t e = cudaSuccess;
  const bool overlap = d.n_prefill_items > 0 && d.n_decode_items > 0 && events == nullptr;
  if (d.n_prefill_items > 0) {
    // the pages the prefill requests read, dequantized into the workspace's
    // staging region (laid out like a bf16 cache with staging page ids), then
    // the bf16 tensor-core prefill over it through the staged block table
    const size_t half = (size_t)d.n_stage_pages * d.n_kv_heads * d.page_size * d.head_dim * 2;
    uint8_t* kst = ws + d.off_stage_kv;
    uint8_t* vst = kst + half;
    CUtensorMap qm, km, vm;
    const cuuint64_t kvdims[2] = {(cuuint64_t)d.head_dim,
                                  (cuuint64_t)d.n_stage_pages * d.n_kv_heads * d.page_size};
    const cuuint64_t kvstr[1] = {(cuuint64_t)d.head_dim * 2};
    const cuuint32_t kvbox[2] = {64, (cuuint32_t)d.page_size};
    const cuuint64_t qdims[3] = {(cuuint64_t)d.head_dim, (cuuint64_t)d.n_q_heads,
                                 (cuuint64_t)d.total_q};
    const cuuint64_t qstr[2] = {(cuuint64_t)d.head_dim * 2,
                                (cuuint64_t)d.n_q_heads * d.head_dim * 2};
    const cuuint32_t qbox[3] = {64, 1, (cuuint32_t)kPrefillTileM};
    if (!make_map(&km, kst, 2, kvdims, kvstr, kvbox) ||
        !make_map(&vm, vst, 2, kvdims, kvstr, kvbox) || !make_map(&qm, q, 3, qdims, qstr, qbox))
      return MB_ERR_CUDA;
    rec(MB_STAGE_PREFILL, 0);
    e = launch_dequant_pages(k_codes, v_codes, k_scale, v_scale,
                             reinterpret_cast<const int32_t*>(ws + d.off_stage_pages),
                             d.n_stage_pages, d.n_kv_heads, d.head_dim, d.page_size,
                             d.num_pages, kst, vst, status, stream);
    if (e != cudaSuccess) return MB_ERR_CUDA;
    PrefillArgs a;
    a.items = reinterpret_cast<const PrefillItem*>(ws + d.off_prefill_items);
    a.n_items = d.n_prefill_items;
    a.block_table = reinterpret_cast<const int32_t*>(ws + d.off_stage_bt);
    a.max_blocks = d.max_blocks;
    a.n_q_heads = d.n_q_heads;
    a.n_kv_heads = d.n_kv_heads;
    a.head_dim = d.head_dim;
    a.page_size = d.page_size;
    a.num_pages = d.n_stage_pages;
    a.scale_log2 = scale_log2;
    a.out = out;
    a.lse = lse;
    a.status = status;
    a.max_ctas = overlap ? d.prefill_ctas : 0;
    a.q_map = &qm;
    a.k_map = &km;
    a.v_map = &vm;
    e = launch_prefill(a, stream);
    rec(MB_STAGE_PREFILL, 1);
    if (e != cudaSuccess) return MB_ERR_CUDA;
  }
  if (d.n_decode_items > 0) {
    // K codes as rows of head_dim bytes, one page of one KV head per box,
    // swizzled into the K-major operand layout of the e4m3 MMA
    CUtensorMap km;
    const cuuint64_t kdims[2] = {(cuuint64_t)d.head_dim,
                                 (cuuint64_t)d.num_pages * d.n_kv_heads * d.page_size};
    const cuuint64_t kstr[1] = {(cuuint64_t)d.head_dim};
    const cuuint32_t kbox[2] = {(cuuint32_t)d.head_dim, (cuuint32_t)d.page_size};
    if (!make_map(&km, k_codes, 2, kdims, kstr, kbox, CU_TENSOR_MAP_DATA_TYPE_UINT8,
                  d.head_dim == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B))
      return MB_ERR_CUDA;
    DecodeFp8Args a;
    a.k_map = &km;
    a.max_rows = d.decode_max_rows;
    a.items = reinterpret_cast<const DecodeItem*>(ws + d.off_decode_items);
    a.rows = reinterpret_cast<const RowDesc*>(ws + d.off_rows);
    a.n_items = d.n_decode_items;
    a.q = q;
    a.k8 = k_codes;
    a.v8 = v_codes;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.block_table = block_table_dev;
    a.max_blocks = d.max_blocks;
    a.n_q_heads = d.n_q_heads;
    a.n_kv_heads = d.n_kv_heads;
    a.head_dim = d.head_dim;
    a.page_size = d.page_size;
    a.num_pages = d.num_pages;
    a.scale_log2 = scale_log2;
    a.out = out;
    a.lse = lse;
    a.part_o = reinterpret_cast<float*>(ws + d.off_part_o);
    a.part_lse = reinterpret_cast<float*>(ws + d.off_part_lse);
    a.row_merge = reinterpret_cast<const MergeRef*>(ws + d.off_row_merge);
    a.combine_count = d.n_combine > 0 ? reinterpret_cast<int32_t*>(ws + d.off_combine_count) : nullptr;
    a.status = status;
    a.after_prefill = d.n_prefill_items > 0 ? 1 : 0;
    a.done_counter = reinterpret_cast<int32_t*>(ws + kDoneCounterOffset);
    rec(MB_STAGE_DECODE, 0);
    // behind the prefill kernel, on the SMs its grid leaves free
    e = launch_decode_fp8(a, stream, overlap);
    rec(MB_STAGE_DECODE, 1);
    if (e != cudaSuccess) return MB_ERR_CUDA;
  }
  // split rows are merged inside the split-KV kernel: the combine stage
  // is recorded as an empty interval
  rec(MB_STAGE_COMBINE, 0);
  rec(MB_STAGE_COMBINE, 1);
  return MB_OK;
}

mb_status_t mb_attn_forward_fp8(const mb_plan_t* plan, const void* q, const void* k_codes,
                                const void* v_codes, const float* k_scale, const float* v_scale,
                                const int32_t* block_table_dev, void* out, float* lse,
                                cudaStream_t stream) {
  return mb_attn_forward_fp8_timed(plan, q, k_codes, v_codes, k_scale, v_scale,
                                   block_table_dev, out, lse, stream, nullptr);
}

mb_status_t mb_rope_table(float* cos_sin, int32_t max_position, int32_t head_dim, float base) {
  if (!cos_sin || max_position <= 0 || head_dim <= 0 || (head_dim & 1) || !(base > 0.0f) ||
      !isfinite(base))
    return MB_ERR_INVALID_ARG;
  const int half = head_dim / 2;
  for (int32_t p = 0; p < max_position; ++p) {
    float* row = cos_sin + (size_t)p * head_dim;
    for (int i = 0; i < half; ++i) {
      // theta_i = base^(-2 i / D); the angle in double, then rounded once
      const double a = (double)p * pow((double)base, -2.0 * i / head_dim);
      row[i] = (float)cos(a);
      row[half + i] = (float)sin(a);
    }
  }
  return MB_OK;
}

mb_status_t mb_rope_kv_append(void* q, void* k_cache, void* v_cache, const void* k_new,
                              const void* v_new, const int32_t* positions,
                              const int32_t* slot_mapping, int32_t T, const float* cos_sin,
                              int32_t max_position, const mb_config_t* cfg, int32_t* status_dev,
                              cudaStream_t stream) {
  mb_status_t st = validate_config(cfg);
  if (st != MB_OK) return st;
  if (T < 0 || max_position <= 0) return MB_ERR_INVALID_ARG;
  if (T == 0) return MB_OK;
  if (!q || !k_cache || !v_cache || !k_new || !v_new || !positions || !slot_mapping || !cos_sin)
    return MB_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_new) ||
      !aligned16(v_new) || !aligned16(cos_sin) ||
      (reinterpret_cast<uintptr_t>(positions) & 3) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 3) ||
      (reinterpret_cast<uintptr_t>(status_dev) & 3))
    return MB_ERR_INVALID_ARG;
  cudaError_t e = launch_rope_append(q, k_cache, v_cache, k_new, v_new, positions, slot_mapping,
                                     T, cfg->n_q_heads, cfg->n_kv_heads, cfg->head_dim,
                                     cfg->page_size, cfg->num_pages, cos_sin, max_position,
                                     status_dev, stream);
  return e == cudaSuccess ? MB_OK : MB_ERR_CUDA;
}

mb_status_t mb_attn_forward_timed(const mb_plan_t* plan, const void* q, const void* k_cache,
                                  const void* v_cache, const int32_t* block_table_dev,
                                  void* out, float* lse, cudaStream_t stream,
                                  cudaEvent_t* events) {
  if (!plan || !plan->workspace) return MB_ERR_INVALID_ARG;
  const PlanDevice& d = plan->dev;
  if (d.total_q == 0) return MB_OK;
  if (!q || !k_cache || !v_cache || !block_table_dev || !out) return MB_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(lse) & 3) ||
      (reinterpret_cast<uintptr_t>(block_table_dev) & 3))
    return MB_ERR_INVALID_ARG;
  uint8_t* ws = static_cast<uint8_t*>(plan->workspace);
  int32_t* status = reinterpret_cast<int32_t*>(ws);
  const float scale_log2 = d.scale * kLog2e;
  auto rec = [&](int stage, int which) {
    if (events && events[2 * stage + which]) cudaEventRecord(events[2 * stage + which], stream);
  };
  cudaError_t e = cudaSuccess;

  // K/V tensor maps (both attention kernels stage pages with TMA)
  CUtensorMap qm, km, vm;
  {
    const cuuint64_t kvdims[2] = {(cuuint64_t)d.head_dim,
                                  (cuuint64_t)d.num_pages * d.n_kv_heads * d.page_size};
    const cuuint64_t kvstr[1] = {(cuuint64_t)d.head_dim * 2};
    const cuuint32_t kvbox[2] = {64, (cuuint32_t)d.page_size};
    if (!make_map(&km, k_cache, 2, kvdims, kvstr, kvbox) ||
        !make_map(&vm, v_cache, 2, kvdims, kvstr, kvbox))
      return MB_ERR_CUDA;
  }
  // With both kinds of work the prefill kernel goes first, its persistent
  // grid on the plan's share of the SMs, and the split-KV kernel is launched
  // to overlap it (programmatic stream serialization): it starts once every
  // prefill CTA has been dispatched, streams its key ranges on the SMs the
  // prefill leaves free and spreads over the rest as the prefill CTAs
  // finish. (The timed variant launches back to back, each kernel on the
  // whole GPU, so that each stage's events bracket that stage alone.)
  const bool overlap = d.n_prefill_items > 0 && d.n_decode_items > 0 && events == nullptr;
  if (d.n_prefill_items > 0) {
    const cuuint64_t qdims[3] = {(cuuint64_t)d.head_dim, (cuuint64_t)d.n_q_heads,
                                 (cuuint64_t)d.total_q};
    const cuuint64_t qstr[2] = {(cuuint64_t)d.head_dim * 2,
                                (cuuint64_t)d.n_q_heads * d.head_dim * 2};
    const cuuint32_t qbox[3] = {64, 1, (cuuint32_t)kPrefillTileM};
    if (!make_map(&qm, q, 3, qdims, qstr, qbox)) return MB_ERR_CUDA;
    PrefillArgs a;
    a.items = reinterpret_cast<const PrefillItem*>(ws + d.off_prefill_items);
    a.n_items = d.n_prefill_items;
    a.block_table = block_table_dev;
    a.max_blocks = d.max_blocks;
    a.n_q_heads = d.n_q_heads;
    a.n_kv_heads = d.n_kv_heads;
    a.head_dim = d.head_dim;
    a.page_size = d.page_size;
    a.num_pages = d.num_pages;
    a.scale_log2 = scale_log2;
    a.out = out;
    a.lse = lse;
    a.status = status;
    a.max_ctas = overlap ? d.prefill_ctas : 0;
    a.q_map = &qm;
    a.k_map = &km;
    a.v_map = &vm;
    rec(MB_STAGE_PREFILL, 0);
    e = launch_prefill(a, stream);
    rec(MB_STAGE_PREFILL, 1);
    if (e != cudaSuccess) return MB_ERR_CUDA;
  }
  if (d.n_decode_items > 0) {
    DecodeArgs a;
    a.items = reinterpret_cast<const DecodeItem*>(ws + d.off_decode_items);
    a.rows = reinterpret_cast<const RowDesc*>(ws + d.off_rows);
    a.n_items = d.n_decode_items;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_table = block_table_dev;
    a.max_blocks = d.max_blocks;
    a.n_q_heads = d.n_q_heads;
    a.n_kv_heads = d.n_kv_heads;
    a.head_dim = d.head_dim;
    a.page_size = d.page_size;
    a.num_pages = d.num_pages;
    a.scale_log2 = scale_log2;
    a.out = out;
    a.lse = lse;
    a.part_o = reinterpret_cast<float*>(ws + d.off_part_o);
    a.part_lse = reinterpret_cast<float*>(ws + d.off_part_lse);
    a.row_merge = reinterpret_cast<const MergeRef*>(ws + d.off_row_merge);
    a.combine_count = d.n_combine > 0 ? reinterpret_cast<int32_t*>(ws + d.off_combine_count) : nullptr;
    a.status = status;
    a.after_prefill = d.n_prefill_items > 0 ? 1 : 0;
    a.done_counter = reinterpret_cast<int32_t*>(ws + kDoneCounterOffset);
    a.copies = d.decode_copies;
    a.k_map = &km;
    a.v_map = &vm;
    rec(MB_STAGE_DECODE, 0);
    // behind the prefill kernel (overlap) or behind whatever came before
    // (the append, whose tail the kernel's history streaming then overlaps)
    e = launch_decode(a, stream, events == nullptr);
    rec(MB_STAGE_DECODE, 1);
    if (e != cudaSuccess) return MB_ERR_CUDA;
  }
  // split rows are merged inside the split-KV kernel: the combine stage
  // is recorded as an empty interval
  rec(MB_STAGE_COMBINE, 0);
  rec(MB_STAGE_COMBINE, 1);
  return MB_OK;
}

mb_status_t mb_attn_forward(const mb_plan_t* plan, const void* q, const void* k_cache,
                            const void* v_cache, const int32_t* block_table_dev, void* out,
                            float* lse, cudaStream_t stream) {
  return mb_attn_forward_timed(plan, q, k_cache, v_cache, block_table_dev, out, lse, stream,
                               nullptr);
}

}  // extern "C"
