// Attention forward for callers that cannot allocate device memory.
//
// Same kernels and launch order as mb_attn_forward; the difference is where
// the scratch lives. mb_attn_forward uses a workspace the caller allocated;
// this entry point uses g_scratch below, a static device array of
// MB_NOALLOC_SCRATCH_BYTES that the library owns. The host plan's work lists
// are copied into it at every call, then the split-KV partials are written
// after them exactly as in a caller workspace.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/mb.h"
#include "kernels.h"
#include "mb_internal.h"
#include "plan_impl.h"

using namespace mb;

namespace {

constexpr size_t kScratchBytes = MB_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;
constexpr float kLog2e = 1.4426950408889634f;

// One copy per GPU that loads the library, kept until the process exits.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Device address of g_scratch on the current device. Host code cannot use
// the symbol itself as a device pointer, so it is looked up once per device
// (with that device current) and cached.
mb_status_t scratch_for_current_device(void** out) {
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess) return MB_ERR_CUDA;
  if (device < 0 || device >= kMaxDevices) return MB_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[device]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess || p == nullptr) return MB_ERR_CUDA;
    g_scratch_ptr[device] = p;
  }
  *out = g_scratch_ptr[device];
  return MB_OK;
}

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

bool make_map(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
              const cuuint64_t* strides, const cuuint32_t* box) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  cuuint32_t elem[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base),
            dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

}  // namespace

extern "C" mb_status_t mb_attn_forward_noalloc(const mb_plan_t* plan, const void* q,
                                               const void* k_cache, const void* v_cache,
                                               const int32_t* block_table_dev, void* out,
                                               float* lse, int32_t* status_dev,
                                               cudaStream_t stream) {
  if (!plan) return MB_ERR_INVALID_ARG;
  const PlanDevice& d = plan->dev;
  if (d.workspace_bytes > kScratchBytes) return MB_ERR_WORKSPACE;
  if (d.total_q == 0) return MB_OK;
  if (!q || !k_cache || !v_cache || !block_table_dev || !out) return MB_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(lse) & 3) ||
      (reinterpret_cast<uintptr_t>(block_table_dev) & 3) ||
      (reinterpret_cast<uintptr_t>(status_dev) & 3))
    return MB_ERR_INVALID_ARG;
  if (plan->host_image.size() != d.metadata_bytes) return MB_ERR_INVALID_ARG;

  void* scratch = nullptr;
  mb_status_t st = scratch_for_current_device(&scratch);
  if (st != MB_OK) return st;
  uint8_t* ws = static_cast<uint8_t*>(scratch);
  int32_t* status = reinterpret_cast<int32_t*>(ws);

  // work lists (and a zero status word) into the static array; the partials
  // behind them need no clearing: every slot is written before it is read
  if (cudaMemcpyAsync(ws, plan->host_image.data(), d.metadata_bytes, cudaMemcpyHostToDevice,
                      stream) != cudaSuccess)
    return MB_ERR_CUDA;

  const float scale_log2 = d.scale * kLog2e;
  CUtensorMap km, vm;
  {
    const cuuint64_t kvdims[2] = {(cuuint64_t)d.head_dim,
                                  (cuuint64_t)d.num_pages * d.n_kv_heads * d.page_size};
    const cuuint64_t kvstr[1] = {(cuuint64_t)d.head_dim * 2};
    const cuuint32_t kvbox[2] = {64, (cuuint32_t)d.page_size};
    if (!make_map(&km, k_cache, 2, kvdims, kvstr, kvbox) ||
        !make_map(&vm, v_cache, 2, kvdims, kvstr, kvbox))
      return MB_ERR_CUDA;
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
    a.k_map = &km;
    a.v_map = &vm;
    if (launch_decode(a, stream) != cudaSuccess) return MB_ERR_CUDA;
  }
  if (d.n_prefill_items > 0) {
    CUtensorMap qm;
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
    a.q_map = &qm;
    a.k_map = &km;
    a.v_map = &vm;
    if (launch_prefill(a, stream) != cudaSuccess) return MB_ERR_CUDA;
  }
  if (status_dev &&
      cudaMemcpyAsync(status_dev, status, sizeof(int32_t), cudaMemcpyDeviceToDevice, stream) !=
          cudaSuccess)
    return MB_ERR_CUDA;
  return MB_OK;
}
