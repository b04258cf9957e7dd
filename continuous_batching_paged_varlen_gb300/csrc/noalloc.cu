// Attention forward for callers that cannot allocate device memory.
//
// Same kernels as mb_attn_forward, launched one after the other (split-KV,
// then prefill) without the overlap mb_attn_forward arranges between them;
// the other difference is where the scratch lives. mb_attn_forward uses a workspace the caller allocated;
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

// The array's device address per device, with the id of the CUDA context it
// was looked up in: a context created later on the same device (after a
// cudaDeviceReset, say) loads the library's module again, at another address.
struct ScratchAddr {
  unsigned long long ctx_id;
  void* ptr;
};
std::mutex g_mu;
ScratchAddr g_scratch_addr[kMaxDevices] = {};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Id of the calling thread's current CUDA context (driver entry points
// cuCtxGetCurrent / cuCtxGetId, reached through the runtime).
bool current_context_id(unsigned long long* id) {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  if (!get_current || !get_id) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_scratch in the current device's context. Host code
// cannot use the symbol itself as a device pointer, so the address is looked
// up (with that device current) once per device and context, and cached.
mb_status_t scratch_for_current_device(void** out) {
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess) return MB_ERR_CUDA;
  if (device < 0 || device >= kMaxDevices) return MB_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  ScratchAddr& a = g_scratch_addr[device];
  unsigned long long ctx = 0;
  const bool have_ctx = current_context_id(&ctx);
  if (!have_ctx || !a.ptr || a.ctx_id != ctx) {
    // the lookup also makes the device's primary context current when no
    // context is yet
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess || p == nullptr) return MB_ERR_CUDA;
    if (!have_ctx && !current_context_id(&ctx)) return MB_ERR_CUDA;
    a.ptr = p;
    a.ctx_id = ctx;
  }
  *out = a.ptr;
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
  if (reinterpret_cast<uintptr_t>(status_dev) & 3) return MB_ERR_INVALID_ARG;
  if (d.total_q == 0) {
    // nothing to run: the caller's status word still reports "no flags"
    if (status_dev && cudaMemsetAsync(status_dev, 0, sizeof(int32_t), stream) != cudaSuccess)
      return MB_ERR_CUDA;
    return MB_OK;
  }
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
    a.after_prefill = 0;
    a.done_counter = reinterpret_cast<int32_t*>(ws + kDoneCounterOffset);
    a.copies = d.decode_copies;
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
    a.max_ctas = 0;
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
