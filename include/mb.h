/*
 * mb.h -- C ABI of the mixed-batch paged attention library (one GB300, sm_103a).
 *
 * The library computes the attention step of one continuous-batching
 * iteration (one layer): a ragged batch of requests, each described by the
 * triple (q_start, q_end, kv_length), whose new query rows attend to their
 * own paged K/V cache.
 *
 *   - Per-request triple, kv_length counted after this iteration's append:
 *     "ORCA and chunked prefill", section 2.
 *   - Mask: the first S0 = kv_length - q_rows key columns are visible to every
 *     new row; over the last q_rows columns only the strict upper triangle is
 *     masked (diagonal kept): "How To Scale Your Model notes (7-8)", section 2;
 *     the same two blocks in "ORCA and chunked prefill", section 4.
 *   - Paged K/V through a per-request block table, pages shareable between
 *     requests: "How To Scale Your Model notes (7-8)", section 3 (paging);
 *     slot mapping ("out_cache_loc") and block tables built by the host:
 *     "GLM-5.3 e2e token ledger", stage 4.
 *   - GQA: g = n_q_heads / n_kv_heads query heads share KV head h / g
 *     (contiguous grouping): "How To Scale Your Model notes (7-8)", section 3.
 *   - Shared prefix read once for all requests that share it, each request
 *     keeping its own softmax state: "How To Scale Your Model notes (7-8)",
 *     section 3 (stored once is not read once).
 *
 * Layouts (all row-major, contiguous, bf16 = IEEE bfloat16 bit patterns):
 *   q, out      [total_q, n_q_heads, head_dim]            bf16
 *   lse         [total_q, n_q_heads]                      fp32 (natural log)
 *   k_new/v_new [T, n_kv_heads, head_dim]                 bf16
 *   k_cache,
 *   v_cache     [num_pages, n_kv_heads, page_size, head_dim] bf16
 *               (one page of one KV head is one contiguous
 *                page_size * head_dim * 2 byte tile)
 *   block_table [n_reqs, max_blocks_per_req]               int32 page ids;
 *               entry b of request r holds logical positions
 *               [b * page_size, (b + 1) * page_size)
 *   slot        page * page_size + position % page_size    int32
 *
 * Ownership: the caller owns every device buffer (caches, q, out, lse,
 * block tables, slot mappings, the workspace) and the stream. The library
 * never allocates device memory and never synchronises the device; a plan
 * owns only host memory. Calls enqueue work on the caller's stream.
 *
 * Errors: host-detectable errors are returned as mb_status_t and nothing is
 * enqueued. Device-detected errors (a slot or page out of range, a bounded
 * wait that ran out) are OR-ed as bit flags (1 << status) into a device
 * int32 status word: the one passed to mb_kv_append, and for attention the
 * first 4 bytes of the plan's workspace. The caller reads it after a sync.
 */
#ifndef MB_H
#define MB_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Bumped whenever a struct or signature below changes (3: mb_plan_info_t
 * gained splitkv_max_rows). */
#define MB_ABI_VERSION 3

typedef enum {
  MB_OK = 0,
  MB_ERR_INVALID_ARG = 1,  /* null pointer, negative size, bad option        */
  MB_ERR_SHAPE = 2,        /* inconsistent triples / block table / config    */
  MB_ERR_UNSUPPORTED = 3,  /* head_dim or page_size outside the built set    */
  MB_ERR_WORKSPACE = 4,    /* workspace missing, too small or misaligned     */
  MB_ERR_CUDA = 5,         /* a CUDA runtime call failed                     */
  MB_ERR_TIMEOUT = 6,      /* device flag: a bounded wait in a kernel ran out */
  MB_ERR_DEVICE_INDEX = 7, /* device flag: slot / page index out of range    */
  MB_ERR_SHARED_PAGE = 8   /* mb_check_append_targets: a new row would land in
                              a page another request also maps              */
} mb_status_t;

/* One request of the iteration ("ORCA and chunked prefill", section 2).
 * q_rows = q_end - q_start new rows at rows [q_start, q_end) of q / out;
 * kv_length = whole context including this iteration's q_rows rows, so the
 * new rows occupy logical positions [kv_length - q_rows, kv_length).
 * q_rows = 0 is allowed (no output). */
typedef struct {
  int32_t q_start;
  int32_t q_end;
  int32_t kv_length;
} mb_request_t;

/* Problem configuration shared by every call of one layer. */
typedef struct {
  int32_t n_q_heads;           /* Hq, multiple of n_kv_heads                  */
  int32_t n_kv_heads;          /* Hkv                                          */
  int32_t head_dim;            /* D: 64 or 128                                 */
  int32_t page_size;           /* tokens per page: 16, 32, 64 or 128           */
  int32_t num_pages;           /* pages in each of k_cache / v_cache           */
  int32_t max_blocks_per_req;  /* columns of the block table                   */
  float scale;                 /* softmax scale; 0 -> 1/sqrt(head_dim)         */
} mb_config_t;

/* Planner knobs (mb_attn_plan_ex). Zero-initialised = defaults. */
typedef struct {
  int32_t prefill_min_rows;  /* requests with q_rows >= this run the tensor-core
                                prefill kernel; 0 -> default (16);
                                < 0 -> never (everything on split-KV)        */
  int32_t kv_chunk;          /* split-KV chunk in keys (multiple of 64, rounded
                                up to whole pages; ranges are cut into equal
                                page-aligned parts no longer than this);
                                0 -> chosen from the batch (>= 1024)         */
  int32_t disable_cascade;   /* 1 -> no shared-prefix grouping               */
  int32_t target_ctas;       /* split-KV work items to aim for; 0 -> auto     */
  int32_t prefill_ctas;      /* when a plan holds both kinds of work, the SMs
                                the persistent prefill grid takes while the
                                split-KV kernel streams on the rest (one CTA
                                per SM each); 0 -> chosen by the planner's
                                cost model; < 0 -> every SM (the split-KV
                                kernel then only fills the prefill's tail) */
  int32_t fp8_cache;         /* 1 -> the plan serves mb_attn_forward_fp8: the
                                pages its prefill requests read get a bf16
                                staging copy in the workspace (see there) */
} mb_plan_options_t;

/* Plan summary (mb_plan_info). */
typedef struct {
  int32_t n_decode_items;    /* CTAs of the split-KV kernel                   */
  int32_t n_decode_rows;     /* row descriptors                               */
  int32_t n_prefill_items;   /* CTAs of the prefill kernel                    */
  int32_t n_combine;         /* output rows merged from split-KV partials     */
  int32_t n_partials;        /* partial (O, LSE) slots                        */
  int32_t n_cascade_groups;  /* shared-prefix groups                          */
  int32_t cascade_keys;      /* keys read once per group (sum over groups)    */
  int32_t kv_chunk;          /* split-KV chunk actually used                  */
  int32_t total_q;           /* max q_end                                     */
  int32_t n_launches;        /* kernels one mb_attn_forward launches          */
  size_t workspace_bytes;
  size_t metadata_bytes;     /* bytes uploaded host->device by the plan       */
  int32_t prefill_ctas;      /* prefill CTAs mb_attn_forward launches beside the
                                split-KV kernel (0: no prefill work)         */
  int32_t staged_pages;      /* fp8 plans: cache pages dequantized to bf16 for
                                the prefill kernel per forward              */
  int32_t splitkv_copies;    /* 1: the split-KV build that spreads each row's
                                keys over copies in the softmax warps (most
                                keys in CTAs of <= 32 rows and >= 8 tiles) */
  int32_t splitkv_max_rows;  /* largest query-row count of a split-KV CTA; an
                                fp8 cache with head_dim 128 runs the few-row
                                form of its split-KV kernel when <= 8        */
} mb_plan_info_t;

typedef struct mb_plan mb_plan_t;

/* Stages timed by mb_attn_forward_timed. MB_STAGE_COMBINE is kept for the
 * event layout: the log-sum-exp merge of split rows runs inside the split-KV
 * kernel, so its two events are recorded back to back (an empty interval). */
#define MB_STAGE_DECODE 0
#define MB_STAGE_COMBINE 1
#define MB_STAGE_PREFILL 2
#define MB_NUM_STAGES 3

int32_t mb_abi_version(void);
const char* mb_status_string(mb_status_t s);

/* Self-test of the failure path every kernel's waits share (no counterpart
 * on the pages). Launches one CTA on stream whose bounded wait, on an
 * mbarrier that nothing completes, runs out after the kernels' 2 s limit; the
 * CTA then sets bit (1 << MB_ERR_TIMEOUT) in *status_dev (device int32,
 * 4-byte aligned) and returns, as a timed-out attention kernel does: no
 * fault, and the context stays usable. Returns MB_ERR_INVALID_ARG for a null status_dev,
 * MB_ERR_CUDA if the launch fails; the caller reads the status after a sync. */
mb_status_t mb_selftest_wait_timeout(int32_t* status_dev, cudaStream_t stream);

/* Host helper: the slot ("out_cache_loc") of every new row, i.e. where
 * mb_kv_append writes it ("GLM-5.3 e2e token ledger", stage 4).
 * New row t of request r sits at logical position p = kv_length - q_rows +
 * (t - q_start), slot = block_table[r][p / page_size] * page_size +
 * p % page_size. slots_out (host, total_q entries) receives -1 for rows no
 * request covers. block_table_host is [n_reqs, cfg->max_blocks_per_req].
 * Errors: MB_ERR_INVALID_ARG, MB_ERR_SHAPE (same checks as mb_attn_plan). */
mb_status_t mb_slot_mapping(const mb_request_t* reqs, int32_t n_reqs,
                            const int32_t* block_table_host,
                            const mb_config_t* cfg, int32_t* slots_out,
                            int32_t total_q);

/* Host helper: the logical position of every new row (what the rotary
 * embedding rotates by): row t of request r is at kv_length - q_rows +
 * (t - q_start) ("ORCA and chunked prefill", section 2: kv_length counts this
 * iteration's rows). positions_out (host, total_q entries) receives -1 for
 * rows no request covers. Errors: MB_ERR_INVALID_ARG (null pointer, negative
 * size), MB_ERR_SHAPE (q_start > q_end, q_rows > kv_length, a range past
 * total_q). */
mb_status_t mb_positions(const mb_request_t* reqs, int32_t n_reqs, int32_t* positions_out,
                         int32_t total_q);

/* Host debug check of the append contract below: no new row of this
 * iteration may land in a page that another request's block table also maps
 * (a shared prefix page is read by every sharer; writing it would change
 * their history). Request r maps pages block_table_host[r][0 ..
 * ceil(kv_length / page_size)); its new rows are its positions [kv_length -
 * q_rows, kv_length). Returns MB_OK, or MB_ERR_SHARED_PAGE with
 * *bad_request_out = the first offending request (else -1); the errors of
 * mb_attn_plan for inconsistent inputs. Host only, no CUDA call. */
mb_status_t mb_check_append_targets(const mb_request_t* reqs, int32_t n_reqs,
                                    const int32_t* block_table_host,
                                    const mb_config_t* cfg, int32_t* bad_request_out);

/* KV append: scatter this iteration's K/V rows into their pages
 * ("ORCA and chunked prefill", section 4: append K, V to the cache before
 * the attention reads it). For t in [0, T): slot = slot_mapping[t];
 * slot < 0 skips the row (padding); otherwise every KV head h gets
 *   k_cache[slot / ps][h][slot % ps][:] = k_new[t][h][:]  (same for V),
 * a bit-exact copy. k_new/v_new [T, Hkv, D] contiguous bf16 (device);
 * slot_mapping int32 [T] (device). Pages written here must not be shared
 * with another request (the caller's contract; mb_check_append_targets
 * checks it on the host). A slot >= num_pages*ps is
 * skipped and sets bit (1 << MB_ERR_DEVICE_INDEX) in *status_dev
 * (nullable device int32). T = 0 enqueues nothing. Asynchronous on stream:
 * the kernel may start under the tail of the launch before it on `stream`
 * (programmatic dependent launch) and waits for that launch to complete
 * before it reads or writes any memory. */
mb_status_t mb_kv_append(void* k_cache, void* v_cache, const void* k_new,
                         const void* v_new, const int32_t* slot_mapping,
                         int32_t T, const mb_config_t* cfg, int32_t* status_dev,
                         cudaStream_t stream);

/* fp8 (e4m3) KV cache ("GLM-5.3 e2e token ledger", the KV layout
 * paragraphs: FP8 K/V with FP32 scales stored beside them, read together by
 * the attention kernel to dequantize). Layout, all device memory:
 *   k_codes, v_codes  [num_pages, n_kv_heads, page_size, head_dim] uint8
 *                     e4m3 codes (1 sign, 4 exponent bits with bias 7,
 *                     3 mantissa bits, no infinities; 0x7F/0xFF are NaN)
 *   k_scale, v_scale  [num_pages, n_kv_heads, page_size] fp32, one scale
 *                     per (token, KV head) row
 * and a row's values are decode(code) * scale.
 *
 * Append with quantization: for every token t with slot = slot_mapping[t]
 * >= 0 and every KV head h, the bf16 row x = k_new[t][h] (and likewise
 * v_new) is stored as scale = amax(|x|) / 448 (fp32 division; 448 = the
 * largest e4m3 value) and code_i = e4m3(x_i / scale) (one IEEE fp32
 * division, round to nearest even, saturating at +-448, the sign kept for
 * values that round to zero); an all-zero row gets scale 0 and codes 0.
 * Slot rules, status bits, alignment (every pointer 16-byte aligned),
 * launch order and errors as for mb_kv_append. */
mb_status_t mb_kv_append_fp8(void* k_codes, void* v_codes, float* k_scale, float* v_scale,
                             const void* k_new, const void* v_new,
                             const int32_t* slot_mapping, int32_t T,
                             const mb_config_t* cfg, int32_t* status_dev,
                             cudaStream_t stream);

/* Attention of every planned request over an fp8 cache (layout above):
 * the same result as mb_attn_forward on the dequantized K/V.
 *   - Split-KV work (decode rows, small chunks, shared-prefix groups) reads
 *     the codes directly: Q K^T on the tensor cores in e4m3 (each query row
 *     written once as two e4m3 rows sq (hi + lo), sq = amax|q| / 448, which
 *     keeps q to about 2^-8 of each value), the K scales applied to the
 *     scores, P V on f16 operands with the V scale and 1 / rho carried by
 *     V' (V' = code * v_scale / rho) or, when every split-KV CTA holds at
 *     most 8 rows and head_dim is 128, by P (P' = p * v_scale / rho, V' =
 *     code), rho a power of two bounding the CTA's V scales; fp32
 *     accumulation. The two forms differ only in where the f16 roundings
 *     fall.
 *   - Prefill work needs a plan built with mb_plan_options_t.fp8_cache = 1
 *     (else MB_ERR_UNSUPPORTED, nothing enqueued). Each forward first
 *     dequantizes the pages the prefill requests read (decode(code) * scale
 *     in fp32, rounded once to bf16) into the plan's workspace, once per
 *     page however many prefill requests map it, then runs the tensor-core
 *     prefill kernel (bf16 operands, fp32 accumulation) over those pages,
 *     with the split-KV kernel beside it as in mb_attn_forward.
 * Other arguments, outputs and errors as for mb_attn_forward; all pointers
 * 16-byte aligned (lse 4). */
mb_status_t mb_attn_forward_fp8(const mb_plan_t* plan, const void* q,
                                const void* k_codes, const void* v_codes,
                                const float* k_scale, const float* v_scale,
                                const int32_t* block_table_dev, void* out,
                                float* lse, cudaStream_t stream);

/* mb_attn_forward_fp8 with per-stage events (MB_STAGE_PREFILL covers the
 * staging dequantization and the prefill kernel; MB_STAGE_DECODE;
 * MB_STAGE_COMBINE empty, as in mb_attn_forward_timed). */
mb_status_t mb_attn_forward_fp8_timed(const mb_plan_t* plan, const void* q,
                                      const void* k_codes, const void* v_codes,
                                      const float* k_scale, const float* v_scale,
                                      const int32_t* block_table_dev, void* out,
                                      float* lse, cudaStream_t stream,
                                      cudaEvent_t* events);

/* Rotary angle table for mb_rope_kv_append (host helper, no CUDA call).
 * cos_sin (host, max_position * head_dim floats) row p receives
 * [cos(p theta_0) .. cos(p theta_{D/2-1}), sin(p theta_0) .. sin(p theta_{D/2-1})],
 * theta_i = base^(-2 i / head_dim), each angle evaluated in double and rounded
 * once to float (the rotary embedding of the Llama-2 family; the pages name
 * the fused "norm + RoPE + write KV" kernel, "GLM-5.3 e2e token ledger",
 * stage 6, without printing the rotation). Errors: MB_ERR_INVALID_ARG (null
 * pointer, max_position <= 0, odd or non-positive head_dim, base <= 0). */
mb_status_t mb_rope_table(float* cos_sin, int32_t max_position, int32_t head_dim, float base);

/* Fused rotary embedding + KV append ("GLM-5.3 e2e token ledger", stage 6:
 * RoPE and the KV write in one kernel that already holds q and k; the append
 * of "ORCA and chunked prefill", section 4). For every token t in [0, T) at
 * position p = positions[t]:
 *   - each query head row q[t][h] (bf16 [T, Hq, D], device) is rotated in
 *     place: for i < D/2 the pair (x_i, x_{i+D/2}) becomes
 *     (x_i c - x_{i+D/2} s, x_{i+D/2} c + x_i s), c, s = cos_sin[p][i],
 *     cos_sin[p][D/2 + i], computed in fp32 and rounded once to bf16;
 *   - if slot = slot_mapping[t] >= 0, each KV head's k_new[t][h] is rotated
 *     the same way into k_cache[slot / ps][h][slot % ps] and v_new[t][h] is
 *     copied bit for bit into v_cache at the same place (k_new, v_new bf16
 *     [T, Hkv, D], device; k_new is not modified).
 * cos_sin: device fp32 [max_position, head_dim] (see mb_rope_table), 16-byte
 * aligned. positions, slot_mapping: device int32 [T]. A position outside
 * [0, max_position) skips the whole token; a slot >= num_pages * ps skips its
 * cache write; both set bit (1 << MB_ERR_DEVICE_INDEX) in *status_dev
 * (nullable device int32). Pages written must not be shared with another
 * request (the caller's contract). T = 0 enqueues nothing. Asynchronous on
 * stream, launch order and host errors as for mb_kv_append. */
mb_status_t mb_rope_kv_append(void* q, void* k_cache, void* v_cache, const void* k_new,
                              const void* v_new, const int32_t* positions,
                              const int32_t* slot_mapping, int32_t T, const float* cos_sin,
                              int32_t max_position, const mb_config_t* cfg, int32_t* status_dev,
                              cudaStream_t stream);

/* Plan one iteration. Host inputs: reqs[n_reqs] and block_table_host
 * [n_reqs, max_blocks_per_req]. Validates: config (Hq % Hkv == 0, head_dim,
 * page_size), 0 <= q_start <= q_end, q_rows <= kv_length, disjoint q
 * ranges, ceil(kv_length / page_size) <= max_blocks_per_req, every used
 * block id in [0, num_pages). Classifies requests (tensor-core prefill vs
 * split-KV), groups requests whose leading cached pages are the same
 * physical pages (shared-prefix cascade), splits long key ranges into
 * split-KV chunks and lays out the workspace.
 * workspace == NULL: size query; *workspace_bytes receives the size and
 * *out_plan is untouched. Otherwise workspace (device, 256-byte aligned,
 * >= that size, owned by the caller, kept alive and unmodified while the
 * plan is used) receives the work lists with one host->device copy on
 * stream, and *out_plan a new plan (free with mb_attn_destroy). The plan
 * may be reused by any number of mb_attn_forward calls (e.g. every layer
 * of the iteration). The copy runs on the host->device copy engine, in the
 * same queue as the caller's input uploads: a loop that uploads the next
 * step's inputs on another stream while this step computes should plan each
 * step on that upload stream, ahead of the step's inputs, with one workspace
 * per step in flight (planned on the compute stream, the small copy waits
 * behind the next step's bulk upload). */
mb_status_t mb_attn_plan(const mb_request_t* reqs, int32_t n_reqs,
                         const int32_t* block_table_host, const mb_config_t* cfg,
                         void* workspace, size_t* workspace_bytes,
                         cudaStream_t stream, mb_plan_t** out_plan);

/* mb_attn_plan with explicit planner knobs (opts may be NULL). */
mb_status_t mb_attn_plan_ex(const mb_request_t* reqs, int32_t n_reqs,
                            const int32_t* block_table_host,
                            const mb_config_t* cfg,
                            const mb_plan_options_t* opts, void* workspace,
                            size_t* workspace_bytes, cudaStream_t stream,
                            mb_plan_t** out_plan);

/* Attention of every planned request. q [total_q, Hq, D] bf16, caches as
 * above (already holding this iteration's rows), block_table_dev: device
 * copy of the planned block table, out [total_q, Hq, D] bf16 (rows no
 * request covers are not written), lse [total_q, Hq] fp32 natural-log
 * log-sum-exp of the scaled visible scores (nullable). No device->host
 * traffic and no allocation: the launch sequence can be captured in a CUDA
 * graph. Launch order (programmatic dependent launch on the same stream):
 * the split-KV kernel starts under the tail of the launch before it (the
 * KV append, say) and streams history key tiles at once, but waits for that
 * launch to complete before it reads q or a key tile holding this step's
 * rows and before it writes anything. When the plan holds both kinds of
 * work, the prefill kernel is launched first on info.prefill_ctas SMs (it
 * starts once the launch before it has completed) and the split-KV kernel
 * runs beside it on the other SMs, then on each SM a prefill CTA leaves;
 * its last CTA waits for the prefill kernel. Whatever is enqueued on
 * `stream` after the call sees out and lse. Device-detected errors go to
 * the workspace status word. */
mb_status_t mb_attn_forward(const mb_plan_t* plan, const void* q,
                            const void* k_cache, const void* v_cache,
                            const int32_t* block_table_dev, void* out,
                            float* lse, cudaStream_t stream);

/* mb_attn_forward that also records events[2*s] / events[2*s+1] on stream
 * around stage s (MB_STAGE_*) when that stage launches. Stages are launched
 * back to back (no overlap) so each pair brackets its stage alone. events:
 * array of 2 * MB_NUM_STAGES created events (entries may be NULL). */
mb_status_t mb_attn_forward_timed(const mb_plan_t* plan, const void* q,
                                  const void* k_cache, const void* v_cache,
                                  const int32_t* block_table_dev, void* out,
                                  float* lse, cudaStream_t stream,
                                  cudaEvent_t* events);

/* Host-only planning: builds the plan (same validation and work lists as
 * mb_attn_plan_ex) without a workspace and without any CUDA call. Such a plan
 * cannot be passed to mb_attn_forward (MB_ERR_INVALID_ARG); it serves
 * mb_plan_info / mb_plan_export_metadata and mb_attn_forward_noalloc. */
mb_status_t mb_attn_plan_host(const mb_request_t* reqs, int32_t n_reqs,
                              const int32_t* block_table_host, const mb_config_t* cfg,
                              const mb_plan_options_t* opts, mb_plan_t** out_plan);

/* Copy the plan's metadata image (the bytes mb_attn_plan uploads to the
 * start of the workspace; info.metadata_bytes long) into host memory dst of
 * dst_bytes. Its layout: int32 status word at 0, then the work lists at the
 * offsets given by mb_plan_layout. */
mb_status_t mb_plan_export_metadata(const mb_plan_t* plan, void* dst, size_t dst_bytes);

/* Byte offsets of the workspace regions: out[0..5] = decode items, row
 * descriptors, prefill items, combine entries, partial LSEs, partial outputs. */
mb_status_t mb_plan_layout(const mb_plan_t* plan, size_t* out6);

/* Summary of a plan (host only). */
mb_status_t mb_plan_info(const mb_plan_t* plan, mb_plan_info_t* info);

/* Attention forward that allocates nothing (no counterpart on the pages:
 * this is a convenience of the library, not part of the method).
 *
 * Who needs it: callers that must not allocate device memory themselves --
 * for example code running under an external memory manager that owns every
 * device allocation, a plug-in that is only handed pointers to its inputs and
 * outputs, or a hot loop where a cudaMalloc (which can synchronise the whole
 * device) is not acceptable. Such a caller builds its plan with
 * mb_attn_plan_host (host memory only) and calls this instead of
 * mb_attn_forward; no workspace is passed.
 *
 * The scratch the forward needs (the plan's work lists and the split-KV
 * partial outputs) lives in one static device array inside the library,
 * MB_NOALLOC_SCRATCH_BYTES long. Every GPU that loads the library holds that
 * array until the process exits. A plan whose info.workspace_bytes exceeds
 * the array is rejected with MB_ERR_WORKSPACE before anything is enqueued.
 *
 * The first call on a device (and the first after that device's CUDA context
 * was re-created) looks up the array's device address with that device
 * current; make that first call outside any stream capture. Each call then
 * copies the plan's work lists into the array with cudaMemcpyAsync on
 * `stream` -- this also clears the device status word. The source is the
 * plan's ordinary (pageable) host memory, so the CUDA runtime may make the
 * calling thread wait until the stream's earlier work has finished before
 * the copy. The call then launches the same kernels as mb_attn_forward, one
 * after the other: unlike mb_attn_forward it does not start the split-KV
 * kernel under the prefill kernel's tail, so a plan with both kinds of work
 * takes a little longer. Every call shares the one array and it keeps the
 * last call's contents: calls whose work overlaps on the GPU (other streams,
 * other host threads) race on it, so serialise them. status_dev (nullable,
 * device int32, 4-byte aligned) receives a copy of the call's device error
 * flags (bits 1 << MB_ERR_TIMEOUT / MB_ERR_DEVICE_INDEX), and zero for a plan
 * with no rows. Inputs, outputs and errors are otherwise as for
 * mb_attn_forward. */
#define MB_NOALLOC_SCRATCH_BYTES (8u << 20)
mb_status_t mb_attn_forward_noalloc(const mb_plan_t* plan, const void* q,
                                    const void* k_cache, const void* v_cache,
                                    const int32_t* block_table_dev, void* out,
                                    float* lse, int32_t* status_dev,
                                    cudaStream_t stream);

/* Release a plan's host memory. NULL is accepted. The workspace stays the
 * caller's. */
mb_status_t mb_attn_destroy(mb_plan_t* plan);

#ifdef __cplusplus
}
#endif

#endif /* MB_H */
