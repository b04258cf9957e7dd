// Internal types shared by the host planner and the kernels.
//
// The planner (plan.cpp) turns the iteration's triples and block tables into
// flat work lists that it uploads into the caller's workspace with one
// host->device copy. Workspace layout (offsets in bytes, each region
// 256-byte aligned):
//
//   [0, 256)            status word (int32, device error flags) + padding
//   decode_items        DecodeItem[n_decode_items]    (split-KV / cascade CTAs)
//   rows                RowDesc[n_decode_rows]        (query rows of those CTAs)
//   prefill_items       PrefillItem[n_prefill_items]  (tensor-core prefill CTAs)
//   combine             CombineEntry[n_combine]       (rows merged from partials)
//   row_merge           MergeRef[n_decode_rows]       (per row: its merge reference)
//   combine_count       int32[n_combine]              (arrival counters, zero)
//   stage_pages         int32[n_stage_pages]          (fp8 plans: cache pages the
//                                                      prefill reads, staged)
//   stage_bt            int32[n_reqs * max_blocks]    (fp8 plans: the prefill
//                                                      requests' block tables
//                                                      in staging page ids)
//   ---- metadata above is uploaded; scratch below is written by kernels ----
//   part_lse            float[n_partials]             (log2-domain LSE per partial)
//   part_o              float[n_partials * head_dim]  (normalised partial outputs)
//   stage_kv            bf16 K then V [n_stage_pages, n_kv_heads, page_size,
//                       head_dim] (fp8 plans: the staged pages, dequantized)
#pragma once

#include <stdint.h>

namespace mb {

constexpr int kStatusBytes = 256;
// int32 at this workspace offset (inside the status region, zero in the
// uploaded image): CTAs of a split-KV launch that finished, counted by the
// kernel launched behind the prefill kernel; its last CTA puts it back to zero
constexpr int kDoneCounterOffset = 4;
constexpr int kRowsPerDecodeItem = 128; // query rows one split-KV CTA owns (TMEM lanes)
constexpr int kPrefillTileM = 128;      // query rows per prefill tile (one TMEM accumulator)
constexpr int kPrefillTileN = 128;      // keys per prefill KV tile
constexpr int kPrefillCtaRows = 256;    // query rows per prefill CTA (two tiles)
constexpr int kCopyMinTiles = 8;        // 128-key tiles from which a split-KV CTA of <= 32
                                        // rows spreads each row's keys over 4 copies

// One CTA of the split-KV kernel: query rows (all of one KV head) against
// the key range [k_begin, k_end) of one block-table row.
struct DecodeItem {
  int32_t bt_row;     // block-table row that addresses the keys
  int32_t kv_head;
  int32_t k_begin;    // logical key range
  int32_t k_end;
  int32_t row_begin;  // first RowDesc
  int32_t n_rows;     // <= kRowsPerDecodeItem
  int32_t k_new;      // keys >= k_new may hold this step's appended rows (k_end: none)
  int32_t pad1;
};

struct RowDesc {
  int32_t q_index;  // flat token row of q / out
  int32_t q_head;
  int32_t vis_end;  // keys j < vis_end are visible to this row (S0 + i + 1)
  int32_t dst;      // >= 0: partial slot; < 0: final row, write out / lse
};

// One CTA of the prefill kernel: up to kPrefillCtaRows consecutive new rows
// of one request and one query head, against keys [0, n_kv_tiles * TileN).
struct PrefillItem {
  int32_t req;         // block-table row
  int32_t q_head;
  int32_t q_row0;      // flat token row of the tile's first row
  int32_t n_rows;      // valid rows in the tile
  int32_t s0;          // cached columns of the request
  int32_t i0;          // index of the tile's first row among the request's new rows
  int32_t kv_length;
  int32_t n_kv_tiles;  // ceil(min(kv_length, s0 + i0 + n_rows) / TileN)
};

struct CombineEntry {
  int32_t q_index;
  int32_t q_head;
  int32_t slot_begin;  // partial slots [slot_begin, slot_begin + n_slots)
  int32_t n_slots;
};

// Per decode row (parallel to the RowDesc array): where a split row's
// partials live and which arrival counter completes it.
struct MergeRef {
  int32_t entry;       // combine entry of the row; -1: the row is final
  int32_t n_slots;     // partials of the output row
  int32_t slot_begin;  // its first partial slot
  int32_t pad;
};

static_assert(sizeof(DecodeItem) == 32, "layout");
static_assert(sizeof(MergeRef) == 16, "layout");
static_assert(sizeof(RowDesc) == 16, "layout");
static_assert(sizeof(PrefillItem) == 32, "layout");
static_assert(sizeof(CombineEntry) == 16, "layout");

// Everything a forward needs from a plan.
struct PlanDevice {
  int32_t n_decode_items, n_decode_rows, n_prefill_items, n_combine, n_partials;
  int32_t n_q_heads, n_kv_heads, head_dim, page_size, num_pages, max_blocks;
  int32_t total_q;
  int32_t prefill_ctas;  // prefill grid when the split-KV kernel runs beside it
  int32_t decode_copies;  // split-KV build with row copies (most keys in long CTAs of <= 32 rows)
  int32_t decode_max_rows;  // largest n_rows of the split-KV CTAs
  float scale;
  size_t off_decode_items, off_rows, off_prefill_items, off_combine, off_row_merge,
      off_combine_count, off_part_lse, off_part_o;
  int32_t n_stage_pages;  // fp8 plans with prefill work: pages staged as bf16
  size_t off_stage_pages, off_stage_bt, off_stage_kv;
  size_t metadata_bytes, workspace_bytes;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace mb
