/*
 * mb_sched.h -- host iteration builder for the mixed-batch attention library.
 *
 * Builds, iteration by iteration, the inputs mb.h's calls take: the ragged
 * batch of (q_start, q_end, kv_length) triples, each request's block table
 * and the slot ("out_cache_loc") and logical position of every new row. Host
 * memory only; no CUDA call.
 *
 * The rules follow the pages:
 *   - iteration-level scheduling: requests join and leave between iterations,
 *     each iteration runs one step of every scheduled request ("ORCA and
 *     chunked prefill", sections 2-3);
 *   - every iteration has a budget of Q rows that decode steps and prefill
 *     chunks share; a long prompt is cut into chunks that piggyback on the
 *     running decodes ("ORCA and chunked prefill", sections 4-5);
 *   - a decode step computes decode_rows rows (1; k + 1 with speculative /
 *     MTP verification) and reuses its tail page until it is full; when the
 *     KV pool has too few free pages, the most recently admitted running
 *     request is preempted: returned to the waiting queue with its KV freed
 *     ("GLM-5.3 e2e token ledger", stage 3);
 *   - a prefix-cache hit does not allocate the matched prefix pages: it adds
 *     a reference to them and only the unmatched tail gets new pages
 *     ("GLM-5.3 e2e token ledger", stage 3, KV pages and prefix hits; "How To
 *     Scale Your Model notes (7-8)", section 3, shared prefixes).
 *
 * Policy where the pages leave it open: decode steps first (in admission
 * order), then the prefill chunks of admitted requests (admission order), then
 * new admissions first come first served; a prefill that does not fit the
 * free pages is shortened to whole free pages or waits (only decode steps
 * preempt, and a step that preempted admits nobody); prefix cache entries no
 * running request uses are dropped before any request is preempted. A
 * preempted request starts over (its KV is recomputed when it is readmitted).
 * After its last prefill chunk a request has its first output token; each
 * decode step then adds decode_rows tokens; it finishes when max_new_tokens
 * are out and its pages are released.
 *
 * Usage per iteration: mb_sched_step (build), run mb_kv_append / plan /
 * forward on its outputs, mb_sched_commit (advance). A step must be committed
 * before the next one. Errors are return codes (mb_status_t of mb.h).
 */
#ifndef MB_SCHED_H
#define MB_SCHED_H

#include <stdint.h>

#include "mb.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int32_t num_pages;           /* pages of the KV pool                           */
  int32_t page_size;           /* tokens per page                                */
  int32_t max_blocks_per_req;  /* block-table width (longest request / page_size) */
  int32_t token_budget;        /* Q rows per iteration (decode steps + chunks)   */
  int32_t max_running;         /* requests holding KV at once; 0 = no cap        */
  int32_t decode_rows;         /* rows per decode step; 0 -> 1                   */
} mb_sched_config_t;

typedef struct {
  int32_t n_reqs;       /* requests in the iteration                        */
  int32_t total_q;      /* Q rows                                           */
  int32_t n_prefill;    /* prefill chunks among them                        */
  int32_t n_decode;     /* decode steps among them                          */
  int32_t n_preempted;  /* requests preempted while building it             */
  int32_t n_prefix_hits;/* admissions that reused cached prefix pages       */
  int32_t n_waiting;    /* after the step                                   */
  int32_t n_running;
  int32_t n_finished;   /* since creation                                   */
  int32_t free_pages;
} mb_sched_stats_t;

/* Request states (mb_sched_request_info). */
#define MB_SCHED_WAITING 0
#define MB_SCHED_PREFILL 1
#define MB_SCHED_DECODE 2
#define MB_SCHED_FINISHED 3

typedef struct mb_sched mb_sched_t;

/* Create a scheduler. Errors: MB_ERR_INVALID_ARG (null, non-positive sizes,
 * page_size not a power of two in [16, 128]). */
mb_status_t mb_sched_create(const mb_sched_config_t* cfg, mb_sched_t** out);

/* Free the scheduler (host memory only). NULL is accepted. */
mb_status_t mb_sched_destroy(mb_sched_t* s);

/* Queue a request: prompt_len prompt tokens, then max_new_tokens outputs
 * (>= 1). prefix_id >= 0 marks the first prefix_len prompt positions as a
 * prefix shared with every request of the same id and the same prefix_len
 * (prefix_len a positive multiple of page_size, < prompt_len); -1: none. *request_id receives the
 * request's id (0, 1, ... in call order). Errors: MB_ERR_INVALID_ARG,
 * MB_ERR_SHAPE (the request can never fit: more blocks than
 * max_blocks_per_req or pages than the pool). */
mb_status_t mb_sched_add(mb_sched_t* s, int32_t prompt_len, int32_t max_new_tokens,
                         int32_t prefix_id, int32_t prefix_len, int32_t* request_id);

/* Build the next iteration into caller-owned host arrays:
 *   reqs_out[cap_reqs]                      triples, flat Q layout in order
 *   ids_out[cap_reqs]                       request id of each triple
 *   block_table_out[cap_reqs * max_blocks]  page ids, -1 past the request's pages
 *   slots_out[cap_rows], positions_out[cap_rows]  per Q row
 * stats (nullable) receives the counters. An empty iteration (nothing to run)
 * returns n_reqs = 0. Errors: MB_ERR_INVALID_ARG (null, a previous step not
 * committed), MB_ERR_WORKSPACE (caps too small: nothing is scheduled; retry
 * with cap_reqs >= live requests and cap_rows >= token_budget). */
mb_status_t mb_sched_step(mb_sched_t* s, mb_request_t* reqs_out, int32_t* ids_out,
                          int32_t* block_table_out, int32_t* slots_out,
                          int32_t* positions_out, int32_t cap_reqs, int32_t cap_rows,
                          mb_sched_stats_t* stats);

/* The built iteration ran: advance every scheduled request, retire finished
 * ones (their pages are released) and write their ids to finished_out
 * (nullable, up to cap entries; *n_finished receives the count). Errors:
 * MB_ERR_INVALID_ARG (no step to commit). */
mb_status_t mb_sched_commit(mb_sched_t* s, int32_t* finished_out, int32_t cap,
                            int32_t* n_finished);

/* Inspection (tests): reference count of every page (refs_out[num_pages]:
 * holders among requests and prefix cache entries; 0 = free). */
mb_status_t mb_sched_page_refs(const mb_sched_t* s, int32_t* refs_out, int32_t num_pages);

/* Inspection (tests): info_out[8] = state (MB_SCHED_*), computed positions,
 * generated tokens, pages held, preemptions, prompt_len, max_new_tokens,
 * prefix_id. Errors: MB_ERR_INVALID_ARG (unknown id). */
mb_status_t mb_sched_request_info(const mb_sched_t* s, int32_t request_id, int32_t* info_out);

#ifdef __cplusplus
}
#endif

#endif /* MB_SCHED_H */
