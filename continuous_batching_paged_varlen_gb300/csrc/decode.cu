// Split-KV attention for rows with few new queries (decode steps, small
// chunks) and for shared-prefix cascade groups.
//
// One CTA owns up to 128 query rows that all read the same KV head -- the g
// query heads of a GQA group ("How To Scale Your Model notes (7-8)",
// section 3: g queries share one KV head, so its K/V bytes are read once for
// all g of them) and, for a cascade group, the rows of every request whose
// block tables share the prefix pages ("How To Scale Your Model notes
// (7-8)", section 3: load a common KV block once, apply it to every sharing
// request's queries, each request keeping its own softmax state). The CTA
// walks the key range [k_begin, k_end) of one block-table row in 128-key
// tiles and keeps, per row, a running max, a running sum and the output
// accumulator; each key is masked by the row's own visibility bound
// (S0 + i + 1, "How To Scale Your Model notes (7-8)", section 2). The result
// is the final row (bf16 out + LSE) or, when the key range was split, a
// normalised partial (fp32 O, log2-domain LSE); the CTA that writes a row's
// last partial merges them all (combine.cuh).
//
// This path is bound by HBM bandwidth, so the design spends everything on
// keeping bytes in flight and almost nothing on issue slots:
//   warp 4      TMA producer: K_j, V_j, K_j+1, ... page by page through the
//               block table into a 7-slot ring (one box per page and 64-column
//               block, one lane per box), 128-byte swizzle. The ring takes all
//               of shared memory: the query rows live in TMEM, so a CTA whose
//               rate is set by its bytes in flight (beside the prefill kernel,
//               or with few rows) streams a seventh faster than with 6 slots.
//   warp 5      TMEM allocation; one lane issues S = Q K^T (M 128 = the
//               gathered rows from TMEM, N 128 keys, K = D) into a
//               double-buffered TMEM tile and O += P V (P from TMEM, V from
//               shared memory). The tensor core is mostly idle: it only
//               spares the CUDA cores.
//   warps 0-3   softmax: TMEM load of a row's scores, mask, online max / sum
//               in the log2 domain, P back into TMEM over the scores, rare O
//               rescale, epilogue. One thread per query row (only warps that
//               own real rows run), or, in the kCopies build for CTAs of at
//               most 32 rows and at least kCopyMinTiles key tiles (a decode
//               step's GQA group), each row copied into one lane of each of
//               the 4 warps, each copy keeping its own online softmax over 32
//               of every tile's 128 keys; the copies merge in the epilogue.
//               One row's exponentials then run on all 4 SM sub-partitions
//               instead of one, which is what paced the 4-row CTAs.
// Launch overlap: the kernel lets the next launch on the stream start at
// once and waits (griddepcontrol) for the launch before it only where it
// must: behind the KV append, before it reads q or a tile that holds this
// step's rows, reuses a ring slot or writes anything, so that history tiles
// stream while the append runs; behind its own forward's prefill kernel it
// runs on the SMs the prefill grid leaves free and its last CTA waits for the
// prefill before the grid completes.
// Every wait is bounded; on a timeout the CTA raises its abort flag, drains
// what it issued, frees its TMEM and returns.
#include <cuda_runtime.h>
#include <math.h>

#include "../../include/mb.h"
#include "combine.cuh"
#include "kernels.h"
#include "mb_device.cuh"

namespace mb {
namespace {

using namespace dev;

constexpr int BM = 128;  // gathered query rows (TMEM lanes)
constexpr int BN = 128;  // keys per tile
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;    // + 128 * buffer
constexpr uint32_t kColO = 256;
constexpr uint32_t kColQ = 384;  // the query rows, bf16 pairs (D / 2 columns)
constexpr float kRescaleThreshold = 8.0f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint64_t kDrainNs = 200000000ull;

enum {
  kSlots = 7,
  B_KV_FULL = 0,              // + slot
  B_KV_EMPTY = kSlots,        // + slot
  B_S_FULL = 2 * kSlots,      // + buffer
  // P(j) written / P(j) V(j) done, one barrier per tile parity: the softmax
  // warps may run a tile ahead of the PV that reads their P, so a single
  // barrier could complete twice before its waiter looks (parity waits
  // cannot tell those apart); per parity, no waiter falls two phases behind
  B_P_FULL = 2 * kSlots + 2,  // + (j & 1)
  B_O_DONE = 2 * kSlots + 4,  // + (j & 1)
  B_VZ_READY = 2 * kSlots + 6,
  B_EPI_FULL = 2 * kSlots + 7,  // the 4 softmax warps parked their copies (R > 1)
  B_COUNT = 2 * kSlots + 8
};

template <int D>
struct Layout {
  static constexpr int kHalves = D / 64;
  static constexpr uint32_t kHalfBytes = 128 * 128;
  static constexpr uint32_t kTileBytes = kHalves * kHalfBytes;
  static constexpr uint32_t kv_off = 0;
  static constexpr uint32_t bar_off = kv_off + kSlots * kTileBytes;
  static constexpr uint32_t misc_off = bar_off + B_COUNT * 8;
  static constexpr uint32_t kBytes = misc_off + 16;
  // + alignment slack; more than half the SM so that one CTA holds the SM's
  // 512 TMEM columns alone
  static constexpr uint32_t kAlloc =
      (kBytes + 1024 > 232448u / 2 + 1024) ? kBytes + 1024 : 232448u / 2 + 1024;
  static_assert(kAlloc <= 232448, "shared memory");
};

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// What the softmax warps share with the rest of the CTA.
struct SoftmaxShared {
  uint64_t* bars;
  volatile int* abort_flag;
  uint32_t tmem;
  float* redo;  // [4 * 32][D + 4]: the copies' O (the idle K/V ring, epilogue only)
  float* redm;  // [4 * 32]: the copies' running max, log2 units
  float* redl;  // [4 * 32]: the copies' running sum
};

// Softmax role of warp `warp` (0-3) for rows of W keys per copy. Rows: group
// g = warp % ngrp of 32 rows, copy c = warp / ngrp, with R = 128 / W copies
// of each row (ngrp = 4 / R groups). The Q tile holds row 32 g + i in TMEM
// lane 32 (g + ngrp c) + i for every copy c, so each copy's lane receives
// the row's scores of every key; copy c takes keys [c W, c W + W) of each
// tile with its own running max, sum and O accumulator (a split of the
// row's keys), writes its share of P and zeros elsewhere, and the epilogue
// merges the copies. Spreading a row over the 4 warps spreads its
// exponentials over the 4 SM sub-partitions: a few rows (a GQA group's g
// heads of one decode step) leave the MUFU of one sub-partition the limit
// otherwise, at ~2k cycles per 128-key tile.
template <int D, int W>
__device__ __forceinline__ void softmax_role(const DecodeArgs& a, const DecodeItem& it,
                                             const SoftmaxShared& sh, const RowDesc rd,
                                             const bool valid, const int n, const int warp,
                                             const int lane) {
  constexpr int R = BN / W;     // copies of a row
  constexpr int NGRP = 4 / R;   // row groups
  constexpr int RR = D + 4;     // floats per row of the epilogue buffer
  uint64_t* bars = sh.bars;
  const int c = warp / NGRP, g = warp % NGRP;
  const int col0 = c * W;  // this copy's first key of each tile
  // visible keys of this row inside the item: [k_begin, min(k_end, vis_end))
  const int vis_hi = min(it.k_end, rd.vis_end);
  const uint32_t lane_addr = (uint32_t)(warp * 32) << 16;
  const uint32_t o_col = sh.tmem + lane_addr + kColO;
  const float cs = a.scale_log2;
  float m = -INFINITY, l = 0.f;
  bool ok = true;
  for (int j = 0; j < n; ++j) {
    const uint32_t s_col = sh.tmem + lane_addr + kColS + 128 * (j & 1);
    ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_S_FULL + (j & 1)], (uint32_t)(j >> 1) & 1u,
                                           sh.abort_flag, a.status));
    if (!ok) break;
    tc_fence_after();
    uint32_t s[W];
    if constexpr (W == 128) {
      tmem_ld128(s_col, *reinterpret_cast<uint32_t(*)[128]>(&s[0]));
      tmem_ld_wait128(*reinterpret_cast<uint32_t(*)[128]>(&s[0]));
    } else {
#pragma unroll
      for (int h = 0; h < W / 32; ++h) {
        tmem_ld32(s_col + col0 + 32 * h, *reinterpret_cast<uint32_t(*)[32]>(&s[32 * h]));
        tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&s[32 * h]));
      }
    }
    const int lim = vis_hi - (it.k_begin + j * BN) - col0;  // keys e < lim are visible
    if (lim < W) {
#pragma unroll
      for (int e = 0; e < W; ++e)
        if (e >= lim) s[e] = __float_as_uint(-INFINITY);
    }
    constexpr int NM = W < 16 ? W : 16;
    float mx[NM];
#pragma unroll
    for (int k = 0; k < NM; ++k) mx[k] = __uint_as_float(s[k]);
#pragma unroll
    for (int e = NM; e < W; e += NM)
#pragma unroll
      for (int k = 0; k < NM; ++k) mx[k] = fmaxf(mx[k], __uint_as_float(s[e + k]));
#pragma unroll
    for (int w2 = NM / 2; w2 > 0; w2 >>= 1)
#pragma unroll
      for (int k = 0; k < w2; ++k) mx[k] = fmaxf(mx[k], mx[k + w2]);
    const float m_new = fmaxf(m, mx[0]);
    float alpha = 1.f;
    bool need = false;
    if (m == -INFINITY) {
      m = m_new;  // nothing accumulated yet (O is written with accumulate off or all-zero P)
    } else if ((m_new - m) * cs > kRescaleThreshold) {
      need = true;
      alpha = fast_exp2((m - m_new) * cs);
      l *= alpha;
      m = m_new;
    }
    const float mc = (m == -INFINITY) ? 0.f : m * cs;
    float sum[4] = {0.f, 0.f, 0.f, 0.f};
    uint32_t pk[W / 2];
#pragma unroll
    for (int e = 0; e < W; e += 2) {
      const float e0 = fast_exp2(fmaf(__uint_as_float(s[e]), cs, -mc));
      const float e1 = fast_exp2(fmaf(__uint_as_float(s[e + 1]), cs, -mc));
      sum[(e >> 1) & 3] += e0 + e1;
      pk[e >> 1] = pack_bf16x2(e0, e1);
    }
    l += (sum[0] + sum[1]) + (sum[2] + sum[3]);
    // P(j) goes over S(j) in buffer j & 1, which PV(j - 2) read last: S(j)
    // was issued after PV(j - 2), so that PV is done. Only a rescale of O
    // must wait for PV(j - 1), which accumulates into O (the only PV that
    // can still run: PV(j) needs this P). So the PV's latency stays off
    // the per-tile chain unless a copy's max grew by more than 2^8.
    if (__any_sync(0xffffffffu, need)) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_O_DONE + ((j - 1) & 1)],
                                             (uint32_t)((j - 1) >> 1) & 1u, sh.abort_flag,
                                             a.status));
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(o_col + cc * 32, o);
        tmem_ld_wait(o);
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
        tmem_st32(o_col + cc * 32, o);
      }
    }
    // P: the first 64 columns of the buffer hold the tile's 128 keys as bf16
    // pairs; this copy's W keys are its W / 2 columns and every other column
    // of its lanes is zero, so the PV sums only its own keys
    if constexpr (W == 128) {
      tmem_st32(s_col, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
      tmem_st32(s_col + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
    } else {
      uint32_t zero[W / 2];
#pragma unroll
      for (int e = 0; e < W / 2; ++e) zero[e] = 0u;
#pragma unroll
      for (int k = 0; k < R; ++k) {  // c is the same in every lane of the warp
        const uint32_t* src = k == c ? pk : zero;
        if constexpr (W == 64) {
          tmem_st32(s_col + 32 * k, *reinterpret_cast<const uint32_t(*)[32]>(src));
        } else {
          tmem_st16(s_col + 16 * k, src);
        }
      }
    }
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars[B_P_FULL + (j & 1)]);
  }
  if (ok && n > 0)
    ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_O_DONE + ((n - 1) & 1)],
                                           (uint32_t)((n - 1) >> 1) & 1u, sh.abort_flag,
                                           a.status));
  if (!ok || n == 0) return;
  tc_fence_after();
  const bool final_row = rd.dst < 0;
  const int64_t orow = (int64_t)rd.q_index * a.n_q_heads + rd.q_head;
  if constexpr (R == 1) {
    const bool any = l > 0.f;
    const float inv = any ? 1.f / l : 0.f;
    const float lse2 = any ? m * cs + log2f(l) : -INFINITY;
    // the TMEM loads are warp-collective: every lane runs them, whatever its
    // row; only the stores depend on the row
    uint4* dst_out = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + orow * D);
    float4* dst_part = reinterpret_cast<float4*>(a.part_o + (int64_t)max(rd.dst, 0) * D);
#pragma unroll
    for (int cc = 0; cc < D / 32; ++cc) {
      uint32_t o[32];
      tmem_ld32(o_col + cc * 32, o);
      tmem_ld_wait(o);
      if (valid && final_row) {
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint4 v;
          v.x = pack_bf16x2(__uint_as_float(o[q4 * 8 + 0]) * inv, __uint_as_float(o[q4 * 8 + 1]) * inv);
          v.y = pack_bf16x2(__uint_as_float(o[q4 * 8 + 2]) * inv, __uint_as_float(o[q4 * 8 + 3]) * inv);
          v.z = pack_bf16x2(__uint_as_float(o[q4 * 8 + 4]) * inv, __uint_as_float(o[q4 * 8 + 5]) * inv);
          v.w = pack_bf16x2(__uint_as_float(o[q4 * 8 + 6]) * inv, __uint_as_float(o[q4 * 8 + 7]) * inv);
          dst_out[cc * 4 + q4] = v;
        }
      } else if (valid) {
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4)
          dst_part[cc * 8 + q4] = make_float4(__uint_as_float(o[q4 * 4 + 0]) * inv,
                                              __uint_as_float(o[q4 * 4 + 1]) * inv,
                                              __uint_as_float(o[q4 * 4 + 2]) * inv,
                                              __uint_as_float(o[q4 * 4 + 3]) * inv);
      }
    }
    if (valid && final_row && a.lse) a.lse[orow] = lse2 * kLn2;
    if (valid && !final_row) {
      a.part_lse[rd.dst] = lse2;
      __threadfence();  // the partial is visible before this CTA counts it
    }
  } else {
    // merge the R copies of each row (splits of its keys): every warp parks
    // its lanes' max, sum and O, then finishes D / R columns of its row group
    // with weights 2^(m_c - M), M the largest copy max
    sh.redm[warp * 32 + lane] = m == -INFINITY ? -INFINITY : m * cs;
    sh.redl[warp * 32 + lane] = l;
    float* mine = sh.redo + (warp * 32 + lane) * RR;
#pragma unroll
    for (int cc = 0; cc < D / 32; ++cc) {
      uint32_t o[32];
      tmem_ld32(o_col + cc * 32, o);
      tmem_ld_wait(o);
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4)
        *reinterpret_cast<float4*>(mine + cc * 32 + q4 * 4) =
            make_float4(__uint_as_float(o[q4 * 4 + 0]), __uint_as_float(o[q4 * 4 + 1]),
                        __uint_as_float(o[q4 * 4 + 2]), __uint_as_float(o[q4 * 4 + 3]));
    }
    // every softmax warp runs when R > 1; a bounded wait, so that a warp
    // that gave up on an earlier wait cannot leave the others here
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars[B_EPI_FULL]);
    if (!__all_sync(0xffffffffu, mbar_wait(&bars[B_EPI_FULL], 0u, sh.abort_flag, a.status)))
      return;
    float mcp[R], wc[R];
    float M = -INFINITY;
#pragma unroll
    for (int cc = 0; cc < R; ++cc) {
      mcp[cc] = sh.redm[(g + NGRP * cc) * 32 + lane];
      M = fmaxf(M, mcp[cc]);
    }
    float lt = 0.f;
#pragma unroll
    for (int cc = 0; cc < R; ++cc) {
      wc[cc] = M == -INFINITY ? 0.f : fast_exp2(mcp[cc] - M);  // 0 for a copy with no key
      lt += wc[cc] * sh.redl[(g + NGRP * cc) * 32 + lane];
    }
    const bool any = lt > 0.f;
    const float inv = any ? 1.f / lt : 0.f;
    const float lse2 = any ? M + log2f(lt) : -INFINITY;
    constexpr int CW = D / R;  // columns this warp finishes
    const int cbeg = c * CW;
    if (valid) {
#pragma unroll 4
      for (int q4 = 0; q4 < CW / 4; ++q4) {
        const int col = cbeg + 4 * q4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int cc = 0; cc < R; ++cc) {
          const float4 v =
              *reinterpret_cast<const float4*>(sh.redo + ((g + NGRP * cc) * 32 + lane) * RR + col);
          acc.x = fmaf(wc[cc], v.x, acc.x);
          acc.y = fmaf(wc[cc], v.y, acc.y);
          acc.z = fmaf(wc[cc], v.z, acc.z);
          acc.w = fmaf(wc[cc], v.w, acc.w);
        }
        if (final_row) {
          uint2 w2;
          w2.x = pack_bf16x2(acc.x * inv, acc.y * inv);
          w2.y = pack_bf16x2(acc.z * inv, acc.w * inv);
          *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + orow * D + col) = w2;
        } else {
          *reinterpret_cast<float4*>(a.part_o + (int64_t)rd.dst * D + col) =
              make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        }
      }
      if (c == 0) {
        if (final_row && a.lse) a.lse[orow] = lse2 * kLn2;
        if (!final_row) a.part_lse[rd.dst] = lse2;
      }
      if (!final_row) __threadfence();  // each copy's columns are visible before the count
    }
  }
}

template <int D, bool kCopies>
__global__ void __launch_bounds__(kThreads, 1)
    splitkv_kernel(const DecodeArgs a, const int ps_shift,
                   const __grid_constant__ CUtensorMap k_map,
                   const __grid_constant__ CUtensorMap v_map) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* skv = smem + L::kv_off;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::bar_off);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::misc_off + 4);

  // the kernel behind this one (the next layer's append, say) may launch now
  pdl_launch_dependents();
  const bool dep_wait = a.after_prefill == 0;
  const DecodeItem it = a.items[blockIdx.x];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nr = it.n_rows;
  const int n = ceil_div(it.k_end - it.k_begin, BN);
  const bool tail_zero = it.k_begin + n * BN > it.k_end;
  // the kernel built with kCopies spreads each row's keys over 4 copies in
  // the 4 softmax warps (see softmax_role) when the CTA has at most 32 rows
  // and a long key range; otherwise one thread per row. The plan picks that
  // build when most of its keys sit in such CTAs: the copies' code makes the
  // kernel larger, which costs a short launch more (instruction fetch) than
  // the copies save it (measured on a shared-prefix step of 5-tile CTAs)
  const bool copies = kCopies && n >= kCopyMinTiles && nr <= 32;
  const int ngrp = copies ? 1 : 4;
  const int active_warps = ngrp < 4 ? 4 : ceil_div(nr, 32);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&bars[B_KV_FULL + s], 1);
      mbar_init(&bars[B_KV_EMPTY + s], 1);
    }
    mbar_init(&bars[B_S_FULL + 0], 1);
    mbar_init(&bars[B_S_FULL + 1], 1);
    mbar_init(&bars[B_P_FULL + 0], active_warps);
    mbar_init(&bars[B_P_FULL + 1], active_warps);
    mbar_init(&bars[B_O_DONE + 0], 1);
    mbar_init(&bars[B_O_DONE + 1], 1);
    mbar_init(&bars[B_VZ_READY], 1);
    mbar_init(&bars[B_EPI_FULL], 4);
    *abort_flag = 0;
    fence_barrier_init();
  }
  // Only the barriers are shared before the producer starts (a short step
  // has few tiles, so setup latencies would otherwise add up in series): it
  // issues K_0 at once, then waits until the other warps have issued their
  // Q loads, so that those enter the memory system ahead of the rest of the
  // ring (behind ~200 KB of copies per SM, a dependent gather waits
  // microseconds). Its first tile's page ids are loaded before the barrier.
  const int32_t* btrow = a.block_table + (int64_t)it.bt_row * a.max_blocks;
  const int last_block = (it.k_end - 1) >> ps_shift;
  const int first_block = it.k_begin >> ps_shift;  // k_begin is page-aligned
  int32_t page0 = 0;
  if (warp == 4 && n > 0 && lane < (BN >> ps_shift))
    page0 = __ldg(btrow + min(first_block + lane, last_block));
  // each softmax lane's row (group warp % ngrp): its descriptor is loaded
  // now, so that its latency overlaps the set-up and the Q gather
  const int my_row = (warp % ngrp) * 32 + lane;
  const bool row_valid = warp < 4 && warp < active_warps && my_row < nr;
  RowDesc rd;
  rd.q_index = 0;
  rd.q_head = 0;
  rd.vis_end = 0;
  rd.dst = -1;
  if (row_valid) rd = a.rows[it.row_begin + my_row];
  // thread t < n_rows counts row t's arrival at the end (split rows): its
  // merge reference and output row, loaded now as well
  MergeRef my_ref = {-1, 0, 0, 0};
  int32_t my_out_row = 0;
  if (a.combine_count && (int)threadIdx.x < nr) {
    my_ref = a.row_merge[it.row_begin + threadIdx.x];
    const RowDesc md = a.rows[it.row_begin + threadIdx.x];
    my_out_row = md.q_index * a.n_q_heads + md.q_head;
  }
  __syncthreads();
  uint32_t tmem = 0;
  if (warp != 4) {
    if (warp == 5) {
      tmem_alloc(tmem_slot, kTmemCols);
      tmem_relinquish();
    }
    // the item's query rows go to TMEM, where the S MMA reads its A operand:
    // softmax warp w writes tile rows 32 w .. 32 w + 31 into its own lanes,
    // tile row t holding item row 32 ((t / 32) % ngrp) + t % 32 (each row
    // once per copy; rows past n_rows zero). The loads are in flight before
    // the producer is released, the stores follow once TMEM is allocated.
    // q may be the kernel ahead's output (a rotary append rewrites it)
    if (dep_wait) pdl_wait();
    constexpr int CH = D / 8;  // 16-byte chunks per row
    uint4 qv[CH];
    if (warp < 4) {
      const uint4* q = static_cast<const uint4*>(a.q);
      const bool qrow = my_row < nr;
      const RowDesc qd = qrow ? a.rows[it.row_begin + my_row] : rd;
      const uint4* src = q + ((int64_t)qd.q_index * a.n_q_heads + qd.q_head) * CH;
#pragma unroll
      for (int c = 0; c < CH; ++c) qv[c] = qrow ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
    }
    named_barrier_arrive(2, kThreads);  // the producer's wait below
    tc_fence_before();
    named_barrier_sync(1, kThreads - 32);
    tc_fence_after();
    tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
    if (warp < 4) {
      const uint32_t qcol = tmem + ((uint32_t)(warp * 32) << 16) + kColQ;
#pragma unroll
      for (int h = 0; h < CH / 8; ++h)
        tmem_st32(qcol + 32 * h, *reinterpret_cast<const uint32_t(*)[32]>(&qv[8 * h]));
      tmem_st_wait();
    }
    tc_fence_before();
    named_barrier_sync(3, kThreads - 32);  // Q in TMEM before the first S MMA
    tc_fence_after();
  }

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    const int ps = 1 << ps_shift;
    const int npg = BN / ps, nbox = npg * L::kHalves;
    const int my_pg = lane % npg, my_h2 = lane / npg;
    int32_t my_y = 0;
    int32_t page_next = page0;  // keys past k_end map to the last page: masked, V zeroed
    int issued = 0;
    // dep_wait: history keys were written before the kernel ahead ran, so
    // the ring fills with them at once; the wait for that kernel comes at the
    // first tile that reaches this step's new rows, or before the first slot
    // is reused (so no bounded wait below runs while the kernel ahead does).
    // Then, as without dep_wait after K_0, the producer lets the Q loads
    // (issued by the other warps right after their own wait) go first.
    bool waited = !dep_wait, q_first = false;
    for (int i = 0; i < 2 * n; ++i) {
      const int j = i >> 1, slot = i % kSlots;
      const uint32_t ph = (uint32_t)(i / kSlots) & 1u;
      if (!waited && (i >= kSlots || it.k_begin + (j + 1) * BN > it.k_new)) {
        pdl_wait();
        waited = true;
      }
      if (!q_first && waited && (dep_wait || i == 1)) {
        named_barrier_sync(2, kThreads);  // every Q load issued
        q_first = true;
      }
      if (i >= kSlots &&
          !__all_sync(0xffffffffu, mbar_wait(&bars[B_KV_EMPTY + slot], ph ^ 1u, abort_flag,
                                             a.status)))
        break;
      if ((i & 1) == 0 && lane < npg) {
        // this lane's page of K_j / V_j, loaded one K tile ahead: the load's
        // latency then overlaps the waits and copies of the tile before it
        // (a dependent load here would stall every refill of the ring)
        int32_t page = page_next;
        if (j + 1 < n)
          page_next = __ldg(btrow + min(first_block + (j + 1) * npg + lane, last_block));
        if ((unsigned)page >= (unsigned)a.num_pages) {
          set_status(a.status, MB_ERR_DEVICE_INDEX);
          page = 0;
        }
        my_y = (page * a.n_kv_heads + it.kv_head) << ps_shift;
      }
      const int32_t y = __shfl_sync(0xffffffffu, my_y, my_pg);
      if (lane == 0) mbar_arrive_expect_tx(&bars[B_KV_FULL + slot], L::kTileBytes);
      __syncwarp();
      if (lane < nbox)
        tma_load_2d(skv + slot * L::kTileBytes + my_h2 * L::kHalfBytes + my_pg * ps * 128,
                    (i & 1) ? &v_map : &k_map, &bars[B_KV_FULL + slot], my_h2 * 64, y);
      issued = i + 1;
    }
    __syncwarp();
    if (tail_zero && issued == 2 * n) {
      // keys >= k_end in the last V tile: zero their rows (P is 0 there, and
      // an unwritten slot may hold a non-finite value)
      const int i = 2 * n - 1, slot = i % kSlots;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_KV_FULL + slot],
                                                        (uint32_t)(i / kSlots) & 1u, abort_flag,
                                                        a.status));
      if (ok) {
        const int r0 = it.k_end - (it.k_begin + (n - 1) * BN);
        const int nz = BN - r0;
        uint8_t* vb = skv + slot * L::kTileBytes;
        for (int idx = lane; idx < nz * L::kHalves * 8; idx += 32) {
          const int c = idx & 7;
          const int rr = idx >> 3;
          const int h2 = rr / nz;
          const int row = r0 + (rr - h2 * nz);
          *reinterpret_cast<uint4*>(vb + h2 * L::kHalfBytes + row * 128 + c * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_VZ_READY]);
    }
    if (lane == 0)
      for (int i = max(0, issued - kSlots); i < issued; ++i)
        mbar_drain(&bars[B_KV_FULL + i % kSlots], (uint32_t)(i / kSlots) & 1u, kDrainNs);
    // this warp also writes merged rows below
    if (!waited) pdl_wait();
    if (!q_first && n > 0) named_barrier_sync(2, kThreads);
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(BM, BN, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(BM, D, false, true);
      const uint32_t kva = smem_u32(skv);
      int last_pv = -1;
      auto wait = [&](int b, uint32_t parity) -> bool {
        const bool ok = mbar_wait(&bars[b], parity, abort_flag, a.status);
        tc_fence_after();
        return ok;
      };
      auto issue_s = [&](int j) -> bool {
        const int ki = 2 * j;
        if (!wait(B_KV_FULL + ki % kSlots, (uint32_t)(ki / kSlots) & 1u)) return false;
        const uint32_t k0 = kva + (ki % kSlots) * L::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * L::kHalfBytes + (kk & 3) * 32;
          umma_bf16_ts(tmem + kColS + 128 * (j & 1), tmem + kColQ + kk * 8,
                       sdesc_sw128(k0 + off, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
        }
        umma_commit(&bars[B_S_FULL + (j & 1)]);
        umma_commit(&bars[B_KV_EMPTY + ki % kSlots]);
        return true;
      };
      bool ok = n > 0 && issue_s(0);
      if (ok && n > 1) ok = issue_s(1);
      for (int j = 0; ok && j < n; ++j) {
        const int vi = 2 * j + 1;
        if (!(ok = wait(B_KV_FULL + vi % kSlots, (uint32_t)(vi / kSlots) & 1u))) break;
        if (j == n - 1 && tail_zero && !(ok = wait(B_VZ_READY, 0))) break;
        if (!(ok = wait(B_P_FULL + (j & 1), (uint32_t)(j >> 1) & 1u))) break;
        const uint32_t v0 = kva + (vi % kSlots) * L::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          const uint64_t bd = sdesc_sw128(v0 + kk * 2048, L::kHalfBytes, 1024);
          umma_bf16_ts(tmem + kColO, tmem + kColS + 128 * (j & 1) + kk * 8, bd, idesc_pv,
                       (j > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&bars[B_O_DONE + (j & 1)]);
        umma_commit(&bars[B_KV_EMPTY + vi % kSlots]);
        last_pv = j;
        // S(j+2) reuses this buffer; it follows PV(j) in issue order
        if (j + 2 < n && !(ok = issue_s(j + 2))) break;
      }
      if (last_pv >= 0)
        mbar_drain(&bars[B_O_DONE + (last_pv & 1)], (uint32_t)(last_pv >> 1) & 1u, kDrainNs);
    }
  } else if (warp < active_warps) {
    // ------------------------------------------------------------ softmax
    SoftmaxShared sh;
    sh.bars = bars;
    sh.abort_flag = abort_flag;
    sh.tmem = tmem;
    // the epilogue's buffers: the K/V ring, idle once the last PV is done
    sh.redo = reinterpret_cast<float*>(skv);
    sh.redm = sh.redo + 128 * (D + 4);
    sh.redl = sh.redm + 128;
    if constexpr (kCopies) {
      if (copies)
        softmax_role<D, 32>(a, it, sh, rd, row_valid, n, warp, lane);
      else
        softmax_role<D, 128>(a, it, sh, rd, row_valid, n, warp, lane);
    } else {
      softmax_role<D, 128>(a, it, sh, rd, row_valid, n, warp, lane);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (a.combine_count) {
    // one arrival per split row (also after an abort: the counters must stay
    // in step for the next launch); the CTA whose arrival completes a row
    // merges it. Every partial write of this CTA was fenced before the
    // barrier above. Scratch: the K/V ring, every copy landed and read.
    dev::MergeArgs mg;
    mg.rows = a.rows + it.row_begin;
    mg.refs = a.row_merge + it.row_begin;
    mg.n_rows = nr;
    mg.count = a.combine_count;
    mg.part_o = a.part_o;
    mg.part_lse = a.part_lse;
    mg.n_q_heads = a.n_q_heads;
    mg.out = static_cast<__nv_bfloat16*>(a.out);
    mg.lse = a.lse;
    dev::merge_completed_rows<D, kThreads>(mg, reinterpret_cast<uint32_t*>(skv), true, my_ref,
                                           my_out_row);
  }
  if (!dep_wait && threadIdx.x == 0) {
    // started under the prefill kernel's tail: the grid must not complete
    // before that kernel does (what follows on the stream counts on it), so
    // the last CTA to finish waits for it
    __threadfence();
    if (atomicAdd(a.done_counter, 1) == (int)gridDim.x - 1) {
      pdl_wait();
      atomicExch(a.done_counter, 0);
    }
  }
}

template <int D, bool kCopies>
cudaError_t launch_d(const DecodeArgs& a, cudaStream_t s, bool overlap_previous, int ps_shift) {
  static OncePerDevice setup;
  cudaError_t e = setup.run([](int) {
    return cudaFuncSetAttribute(splitkv_kernel<D, kCopies>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)Layout<D>::kAlloc);
  });
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.n_items);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Layout<D>::kAlloc;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap_previous ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, splitkv_kernel<D, kCopies>, a, ps_shift, *a.k_map, *a.v_map);
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s, bool overlap_previous) {
  if (a.n_items <= 0) return cudaSuccess;
  const int ps_shift = __builtin_ctz((unsigned)a.page_size);
  if (a.head_dim == 128)
    return a.copies ? launch_d<128, true>(a, s, overlap_previous, ps_shift)
                    : launch_d<128, false>(a, s, overlap_previous, ps_shift);
  return a.copies ? launch_d<64, true>(a, s, overlap_previous, ps_shift)
                  : launch_d<64, false>(a, s, overlap_previous, ps_shift);
}

}  // namespace mb
