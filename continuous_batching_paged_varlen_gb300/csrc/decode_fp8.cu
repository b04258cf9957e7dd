// Split-KV attention over an fp8 (e4m3) KV cache with per-row fp32 scales.
//
// "GLM-5.3 e2e token ledger", the KV layout paragraphs: the cache holds K/V
// as FP8 codes with FP32 scales stored beside them, and the attention kernel
// reads both to dequantize. Here every (token, KV head) row of D codes has
// one scale: k = decode(code) * scale. The work lists are the ones the
// bf16 split-KV kernel runs (one CTA = up to 128 query rows of one KV head
// against the key range [k_begin, k_end) of one block-table row, "How To
// Scale Your Model notes (7-8)", section 3), and the results are the same
// final rows or normalised partials, merged by the CTA that completes a row
// (combine.cuh).
//
// The scales of key j factor out of both products:
//   S[r][j] = ks_j sq_r (qc_r . kcode_j)    O[r] = rho sum_j p[r][j] (vs_j / rho) vcode_j
//   * Q K^T runs on the raw e4m3 K codes (kind::f8f6f4, fp32 accumulation):
//     each query row q is written as sq (hi + lo) with sq = amax|q| / 448,
//     hi = e4m3(q / sq) and lo = e4m3(q / sq - hi), two e4m3 rows whose
//     products with the K tile add up in the same accumulator. hi + lo holds
//     q to about 2^-8 of each value (near bf16's 2^-9), so the split costs
//     the scores about what bf16 Q costs them, and no K value is converted.
//   * P V' runs on f16 operands: V' = vcode_j (vs_j / rho) and P = p. rho is
//     the smallest power of two at least as large as every V scale of the
//     CTA's keys, so V' stays within +-448 whatever the magnitude of V, and
//     O = rho (P V') / l.
//   The softmax applies ks_j sq_r (times log2(e) and the softmax scale) to
//   the scores.
//
// Roles (352 threads):
//   warp 8      K copies: K tiles by TMA, one box per page, straight into the
//               128-byte (64-byte for D = 64) swizzled K-major operand layout
//               of a 4-slot ring (8 for D = 64), each page's ps scales by bulk
//               copy beside them.
//   warp 10     V copies: V codes and scales by bulk copy into a 5-slot
//               staging ring (6). Two streams, each paced by its own ring: one
//               warp issuing both kept the rings from running ahead (each of
//               its waits and issues took ~500 cycles beside the converters'
//               shared-memory traffic; one K + V pair per tile period).
//   warps 4-7   V converters: first the item's largest V scale (read from
//               the scale array) sets rho; then 16 staged codes -> 8 f16x2
//               words per task, times the key's vs / rho, into the operand
//               tiles of a 2-slot ring (rows past k_end zeroed).
//   warp 9      TMEM allocation; one lane issues S = Q K^T (the hi and lo
//               rows of Q from TMEM) and O += P' V (P' from TMEM). S has one
//               buffer: S(j+1) is issued, ahead of PV(j), as soon as the
//               softmax warps have read S(j) into registers. P has two (by
//               tile parity), so the softmax of tile j waits only for
//               PV(j-2) before writing its P (and for PV(j-1) when it must
//               rescale O).
//   warps 0-3   softmax; each thread first writes its query row's hi / lo
//               codes to TMEM. With few rows (a decode step's g query heads),
//               each row is copied into 4 (or 2) TMEM lanes of different
//               warps and each copy handles 32 (or 64) of the tile's 128
//               keys, so the exponentials of one row spread over the 4 SM
//               sub-partitions. Each copy keeps its own running max, sum and
//               accumulator (a split-KV partition of the row's keys); the
//               epilogue merges them.
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

constexpr int BM = 128;  // TMEM lanes (query rows, possibly copied)
constexpr int BN = 128;  // keys per tile
constexpr int kThreads = 352;  // warps 0-9 as below, warp 10 the V copy stream
constexpr uint32_t kQBarCount = 128 + 2 * 32;  // softmax warps + the two copy streams
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;    // S: one 128-key tile, read out by the softmax before S(j+1)
constexpr uint32_t kColO = 256;  // D columns
constexpr uint32_t kColQ = 384;  // hi codes (D / 4 columns), then lo codes
constexpr uint32_t kColP = 128;  // P: two buffers of 64 f16x2 columns (128 keys), by tile parity
constexpr float kRescaleThreshold = 8.0f;
constexpr uint64_t kDrainNs = 200000000ull;
constexpr int kVOpSlots = 2;          // f16 V operand tiles: V_j in slot j % 2, freed by PV(j)'s
                                      // barrier of the same parity (B_O_DONE + j % 2)
constexpr int kMaxSlots = 8;

enum {
  B_K_FULL = 0,                          // + K slot
  B_K_EMPTY = B_K_FULL + kMaxSlots,      // + K slot (the 4 softmax warps, after S(j))
  B_VS_FULL = B_K_EMPTY + kMaxSlots,     // + V staging slot
  B_VS_EMPTY = B_VS_FULL + kMaxSlots,    // + V staging slot
  B_S_FULL = B_VS_EMPTY + kMaxSlots,     // S(j) computed
  B_S_FREE = B_S_FULL + 1,               // the 4 softmax warps have read S(j) out
  B_PV_READY = B_S_FREE + 1,             // + P buffer: P(j) written (4 softmax warps) and
                                         // V_j converted (4 converter warps), j of that parity
  B_O_DONE = B_PV_READY + 2,             // + P buffer: P(j) V(j) done, j of that parity
  B_RHO_READY = B_O_DONE + 2,            // converters' partial maxima of the V scales
  B_EPI_FULL = B_RHO_READY + 1,
  B_Q_READY = B_EPI_FULL + 1,
  B_MMA_DONE = B_Q_READY + 1,
  // the few-row kernel's own: S buffers full / read out, and the softmax
  // warps' per-tile exchange of row maxima (two of each, by tile parity)
  B_T_S_FULL = B_MMA_DONE + 1,
  B_T_S_FREE = B_T_S_FULL + 2,
  B_RED_FULL = B_T_S_FREE + 2,
  B_COUNT = B_RED_FULL + 2
};

template <int D>
struct Layout {
  static constexpr int kHalves = D / 64;
  static constexpr uint32_t kHalfBytes = 128 * 128;  // 128 rows x 64 16-bit values
  static constexpr uint32_t kVOpBytes = kHalves * kHalfBytes;
  static constexpr uint32_t kCodes = BN * D;  // e4m3 codes of one tile
  // K slot: the swizzled code tile, then its scales, padded to 1024 bytes
  static constexpr uint32_t kKSlot = (kCodes + BN * 4 + 1023) & ~1023u;
  // K ring and V staging in the same shared memory: the V stream's depth
  // paces the kernel more than the K ring's (measured 4 / 5 against 6 / 3:
  // 2 % faster on the 256-decode batch)
  static constexpr int kKSlots = D == 128 ? 4 : 8;
  static constexpr uint32_t kVStBytes = kCodes + BN * 4;
  static constexpr int kVStSlots = D == 128 ? 5 : 6;
  static constexpr uint32_t k_off = 0;
  static constexpr uint32_t vop_off = k_off + kKSlots * kKSlot;
  static constexpr uint32_t vst_off = vop_off + kVOpSlots * kVOpBytes;
  static constexpr uint32_t redm_off = vst_off + kVStSlots * kVStBytes;  // float [4][32]
  static constexpr uint32_t redl_off = redm_off + 4 * 32 * 4;             // float [4][32]
  static constexpr uint32_t bar_off = redl_off + 4 * 32 * 4;
  // TMEM address, abort flag, the converters' 4 partial maxima of the V scales
  static constexpr uint32_t misc_off = (bar_off + B_COUNT * 8 + 15) & ~15u;
  static constexpr uint32_t kBytes = misc_off + 32;
  // more than half the SM so that one CTA holds the SM's 512 TMEM columns
  static constexpr uint32_t kAlloc =
      (kBytes + 1024 > 232448u / 2 + 1024) ? kBytes + 1024 : 232448u / 2 + 1024;
  // the epilogue adds the row copies' outputs in the (then idle) K ring
  static constexpr int kRedRow = D + 4;  // floats per row, padded against bank conflicts
  static_assert(kKSlots <= kMaxSlots && kVStSlots <= kMaxSlots, "rings");
  static_assert(kVOpSlots == 2, "V operand slots are freed by the P-buffer barriers");
  static_assert(4 * 32 * kRedRow * 4 <= kKSlots * kKSlot, "reduction buffer");
  static_assert(kAlloc <= 232448, "shared memory");
  static_assert(misc_off % 16 == 0, "misc alignment");
};

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// (lo, hi) fp32 -> two e4m3 codes (lo in the low byte), nearest, saturating.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// Smallest power of two >= x, for finite x > 0.
__device__ __forceinline__ float pow2_ceil(float x) {
  const uint32_t b = __float_as_uint(x);
  uint32_t e = b & 0x7f800000u;
  if ((b & 0x007fffffu) != 0u || e == 0u) e += 0x00800000u;
  return __uint_as_float(e);
}
// Four scaled values y0..y3 -> hi codes and lo codes (lo = e4m3(y - hi)),
// one 32-bit word each, y0 in the lowest byte.
__device__ __forceinline__ void split4(float y0, float y1, float y2, float y3, uint32_t& hi,
                                       uint32_t& lo) {
  const uint32_t h01 = f32x2_to_e4m3x2(y0, y1), h23 = f32x2_to_e4m3x2(y2, y3);
  float d0, d1, d2, d3;
  f16x2_to_f32x2(e4m3x2_to_f16x2(h01), d0, d1);
  f16x2_to_f32x2(e4m3x2_to_f16x2(h23), d2, d3);
  hi = h01 | (h23 << 16);
  lo = f32x2_to_e4m3x2(y0 - d0, y1 - d1) | (f32x2_to_e4m3x2(y2 - d2, y3 - d3) << 16);
}

// Shared-memory loads by shared-window address. The softmax reaches its
// buffers through a struct of pointers, where the compiler cannot see the
// state space and would issue generic loads; these stay ld.shared. They are
// volatile so that none moves above the barrier wait that publishes the data.
__device__ __forceinline__ float4 lds4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ uint4 lds4u(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts4u(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ float lds1(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}

struct Shared {
  uint64_t* bars;
  volatile int* abort_flag;
  const uint8_t* kring;  // K slots (codes, then scales)
  const float* rho4;     // the converters' 4 partial maxima of the V scales
  float* redm;           // [4][32]
  float* redl;           // [4][32]
  float* redo;           // [4][32][D + 4] (K ring, epilogue only)
  uint32_t tmem;
};

// rho: the smallest power of two >= every V scale of the item (0 when all
// are 0), from the converters' partial maxima.
__device__ __forceinline__ float rho_of(const float* rho4) {
  const float4 v = lds4(smem_u32(rho4));
  const float mx = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
  return mx > 0.f ? pow2_ceil(mx) : 0.f;
}

// Softmax role of warp `warp` (0-3). Rows: group g = warp % ngrp of 32 rows,
// copy c = warp / ngrp; W = 128 / R keys of every tile per copy (R = 4 / ngrp
// copies of each row). Each copy runs its own online softmax over its keys
// (its own running max m, sum l and TMEM accumulator lane): the copies of a
// row are split-KV partitions by key, merged in the epilogue.
template <int D, int W>
__device__ __forceinline__ void softmax_role(const DecodeFp8Args& a, const DecodeItem& it,
                                             const Shared& sh, int n, int warp, int lane) {
  constexpr int R = BN / W;
  constexpr int ngrp = 4 / R;
  using L = Layout<D>;
  uint64_t* bars = sh.bars;
  const int g = warp % ngrp, c = warp / ngrp;
  const int r = 32 * g + lane;
  const bool valid = r < it.n_rows;
  RowDesc rd;
  rd.q_index = 0;
  rd.q_head = 0;
  rd.vis_end = 0;
  rd.dst = -1;
  if (valid) rd = a.rows[it.row_begin + r];
  const uint32_t lane_addr = (uint32_t)(warp * 32) << 16;

  // this lane's query row as sq * (hi + lo), the hi / lo codes into TMEM
  // (the A operands of Q K^T); lanes without a row hold zeros. The row's
  // loads are all issued before the copy streams pass their first tile,
  // so they reach memory ahead of the rest of the ring.
  float sq = 0.f;
  {
    const uint4* qrow = static_cast<const uint4*>(a.q) +
                        ((int64_t)rd.q_index * a.n_q_heads + rd.q_head) * (D / 8);
    uint4 qb[D / 8];
#pragma unroll
    for (int k = 0; k < D / 8; ++k) qb[k] = valid ? __ldg(qrow + k) : make_uint4(0u, 0u, 0u, 0u);
    named_barrier_arrive(2, kQBarCount);  // the copy streams' wait
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < D / 8; ++k) {
      const uint32_t wv[4] = {qb[k].x, qb[k].y, qb[k].z, qb[k].w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        amax = fmax3(amax, fabsf(bf16_lo(wv[e])), fabsf(bf16_hi(wv[e])));
    }
    sq = amax * (1.f / 448.f);
    const float inv = amax > 0.f ? 448.f / amax : 0.f;
    constexpr int QW = D / 4;  // 32-bit columns per code row
    constexpr int QH = QW < 32 ? QW : 32;
#pragma unroll
    for (int hh = 0; hh < QW / QH; ++hh) {
      uint32_t hi[QH], lo[QH];
#pragma unroll
      for (int k = 0; k < QH / 2; ++k) {  // one 16-byte chunk = 8 values = 2 columns
        uint4 b = make_uint4(0u, 0u, 0u, 0u);  // the row again, from L1
        if (valid) b = __ldg(qrow + hh * (QH / 2) + k);
        split4(bf16_lo(b.x) * inv, bf16_hi(b.x) * inv, bf16_lo(b.y) * inv, bf16_hi(b.y) * inv,
               hi[2 * k], lo[2 * k]);
        split4(bf16_lo(b.z) * inv, bf16_hi(b.z) * inv, bf16_lo(b.w) * inv, bf16_hi(b.w) * inv,
               hi[2 * k + 1], lo[2 * k + 1]);
      }
      if constexpr (QH == 32) {
        tmem_st32(sh.tmem + lane_addr + kColQ + 32 * hh, hi);
        tmem_st32(sh.tmem + lane_addr + kColQ + QW + 32 * hh, lo);
      } else {
        tmem_st16(sh.tmem + lane_addr + kColQ, hi);
        tmem_st16(sh.tmem + lane_addr + kColQ + QW, lo);
      }
    }
    // P starts as zeros; each copy then rewrites only its own keys' columns
    {
      uint32_t zero[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) zero[e] = 0u;
#pragma unroll
      for (int z = 0; z < 4; ++z) tmem_st32(sh.tmem + lane_addr + kColP + 32 * z, zero);
    }
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars[B_Q_READY]);
  }

  const int vis_hi = min(it.k_end, rd.vis_end);
  const uint32_t o_col = sh.tmem + lane_addr + kColO;
  const uint32_t p_base = sh.tmem + lane_addr + kColP;
  const int col0 = c * W;
  const float crow = a.scale_log2 * sq;  // this row's factor of every score
  float m = -INFINITY, l = 0.f;
  bool ok = true;
  for (int j = 0; j < n; ++j) {
    const int ks_slot = j % L::kKSlots;
    const uint32_t p_col = sh.tmem + lane_addr + kColS;
    const uint32_t p_buf = p_base + 64 * (j & 1);  // this tile's P buffer
    ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_S_FULL], (uint32_t)j & 1u, sh.abort_flag,
                                           a.status));
    if (!ok) break;
    tc_fence_after();
    // K_j (its scales arrive with its codes) and K_(j+1): the MMA thread
    // issues S(j+1) on this warp's release of S(j) alone. K_j was waited
    // for one tile earlier, except the first.
    for (int jj = j == 0 ? 0 : j + 1; jj <= j + 1 && jj < n; ++jj) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_K_FULL + jj % L::kKSlots],
                                             (uint32_t)(jj / L::kKSlots) & 1u, sh.abort_flag,
                                             a.status));
      if (!ok) break;
    }
    if (!ok) break;
    // scores in the log2 domain: ks_j sq log2(e) scale (qc . kcode_j), keys
    // past the row's visibility bound at -inf
    const uint32_t kf = smem_u32(sh.kring + ks_slot * L::kKSlot + L::kCodes) + 4 * col0;
    const int lim = vis_hi - (it.k_begin + j * BN) - col0;  // columns e < lim are visible
    // up to 64 columns stay in registers; 128 take a second pass over TMEM
    // (the max first, then the exponentials), which keeps the role within
    // the 168 registers a 320-thread CTA has per thread
    constexpr int KEEP = W <= 64 ? W : 32;
    uint32_t s[KEEP];
    auto scaled_chunk = [&](int h, uint32_t* x) {
      tmem_ld32(p_col + col0 + 32 * h, *reinterpret_cast<uint32_t(*)[32]>(x));
      tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(x));
#pragma unroll
      for (int e4 = 0; e4 < 8; ++e4) {
        const float4 f = lds4(kf + 4 * (32 * h + 4 * e4));
        const float fv[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int e = 4 * e4 + q;
          x[e] = __float_as_uint(32 * h + e < lim ? __uint_as_float(x[e]) * (fv[q] * crow)
                                                  : -INFINITY);
        }
      }
    };
    float mx = -INFINITY;
#pragma unroll
    for (int h = 0; h < W / 32; ++h) {
      uint32_t* x = W <= 64 ? &s[32 * h] : s;
      scaled_chunk(h, x);
#pragma unroll
      for (int e = 0; e < 32; ++e) mx = fmaxf(mx, __uint_as_float(x[e]));
    }
    // S is in registers: S(j+1) may overwrite it (W = 128 reads it again
    // below); K_(j+1) has landed (waited for above)
    auto s_free = [&]() {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_S_FREE]);
    };
    if constexpr (W <= 64) s_free();
    const float m_new = fmaxf(m, mx);
    float alpha = 1.f;
    bool need = false;
    if (m == -INFINITY) {
      m = m_new;
    } else if (m_new - m > kRescaleThreshold) {
      need = true;
      alpha = fast_exp2(m - m_new);
      l *= alpha;
      m = m_new;
    }
    const float mc = (m == -INFINITY) ? 0.f : m;
    // P = p in f16 (V carries vs / rho) for this copy's keys, into the P
    // columns once P(j-1) V(j-1) has read them; the other copies' columns
    // stay zero
    constexpr int kChunks = W / 32;  // 32-key chunks of this copy
    float sum[2] = {0.f, 0.f};
    auto exps = [&](const uint32_t* x, uint32_t* pk) {
#pragma unroll
      for (int e4 = 0; e4 < 8; ++e4) {
        const float p0 = fast_exp2(__uint_as_float(x[4 * e4]) - mc);
        const float p1 = fast_exp2(__uint_as_float(x[4 * e4 + 1]) - mc);
        const float p2 = fast_exp2(__uint_as_float(x[4 * e4 + 2]) - mc);
        const float p3 = fast_exp2(__uint_as_float(x[4 * e4 + 3]) - mc);
        sum[0] += p0 + p2;
        sum[1] += p1 + p3;
        pk[2 * e4] = pack_f16x2(p0, p1);
        pk[2 * e4 + 1] = pack_f16x2(p2, p3);
      }
    };
    // P(j-2) V(j-2) done: this tile's P buffer may be rewritten; when the
    // warp rescales O, P(j-1) V(j-1) too (O is stable; P has two buffers, so
    // it may still run otherwise). Each P buffer's barrier completes every
    // other tile and is waited for at every completion, so no wait is two
    // phases ahead.
    const bool rescale = j > 0 && __any_sync(0xffffffffu, need);
    auto wait_pv = [&]() -> bool {
      const int jj = rescale ? j - 1 : j - 2;  // the PV that must be done
      if (jj >= 0 && !__all_sync(0xffffffffu, mbar_wait(&bars[B_O_DONE + (jj & 1)],
                                                        (uint32_t)(jj >> 1) & 1u, sh.abort_flag,
                                                        a.status)))
        return false;
      tc_fence_after();
      return true;
    };
    if constexpr (W <= 64) {
      // the exponentials overlap P(j-1) V(j-1)
      uint32_t pk[W / 2];
#pragma unroll
      for (int h = 0; h < kChunks; ++h) exps(&s[32 * h], &pk[16 * h]);
      if (!(ok = wait_pv())) break;
#pragma unroll
      for (int h = 0; h < kChunks; ++h) tmem_st16(p_buf + (col0 >> 1) + 16 * h, &pk[16 * h]);
    } else {
      // second pass over S, 32 keys at a time, straight into P
      if (!(ok = wait_pv())) break;
#pragma unroll
      for (int h = 0; h < kChunks; ++h) {
        uint32_t pk[16];
        scaled_chunk(h, s);
        exps(s, pk);
        tmem_st16(p_buf + 16 * h, pk);
      }
      tmem_st_wait();
      s_free();
    }
    l += sum[0] + sum[1];
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars[B_K_EMPTY + ks_slot]);  // done with the K tile's scales
    if (rescale) {
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
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars[B_PV_READY + (j & 1)]);
  }
  if (ok && n > 0)  // P(n-1) V(n-1) done, and with it every PV before it
    ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_O_DONE + ((n - 1) & 1)],
                                           (uint32_t)((n - 1) >> 1) & 1u, sh.abort_flag,
                                           a.status));
  // the V operand carries vs / rho: O = rho * (P V') / l
  if (ok && n > 0)
    ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_RHO_READY], 0u, sh.abort_flag, a.status));
  if (!ok || n == 0) return;
  tc_fence_after();
  const float rho = rho_of(sh.rho4);
  const bool final_row = rd.dst < 0;
  const int64_t orow = (int64_t)rd.q_index * a.n_q_heads + rd.q_head;
  if constexpr (R == 1) {
    const bool any = l > 0.f;
    const float inv = any ? rho / l : 0.f;
    const float lse2 = any ? m + log2f(l) : -INFINITY;
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
    if (valid && final_row && a.lse) a.lse[orow] = lse2 * 0.6931471805599453f;
    if (valid && !final_row) {
      a.part_lse[rd.dst] = lse2;
      __threadfence();  // the partial is visible before this CTA counts it
    }
  } else {
    // merge the R copies (split-KV partitions of the row's keys): every warp
    // parks its lanes' m, l and O, then finishes D / R columns of its row
    // group with weights 2^(m_c - M), M the largest m_c
    constexpr int RR = L::kRedRow;
    sh.redl[warp * 32 + lane] = l;
    sh.redm[warp * 32 + lane] = m;
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
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars[B_EPI_FULL]);
    if (!__all_sync(0xffffffffu, mbar_wait(&bars[B_EPI_FULL], 0u, sh.abort_flag, a.status)))
      return;
    float mcp[R], wc[R];
    float M = -INFINITY;
#pragma unroll
    for (int cc = 0; cc < R; ++cc) {
      mcp[cc] = lds1(smem_u32(sh.redm + (g + ngrp * cc) * 32 + lane));
      M = fmaxf(M, mcp[cc]);
    }
    float lt = 0.f;
#pragma unroll
    for (int cc = 0; cc < R; ++cc) {
      wc[cc] = M == -INFINITY ? 0.f : fast_exp2(mcp[cc] - M);  // 0 for a copy with no key
      lt += wc[cc] * lds1(smem_u32(sh.redl + (g + ngrp * cc) * 32 + lane));
    }
    const bool any = lt > 0.f;
    const float inv = any ? rho / lt : 0.f;
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
          const float4 v = lds4(smem_u32(sh.redo + ((g + ngrp * cc) * 32 + lane) * RR + col));
          acc.x = fmaf(wc[cc], v.x, acc.x);
          acc.y = fmaf(wc[cc], v.y, acc.y);
          acc.z = fmaf(wc[cc], v.z, acc.z);
          acc.w = fmaf(wc[cc], v.w, acc.w);
        }
        if (final_row) {
          uint2 w;
          w.x = pack_bf16x2(acc.x * inv, acc.y * inv);
          w.y = pack_bf16x2(acc.z * inv, acc.w * inv);
          *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + orow * D + col) = w;
        } else {
          *reinterpret_cast<float4*>(a.part_o + (int64_t)rd.dst * D + col) =
              make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        }
      }
      if (c == 0) {
        if (final_row && a.lse) a.lse[orow] = lse2 * 0.6931471805599453f;
        if (!final_row) a.part_lse[rd.dst] = lse2;
      }
      if (!final_row) __threadfence();  // each copy's columns are visible before the count
    }
  }
}

// One copy stream of the split-KV kernels, one warp each: the K tiles (a TMA
// box per page, and the pages' K scales) or the V tiles (codes and scales by
// bulk copy), each paced by its own ring alone. Both streams wait, after
// their first tile, until the softmax warps have issued their Q loads.
template <int D, class L, bool kV>
__device__ __forceinline__ void stream_role(const DecodeFp8Args& a, const DecodeItem& it,
                                            const int n, const int lane, const int ps_shift,
                                            const CUtensorMap* k_map, uint8_t* sk, uint8_t* svs,
                                            uint64_t* bars, volatile int* abort_flag,
                                            const int32_t page0, const uint32_t q_bar_count) {
  constexpr int kSlots = kV ? L::kVStSlots : L::kKSlots;
  const int ps = 1 << ps_shift;
  const int npg = BN / ps;
  const int32_t* btrow = a.block_table + (int64_t)it.bt_row * a.max_blocks;
  const int last_block = (it.k_end - 1) >> ps_shift;
  const int first_block = it.k_begin >> ps_shift;  // k_begin is page-aligned
  // lane < npg owns one page of every tile; its block-table entry is loaded
  // one tile ahead
  auto page_of = [&](int j) -> int32_t {
    int b = first_block + j * npg + lane;
    if (b > last_block) b = last_block;  // keys past k_end: masked, V zeroed
    return __ldg(btrow + b);
  };
  int32_t next_page = lane < npg ? page0 : 0;
  int issued = 0;
  for (int j = 0; j < n; ++j) {
    if (j == 1) named_barrier_sync(2, q_bar_count);
    const int slot = j % kSlots;
    if (j >= kSlots &&
        !__all_sync(0xffffffffu, mbar_wait(&bars[(kV ? B_VS_EMPTY : B_K_EMPTY) + slot],
                                           ((uint32_t)(j / kSlots) & 1u) ^ 1u, abort_flag,
                                           a.status)))
      break;
    int64_t my_row = 0;  // first cache row of this lane's page (rows of D codes)
    if (lane < npg) {
      int32_t page = next_page;
      if (j + 1 < n) next_page = page_of(j + 1);
      if ((unsigned)page >= (unsigned)a.num_pages) {
        set_status(a.status, MB_ERR_DEVICE_INDEX);
        page = 0;
      }
      my_row = ((int64_t)page * a.n_kv_heads + it.kv_head) << ps_shift;
    }
    uint64_t* full = &bars[(kV ? B_VS_FULL : B_K_FULL) + slot];
    if (lane == 0) mbar_arrive_expect_tx(full, L::kCodes + BN * 4);
    __syncwarp();
    if (lane < npg) {
      if constexpr (!kV) {
        uint8_t* dst = sk + slot * L::kKSlot;
        tma_load_2d(dst + lane * ps * D, k_map, full, 0, (int32_t)my_row);
        bulk_load(dst + L::kCodes + lane * ps * 4, a.k_scale + my_row, (uint32_t)(ps * 4), full);
      } else {
        uint8_t* dst = svs + slot * L::kVStBytes;
        bulk_load(dst + lane * ps * D, static_cast<const uint8_t*>(a.v8) + my_row * D,
                  (uint32_t)(ps * D), full);
        bulk_load(dst + L::kCodes + lane * ps * 4, a.v_scale + my_row, (uint32_t)(ps * 4), full);
      }
    }
    ++issued;
  }
  if (n == 1) named_barrier_sync(2, q_bar_count);
  __syncwarp();
  if (lane == 0)
    for (int j = max(0, issued - kSlots); j < issued; ++j)
      mbar_drain(&bars[(kV ? B_VS_FULL : B_K_FULL) + j % kSlots], (uint32_t)(j / kSlots) & 1u,
                 kDrainNs);
}

// V converter role (kConv warps; converter ci = 0 .. kConv - 1): rho from
// the item's V scales (converters 0-3), then every staged V tile -> the f16
// operand ring (keys past k_end zeroed), in the MN-major 128-byte-swizzled
// layout of [key][D] rows. kScaled: each key's vs / rho multiplied in here;
// otherwise the codes are converted as they are (exactly) and the softmax
// folds vs / rho into P.
template <int D, class L, bool kScaled = true, int kConv = 4>
__device__ __forceinline__ void converter_role(const DecodeFp8Args& a, const DecodeItem& it,
                                               const int n, const int ci, const int lane,
                                               const int ps_shift, uint8_t* svo, uint8_t* svs,
                                               float* rho4, uint64_t* bars,
                                               volatile int* abort_flag) {
  const int ct = ci * 32 + lane;
  constexpr int CPR = D / 16;       // 16-code chunks per key row
  constexpr int TASKS = BN * CPR;   // per tile
  // rho first: the largest V scale of the item's keys, read straight from
  // the scale array (4 bytes per key, beside the 128 bytes of codes the
  // V copy stream is already fetching); each of the first 4 converters'
  // maximum goes to shared memory, and every consumer takes the power of
  // two >= the largest
  if (ci < 4) {
    const int ps = 1 << ps_shift;
    const int32_t* btrow = a.block_table + (int64_t)it.bt_row * a.max_blocks;
    const int last_block = (it.k_end - 1) >> ps_shift;
    float vmx = 0.f;
    for (int b = (it.k_begin >> ps_shift) + ct; b <= last_block; b += 128) {
      const int32_t page = __ldg(btrow + b);
      if ((unsigned)page >= (unsigned)a.num_pages) continue;  // flagged by the copy streams
      const float4* sp = reinterpret_cast<const float4*>(
          a.v_scale + (((int64_t)page * a.n_kv_heads + it.kv_head) << ps_shift));
      const int nk = min(ps, it.k_end - (b << ps_shift));  // keys of the page below k_end
#pragma unroll 4
      for (int e4 = 0; e4 < ps / 4; ++e4) {
        const float4 v = __ldg(sp + e4);
        if (4 * e4 + 0 < nk) vmx = fmaxf(vmx, v.x);
        if (4 * e4 + 1 < nk) vmx = fmaxf(vmx, v.y);
        if (4 * e4 + 2 < nk) vmx = fmaxf(vmx, v.z);
        if (4 * e4 + 3 < nk) vmx = fmaxf(vmx, v.w);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
      vmx = fmaxf(vmx, __shfl_xor_sync(0xffffffffu, vmx, off));
    if (lane == 0) rho4[ci] = vmx;
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars[B_RHO_READY]);
  }
  const bool rho_ok =
      __all_sync(0xffffffffu, mbar_wait(&bars[B_RHO_READY], 0u, abort_flag, a.status));
  const float rho = rho_ok ? rho_of(rho4) : 0.f;
  const float inv_rho = rho > 0.f ? 1.f / rho : 0.f;
  for (int j = 0; rho_ok && j < n; ++j) {
    const int vs = j % L::kVStSlots, vo = j % kVOpSlots;
    if (!__all_sync(0xffffffffu, mbar_wait(&bars[B_VS_FULL + vs],
                                           (uint32_t)(j / L::kVStSlots) & 1u, abort_flag,
                                           a.status)))
      break;
    // operand slot j % 2 is free once PV(j-2) is done
    if (j >= kVOpSlots &&
        !__all_sync(0xffffffffu, mbar_wait(&bars[B_O_DONE + (j & 1)],
                                           (uint32_t)((j >> 1) - 1) & 1u, abort_flag,
                                           a.status)))
      break;
    tc_fence_after();
    const uint8_t* stg = svs + vs * L::kVStBytes;
    const uint32_t stg_s = smem_u32(stg);
    const uint32_t op_s = smem_u32(svo + vo * L::kVOpBytes);
    const int nvalid = min(BN, it.k_end - (it.k_begin + j * BN));
    // task t: key t / CPR, codes [16 q, 16 q + 16) -> f16 chunks 2q', 2q'+1
    // of half q / 4 (q' = q % 4 for D = 128), each value times the key's
    // vs / rho (f16, at most 1) when kScaled. The lanes of a store phase hit distinct
    // banks: for D = 128 lanes with q >= 4 store their second chunk first;
    // for D = 64 the phase's two keys swizzle apart.
#pragma unroll
    for (int t = ct; t < TASKS; t += kConv * 32) {
      const int key = t / CPR, q = t % CPR;
      uint4 raw = lds4u(stg_s + key * D + q * 16);
      // rows past k_end (their bits, scale included, may be anything): 0
      if (key >= nvalid) raw = make_uint4(0u, 0u, 0u, 0u);
      const bool swap = D == 128 && q >= 4;
      const uint32_t w0 = swap ? raw.z : raw.x, w1 = swap ? raw.w : raw.y;
      const uint32_t w2 = swap ? raw.x : raw.z, w3 = swap ? raw.y : raw.w;
      uint4 first, second;
      first.x = e4m3x2_to_f16x2(w0);
      first.y = e4m3x2_to_f16x2(w0 >> 16);
      first.z = e4m3x2_to_f16x2(w1);
      first.w = e4m3x2_to_f16x2(w1 >> 16);
      second.x = e4m3x2_to_f16x2(w2);
      second.y = e4m3x2_to_f16x2(w2 >> 16);
      second.z = e4m3x2_to_f16x2(w3);
      second.w = e4m3x2_to_f16x2(w3 >> 16);
      if constexpr (kScaled) {
        const float fk = lds1(stg_s + L::kCodes + 4 * key) * inv_rho;
        const uint32_t f2 = key < nvalid ? pack_f16x2(fk, fk) : 0u;
        first.x = hmul2(first.x, f2);
        first.y = hmul2(first.y, f2);
        first.z = hmul2(first.z, f2);
        first.w = hmul2(first.w, f2);
        second.x = hmul2(second.x, f2);
        second.y = hmul2(second.y, f2);
        second.z = hmul2(second.z, f2);
        second.w = hmul2(second.w, f2);
      }
      const int half = D == 128 ? (q >> 2) : 0;
      const int c0 = 2 * (D == 128 ? (q & 3) : q);
      const int sw = key & 7;
      const uint32_t rowp = op_s + half * L::kHalfBytes + key * 128;
      sts4u(rowp + (((c0 + (swap ? 1 : 0)) ^ sw) << 4), first);
      sts4u(rowp + (((c0 + (swap ? 0 : 1)) ^ sw) << 4), second);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&bars[B_VS_EMPTY + vs]);
      mbar_arrive(&bars[B_PV_READY + (j & 1)]);  // V_j in operand slot j % 2
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    splitkv_fp8_kernel(const DecodeFp8Args a, const int ps_shift,
                       const __grid_constant__ CUtensorMap k_map) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sk = smem + L::k_off;
  uint8_t* svo = smem + L::vop_off;
  uint8_t* svs = smem + L::vst_off;
  float* rho4 = reinterpret_cast<float*>(smem + L::misc_off + 16);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::bar_off);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::misc_off + 4);

  // the kernel behind this one (the next layer's append, say) may launch now
  pdl_launch_dependents();
  const DecodeItem it = a.items[blockIdx.x];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nr = it.n_rows;
  const int n = ceil_div(it.k_end - it.k_begin, BN);
  const int nw = ceil_div(nr, 32);
  const int ngrp = nw <= 1 ? 1 : (nw == 2 ? 2 : 4);  // row groups; 4 / ngrp copies per row
  // the copy streams' first block-table entries load while the CTA sets up
  int32_t page0 = 0;
  if ((warp == 8 || warp == 10) && n > 0 && lane < (BN >> ps_shift))
    page0 = __ldg(a.block_table + (int64_t)it.bt_row * a.max_blocks +
                  min((it.k_begin >> ps_shift) + lane, (it.k_end - 1) >> ps_shift));

  if (threadIdx.x == 0) {
    for (int s = 0; s < L::kKSlots; ++s) {
      mbar_init(&bars[B_K_FULL + s], 1);
      mbar_init(&bars[B_K_EMPTY + s], 4);
    }
    for (int s = 0; s < L::kVStSlots; ++s) {
      mbar_init(&bars[B_VS_FULL + s], 1);
      mbar_init(&bars[B_VS_EMPTY + s], 4);
    }
    mbar_init(&bars[B_S_FULL], 1);
    mbar_init(&bars[B_S_FREE], 4);
    mbar_init(&bars[B_PV_READY + 0], 8);
    mbar_init(&bars[B_PV_READY + 1], 8);
    mbar_init(&bars[B_O_DONE + 0], 1);
    mbar_init(&bars[B_O_DONE + 1], 1);
    mbar_init(&bars[B_RHO_READY], 4);
    mbar_init(&bars[B_EPI_FULL], 4);
    mbar_init(&bars[B_Q_READY], 4);
    mbar_init(&bars[B_MMA_DONE], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    stream_role<D, L, false>(a, it, n, lane, ps_shift, &k_map, sk, svs, bars, abort_flag, page0,
                             kQBarCount);
  } else if (warp == 10) {
    stream_role<D, L, true>(a, it, n, lane, ps_shift, &k_map, sk, svs, bars, abort_flag, page0,
                            kQBarCount);
  } else if (warp >= 4 && warp < 8) {
    converter_role<D, L>(a, it, n, warp - 4, lane, ps_shift, svo, svs, rho4, bars, abort_flag);
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // with kind::f8f6f4 format code 0 is e4m3: S = (hi | lo)(e4m3) x K(e4m3)
      constexpr uint32_t idesc_qk = idesc_f16_f32(BM, BN, false, false);
      constexpr uint32_t idesc_pv = idesc_f16_f32(BM, D, false, true);
      const uint32_t ka = smem_u32(sk);
      const uint32_t voa = smem_u32(svo);
      auto wait = [&](int b, uint32_t parity) -> bool {
        const bool ok = mbar_wait(&bars[b], parity, abort_flag, a.status);
        tc_fence_after();
        return ok;
      };
      auto issue_s = [&](int j) -> bool {
        const int slot = j % L::kKSlots;
        // K_j landed: waited for here for the first tile; for the others the
        // softmax warps waited before releasing S(j - 1)
        if (j == 0 && !wait(B_K_FULL + slot, 0u)) return false;
        const uint32_t k0 = ka + slot * L::kKSlot;
#pragma unroll
        for (int part = 0; part < 2; ++part)  // hi codes, then lo codes of Q
#pragma unroll
          for (int kk = 0; kk < D / 32; ++kk) {  // 32 e4m3 values (32 bytes) per MMA
            const uint64_t bd = D == 128 ? sdesc_sw128(k0 + kk * 32, 16, 1024)
                                         : sdesc_sw64(k0 + kk * 32, 16, 512);
            umma_f8_ts(tmem + kColS, tmem + kColQ + part * (D / 4) + kk * 8, bd, idesc_qk,
                       (part | kk) ? 1u : 0u);
          }
        umma_commit(&bars[B_S_FULL]);
        return true;
      };
      bool ok = n > 0 && wait(B_Q_READY, 0u);
      if (ok) ok = issue_s(0);
      for (int j = 0; ok && j < n; ++j) {
        // S(j+1) overwrites S(j) once the softmax warps have read it out,
        // ahead of PV(j): the next tile's scores overlap this tile's softmax
        if (j + 1 < n) {
          if (!(ok = wait(B_S_FREE, (uint32_t)j & 1u))) break;
          if (!(ok = issue_s(j + 1))) break;
        }
        const int vo = j % kVOpSlots;
        // P(j) written and V_j converted: one barrier per P buffer (the
        // softmax may already have written P(j+1) -- S(j+1) went ahead of
        // PV(j) -- never P(j+2); V_(j+2) waits for PV(j))
        if (!(ok = wait(B_PV_READY + (j & 1), (uint32_t)(j >> 1) & 1u))) break;
        const uint32_t v0 = voa + vo * L::kVOpBytes;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          const uint64_t bd = sdesc_sw128(v0 + kk * 2048, L::kHalfBytes, 1024);
          umma_bf16_ts(tmem + kColO, tmem + kColP + 64 * (j & 1) + kk * 8, bd, idesc_pv,
                       (j > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&bars[B_O_DONE + (j & 1)]);  // also frees V operand slot j % 2
      }
      // everything issued has completed before TMEM is freed
      umma_commit(&bars[B_MMA_DONE]);
      mbar_drain(&bars[B_MMA_DONE], 0u, kDrainNs);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ softmax
    Shared sh;
    sh.bars = bars;
    sh.abort_flag = abort_flag;
    sh.kring = sk;
    sh.rho4 = rho4;
    sh.redm = reinterpret_cast<float*>(smem + L::redm_off);
    sh.redl = reinterpret_cast<float*>(smem + L::redl_off);
    sh.redo = reinterpret_cast<float*>(sk);
    sh.tmem = tmem;
    if (ngrp == 1)
      softmax_role<D, 32>(a, it, sh, n, warp, lane);
    else if (ngrp == 2)
      softmax_role<D, 64>(a, it, sh, n, warp, lane);
    else
      softmax_role<D, 128>(a, it, sh, n, warp, lane);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (a.combine_count) {
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
    // the K ring is no longer written (every copy has landed) nor read
    dev::merge_completed_rows<D, kThreads>(mg, reinterpret_cast<uint32_t*>(sk));
  }
  if (a.after_prefill && threadIdx.x == 0) {
    // started under the prefill kernel's tail: the grid must not complete
    // before that kernel does, so the last CTA to finish waits for it
    __threadfence();
    if (atomicAdd(a.done_counter, 1) == (int)gridDim.x - 1) {
      pdl_wait();
      atomicExch(a.done_counter, 0);
    }
  }
}


// ============================================================================
// Few-row form: S^T = K Q^T and O^T = V'^T P^T.
//
// A CTA of a few query rows (a decode step's g query heads: at most 8 rows
// here) leaves most of a 128-row MMA idle, and the form above pays for that
// in its per-tile chain: each softmax copy loads, scales and exponentiates
// 32 scores in a row, with 4 of a warp's 32 lanes busy. Here the tile's 128
// keys are the MMA's M and the rows its N (16):
//   * S^T[key][n] = sum_d kcode[key][d] qcode[n][d]: kind::f8f6f4 with the
//     K tile as A (the TMA box already is the K-major swizzled layout) and
//     Q's code rows as B, in shared memory: the R rows' hi codes in columns
//     n < R, their lo codes in columns R + r, so one product reads the K
//     tile once and the softmax adds the two halves of each score;
//   * O^T[d][r] += sum_key vcode[key][d] P'[key][r]: kind::f16 with the V
//     codes converted to f16 (exactly, no scale: the converter warps' only
//     work) as an MN-major A operand and P'^T = (p vs_key / rho)^T (f16,
//     K-major) as B: each softmax thread folds its key's V scale into P.
// A softmax thread owns one key of the tile (its TMEM lane): it reads its N
// scores, its key's scale, and writes one P value per row. The row maxima
// are reduced across the 128 keys (a warp reduction, then the 4 warps'
// maxima through shared memory and an mbarrier, both bounded); every
// thread then holds the same reference max per row, so all p of a tile
// share it, as the PV product needs. O^T is rescaled in TMEM (every thread
// its d = lane) only when a row's max grew by more than 2^8, as above; each
// thread keeps its key's share of every row sum, added up at the end.
// D = 128 only.

// 8-bit-float product with both operands in shared memory.
__device__ __forceinline__ void umma_f8_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// N (4, 8, 16 or 32) consecutive 32-bit columns of this thread's TMEM lane,
// and the wait that completes the load (the registers are its operands, so
// no use is scheduled before it).
template <int N>
__device__ __forceinline__ void tmem_ldn(uint32_t taddr, uint32_t* r);
template <>
__device__ __forceinline__ void tmem_ldn<4>(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr)
               : "memory");
}
template <>
__device__ __forceinline__ void tmem_ldn<8>(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
}
template <>
__device__ __forceinline__ void tmem_ldn<16>(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
template <>
__device__ __forceinline__ void tmem_ldn<32>(uint32_t taddr, uint32_t* r) {
  tmem_ld32(taddr, *reinterpret_cast<uint32_t(*)[32]>(r));
}
template <int N>
__device__ __forceinline__ void tmem_ldn_wait(uint32_t* r);
template <>
__device__ __forceinline__ void tmem_ldn_wait<4>(uint32_t* r) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3])
               :
               : "memory");
}
template <>
__device__ __forceinline__ void tmem_ldn_wait<8>(uint32_t* r) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7])
               :
               : "memory");
}
template <>
__device__ __forceinline__ void tmem_ldn_wait<16>(uint32_t* r) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}
template <>
__device__ __forceinline__ void tmem_ldn_wait<32>(uint32_t* r) {
  tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(r));
}
template <int N>
__device__ __forceinline__ void tmem_stn(uint32_t taddr, const uint32_t* r);
template <>
__device__ __forceinline__ void tmem_stn<4>(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
               : "memory");
}
template <>
__device__ __forceinline__ void tmem_stn<8>(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(
                   taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
               "r"(r[7])
               : "memory");
}
template <>
__device__ __forceinline__ void tmem_stn<16>(uint32_t taddr, const uint32_t* r) {
  tmem_st16(taddr, r);
}
template <>
__device__ __forceinline__ void tmem_stn<32>(uint32_t taddr, const uint32_t* r) {
  tmem_st32(taddr, *reinterpret_cast<const uint32_t(*)[32]>(r));
}

// Largest value over the warp (finite or -inf inputs): the fp32 bits mapped
// to integers of the same order (negative values: the low 31 bits flipped),
// one integer reduction, mapped back.
__device__ __forceinline__ float warp_max(float v) {
  int i = __float_as_int(v);
  i = i < 0 ? (i ^ 0x7fffffff) : i;
  i = __reduce_max_sync(0xffffffffu, i);
  return __int_as_float(i < 0 ? (i ^ 0x7fffffff) : i);
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}
__device__ __forceinline__ void sts_f16(uint32_t addr, float x) {
  unsigned short h;
  asm("cvt.rn.f16.f32 %0, %1;" : "=h"(h) : "f"(x));
  asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(h) : "memory");
}

// Shared memory of the few-row kernel (D = 128, NQ = the MMA's N).
template <int NQ>
struct LayoutT {
  static constexpr int D = 128;
  static constexpr int kHalves = 2;
  static constexpr uint32_t kHalfBytes = 128 * 128;  // 128 keys x 64 f16 values
  static constexpr uint32_t kVOpBytes = kHalves * kHalfBytes;
  static constexpr uint32_t kCodes = BN * D;
  static constexpr uint32_t kKSlot = (kCodes + BN * 4 + 1023) & ~1023u;
  static constexpr int kKSlots = 4;
  static constexpr uint32_t kVStBytes = kCodes + BN * 4;
  static constexpr int kVStSlots = 4;
  static constexpr uint32_t kQBytes = NQ * 128;      // NQ 128-byte code rows (hi, lo, zeros)
  static constexpr uint32_t kPHalf = NQ * 128;       // P^T: NQ rows x 64 keys (f16)
  static constexpr uint32_t kPBytes = 2 * kPHalf;    // one tile's P^T
  static constexpr uint32_t k_off = 0;
  static constexpr uint32_t vop_off = k_off + kKSlots * kKSlot;
  static constexpr uint32_t vst_off = vop_off + kVOpSlots * kVOpBytes;
  static constexpr uint32_t q_off = vst_off + kVStSlots * kVStBytes;  // Q codes, B of S^T
  static constexpr uint32_t p_off = q_off + kQBytes;                  // two P^T buffers
  static constexpr uint32_t par_off = p_off + 2 * kPBytes;
  // per row: crow (float), lim (int), q_index, q_head, dst
  static constexpr uint32_t redm_off = par_off + 5 * 32 * 4;  // float [2][32][4]
  static constexpr uint32_t redl_off = redm_off + 2 * 32 * 4 * 4;  // float [32][4]
  static constexpr uint32_t bar_off = redl_off + 32 * 4 * 4;
  static constexpr uint32_t misc_off = (bar_off + B_COUNT * 8 + 15) & ~15u;
  static constexpr uint32_t kBytes = misc_off + 32;
  static constexpr uint32_t kAlloc = kBytes + 1024;
  static_assert(kKSlots <= kMaxSlots && kVStSlots <= kMaxSlots, "rings");
  static_assert(vop_off % 1024 == 0 && q_off % 1024 == 0 && p_off % 1024 == 0,
                "operand tiles are 1024-byte aligned (128-byte swizzle atoms)");
  static_assert(kAlloc <= 232448, "shared memory");
};
// Rows up to which the few-row form is used. Its per-key work grows with the
// rows (a reduction, an exponential and a store per row); measured on this
// GPU it is 3.5 % faster than the form above at 4 rows (256 decodes, GQA 4),
// and 1.3x / 2.1x slower at 16 / 24 rows (speculative and shared-prefix
// batches).
constexpr int kFewRowsMax = 8;
constexpr int kThreadsT = 384;  // the few-row kernel's CTA
constexpr int kConvT = 5;       // its V converter warps (4-7 and 11)
constexpr uint32_t kQBarCountT = 128 + 2 * 32;  // softmax warps + the two copy streams
constexpr uint32_t kTmemColsT = 128;
constexpr uint32_t kColST = 0;   // S^T: two buffers of NQ columns, by tile parity
constexpr uint32_t kColOT = 64;  // O^T: NQ columns (lane = d)

struct SharedT {
  uint64_t* bars;
  volatile int* abort_flag;
  const uint8_t* kring;  // K slots (codes, then scales)
  const uint8_t* vring;  // V staging slots (codes, then scales)
  int nvalid_rel;        // k_end - k_begin: keys at or past it are padding
  const float* rho4;     // the converters' 4 partial maxima of the V scales
  uint32_t q_s;          // shared address of Q's code rows (hi rows, lo rows, zeros)
  uint32_t p_s;          // shared address of the first P^T buffer
  float* crow;           // [32] per row: scale_log2 * sq (0 past n_rows)
  int* lim;              // [32] keys j < lim (relative to k_begin) are visible
  int* qidx;             // [32] flat token row
  int* qhead;            // [32]
  int* dst;              // [32] partial slot, or < 0 for a final row
  float* redm;           // [2][32][4] the 4 warps' maxima of every row, by tile parity
  float* redl;           // [32][4] the 4 warps' shares of every row sum
  uint32_t tmem;
};

// Softmax role of the few-row kernel (warps 0-3; thread t = key t of every
// tile and d = t of O^T). R: rows the build holds (>= it.n_rows).
template <int R>
__device__ __forceinline__ void softmax_t(const DecodeFp8Args& a, const DecodeItem& it,
                                          const SharedT& sh, const int n, const int warp,
                                          const int lane) {
  constexpr int NQ = 16;
  static_assert(2 * R <= NQ, "hi and lo rows of every query row in one B operand");
  using L = LayoutT<NQ>;
  uint64_t* bars = sh.bars;
  const int t = warp * 32 + lane;
  const int nr = it.n_rows;
  const uint32_t lane_addr = (uint32_t)(warp * 32) << 16;

  // thread r < R writes row r's hi codes (B row r) and lo codes (B row
  // R + r), zeros past n_rows, and the row's constants; threads 2R..NQ-1
  // zero the remaining B rows. The row's loads are issued before the
  // copy streams pass their first tile
  {
    const bool valid = t < nr;
    RowDesc rd;
    rd.q_index = 0;
    rd.q_head = 0;
    rd.vis_end = 0;
    rd.dst = -1;
    if (valid) rd = a.rows[it.row_begin + t];
    const uint4* qrow = static_cast<const uint4*>(a.q) +
                        ((int64_t)rd.q_index * a.n_q_heads + rd.q_head) * (L::D / 8);
    uint4 qb[L::D / 8];
#pragma unroll
    for (int k = 0; k < L::D / 8; ++k) qb[k] = valid ? __ldg(qrow + k) : make_uint4(0u, 0u, 0u, 0u);
    named_barrier_arrive(2, kQBarCountT);  // the copy streams' wait
    if (t >= 2 * R && t < NQ) {
#pragma unroll
      for (int c = 0; c < 8; ++c) sts4u(sh.q_s + (uint32_t)t * 128u + 16u * c, make_uint4(0u, 0u, 0u, 0u));
    }
    if (t < R) {
      float amax = 0.f;
#pragma unroll
      for (int k = 0; k < L::D / 8; ++k) {
        const uint32_t wv[4] = {qb[k].x, qb[k].y, qb[k].z, qb[k].w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          amax = fmax3(amax, fabsf(bf16_lo(wv[e])), fabsf(bf16_hi(wv[e])));
      }
      const float sq = amax * (1.f / 448.f);
      const float inv = amax > 0.f ? 448.f / amax : 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) {  // 16 codes per 16-byte chunk
        uint4 h, l;
        const uint4 b0 = qb[2 * c], b1 = qb[2 * c + 1];
        split4(bf16_lo(b0.x) * inv, bf16_hi(b0.x) * inv, bf16_lo(b0.y) * inv, bf16_hi(b0.y) * inv,
               h.x, l.x);
        split4(bf16_lo(b0.z) * inv, bf16_hi(b0.z) * inv, bf16_lo(b0.w) * inv, bf16_hi(b0.w) * inv,
               h.y, l.y);
        split4(bf16_lo(b1.x) * inv, bf16_hi(b1.x) * inv, bf16_lo(b1.y) * inv, bf16_hi(b1.y) * inv,
               h.z, l.z);
        split4(bf16_lo(b1.z) * inv, bf16_hi(b1.z) * inv, bf16_lo(b1.w) * inv, bf16_hi(b1.w) * inv,
               h.w, l.w);
        const int tl = R + t;  // the lo row
        sts4u(sh.q_s + (uint32_t)t * 128u + ((uint32_t)(c ^ (t & 7)) << 4), h);
        sts4u(sh.q_s + (uint32_t)tl * 128u + ((uint32_t)(c ^ (tl & 7)) << 4), l);
      }
      sh.crow[t] = valid ? a.scale_log2 * sq : 0.f;
      sh.lim[t] = valid ? min(it.k_end, rd.vis_end) - it.k_begin : 0;
      sh.qidx[t] = rd.q_index;
      sh.qhead[t] = rd.q_head;
      sh.dst[t] = rd.dst;
    }
    // P^T starts as zeros: the rows past R are never written
    for (uint32_t o = (uint32_t)t * 16u; o < 2u * L::kPBytes; o += 128u * 16u)
      sts4u(sh.p_s + o, make_uint4(0u, 0u, 0u, 0u));
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars[B_Q_READY]);
  }
  bool ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_Q_READY], 0u, sh.abort_flag, a.status));

  // P carries each key's vs / rho (the converters leave V' = the codes):
  // O = rho (P' V') / l
  if (ok && n > 0)
    ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_RHO_READY], 0u, sh.abort_flag, a.status));
  const float rho = ok ? rho_of(sh.rho4) : 0.f;
  const float inv_rho = rho > 0.f ? 1.f / rho : 0.f;
  float m[R], l[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
  }
  // this thread's P^T element of row r: half t / 64, 16-byte chunk (t % 64) / 8
  // swizzled by r % 8, element t % 8
  const uint32_t p_half = (uint32_t)(t >> 6) * L::kPHalf;
  const uint32_t p_chunk = (uint32_t)((t & 63) >> 3), p_elem = (uint32_t)(t & 7) * 2u;
  for (int j = 0; ok && j < n; ++j) {
    const int b = j & 1;
    const int ks_slot = j % L::kKSlots;
    ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_T_S_FULL + b], (uint32_t)(j >> 1) & 1u,
                                           sh.abort_flag, a.status));
    if (!ok) break;
    // K_j's scales arrived with its codes
    ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_K_FULL + ks_slot],
                                           (uint32_t)(j / L::kKSlots) & 1u, sh.abort_flag,
                                           a.status));
    if (!ok) break;
    tc_fence_after();
    uint32_t s[2 * R];  // hi halves, then lo halves
    tmem_ldn<2 * R>(sh.tmem + lane_addr + kColST + (uint32_t)(b * NQ), s);
    const float ks = lds1(smem_u32(sh.kring + ks_slot * L::kKSlot + L::kCodes) + 4u * (uint32_t)t);
    tmem_ldn_wait<2 * R>(s);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars[B_T_S_FREE + b]);  // S(j + 2) may overwrite the buffer
    // this key's scores in the log2 domain, -inf where the row does not see it
    const int kpos = j * BN + t;
    float v[R];
#pragma unroll
    for (int r4 = 0; r4 < (R + 3) / 4; ++r4) {
      const float4 c4 = lds4(smem_u32(sh.crow + 4 * r4));
      const uint4 l4 = lds4u(smem_u32(sh.lim + 4 * r4));
      const float cr[4] = {c4.x, c4.y, c4.z, c4.w};
      const int li[4] = {(int)l4.x, (int)l4.y, (int)l4.z, (int)l4.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int r = 4 * r4 + q;
        if (r < R)
          v[r] = kpos < li[q]
                     ? (__uint_as_float(s[r]) + __uint_as_float(s[R + r])) * (ks * cr[q])
                     : -INFINITY;
      }
    }
    // every row's maximum over the tile's 128 keys
    float* red = sh.redm + b * (32 * 4);
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float mw = warp_max(v[r]);
      if (lane == 0) red[r * 4 + warp] = mw;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars[B_RED_FULL + b]);
    ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_RED_FULL + b], (uint32_t)(j >> 1) & 1u,
                                           sh.abort_flag, a.status));
    if (!ok) break;
    // the reference max moves only when a row's max grew by more than 2^8
    // (every thread takes the same decision from the same values)
    float alpha[R];
    bool need = false;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float4 q4 = lds4(smem_u32(red + r * 4));
      const float mt = fmaxf(fmaxf(q4.x, q4.y), fmaxf(q4.z, q4.w));
      alpha[r] = 1.f;
      if (mt > m[r] + kRescaleThreshold) {  // also the first tile the row sees a key in
        if (m[r] != -INFINITY) {
          alpha[r] = fast_exp2(m[r] - mt);
          need = true;
        }
        l[r] *= alpha[r];
        m[r] = mt;
      }
    }
    // this tile's P^T buffer was read by P V(j - 2); when O is rescaled,
    // P V(j - 1) must be done too. The barrier of a buffer completes every
    // other tile and the PV after the one waited for needs this tile's P,
    // so no wait is two phases ahead.
    const int jj = need ? j - 1 : j - 2;
    if (jj >= 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_O_DONE + (jj & 1)],
                                             (uint32_t)(jj >> 1) & 1u, sh.abort_flag, a.status));
      if (!ok) break;
      tc_fence_after();
    }
    // this key's V scale (its staging slot holds the scales beside the codes)
    const int vs_slot = j % L::kVStSlots;
    ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_VS_FULL + vs_slot],
                                           (uint32_t)(j / L::kVStSlots) & 1u, sh.abort_flag,
                                           a.status));
    if (!ok) break;
    const float vsc = lds1(smem_u32(sh.vring + vs_slot * L::kVStBytes + L::kCodes) + 4u * (uint32_t)t);
    const float fv = kpos < sh.nvalid_rel ? vsc * inv_rho : 0.f;  // keys past k_end: 0
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars[B_VS_EMPTY + vs_slot]);
    const uint32_t pbuf = sh.p_s + (uint32_t)b * L::kPBytes + p_half + p_elem;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float p = m[r] == -INFINITY ? 0.f : fast_exp2(v[r] - m[r]);
      l[r] += p;
      sts_f16(pbuf + (uint32_t)r * 128u + ((p_chunk ^ (uint32_t)(r & 7)) << 4), p * fv);
    }
    if (need) {
      uint32_t o[R];
      tmem_ldn<R>(sh.tmem + lane_addr + kColOT, o);
      tmem_ldn_wait<R>(o);
#pragma unroll
      for (int r = 0; r < R; ++r) o[r] = __float_as_uint(__uint_as_float(o[r]) * alpha[r]);
      tmem_stn<R>(sh.tmem + lane_addr + kColOT, o);
      tmem_st_wait();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&bars[B_K_EMPTY + ks_slot]);  // the scale is read, S(j) is done
      mbar_arrive(&bars[B_PV_READY + b]);
    }
  }
  if (ok && n > 0)  // P V(n-1) done, and with it every PV before it
    ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_O_DONE + ((n - 1) & 1)],
                                           (uint32_t)((n - 1) >> 1) & 1u, sh.abort_flag,
                                           a.status));
  if (!ok || n == 0) return;
  tc_fence_after();
  // every row's sum over the 128 keys' shares
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const float lw = warp_sum(l[r]);
    if (lane == 0) sh.redl[r * 4 + warp] = lw;
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(&bars[B_EPI_FULL]);
  if (!__all_sync(0xffffffffu, mbar_wait(&bars[B_EPI_FULL], 0u, sh.abort_flag, a.status)))
    return;
  uint32_t o[R];
  tmem_ldn<R>(sh.tmem + lane_addr + kColOT, o);
  tmem_ldn_wait<R>(o);
  bool partial = false;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (r >= nr) break;
    const float4 q4 = lds4(smem_u32(sh.redl + r * 4));
    const float lt = (q4.x + q4.y) + (q4.z + q4.w);
    const bool any = lt > 0.f;
    const float inv = any ? rho / lt : 0.f;
    const float lse2 = any ? m[r] + log2f(lt) : -INFINITY;
    const int dst = sh.dst[r];
    const int64_t orow = (int64_t)sh.qidx[r] * a.n_q_heads + sh.qhead[r];
    const float x = __uint_as_float(o[r]) * inv;  // O[r][d = t]
    if (dst < 0) {
      reinterpret_cast<unsigned short*>(a.out)[orow * L::D + t] =
          (unsigned short)(pack_bf16x2(x, 0.f) & 0xffffu);
      if (t == 0 && a.lse) a.lse[orow] = lse2 * 0.6931471805599453f;
    } else {
      a.part_o[(int64_t)dst * L::D + t] = x;
      if (t == 0) a.part_lse[dst] = lse2;
      partial = true;
    }
  }
  if (partial) __threadfence();  // the partials are visible before this CTA counts them
}


// Roles: softmax warps 0-3, V converters 4-7 and 11, K copies warp 8, MMA
// lane of warp 9, V copies warp 10; R = the build's rows (4 or 8).
template <int R>
__global__ void __launch_bounds__(kThreadsT, 1)
    splitkv_fp8t_kernel(const DecodeFp8Args a, const int ps_shift,
                        const __grid_constant__ CUtensorMap k_map) {
  constexpr int D = 128;
  constexpr int NQ = 16;
  using L = LayoutT<NQ>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sk = smem + L::k_off;
  uint8_t* svo = smem + L::vop_off;
  uint8_t* svs = smem + L::vst_off;
  float* rho4 = reinterpret_cast<float*>(smem + L::misc_off + 16);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::bar_off);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::misc_off + 4);

  // the kernel behind this one may launch now
  pdl_launch_dependents();
  const DecodeItem it = a.items[blockIdx.x];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int n = ceil_div(it.k_end - it.k_begin, BN);
  if (it.n_rows > R) {  // the plan sizes the build to its largest CTA
    if (threadIdx.x == 0) set_status(a.status, MB_ERR_DEVICE_INDEX);
    n = 0;
  }
  int32_t page0 = 0;
  if ((warp == 8 || warp == 10) && n > 0 && lane < (BN >> ps_shift))
    page0 = __ldg(a.block_table + (int64_t)it.bt_row * a.max_blocks +
                  min((it.k_begin >> ps_shift) + lane, (it.k_end - 1) >> ps_shift));

  if (threadIdx.x == 0) {
    for (int s = 0; s < L::kKSlots; ++s) {
      mbar_init(&bars[B_K_FULL + s], 1);
      mbar_init(&bars[B_K_EMPTY + s], 4);
    }
    for (int s = 0; s < L::kVStSlots; ++s) {
      mbar_init(&bars[B_VS_FULL + s], 1);
      mbar_init(&bars[B_VS_EMPTY + s], 4 + kConvT);  // converters, softmax (the V scales)
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars[B_T_S_FULL + b], 1);
      mbar_init(&bars[B_T_S_FREE + b], 4);
      mbar_init(&bars[B_PV_READY + b], 4 + kConvT);
      mbar_init(&bars[B_O_DONE + b], 1);
      mbar_init(&bars[B_RED_FULL + b], 4);
    }
    mbar_init(&bars[B_RHO_READY], 4);
    mbar_init(&bars[B_EPI_FULL], 4);
    mbar_init(&bars[B_Q_READY], 4);
    mbar_init(&bars[B_MMA_DONE], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, kTmemColsT);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    stream_role<D, L, false>(a, it, n, lane, ps_shift, &k_map, sk, svs, bars, abort_flag, page0,
                             kQBarCountT);
  } else if (warp == 10) {
    stream_role<D, L, true>(a, it, n, lane, ps_shift, &k_map, sk, svs, bars, abort_flag, page0,
                            kQBarCountT);
  } else if ((warp >= 4 && warp < 8) || warp == 11) {
    converter_role<D, L, false, kConvT>(a, it, n, warp == 11 ? 4 : warp - 4, lane, ps_shift, svo,
                                        svs, rho4, bars, abort_flag);
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // kind::f8f6f4 with format code 0: e4m3 x e4m3; kind::f16: f16 x f16
      constexpr uint32_t idesc_qk = idesc_f16_f32(128, NQ, false, false);
      constexpr uint32_t idesc_pv = idesc_f16_f32(128, NQ, true, false);
      const uint32_t ka = smem_u32(sk), voa = smem_u32(svo);
      const uint32_t qa = smem_u32(smem + L::q_off), pa = smem_u32(smem + L::p_off);
      auto wait = [&](int b, uint32_t parity) -> bool {
        const bool ok = mbar_wait(&bars[b], parity, abort_flag, a.status);
        tc_fence_after();
        return ok;
      };
      // S^T(j) = K_j (A: 128 keys x D codes) x Q^T (B: NQ code rows x D)
      auto issue_s = [&](int j) -> bool {
        const int slot = j % L::kKSlots;
        if (!wait(B_K_FULL + slot, (uint32_t)(j / L::kKSlots) & 1u)) return false;
        const uint32_t k0 = ka + slot * L::kKSlot;
#pragma unroll
        for (int kk = 0; kk < D / 32; ++kk)  // 32 codes (32 bytes) per MMA
          umma_f8_ss(tmem + kColST + (uint32_t)((j & 1) * NQ), sdesc_sw128(k0 + kk * 32, 16, 1024),
                     sdesc_sw128(qa + kk * 32, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
        umma_commit(&bars[B_T_S_FULL + (j & 1)]);
        return true;
      };
      bool ok = n > 0 && wait(B_Q_READY, 0u);
      if (ok) ok = issue_s(0);
      for (int j = 0; ok && j < n; ++j) {
        // S^T(j+1) ahead of PV(j), into the other buffer once the softmax
        // has read S^T(j-1) out of it
        if (j + 1 < n) {
          const int jn = j + 1;
          if (jn >= 2 && !(ok = wait(B_T_S_FREE + (jn & 1), (uint32_t)((jn >> 1) - 1) & 1u)))
            break;
          if (!(ok = issue_s(jn))) break;
        }
        // P^T(j) written and V_j converted
        if (!(ok = wait(B_PV_READY + (j & 1), (uint32_t)(j >> 1) & 1u))) break;
        const uint32_t v0 = voa + (uint32_t)(j % kVOpSlots) * L::kVOpBytes;
        const uint32_t p0 = pa + (uint32_t)(j & 1) * L::kPBytes;
        // O^T += V'^T (A: D x 16 keys, MN-major) x P^T (B: 16 keys x NQ rows)
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          umma_bf16_ss(tmem + kColOT, sdesc_sw128(v0 + kk * 2048, L::kHalfBytes, 1024),
                       sdesc_sw128(p0 + (kk >> 2) * L::kPHalf + (kk & 3) * 32, 16, 1024),
                       idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&bars[B_O_DONE + (j & 1)]);  // also frees V operand slot j % 2
      }
      umma_commit(&bars[B_MMA_DONE]);
      mbar_drain(&bars[B_MMA_DONE], 0u, kDrainNs);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ softmax
    SharedT sh;
    sh.bars = bars;
    sh.abort_flag = abort_flag;
    sh.kring = sk;
    sh.vring = svs;
    sh.nvalid_rel = it.k_end - it.k_begin;
    sh.rho4 = rho4;
    sh.q_s = smem_u32(smem + L::q_off);
    sh.p_s = smem_u32(smem + L::p_off);
    sh.crow = reinterpret_cast<float*>(smem + L::par_off);
    sh.lim = reinterpret_cast<int*>(smem + L::par_off + 128);
    sh.qidx = reinterpret_cast<int*>(smem + L::par_off + 256);
    sh.qhead = reinterpret_cast<int*>(smem + L::par_off + 384);
    sh.dst = reinterpret_cast<int*>(smem + L::par_off + 512);
    sh.redm = reinterpret_cast<float*>(smem + L::redm_off);
    sh.redl = reinterpret_cast<float*>(smem + L::redl_off);
    sh.tmem = tmem;
    softmax_t<R>(a, it, sh, n, warp, lane);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemColsT);
  }
  if (a.combine_count) {
    dev::MergeArgs mg;
    mg.rows = a.rows + it.row_begin;
    mg.refs = a.row_merge + it.row_begin;
    mg.n_rows = it.n_rows;
    mg.count = a.combine_count;
    mg.part_o = a.part_o;
    mg.part_lse = a.part_lse;
    mg.n_q_heads = a.n_q_heads;
    mg.out = static_cast<__nv_bfloat16*>(a.out);
    mg.lse = a.lse;
    // the K ring is no longer written (every copy has landed) nor read
    dev::merge_completed_rows<D, kThreadsT>(mg, reinterpret_cast<uint32_t*>(sk));
  }
  if (a.after_prefill && threadIdx.x == 0) {
    // started under the prefill kernel's tail: the grid must not complete
    // before that kernel does, so the last CTA to finish waits for it
    __threadfence();
    if (atomicAdd(a.done_counter, 1) == (int)gridDim.x - 1) {
      pdl_wait();
      atomicExch(a.done_counter, 0);
    }
  }
}

template <int R>
cudaError_t launch_fp8t(const DecodeFp8Args& a, cudaStream_t s, bool overlap_previous,
                        int ps_shift) {
  using L = LayoutT<16>;
  static OncePerDevice setup;
  const cudaError_t e = setup.run([](int) {
    return cudaFuncSetAttribute(splitkv_fp8t_kernel<R>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::kAlloc);
  });
  if (e != cudaSuccess) return e;
  if (overlap_previous)
    return launch_programmatic(splitkv_fp8t_kernel<R>, dim3((unsigned)a.n_items),
                               dim3(kThreadsT), L::kAlloc, s, a, ps_shift, *a.k_map);
  splitkv_fp8t_kernel<R><<<(unsigned)a.n_items, kThreadsT, L::kAlloc, s>>>(a, ps_shift, *a.k_map);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_fp8(const DecodeFp8Args& a, cudaStream_t s, bool overlap_previous) {
  if (a.n_items <= 0) return cudaSuccess;
  const int ps_shift = __builtin_ctz((unsigned)a.page_size);
  // CTAs of at most 8 rows: the few-row form, sized to the largest
  if (a.head_dim == 128 && a.max_rows > 0 && a.max_rows <= kFewRowsMax) {
    if (a.max_rows <= 4) return launch_fp8t<4>(a, s, overlap_previous, ps_shift);
    return launch_fp8t<8>(a, s, overlap_previous, ps_shift);
  }
  static OncePerDevice setup128, setup64;
  cudaError_t e;
  if (a.head_dim == 128) {
    e = setup128.run([](int) {
      return cudaFuncSetAttribute(splitkv_fp8_kernel<128>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)Layout<128>::kAlloc);
    });
    if (e != cudaSuccess) return e;
    if (overlap_previous)
      return launch_programmatic(splitkv_fp8_kernel<128>, dim3((unsigned)a.n_items),
                                 dim3(kThreads), Layout<128>::kAlloc, s, a, ps_shift, *a.k_map);
    splitkv_fp8_kernel<128><<<(unsigned)a.n_items, kThreads, Layout<128>::kAlloc, s>>>(
        a, ps_shift, *a.k_map);
    return cudaGetLastError();
  }
  e = setup64.run([](int) {
    return cudaFuncSetAttribute(splitkv_fp8_kernel<64>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)Layout<64>::kAlloc);
  });
  if (e != cudaSuccess) return e;
  if (overlap_previous)
    return launch_programmatic(splitkv_fp8_kernel<64>, dim3((unsigned)a.n_items),
                               dim3(kThreads), Layout<64>::kAlloc, s, a, ps_shift, *a.k_map);
  splitkv_fp8_kernel<64><<<(unsigned)a.n_items, kThreads, Layout<64>::kAlloc, s>>>(
      a, ps_shift, *a.k_map);
  return cudaGetLastError();
}

}  // namespace mb
