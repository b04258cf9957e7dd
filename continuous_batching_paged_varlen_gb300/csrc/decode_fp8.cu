// Split-KV attention over an fp8 (e4m3) KV cache with per-row fp32 scales.
//
// "GLM-5.3 e2e token ledger", the KV layout paragraphs: the cache holds K/V
// as FP8 codes with FP32 scales stored beside them, and the attention kernel
// reads both to dequantize. Here every (token, KV head) row of D codes has
// one scale: k = decode(code) * scale. The work lists are the ones the
// bf16 split-KV kernel runs (one CTA = up to 128 query rows of one KV head
// against the key range [k_begin, k_end) of one block-table row, "How To
// Scale Your Model notes (7-8)", section 3), and the results are the same
// final rows or normalised partials for the combine kernel.
//
// The scale of key j factors out of both products:
//   S[r][j] = ks_j * (q_r . kcode_j)       O[r] = sum_j (p[r][j] * vs_j) vcode_j
// so the tensor core multiplies raw codes and the softmax applies ks_j to
// the scores and folds vs_j into P. Every e4m3 value is exact in f16 and in
// bf16, so the operands lose nothing: Q K^T runs on f16 operands (Q is
// rounded from bf16 to f16 once, saturating at +-65504) and P V on bf16
// operands, both with fp32 accumulation in TMEM.
//
// Half the bytes of the bf16 cache per key, so the pipeline adds a stage
// that turns the staged codes into MMA operands:
//   warp 8      producer: for each 128-key tile, one bulk copy per page of
//               codes (a page of one KV head is ps * D contiguous bytes) and
//               one of its ps scales, K then V, into a staging ring.
//   warps 4-7   converters: staged codes -> 16-bit operand tiles in the
//               128-byte-swizzled K-major layout (K as f16, V as bf16, V rows
//               past k_end zeroed), and the tile's scales (ks * log2(e) *
//               softmax scale, vs) into a small ring the softmax reads.
//   warp 9      TMEM allocation; one lane issues S = Q K^T and O += P V.
//   warps 0-3   softmax. With few rows (a decode step's g query heads), each
//               row is copied into 4 (or 2) TMEM lanes of different warps and
//               each copy handles 32 (or 64) of the tile's 128 keys, so the
//               exponentials of one row spread over 4 SM sub-partitions; the
//               copies agree on the running max through shared memory every
//               tile and add their partial sums and outputs at the end.
// Every wait is bounded; on a timeout the CTA raises its abort flag, drains
// what it issued, frees its TMEM and returns.
#include <cuda_runtime.h>
#include <math.h>

#include "../../include/mb.h"
#include "kernels.h"
#include "mb_device.cuh"

namespace mb {
namespace {

using namespace dev;

constexpr int BM = 128;  // TMEM lanes (query rows, possibly copied)
constexpr int BN = 128;  // keys per tile
constexpr int kThreads = 320;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;  // + 128 * buffer
constexpr uint32_t kColO = 256;
constexpr float kRescaleThreshold = 8.0f;
constexpr uint64_t kDrainNs = 200000000ull;
constexpr int kOpSlots = 3;   // 16-bit operand tiles: K_j, V_j, K_j+1, ...
constexpr int kScSlots = 4;   // per-tile scale vectors
constexpr int kMaxStSlots = 8;

enum {
  B_ST_FULL = 0,                           // + staging slot
  B_ST_EMPTY = B_ST_FULL + kMaxStSlots,    // + staging slot
  B_OP_FULL = B_ST_EMPTY + kMaxStSlots,    // + operand slot
  B_OP_EMPTY = B_OP_FULL + kOpSlots,       // + operand slot
  B_SCK_FULL = B_OP_EMPTY + kOpSlots,      // + scale slot
  B_SCV_FULL = B_SCK_FULL + kScSlots,      // + scale slot
  B_SC_EMPTY = B_SCV_FULL + kScSlots,      // + scale slot
  B_S_FULL = B_SC_EMPTY + kScSlots,        // + S buffer
  B_P_FULL = B_S_FULL + 2,
  B_O_DONE = B_P_FULL + 1,
  B_RED_FULL = B_O_DONE + 1,               // + buffer
  B_EPI_FULL = B_RED_FULL + 2,
  B_MMA_DONE = B_EPI_FULL + 1,
  B_COUNT = B_MMA_DONE + 1
};

template <int D>
struct Layout {
  static constexpr int kHalves = D / 64;
  static constexpr uint32_t kHalfBytes = 128 * 128;  // 128 rows x 64 16-bit values
  static constexpr uint32_t kTileBytes = kHalves * kHalfBytes;
  static constexpr int kStSlots = D == 128 ? 4 : 8;
  static constexpr uint32_t kStCodes = BN * D;             // codes of one staged tile
  static constexpr uint32_t kStBytes = kStCodes + BN * 4;  // + its scales
  static constexpr uint32_t q_off = 0;
  static constexpr uint32_t op_off = kTileBytes;
  static constexpr uint32_t st_off = op_off + kOpSlots * kTileBytes;
  static constexpr uint32_t sc_off = st_off + kStSlots * kStBytes;
  static constexpr uint32_t redm_off = sc_off + kScSlots * 2 * BN * 4;  // float [2][4][32]
  static constexpr uint32_t redl_off = redm_off + 2 * 4 * 32 * 4;       // float [4][32]
  static constexpr uint32_t bar_off = redl_off + 4 * 32 * 4;
  static constexpr uint32_t misc_off = bar_off + B_COUNT * 8;
  static constexpr uint32_t kBytes = misc_off + 16;
  // more than half the SM so that one CTA holds the SM's 512 TMEM columns
  static constexpr uint32_t kAlloc =
      (kBytes + 1024 > 232448u / 2 + 1024) ? kBytes + 1024 : 232448u / 2 + 1024;
  // the epilogue adds the row copies' outputs in the (then idle) operand ring
  static constexpr int kRedRow = D + 4;  // floats per row, padded against bank conflicts
  static_assert(kStSlots <= kMaxStSlots, "staging ring");
  static_assert(4 * 32 * kRedRow * 4 <= kOpSlots * kTileBytes, "reduction buffer");
  static_assert(kAlloc <= 232448, "shared memory");
};

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Two e4m3 codes (low byte first) -> f16x2 (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((unsigned short)(two & 0xffffu)));
  return r;
}
// f16x2 -> bf16x2, exact for values that fit both formats (every e4m3 value).
__device__ __forceinline__ uint32_t f16x2_to_bf16x2(uint32_t h) {
  float lo, hi;
  asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(h));
  return pack_bf16x2(lo, hi);
}
// bf16x2 -> f16x2, round to nearest, saturating at +-65504.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t u) {
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(bf16_hi(u)), "f"(bf16_lo(u)));
  return r;
}

struct Shared {
  uint64_t* bars;
  volatile int* abort_flag;
  const float* sc;  // [kScSlots][2][BN]: ks * scale_log2, vs
  float* redm;      // [2][4][32]
  float* redl;      // [4][32]
  float* redo;      // [4][32][D + 4] (operand ring, epilogue only)
  uint32_t tmem;
};

// Softmax role of warp `warp` (0-3). Rows: group g = warp % ngrp of 32 rows,
// copy c = warp / ngrp; W = 128 / R keys of every tile per copy (R = 4 / ngrp
// copies of each row).
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
  const int vis_hi = min(it.k_end, rd.vis_end);
  const uint32_t lane_addr = (uint32_t)(warp * 32) << 16;
  const uint32_t o_col = sh.tmem + lane_addr + kColO;
  const int col0 = c * W;
  float m = -INFINITY, l = 0.f;
  bool ok = true;
  for (int j = 0; j < n; ++j) {
    const int sc = j % kScSlots;
    const uint32_t scph = (uint32_t)(j / kScSlots) & 1u;
    const uint32_t p_col = sh.tmem + lane_addr + kColS + 128 * (j & 1);
    ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_S_FULL + (j & 1)], (uint32_t)(j >> 1) & 1u,
                                           sh.abort_flag, a.status));
    if (!ok) break;
    tc_fence_after();
    ok = __all_sync(0xffffffffu,
                    mbar_wait(&bars[B_SCK_FULL + sc], scph, sh.abort_flag, a.status));
    if (!ok) break;
    // scores in the log2 domain: ks_j * log2(e) * scale * (q . kcode_j),
    // keys past the row's visibility bound at -inf
    const float* kf = sh.sc + sc * 2 * BN + col0;
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
        const float4 f = reinterpret_cast<const float4*>(kf + 32 * h)[e4];
        const float fv[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int e = 4 * e4 + q;
          x[e] = __float_as_uint(32 * h + e < lim ? __uint_as_float(x[e]) * fv[q] : -INFINITY);
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
    if constexpr (R > 1) {
      // the copies of a row agree on the tile max
      float* red = sh.redm + (j & 1) * 128;
      red[warp * 32 + lane] = mx;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_RED_FULL + (j & 1)]);
      ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_RED_FULL + (j & 1)],
                                             (uint32_t)(j >> 1) & 1u, sh.abort_flag, a.status));
      if (!ok) break;
#pragma unroll
      for (int cc = 0; cc < R; ++cc) mx = fmaxf(mx, red[(g + ngrp * cc) * 32 + lane]);
    }
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
    ok = __all_sync(0xffffffffu,
                    mbar_wait(&bars[B_SCV_FULL + sc], scph, sh.abort_flag, a.status));
    if (!ok) break;
    // P' = p * vs_j in bf16, stored 16 packed columns (32 keys) at a time
    // into S buffer j & 1 (P(j-1) V(j-1) reads the other one); the other
    // copies' columns are zero
    const float4* vf = reinterpret_cast<const float4*>(sh.sc + sc * 2 * BN + BN + col0);
    float sum[2] = {0.f, 0.f};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      constexpr int kChunks = W / 32;  // 32-key chunks of this copy
      const int owner = q / kChunks;   // copy whose keys fill packed columns [16q, 16q+16)
      uint32_t pk[16];
      if (owner == c) {
        const int h = q % kChunks;
        uint32_t* x = W <= 64 ? &s[32 * h] : s;
        if (W > 64) scaled_chunk(h, x);
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          const float4 f = vf[8 * h + e4];
          const float p0 = fast_exp2(__uint_as_float(x[4 * e4]) - mc);
          const float p1 = fast_exp2(__uint_as_float(x[4 * e4 + 1]) - mc);
          const float p2 = fast_exp2(__uint_as_float(x[4 * e4 + 2]) - mc);
          const float p3 = fast_exp2(__uint_as_float(x[4 * e4 + 3]) - mc);
          sum[0] += p0 + p2;
          sum[1] += p1 + p3;
          pk[2 * e4] = pack_bf16x2(p0 * f.x, p1 * f.y);
          pk[2 * e4 + 1] = pack_bf16x2(p2 * f.z, p3 * f.w);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) pk[e] = 0u;
      }
      tmem_st16(p_col + 16 * q, pk);
    }
    l += sum[0] + sum[1];
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars[B_SC_EMPTY + sc]);
    // O may be rescaled once P(j-1) V(j-1) completed; waiting every tile
    // also keeps this barrier's phases in step
    if (j > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_O_DONE], (uint32_t)(j - 1) & 1u,
                                             sh.abort_flag, a.status));
      if (!ok) break;
    }
    tc_fence_after();
    if (__any_sync(0xffffffffu, need)) {
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
    if (lane == 0) mbar_arrive(&bars[B_P_FULL]);
  }
  if (ok && n > 0)
    ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_O_DONE], (uint32_t)(n - 1) & 1u,
                                           sh.abort_flag, a.status));
  if (!ok || n == 0) return;
  tc_fence_after();
  const bool final_row = rd.dst < 0;
  const int64_t orow = (int64_t)rd.q_index * a.n_q_heads + rd.q_head;
  if constexpr (R == 1) {
    const bool any = l > 0.f;
    const float inv = any ? 1.f / l : 0.f;
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
    if (valid && !final_row) a.part_lse[rd.dst] = lse2;
  } else {
    // add the R copies: every warp parks its lanes' l and O, then finishes
    // D / R columns of its row group
    constexpr int RR = L::kRedRow;
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
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars[B_EPI_FULL]);
    if (!__all_sync(0xffffffffu, mbar_wait(&bars[B_EPI_FULL], 0u, sh.abort_flag, a.status)))
      return;
    float lt = 0.f;
#pragma unroll
    for (int cc = 0; cc < R; ++cc) lt += sh.redl[(g + ngrp * cc) * 32 + lane];
    const bool any = lt > 0.f;
    const float inv = any ? 1.f / lt : 0.f;
    const float lse2 = any ? m + log2f(lt) : -INFINITY;
    constexpr int CW = D / R;  // columns this warp finishes
    const int cbeg = c * CW;
    if (valid) {
#pragma unroll 4
      for (int q4 = 0; q4 < CW / 4; ++q4) {
        const int col = cbeg + 4 * q4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int cc = 0; cc < R; ++cc) {
          const float4 v = *reinterpret_cast<const float4*>(
              sh.redo + ((g + ngrp * cc) * 32 + lane) * RR + col);
          acc.x += v.x;
          acc.y += v.y;
          acc.z += v.z;
          acc.w += v.w;
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
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    splitkv_fp8_kernel(const DecodeFp8Args a, const int ps_shift) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sq = smem + L::q_off;
  uint8_t* sop = smem + L::op_off;
  uint8_t* sst = smem + L::st_off;
  float* ssc = reinterpret_cast<float*>(smem + L::sc_off);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::bar_off);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::misc_off + 4);

  // the combine kernel launched after this one may be scheduled now; it
  // waits for this grid to finish before it reads the partials
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const DecodeItem it = a.items[blockIdx.x];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nr = it.n_rows;
  const int n = ceil_div(it.k_end - it.k_begin, BN);
  const int nw = ceil_div(nr, 32);
  const int ngrp = nw <= 1 ? 1 : (nw == 2 ? 2 : 4);  // row groups; 4 / ngrp copies per row

  if (threadIdx.x == 0) {
    for (int s = 0; s < L::kStSlots; ++s) {
      mbar_init(&bars[B_ST_FULL + s], 1);
      mbar_init(&bars[B_ST_EMPTY + s], 4);
    }
    for (int o = 0; o < kOpSlots; ++o) {
      mbar_init(&bars[B_OP_FULL + o], 4);
      mbar_init(&bars[B_OP_EMPTY + o], 1);
    }
    for (int c = 0; c < kScSlots; ++c) {
      mbar_init(&bars[B_SCK_FULL + c], 4);
      mbar_init(&bars[B_SCV_FULL + c], 4);
      mbar_init(&bars[B_SC_EMPTY + c], 4);
    }
    mbar_init(&bars[B_S_FULL + 0], 1);
    mbar_init(&bars[B_S_FULL + 1], 1);
    mbar_init(&bars[B_P_FULL], 4);
    mbar_init(&bars[B_O_DONE], 1);
    mbar_init(&bars[B_RED_FULL + 0], 4);
    mbar_init(&bars[B_RED_FULL + 1], 4);
    mbar_init(&bars[B_EPI_FULL], 4);
    mbar_init(&bars[B_MMA_DONE], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  // Q tile (f16, K-major, 128-byte swizzle). TMEM lane 32w + l holds row
  // 32 (w % ngrp) + l; lanes without a row are zero.
  {
    const uint4* q = static_cast<const uint4*>(a.q);
    constexpr int CH = D / 8;  // 16-byte chunks per row
    for (int idx = threadIdx.x; idx < BM * CH; idx += kThreads) {
      const int r = idx / CH, c = idx - r * CH;
      const int src = 32 * ((r >> 5) % ngrp) + (r & 31);
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (src < nr) {
        const RowDesc rd = a.rows[it.row_begin + src];
        const uint4 b = __ldg(q + ((int64_t)rd.q_index * a.n_q_heads + rd.q_head) * CH + c);
        v.x = bf16x2_to_f16x2(b.x);
        v.y = bf16x2_to_f16x2(b.y);
        v.z = bf16x2_to_f16x2(b.z);
        v.w = bf16x2_to_f16x2(b.w);
      }
      const int half = c >> 3, c8 = c & 7;
      *reinterpret_cast<uint4*>(sq + half * L::kHalfBytes + r * 128 + ((c8 ^ (r & 7)) << 4)) = v;
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    const int ps = 1 << ps_shift;
    const int npg = BN / ps;
    const int32_t* btrow = a.block_table + (int64_t)it.bt_row * a.max_blocks;
    const int last_block = (it.k_end - 1) >> ps_shift;
    const int first_block = it.k_begin >> ps_shift;  // k_begin is page-aligned
    int64_t my_row = 0;  // first cache row of this lane's page (rows of D codes)
    int issued = 0;
    for (int i = 0; i < 2 * n; ++i) {
      const int j = i >> 1, s = i % L::kStSlots;
      const uint32_t ph = (uint32_t)(i / L::kStSlots) & 1u;
      if (i >= L::kStSlots &&
          !__all_sync(0xffffffffu, mbar_wait(&bars[B_ST_EMPTY + s], ph ^ 1u, abort_flag,
                                             a.status)))
        break;
      if ((i & 1) == 0 && lane < npg) {
        int b = first_block + j * npg + lane;
        if (b > last_block) b = last_block;  // keys past k_end: masked, V zeroed
        int32_t page = __ldg(btrow + b);
        if ((unsigned)page >= (unsigned)a.num_pages) {
          set_status(a.status, MB_ERR_DEVICE_INDEX);
          page = 0;
        }
        my_row = ((int64_t)page * a.n_kv_heads + it.kv_head) << ps_shift;
      }
      if (lane == 0) mbar_arrive_expect_tx(&bars[B_ST_FULL + s], L::kStBytes);
      __syncwarp();
      if (lane < npg) {
        uint8_t* dst = sst + s * L::kStBytes;
        const uint8_t* codes = static_cast<const uint8_t*>((i & 1) ? a.v8 : a.k8);
        const float* scales = (i & 1) ? a.v_scale : a.k_scale;
        bulk_load(dst + lane * ps * D, codes + my_row * D, (uint32_t)(ps * D),
                  &bars[B_ST_FULL + s]);
        bulk_load(dst + L::kStCodes + lane * ps * 4, scales + my_row, (uint32_t)(ps * 4),
                  &bars[B_ST_FULL + s]);
      }
      issued = i + 1;
    }
    __syncwarp();
    if (lane == 0)
      for (int i = max(0, issued - L::kStSlots); i < issued; ++i)
        mbar_drain(&bars[B_ST_FULL + i % L::kStSlots], (uint32_t)(i / L::kStSlots) & 1u,
                   kDrainNs);
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ converters
    const int ct = threadIdx.x - 128;
    constexpr int TPR = D / 8;  // 8-code tasks per key row
    for (int i = 0; i < 2 * n; ++i) {
      const int j = i >> 1, s = i % L::kStSlots, o = i % kOpSlots, sc = j % kScSlots;
      const bool is_v = i & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&bars[B_ST_FULL + s],
                                             (uint32_t)(i / L::kStSlots) & 1u, abort_flag,
                                             a.status)))
        break;
      if (i >= kOpSlots &&
          !__all_sync(0xffffffffu, mbar_wait(&bars[B_OP_EMPTY + o],
                                             ((uint32_t)(i / kOpSlots) & 1u) ^ 1u, abort_flag,
                                             a.status)))
        break;
      if (!is_v && j >= kScSlots &&
          !__all_sync(0xffffffffu, mbar_wait(&bars[B_SC_EMPTY + sc],
                                             ((uint32_t)(j / kScSlots) & 1u) ^ 1u, abort_flag,
                                             a.status)))
        break;
      tc_fence_after();
      const uint8_t* st = sst + s * L::kStBytes;
      uint8_t* op = sop + o * L::kTileBytes;
      const int nvalid = min(BN, it.k_end - (it.k_begin + j * BN));
      if (!is_v) {
#pragma unroll 4
        for (int idx = ct; idx < BN * TPR; idx += 128) {
          const int key = idx / TPR, e8 = idx % TPR;
          const uint2 raw = *reinterpret_cast<const uint2*>(st + key * D + e8 * 8);
          uint4 v;
          v.x = e4m3x2_to_f16x2(raw.x);
          v.y = e4m3x2_to_f16x2(raw.x >> 16);
          v.z = e4m3x2_to_f16x2(raw.y);
          v.w = e4m3x2_to_f16x2(raw.y >> 16);
          const int half = e8 >> 3, c8 = e8 & 7;
          *reinterpret_cast<uint4*>(op + half * L::kHalfBytes + key * 128 +
                                    ((c8 ^ (key & 7)) << 4)) = v;
        }
      } else {
#pragma unroll 4
        for (int idx = ct; idx < BN * TPR; idx += 128) {
          const int key = idx / TPR, e8 = idx % TPR;
          uint4 v = make_uint4(0u, 0u, 0u, 0u);
          if (key < nvalid) {  // rows past k_end may hold any bits (P is 0 there)
            const uint2 raw = *reinterpret_cast<const uint2*>(st + key * D + e8 * 8);
            v.x = f16x2_to_bf16x2(e4m3x2_to_f16x2(raw.x));
            v.y = f16x2_to_bf16x2(e4m3x2_to_f16x2(raw.x >> 16));
            v.z = f16x2_to_bf16x2(e4m3x2_to_f16x2(raw.y));
            v.w = f16x2_to_bf16x2(e4m3x2_to_f16x2(raw.y >> 16));
          }
          const int half = e8 >> 3, c8 = e8 & 7;
          *reinterpret_cast<uint4*>(op + half * L::kHalfBytes + key * 128 +
                                    ((c8 ^ (key & 7)) << 4)) = v;
        }
      }
      {
        const float x = reinterpret_cast<const float*>(st + L::kStCodes)[ct];
        float* dst = ssc + sc * 2 * BN + (is_v ? BN : 0);
        dst[ct] = is_v ? (ct < nvalid ? x : 0.f) : x * a.scale_log2;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars[B_ST_EMPTY + s]);
        mbar_arrive(&bars[B_OP_FULL + o]);
        mbar_arrive(&bars[(is_v ? B_SCV_FULL : B_SCK_FULL) + sc]);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_f16_f32(BM, BN, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(BM, D, false, true);
      const uint32_t qa = smem_u32(sq);
      const uint32_t opa = smem_u32(sop);
      auto wait = [&](int b, uint32_t parity) -> bool {
        const bool ok = mbar_wait(&bars[b], parity, abort_flag, a.status);
        tc_fence_after();
        return ok;
      };
      auto issue_s = [&](int j) -> bool {
        const int ki = 2 * j, o = ki % kOpSlots;
        if (!wait(B_OP_FULL + o, (uint32_t)(ki / kOpSlots) & 1u)) return false;
        const uint32_t k0 = opa + o * L::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * L::kHalfBytes + (kk & 3) * 32;
          umma_bf16_ss(tmem + kColS + 128 * (j & 1), sdesc_sw128(qa + off, 16, 1024),
                       sdesc_sw128(k0 + off, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
        }
        umma_commit(&bars[B_S_FULL + (j & 1)]);
        umma_commit(&bars[B_OP_EMPTY + o]);
        return true;
      };
      bool ok = n > 0 && issue_s(0);
      if (ok && n > 1) ok = issue_s(1);
      for (int j = 0; ok && j < n; ++j) {
        const int vi = 2 * j + 1, o = vi % kOpSlots;
        if (!(ok = wait(B_OP_FULL + o, (uint32_t)(vi / kOpSlots) & 1u))) break;
        if (!(ok = wait(B_P_FULL, (uint32_t)j & 1u))) break;
        const uint32_t v0 = opa + o * L::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          const uint64_t bd = sdesc_sw128(v0 + kk * 2048, L::kHalfBytes, 1024);
          umma_bf16_ts(tmem + kColO, tmem + kColS + 128 * (j & 1) + kk * 8, bd, idesc_pv,
                       (j > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&bars[B_O_DONE]);
        umma_commit(&bars[B_OP_EMPTY + o]);
        // S(j+2) reuses this S buffer; it follows PV(j) in issue order
        if (j + 2 < n && !(ok = issue_s(j + 2))) break;
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
    sh.sc = ssc;
    sh.redm = reinterpret_cast<float*>(smem + L::redm_off);
    sh.redl = reinterpret_cast<float*>(smem + L::redl_off);
    sh.redo = reinterpret_cast<float*>(sop);
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
}

}  // namespace

cudaError_t launch_decode_fp8(const DecodeFp8Args& a, cudaStream_t s) {
  if (a.n_items <= 0) return cudaSuccess;
  const int ps_shift = __builtin_ctz((unsigned)a.page_size);
  cudaError_t e;
  if (a.head_dim == 128) {
    e = cudaFuncSetAttribute(splitkv_fp8_kernel<128>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)Layout<128>::kAlloc);
    if (e != cudaSuccess) return e;
    splitkv_fp8_kernel<128><<<(unsigned)a.n_items, kThreads, Layout<128>::kAlloc, s>>>(a, ps_shift);
    return cudaGetLastError();
  }
  e = cudaFuncSetAttribute(splitkv_fp8_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)Layout<64>::kAlloc);
  if (e != cudaSuccess) return e;
  splitkv_fp8_kernel<64><<<(unsigned)a.n_items, kThreads, Layout<64>::kAlloc, s>>>(a, ps_shift);
  return cudaGetLastError();
}

}  // namespace mb
