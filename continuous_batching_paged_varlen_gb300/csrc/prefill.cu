// Prefill / chunk attention on the 5th-generation tensor cores (tcgen05).
//
// One CTA owns 128 consecutive new rows of one request and one query head
// and walks that request's keys in 128-key tiles ("ORCA and chunked
// prefill", section 4: a chunk of C rows attends to the S cached keys with
// no mask and to its own C keys causally). Tiles that lie wholly above the
// causal frontier of every row in the CTA are never visited; only tiles
// that straddle it apply the mask (key j visible to new row i iff
// j <= S0 + i, "How To Scale Your Model notes (7-8)", section 2).
//
// Data movement and roles (192 threads):
//   warp 0      TMA producer: Q tile once (3-D tensor map over [total_q, Hq, D]),
//               then K and V tiles page by page through the block table
//               (2-D tensor map over the [pages * Hkv * page_size, D] cache
//               view), 2-stage ring, 128-byte swizzle.
//   warp 1      allocates 512 TMEM columns; one lane issues the MMAs:
//               S = Q K^T (M 128, N 128, K = D) into a double-buffered TMEM
//               score tile, O += P V (M 128, N = D, K 128) into the TMEM
//               accumulator.
//   warps 2-5   softmax, one thread per query row (TMEM lane = row): load the
//               score row, mask, online max / sum in the log2 domain, write
//               P (bf16, swizzled K-major) to shared memory, rescale O in
//               TMEM only when the running max grew by more than 2^8, and at
//               the end normalise O and store the bf16 row and its LSE.
//
// Every wait is bounded (see mb_device.cuh); on a timeout the CTA raises
// its abort flag, drains the copies it issued, frees its TMEM and returns.
#include <cuda_runtime.h>
#include <math.h>

#include "../../include/mb.h"
#include "kernels.h"
#include "mb_device.cuh"

namespace mb {
namespace {

using namespace dev;

constexpr int BM = kPrefillTileM;
constexpr int BN = kPrefillTileN;
constexpr int kThreads = 192;
constexpr int kStages = 2;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P may reach 2^8 before O is rescaled
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint64_t kDrainNs = 200000000ull;

// barrier slots
enum {
  B_Q_FULL = 0,
  B_K_FULL = 1,    // +stage
  B_K_EMPTY = 3,   // +stage
  B_V_FULL = 5,    // +stage
  B_V_EMPTY = 7,   // +stage
  B_S_FULL = 9,    // +buffer
  B_S_FREE = 11,   // +buffer
  B_P_FULL = 13,
  B_PV_DONE = 14,
  B_VZ_READY = 15,
  B_COUNT = 16
};

template <int D>
struct Layout {
  static constexpr int kHalves = D / 64;                      // 64-element (128 B) column blocks
  static constexpr uint32_t kHalfBytes = 128 * 128;           // 128 rows x 128 B
  static constexpr uint32_t kQBytes = kHalves * kHalfBytes;
  static constexpr uint32_t kKVBytes = kHalves * kHalfBytes;  // one stage of K (or V)
  static constexpr uint32_t kPBytes = 2 * kHalfBytes;         // 128 keys = two 64-key blocks
  static constexpr uint32_t q_off = 0;
  static constexpr uint32_t k_off = q_off + kQBytes;
  static constexpr uint32_t v_off = k_off + kStages * kKVBytes;
  static constexpr uint32_t p_off = v_off + kStages * kKVBytes;
  static constexpr uint32_t bar_off = p_off + kPBytes;
  static constexpr uint32_t misc_off = bar_off + B_COUNT * 8;
  static constexpr uint32_t kBytes = misc_off + 16;
  // + alignment slack; at least 118 KB so that two CTAs never share an SM
  // (each holds all 512 TMEM columns)
  static constexpr uint32_t kAlloc = (kBytes + 1024 > 118u * 1024u) ? kBytes + 1024 : 118u * 1024u;
};

struct Params {
  const PrefillItem* items;
  const int32_t* block_table;
  int32_t max_blocks, n_q_heads, n_kv_heads, num_pages, group, ps_shift;
  float scale_log2;
  __nv_bfloat16* out;
  float* lse;
  int32_t* status;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const Params p, const __grid_constant__ CUtensorMap q_map,
                   const __grid_constant__ CUtensorMap k_map,
                   const __grid_constant__ CUtensorMap v_map) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sq = smem + L::q_off;
  uint8_t* sk = smem + L::k_off;
  uint8_t* sv = smem + L::v_off;
  uint8_t* sp = smem + L::p_off;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::bar_off);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::misc_off + 4);

  const PrefillItem it = p.items[blockIdx.x];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tiles = it.n_kv_tiles;
  const bool tail_zero = n_tiles * BN > it.kv_length;  // last tile holds keys >= kv_length

  if (threadIdx.x == 0) {
    mbar_init(&bars[B_Q_FULL], 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars[B_K_FULL + s], 1);
      mbar_init(&bars[B_K_EMPTY + s], 1);
      mbar_init(&bars[B_V_FULL + s], 1);
      mbar_init(&bars[B_V_EMPTY + s], 1);
      mbar_init(&bars[B_S_FULL + s], 1);
      mbar_init(&bars[B_S_FREE + s], 4);
    }
    mbar_init(&bars[B_P_FULL], 4);
    mbar_init(&bars[B_PV_DONE], 1);
    mbar_init(&bars[B_VZ_READY], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int last_issued = -1;
    const int ps = 1 << p.ps_shift;
    if (lane == 0) {
      prefetch_tensormap(&q_map);
      prefetch_tensormap(&k_map);
      prefetch_tensormap(&v_map);
      mbar_arrive_expect_tx(&bars[B_Q_FULL], L::kQBytes);
      for (int h2 = 0; h2 < L::kHalves; ++h2)
        tma_load_3d(sq + h2 * L::kHalfBytes, &q_map, &bars[B_Q_FULL], h2 * 64, it.q_head,
                    it.q_row0);
      const int32_t* btrow = p.block_table + (int64_t)it.req * p.max_blocks;
      const int last_block = (it.kv_length - 1) >> p.ps_shift;
      const int kv_head = it.q_head / p.group;
      for (int j = 0; j < n_tiles; ++j) {
        const int st = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        if (j >= kStages && !mbar_wait(&bars[B_K_EMPTY + st], ph ^ 1, abort_flag, p.status))
          break;
        mbar_arrive_expect_tx(&bars[B_K_FULL + st], L::kKVBytes);
        int32_t ys[BN / 16];
        for (int pg = 0; pg < BN / ps; ++pg) {
          int b = ((j * BN) >> p.ps_shift) + pg;
          if (b > last_block) b = last_block;  // keys past kv_length: masked / zeroed
          int32_t page = __ldg(btrow + b);
          if ((unsigned)page >= (unsigned)p.num_pages) {
            set_status(p.status, MB_ERR_DEVICE_INDEX);
            page = 0;
          }
          ys[pg] = (page * p.n_kv_heads + kv_head) << p.ps_shift;
          for (int h2 = 0; h2 < L::kHalves; ++h2)
            tma_load_2d(sk + st * L::kKVBytes + h2 * L::kHalfBytes + pg * ps * 128, &k_map,
                        &bars[B_K_FULL + st], h2 * 64, ys[pg]);
        }
        if (j >= kStages && !mbar_wait(&bars[B_V_EMPTY + st], ph ^ 1, abort_flag, p.status)) {
          last_issued = j;  // K of tile j is in flight
          break;
        }
        mbar_arrive_expect_tx(&bars[B_V_FULL + st], L::kKVBytes);
        for (int pg = 0; pg < BN / ps; ++pg)
          for (int h2 = 0; h2 < L::kHalves; ++h2)
            tma_load_2d(sv + st * L::kKVBytes + h2 * L::kHalfBytes + pg * ps * 128, &v_map,
                        &bars[B_V_FULL + st], h2 * 64, ys[pg]);
        last_issued = j;
      }
    }
    __syncwarp();
    last_issued = __shfl_sync(0xffffffffu, last_issued, 0);
    if (tail_zero && last_issued == n_tiles - 1) {
      // keys >= kv_length of the last tile: zero their V rows so that a
      // non-finite value in an unwritten slot cannot reach O through P = 0
      const int j = n_tiles - 1, st = j & 1;
      const bool ok =
          __all_sync(0xffffffffu, mbar_wait(&bars[B_V_FULL + st], (j >> 1) & 1, abort_flag,
                                            p.status));
      if (ok) {
        const int r0 = it.kv_length - j * BN;
        const int nz = BN - r0;
        uint8_t* vb = sv + st * L::kKVBytes;
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
    if (lane == 0) {
      // drain every copy still in flight before the CTA may exit
      mbar_drain(&bars[B_Q_FULL], 0, kDrainNs);
      for (int j = last_issued - 1; j <= last_issued; ++j) {
        if (j < 0) continue;
        mbar_drain(&bars[B_K_FULL + (j & 1)], (j >> 1) & 1, kDrainNs);
        mbar_drain(&bars[B_V_FULL + (j & 1)], (j >> 1) & 1, kDrainNs);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(BM, BN, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(BM, D, false, true);
      const uint32_t qa = smem_u32(sq);
      const uint32_t pa = smem_u32(sp);
      int last_pv = -1, last_s = -1;
      auto issue_pv = [&](int t) -> bool {
        const int st = t & 1;
        if (!mbar_wait(&bars[B_P_FULL], t & 1, abort_flag, p.status)) return false;
        if (!mbar_wait(&bars[B_V_FULL + st], (t >> 1) & 1, abort_flag, p.status)) return false;
        if (t == n_tiles - 1 && tail_zero &&
            !mbar_wait(&bars[B_VZ_READY], 0, abort_flag, p.status))
          return false;
        tc_fence_after();
        const uint32_t va = smem_u32(sv + st * L::kKVBytes);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          // A = P [128 rows x 128 keys], K-major: 64-key block kk/4, 32 B step inside it
          const uint64_t ad = sdesc_sw128(pa + (kk >> 2) * L::kHalfBytes + (kk & 3) * 32, 16, 1024);
          // B = V [128 keys x D], MN-major: 16 keys = two 8-row groups (SBO 1024),
          // next 64 head dims one half further (LBO)
          const uint64_t bd = sdesc_sw128(va + kk * 2048, L::kHalfBytes, 1024);
          umma_bf16_ss(tmem + kColO, ad, bd, idesc_pv, (t > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&bars[B_PV_DONE]);
        umma_commit(&bars[B_V_EMPTY + st]);
        last_pv = t;
        return true;
      };
      bool ok = mbar_wait(&bars[B_Q_FULL], 0, abort_flag, p.status);
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int st = j & 1;
        if (!mbar_wait(&bars[B_K_FULL + st], (j >> 1) & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        if (j >= 2 && !mbar_wait(&bars[B_S_FREE + st], ((j - 2) >> 1) & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t ka = smem_u32(sk + st * L::kKVBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * L::kHalfBytes + (kk & 3) * 32;
          umma_bf16_ss(tmem + (st ? kColS1 : kColS0), sdesc_sw128(qa + off, 16, 1024),
                       sdesc_sw128(ka + off, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
        }
        umma_commit(&bars[B_S_FULL + st]);
        umma_commit(&bars[B_K_EMPTY + st]);
        last_s = j;
        if (j >= 1 && !issue_pv(j - 1)) ok = false;
      }
      if (ok) issue_pv(n_tiles - 1);
      // wait for the tensor core to finish what was issued
      if (last_pv >= 0) mbar_drain(&bars[B_PV_DONE], last_pv & 1, kDrainNs);
      if (last_s >= 0) mbar_drain(&bars[B_S_FULL + (last_s & 1)], (last_s >> 1) & 1, kDrainNs);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int wq = warp & 3;  // TMEM sub-partition this warp may access
    const int r = wq * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(wq * 32) << 16;
    const int vis_last = it.s0 + it.i0 + r;       // last key this row sees
    const int tile_first_vis = it.s0 + it.i0;     // ... for the CTA's first row
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      const int sb = j & 1;
      ok = __all_sync(0xffffffffu,
                      mbar_wait(&bars[B_S_FULL + sb], (j >> 1) & 1, abort_flag, p.status));
      if (!ok) break;
      tc_fence_after();
      uint32_t s[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        tmem_ld32(tmem + lane_addr + (sb ? kColS1 : kColS0) + c * 32, s[c]);
        tmem_ld_wait(s[c]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_S_FREE + sb]);

      const int key0 = j * BN;
      const bool need_mask = key0 + BN - 1 > tile_first_vis;
      float mt = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          float v = __uint_as_float(s[c][e]) * p.scale_log2;
          if (need_mask && key0 + c * 32 + e > vis_last) v = -INFINITY;
          s[c][e] = __float_as_uint(v);
          mt = fmaxf(mt, v);
        }
      const float m_new = fmaxf(m, mt);
      if (j >= 1) {
        ok = __all_sync(0xffffffffu,
                        mbar_wait(&bars[B_PV_DONE], (j - 1) & 1, abort_flag, p.status));
        if (!ok) break;
      }
      if (j == 0) {
        m = m_new;
      } else {
        const bool need = m_new > m + kRescaleThreshold;
        if (__any_sync(0xffffffffu, need)) {
          const float alpha = need ? fast_exp2(m - m_new) : 1.f;
          if (need) {
            l *= alpha;
            m = m_new;
          }
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_addr + kColO + c * 32, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tmem + lane_addr + kColO + c * 32, o);
          }
          tmem_st_wait();
        }
      }
      const float mx = (m == -INFINITY) ? 0.f : m;
      float rowsum = 0.f;
#pragma unroll
      for (int ch = 0; ch < BN / 8; ++ch) {
        float e8[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          e8[t] = fast_exp2(__uint_as_float(s[ch >> 2][(ch & 3) * 8 + t]) - mx);
          rowsum += e8[t];
        }
        uint4 pk;
        pk.x = pack_bf16x2(e8[0], e8[1]);
        pk.y = pack_bf16x2(e8[2], e8[3]);
        pk.z = pack_bf16x2(e8[4], e8[5]);
        pk.w = pack_bf16x2(e8[6], e8[7]);
        const int half = ch >> 3, c8 = ch & 7;
        *reinterpret_cast<uint4*>(sp + half * L::kHalfBytes + r * 128 + ((c8 ^ (r & 7)) << 4)) =
            pk;
      }
      l += rowsum;
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_P_FULL]);
    }
    if (ok)
      ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_PV_DONE], (n_tiles - 1) & 1, abort_flag,
                                             p.status));
    if (ok) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const bool valid = r < it.n_rows;
      const int64_t orow = (int64_t)(it.q_row0 + r) * p.n_q_heads + it.q_head;
      uint4* dst = reinterpret_cast<uint4*>(p.out + orow * D);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_addr + kColO + c * 32, o);
        tmem_ld_wait(o);
        if (valid) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(o[q4 * 8 + 0]) * inv, __uint_as_float(o[q4 * 8 + 1]) * inv);
            v.y = pack_bf16x2(__uint_as_float(o[q4 * 8 + 2]) * inv, __uint_as_float(o[q4 * 8 + 3]) * inv);
            v.z = pack_bf16x2(__uint_as_float(o[q4 * 8 + 4]) * inv, __uint_as_float(o[q4 * 8 + 5]) * inv);
            v.w = pack_bf16x2(__uint_as_float(o[q4 * 8 + 6]) * inv, __uint_as_float(o[q4 * 8 + 7]) * inv);
            dst[c * 4 + q4] = v;
          }
        }
      }
      if (valid && p.lse) p.lse[orow] = (m + log2f(l)) * kLn2;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
cudaError_t launch_d(const PrefillArgs& a, cudaStream_t s) {
  Params p;
  p.items = a.items;
  p.block_table = a.block_table;
  p.max_blocks = a.max_blocks;
  p.n_q_heads = a.n_q_heads;
  p.n_kv_heads = a.n_kv_heads;
  p.group = a.n_q_heads / a.n_kv_heads;
  p.ps_shift = __builtin_ctz((unsigned)a.page_size);
  p.scale_log2 = a.scale_log2;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.lse = a.lse;
  p.status = a.status;
  p.num_pages = a.num_pages;
  constexpr uint32_t smem = Layout<D>::kAlloc;
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  prefill_kernel<D><<<a.n_items, kThreads, smem, s>>>(p, *a.q_map, *a.k_map, *a.v_map);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t s) {
  if (a.n_items <= 0) return cudaSuccess;
  return a.head_dim == 128 ? launch_d<128>(a, s) : launch_d<64>(a, s);
}

}  // namespace mb
