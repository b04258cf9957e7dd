// Prefill / chunk attention on the 5th-generation tensor cores (tcgen05).
//
// A work item is up to 256 consecutive new rows of one request and one query
// head, as two 128-row tiles A and B, against the request's keys in 128-key
// tiles ("ORCA and chunked prefill", section 4: a chunk of C rows attends to
// the S cached keys with no mask and to its own C keys causally). A tile of
// keys that lies wholly above the causal frontier of every row of a query
// tile is never computed for it; only key tiles that straddle the frontier
// apply the mask (key j visible to new row i iff j <= S0 + i, "How To Scale
// Your Model notes (7-8)", section 2).
//
// The grid is persistent: one CTA per SM (each holds its SM's 512 TMEM
// columns) walks a share of the planner's heavy-first item list, so the next
// item's Q and first K/V tiles load, and its first S MMAs run, while the
// current item's last tiles and epilogue finish. When the iteration also has
// split-KV work, the plan may cap the grid below the SM count: the split-KV
// kernel, launched behind this one, starts at once on the SMs left free and
// takes each SM whose CTA has finished its share.
//
// Roles (384 threads, three warpgroups):
//   warps 0-3   softmax of query tile A, warps 4-7 softmax of tile B: one
//               thread per query row (TMEM lane = row). Load the 128 scores of
//               the row in one TMEM load, mask, take the running max (three-
//               input max), scale and shift two scores per packed f32x2 FMA
//               before ex2 (log2 domain), sum in packed adds, write P as
//               bf16 back into TMEM over the row's own scores (the PV MMA
//               reads its A operand from there), and rescale O in TMEM only
//               when a row's max grew by more than 2^8. At the end of an item
//               read O out of TMEM, release it to the next item's PV, then
//               normalise and store the bf16 rows and their LSE. These
//               warpgroups take registers from the third one (setmaxnreg) so
//               the 128 scores of a row stay in registers.
//   warp 8      TMA producer: both Q tiles of an item (3-D tensor map over
//               [total_q, Hq, D]) once the previous item's S MMAs are done,
//               then K_j, V_j, K_j+1, ... page by page through the block
//               table (2-D tensor map over the [pages * Hkv * page_size, D]
//               cache view) into a 5/6-slot ring shared by the two query
//               tiles; 128-byte swizzle. Each lane looks up one page and issues
//               that page's boxes, so a tile of 16-token pages is in flight
//               after one round of issues.
//   warp 9      allocates all 512 TMEM columns (S_A, S_B, O_A, O_B); one lane
//               issues every MMA: S_X = Q_X K^T (M 128, N 128, K = D, both
//               operands in shared memory) and O_X += P_X V (M 128, N = D,
//               K 128, P from TMEM, V from shared memory), ordered
//                   PV_A(j), S_A(j+1), PV_B(j), S_B(j+1)
//               so that each softmax group has two MMAs' time to turn its
//               scores into probabilities while the tensor core works for the
//               other group. S_X(j+1) overwrites the columns PV_X(j) reads P
//               from; the tensor core runs one thread's MMAs in issue order.
//               This thread paces the kernel (it shares its SM sub-partition
//               with two softmax warps): each MMA costs one integer add per
//               descriptor, a commit is issued only where a waiter needs it,
//               and waits probe the barrier before blocking.
//   warps 10-11 idle.
//
// Every wait is bounded (see mb_device.cuh); on a timeout the CTA raises its
// abort flag, drains the copies and MMAs it issued, frees its TMEM and returns.
#include <cuda_runtime.h>
#include <math.h>

#include "../../include/mb.h"
#include "kernels.h"
#include "mb_device.cuh"

namespace mb {
namespace {

using namespace dev;

constexpr int BM = kPrefillTileM;  // rows of one query tile
constexpr int BN = kPrefillTileN;  // keys of one KV tile
constexpr int kThreads = 384;
// registers per thread: at launch (ptxas' count under the launch bounds, checked
// on the host before every launch), then after the re-allocation
constexpr int kLaunchRegs = 168;
constexpr int kProducerRegs = 88;
constexpr int kSoftmaxRegs = 208;
static_assert(2 * 128 * kSoftmaxRegs + 128 * kProducerRegs <= kThreads * kLaunchRegs,
              "register split exceeds the launch's register pool");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;      // + 128 * tile
constexpr uint32_t kColO = 256;    // + 128 * tile
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P may reach 2^8 before O is rescaled
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint64_t kDrainNs = 200000000ull;

enum {
  kMaxSlots = 6,
  B_Q_FULL = 0,
  B_Q_EMPTY = 1,
  B_KV_FULL = 2,                   // + slot
  B_KV_EMPTY = 2 + kMaxSlots,      // + slot
  B_S_FULL = 2 + 2 * kMaxSlots,    // + tile
  B_P_FULL = 4 + 2 * kMaxSlots,    // + tile
  B_O_DONE = 6 + 2 * kMaxSlots,    // + tile
  B_O_FREE = 8 + 2 * kMaxSlots,    // + tile
  B_VZ_READY = 10 + 2 * kMaxSlots, // + (tail count & 1)
  B_MMA_DONE = 12 + 2 * kMaxSlots, // every MMA the CTA issued has completed
  B_COUNT = 13 + 2 * kMaxSlots
};

template <int D>
struct Layout {
  static constexpr int kHalves = D / 64;                       // 64-element (128 B) column blocks
  static constexpr uint32_t kHalfBytes = 128 * 128;            // 128 rows x 128 B
  static constexpr uint32_t kTileBytes = kHalves * kHalfBytes;  // a Q tile or a K/V slot
  static constexpr int kSlots = D == 128 ? 5 : 6;               // K/V ring slots
  static_assert(kSlots <= kMaxSlots, "barrier slots");
  static constexpr uint32_t q_off = 0;                         // Q_A, Q_B
  static constexpr uint32_t kv_off = q_off + 2 * kTileBytes;   // ring slots
  static constexpr uint32_t bar_off = kv_off + kSlots * kTileBytes;
  static constexpr uint32_t misc_off = bar_off + B_COUNT * 8;
  static constexpr uint32_t kBytes = misc_off + 16;
  static constexpr uint32_t kAlloc = kBytes + 1024;  // + slack for 1024-byte alignment
  static_assert(kAlloc <= 232448, "shared memory");
  static_assert(kAlloc > 232448 / 2, "one CTA per SM (it holds all 512 TMEM columns)");
};

struct Params {
  const PrefillItem* items;
  int32_t n_items;
  const int32_t* block_table;
  int32_t max_blocks, n_q_heads, n_kv_heads, num_pages, group, ps_shift;
  float scale_log2;
  __nv_bfloat16* out;
  float* lse;
  int32_t* status;
};

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// The k-th work item of this CTA. The planner lists items heaviest first; the
// persistent grid takes them in rounds of gridDim.x, walking every other round
// backwards (a snake), so each CTA pairs a heavy item with a light one.
__device__ __forceinline__ int item_of(int k) {
  const int g = (int)gridDim.x, b = (int)blockIdx.x;
  return k * g + ((k & 1) ? g - 1 - b : b);
}

// What one work item needs: rows in query tiles A and B, the KV tiles each
// tile visits (keys up to its last row's causal frontier) and whether the
// last KV tile runs past kv_length.
struct ItemShape {
  int rows_a, rows_b, nA, nB, n;
  bool tail_zero;
};
__device__ __forceinline__ ItemShape shape_of(const PrefillItem& it) {
  ItemShape sh;
  sh.rows_a = min(BM, it.n_rows);
  sh.rows_b = max(0, it.n_rows - BM);
  sh.nA = ceil_div(min(it.kv_length, it.s0 + it.i0 + sh.rows_a), BN);
  sh.nB = sh.rows_b > 0 ? ceil_div(min(it.kv_length, it.s0 + it.i0 + BM + sh.rows_b), BN) : 0;
  sh.n = max(sh.nA, sh.nB);
  sh.tail_zero = sh.n * BN > it.kv_length;
  return sh;
}

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
  uint8_t* skv = smem + L::kv_off;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::bar_off);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::misc_off + 4);

  // a kernel launched after this one with programmatic stream serialization
  // (the split-KV kernel of the same iteration) may start once every CTA of
  // this grid has been dispatched; it reads nothing this kernel writes
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&bars[B_Q_FULL], 1);
    mbar_init(&bars[B_Q_EMPTY], 1);
    for (int s = 0; s < L::kSlots; ++s) {
      mbar_init(&bars[B_KV_FULL + s], 1);
      mbar_init(&bars[B_KV_EMPTY + s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars[B_S_FULL + t], 1);
      mbar_init(&bars[B_P_FULL + t], 4);
      mbar_init(&bars[B_O_DONE + t], 1);
      mbar_init(&bars[B_O_FREE + t], 4);
      mbar_init(&bars[B_VZ_READY + t], 1);
    }
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

  // Phases are counted across all of the CTA's items: ring item g (K_j of an
  // item is its ring item 2j, V_j 2j + 1) lives in slot g % kSlots; the
  // Q buffer, the S/P/O barriers of each query tile and the V-tail barriers
  // advance once per use. The proofs that no waiter ever falls two phases
  // behind (which parity waits could not tell apart) are in the comments at
  // the waits.
  if (warp >= 8) {
    regs_dec<kProducerRegs>();
  }
  if (warp == 8) {
    // ------------------------------------------------------------ producer
    const int ps = 1 << p.ps_shift;
    const int npg = BN / ps;                    // pages per KV tile
    const int nbox = npg * L::kHalves;          // TMA boxes per K or V tile (<= 16)
    // lane l issues box (page l % npg, column block l / npg) of every tile
    const int my_pg = lane % npg, my_h2 = lane / npg;
    if (lane == 0) {
      prefetch_tensormap(&q_map);
      prefetch_tensormap(&k_map);
      prefetch_tensormap(&v_map);
    }
    int ri = 0;  // ring items issued (counted one by one: an abort drains exactly these)
    int nq = 0;  // Q loads issued
    int zc = 0;  // V tails zeroed
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int idx = item_of(k);
      if (idx >= p.n_items) break;
      const PrefillItem it = p.items[idx];
      const ItemShape sh = shape_of(it);
      // the Q buffer is free once every S MMA of the previous item has run
      if (nq > 0 && !(ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_Q_EMPTY], (uint32_t)(nq - 1) & 1u,
                                                           abort_flag, p.status))))
        break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars[B_Q_FULL], 2 * L::kTileBytes);
        for (int t = 0; t < 2; ++t)
          for (int h2 = 0; h2 < L::kHalves; ++h2)
            tma_load_3d(sq + t * L::kTileBytes + h2 * L::kHalfBytes, &q_map, &bars[B_Q_FULL],
                        h2 * 64, it.q_head, it.q_row0 + t * BM);
      }
      ++nq;
      const int32_t* btrow = p.block_table + (int64_t)it.req * p.max_blocks;
      const int last_block = (it.kv_length - 1) >> p.ps_shift;
      const int kv_head = it.q_head / p.group;
      int32_t my_y = 0;
      for (int i = 0; i < 2 * sh.n; ++i) {
        const int g = ri, slot = g % L::kSlots;
        const int j = i >> 1;
        if (g >= L::kSlots &&
            !(ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_KV_EMPTY + slot],
                                                     ((uint32_t)(g / L::kSlots) & 1u) ^ 1u,
                                                     abort_flag, p.status))))
          break;
        if ((i & 1) == 0 && lane < npg) {  // page of this lane for K_j and V_j
          int b = ((j * BN) >> p.ps_shift) + lane;
          if (b > last_block) b = last_block;  // keys past kv_length: masked, V zeroed
          int32_t page = __ldg(btrow + b);
          if ((unsigned)page >= (unsigned)p.num_pages) {
            set_status(p.status, MB_ERR_DEVICE_INDEX);
            page = 0;
          }
          my_y = (page * p.n_kv_heads + kv_head) << p.ps_shift;
        }
        const int32_t y = __shfl_sync(0xffffffffu, my_y, my_pg);
        if (lane == 0) mbar_arrive_expect_tx(&bars[B_KV_FULL + slot], L::kTileBytes);
        __syncwarp();
        if (lane < nbox)
          tma_load_2d(skv + slot * L::kTileBytes + my_h2 * L::kHalfBytes + my_pg * ps * 128,
                      (i & 1) ? &v_map : &k_map, &bars[B_KV_FULL + slot], my_h2 * 64, y);
        ++ri;
      }
      if (!ok) break;
      __syncwarp();
      if (sh.tail_zero) {
        // keys >= kv_length in the item's last V tile: zero their rows so that
        // a non-finite value in an unwritten slot cannot reach O through P = 0
        const int g = ri - 1, slot = g % L::kSlots;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_KV_FULL + slot],
                                                     (uint32_t)(g / L::kSlots) & 1u, abort_flag,
                                                     p.status))))
          break;
        const int r0 = it.kv_length - (sh.n - 1) * BN;
        const int nz = BN - r0;
        uint8_t* vb = skv + slot * L::kTileBytes;
        for (int e = lane; e < nz * L::kHalves * 8; e += 32) {
          const int c = e & 7;
          const int rr = e >> 3;
          const int h2 = rr / nz;
          const int row = r0 + (rr - h2 * nz);
          *reinterpret_cast<uint4*>(vb + h2 * L::kHalfBytes + row * 128 + c * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
        // two tail barriers in turn: the MMA thread may not have waited for
        // this item's predecessor yet, never for one further back (this item's
        // Q load needed the predecessor's S MMAs, issued after that wait)
        if (lane == 0) mbar_arrive(&bars[B_VZ_READY + (zc & 1)]);
        ++zc;
      }
    }
    __syncwarp();
    if (lane == 0) {
      // every copy still in flight must land before the CTA may exit
      if (nq > 0) mbar_drain(&bars[B_Q_FULL], (uint32_t)(nq - 1) & 1u, kDrainNs);
      for (int g = max(0, ri - L::kSlots); g < ri; ++g)
        mbar_drain(&bars[B_KV_FULL + g % L::kSlots], (uint32_t)(g / L::kSlots) & 1u, kDrainNs);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
      constexpr uint32_t idesc_qk = idesc_bf16_f32(BM, BN, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(BM, D, false, true);
      // Descriptor words (sdesc_sw128): every operand here shares the high
      // word (SBO 1024); the low words hold the tile's start address and LBO.
      // Each MMA then costs one integer add per operand: the issuing thread is
      // latency-bound (it shares its SM sub-partition with two softmax warps),
      // so every instruction between two MMAs shows up in the step time.
      const uint32_t d_hi = (uint32_t)(sdesc_sw128(0, 0, 1024) >> 32);
      const uint32_t q_lo = (uint32_t)sdesc_sw128(smem_u32(sq), 16, 1024);
      const uint32_t k_lo = (uint32_t)sdesc_sw128(smem_u32(skv), 16, 1024);
      const uint32_t v_lo = (uint32_t)sdesc_sw128(smem_u32(skv), L::kHalfBytes, 1024);
      constexpr uint32_t kTileW = L::kTileBytes >> 4;  // one tile in descriptor address units
      constexpr uint32_t kHalfW = L::kHalfBytes >> 4;
      auto issue_s = [&](int t, int kslot) {
        const uint32_t a0 = q_lo + t * kTileW;
        const uint32_t b0 = k_lo + kslot * kTileW;
        const uint32_t d = tmem + kColS + 128 * t;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          // K-major operands: 64-element block kk / 4, 32-byte step inside it
          const uint32_t o = (kk >> 2) * kHalfW + (kk & 3) * 2;
          umma_bf16_ss_w(d, a0 + o, b0 + o, d_hi, idesc_qk, (uint32_t)kk);
        }
        umma_commit(&bars[B_S_FULL + t]);
      };
      auto issue_pv = [&](int t, int vslot, bool first, bool last) {
        // A = P [128 rows x 128 keys] in TMEM over S_X: 16 keys = 8 columns;
        // B = V [128 keys x D], MN-major: 16 keys = two 8-row groups (SBO,
        // 2048 bytes), next 64 head dims one half further (LBO)
        const uint32_t b0 = v_lo + vslot * kTileW;
        const uint32_t a0 = tmem + kColS + 128 * t;
        const uint32_t d = tmem + kColO + 128 * t;
        const uint32_t acc = first ? 0u : 1u;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          umma_bf16_ts_w(d, a0 + kk * 8, b0 + kk * 128, d_hi, idesc_pv, acc | (uint32_t)kk);
        if (last) umma_commit(&bars[B_O_DONE + t]);  // the epilogue's signal, once per item
      };
      // Waits on what other threads wrote to TMEM (P, the released O) need the
      // tcgen05 fence; waits on TMA completions do not (copy and MMA are both
      // async-proxy accesses ordered by the mbarrier). The non-blocking probe
      // first: most of this thread's waits find the phase already complete.
      auto wait = [&](int b, uint32_t parity) -> bool {
        const bool ok =
            mbar_test(&bars[b], parity) || mbar_wait(&bars[b], parity, abort_flag, p.status);
        tc_fence_after();
        return ok;
      };
      auto wait_tma = [&](int b, uint32_t parity) -> bool {
        return mbar_test(&bars[b], parity) || mbar_wait(&bars[b], parity, abort_flag, p.status);
      };
      int ri = 0, nq = 0, zc = 0;
      int pc[2] = {0, 0};  // PV MMAs issued per query tile (= P tiles consumed)
      int oc[2] = {0, 0};  // items whose O each query tile accumulated
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int idx = item_of(k);
        if (idx >= p.n_items) break;
        const ItemShape sh = shape_of(p.items[idx]);
        if (!(ok = wait_tma(B_Q_FULL, (uint32_t)nq & 1u))) break;
        ++nq;
        const int g0 = ri;
        if (!(ok = wait_tma(B_KV_FULL + g0 % L::kSlots, (uint32_t)(g0 / L::kSlots) & 1u))) break;
        // S_X(0) overwrites the columns the previous item's last PV_X read P
        // from: it follows that PV in this thread's issue order
        if (sh.nA > 0) issue_s(0, g0 % L::kSlots);
        if (sh.nB > 0) issue_s(1, g0 % L::kSlots);
        if (sh.n == 1) umma_commit(&bars[B_Q_EMPTY]);  // every S MMA of the item issued
        umma_commit(&bars[B_KV_EMPTY + g0 % L::kSlots]);
        for (int j = 0; j < sh.n; ++j) {
          const int gv = g0 + 2 * j + 1, gk = gv + 1;
          const int vs = gv % L::kSlots, ks = gk % L::kSlots;
          if (!(ok = wait_tma(B_KV_FULL + vs, (uint32_t)(gv / L::kSlots) & 1u))) break;
          if (j == sh.n - 1 && sh.tail_zero &&
              !(ok = wait(B_VZ_READY + (zc & 1), (uint32_t)(zc >> 1) & 1u)))
            break;
          // the first PV of an item overwrites O_t: the softmax warps must have
          // read out the previous item's O_t (they release it once per item,
          // and each wait here consumes one release)
          if (j < sh.nA) {
            if (j == 0 && oc[0] > 0 && !(ok = wait(B_O_FREE + 0, (uint32_t)(oc[0] - 1) & 1u)))
              break;
            if (!(ok = wait(B_P_FULL + 0, (uint32_t)pc[0] & 1u))) break;
            issue_pv(0, vs, j == 0, j + 1 == sh.nA);
            ++pc[0];
          }
          if (j + 1 < sh.n && !(ok = wait_tma(B_KV_FULL + ks, (uint32_t)(gk / L::kSlots) & 1u))) break;
          if (j + 1 < sh.nA) issue_s(0, ks);  // after PV_A(j) in issue order
          if (j < sh.nB) {
            if (j == 0 && oc[1] > 0 && !(ok = wait(B_O_FREE + 1, (uint32_t)(oc[1] - 1) & 1u)))
              break;
            if (!(ok = wait(B_P_FULL + 1, (uint32_t)pc[1] & 1u))) break;
            issue_pv(1, vs, j == 0, j + 1 == sh.nB);
            ++pc[1];
          }
          umma_commit(&bars[B_KV_EMPTY + vs]);  // V_j free once both PVs finish
          if (j + 1 < sh.nB) issue_s(1, ks);    // after PV_B(j) in issue order
          if (j + 2 == sh.n) umma_commit(&bars[B_Q_EMPTY]);  // every S MMA of the item issued
          if (j + 1 < sh.n) umma_commit(&bars[B_KV_EMPTY + ks]);  // K_j+1 after its S MMAs
        }
        if (!ok) break;
        ri += 2 * sh.n;
        if (sh.tail_zero) ++zc;
        if (sh.nA > 0) ++oc[0];
        if (sh.nB > 0) ++oc[1];
      }
      // let the tensor core finish everything this thread issued before the
      // CTA frees TMEM and exits (also after an abort)
      umma_commit(&bars[B_MMA_DONE]);
      mbar_drain(&bars[B_MMA_DONE], 0, kDrainNs);
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax
    regs_inc<kSoftmaxRegs>();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
    const int t = warp >> 2;           // query tile: warps 0-3 -> A, 4-7 -> B
    const int sub = warp & 3;          // TMEM sub-partition this warp may access
    const int r = sub * 32 + lane;     // row within the tile
    const uint32_t lane_addr = (uint32_t)(sub * 32) << 16;
    const uint32_t s_col = tmem + lane_addr + kColS + 128 * t;
    const uint32_t o_col = tmem + lane_addr + kColO + 128 * t;
    const float c = p.scale_log2;
    int sc = 0;  // S tiles of this query tile consumed, all items
    int oi = 0;  // items whose O this tile finished (O_DONE / O_FREE phases)
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int idx = item_of(k);
      if (idx >= p.n_items) break;
      const PrefillItem it = p.items[idx];
      const ItemShape sh = shape_of(it);
      const int n_t = t ? sh.nB : sh.nA;
      if (n_t == 0) continue;
      const int rows_t = t ? sh.rows_b : sh.rows_a;
      const int first_vis = it.s0 + it.i0 + t * BM;  // last key visible to the tile's row 0
      const int vis_last = first_vis + r;            // ... to this row
      float m = -INFINITY, l = 0.f;  // running max (raw score units), running sum
      for (int j = 0; j < n_t; ++j) {
        // S_t(j) complete implies PV_t(j-1) complete (issued before it by the
        // same thread), so O_t and the P columns are free to touch
        ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_S_FULL + t], (uint32_t)sc & 1u, abort_flag,
                                               p.status));
        if (!ok) break;
        ++sc;
        tc_fence_after();
        uint32_t s[128];
        tmem_ld128(s_col, s);
        tmem_ld_wait128(s);

        const int key0 = j * BN;
        if (key0 + BN - 1 > first_vis) {  // tile straddles the causal frontier
          const int lim = vis_last - key0;
#pragma unroll
          for (int e = 0; e < 128; ++e)
            if (e > lim) s[e] = __float_as_uint(-INFINITY);
        }
        // row max: three-input max over 128 scores, 8 independent chains
        float mx[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
          mx[q] = fmax3(__uint_as_float(s[q]), __uint_as_float(s[q + 8]), __uint_as_float(s[q + 16]));
#pragma unroll
        for (int e = 24; e < 120; e += 16)
#pragma unroll
          for (int q = 0; q < 8; ++q)
            mx[q] = fmax3(mx[q], __uint_as_float(s[e + q]), __uint_as_float(s[e + 8 + q]));
#pragma unroll
        for (int q = 0; q < 8; ++q) mx[q] = fmaxf(mx[q], __uint_as_float(s[120 + q]));
        const float tmax =
            fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
        const float m_new = fmaxf(m, tmax);
        // lazy rescale: keep the old max unless it grew by more than 2^8
        float alpha = 1.f;
        bool need = false;
        if (j == 0) {
          m = m_new;
        } else {
          need = (m_new - m) * c > kRescaleThreshold;
          if (need) {
            alpha = fast_exp2((m - m_new) * c);
            l *= alpha;
            m = m_new;
          }
        }
        const float mc = (m == -INFINITY) ? 0.f : m * c;
        // p = 2^(s * c - m * c): the scale-and-shift of two scores in one
        // packed FMA, the row sum in two packed accumulators
        const uint64_t c2 = f32x2(c, c), nmc2 = f32x2(-mc, -mc);
        uint64_t acc[2] = {0ull, 0ull};
        uint32_t pk[64];
#pragma unroll
        for (int e = 0; e < 128; e += 2) {
          float x0, x1;
          f32x2_split(ffma_x2(f32x2(__uint_as_float(s[e]), __uint_as_float(s[e + 1])), c2, nmc2),
                      x0, x1);
          const float e0 = fast_exp2(x0);
          const float e1 = fast_exp2(x1);
          acc[(e >> 1) & 1] = fadd_x2(acc[(e >> 1) & 1], f32x2(e0, e1));
          pk[e >> 1] = pack_bf16x2(e0, e1);
        }
        float sum_lo, sum_hi;
        f32x2_split(fadd_x2(acc[0], acc[1]), sum_lo, sum_hi);
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
        // P (bf16 pairs) over the first 64 columns of the row's scores
        tmem_st32(s_col, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
        tmem_st32(s_col + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
        tmem_st_wait();
        l += sum_lo + sum_hi;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[B_P_FULL + t]);
      }
      if (!ok) break;
      // the item's last PV (the MMA thread issues no further PV_t before this
      // tile releases O_t below, so O_DONE is at most one phase behind)
      ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_O_DONE + t], (uint32_t)oi & 1u,
                                             abort_flag, p.status));
      if (!ok) break;
      tc_fence_after();
      // read O_t out of TMEM, release it to the next item's PV, then finish
      // the rows from registers while the tensor core moves on
      // (every load's registers pass through its wait, so no use of them can
      // be scheduled before the data lands)
      uint32_t o[D];
      if constexpr (D == 128) {
        tmem_ld128(o_col, *reinterpret_cast<uint32_t(*)[128]>(&o[0]));
        tmem_ld_wait128(*reinterpret_cast<uint32_t(*)[128]>(&o[0]));
      } else {
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          tmem_ld32(o_col + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&o[cc * 32]));
          tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&o[cc * 32]));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_O_FREE + t]);
      ++oi;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      if (r < rows_t) {
        const int64_t orow = (int64_t)(it.q_row0 + t * BM + r) * p.n_q_heads + it.q_head;
        uint4* dst = reinterpret_cast<uint4*>(p.out + orow * D);
#pragma unroll
        for (int q4 = 0; q4 < D / 8; ++q4) {
          uint4 v;
          v.x = pack_bf16x2(__uint_as_float(o[q4 * 8 + 0]) * inv, __uint_as_float(o[q4 * 8 + 1]) * inv);
          v.y = pack_bf16x2(__uint_as_float(o[q4 * 8 + 2]) * inv, __uint_as_float(o[q4 * 8 + 3]) * inv);
          v.z = pack_bf16x2(__uint_as_float(o[q4 * 8 + 4]) * inv, __uint_as_float(o[q4 * 8 + 5]) * inv);
          v.w = pack_bf16x2(__uint_as_float(o[q4 * 8 + 6]) * inv, __uint_as_float(o[q4 * 8 + 7]) * inv);
          dst[q4] = v;
        }
        if (p.lse) p.lse[orow] = (m * c + log2f(l)) * kLn2;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(*reinterpret_cast<volatile uint32_t*>(tmem_slot), kTmemCols);
  }
}

template <int D>
cudaError_t launch_d(const PrefillArgs& a, cudaStream_t s) {
  Params p;
  p.items = a.items;
  p.n_items = a.n_items;
  p.block_table = a.block_table;
  p.max_blocks = a.max_blocks;
  p.n_q_heads = a.n_q_heads;
  p.n_kv_heads = a.n_kv_heads;
  p.num_pages = a.num_pages;
  p.group = a.n_q_heads / a.n_kv_heads;
  p.ps_shift = __builtin_ctz((unsigned)a.page_size);
  p.scale_log2 = a.scale_log2;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.lse = a.lse;
  p.status = a.status;
  constexpr uint32_t smem = Layout<D>::kAlloc;
  // once per device: the register split assumes the kernel launches with
  // kLaunchRegs per thread (with fewer, a warpgroup's increase could never be
  // satisfied); the dynamic shared memory; the SM count
  static OncePerDevice setup;
  static std::atomic<int> sm_count[64];
  cudaError_t e = setup.run([](int dev) -> cudaError_t {
    cudaFuncAttributes fa;
    cudaError_t r = cudaFuncGetAttributes(&fa, prefill_kernel<D>);
    if (r != cudaSuccess) return r;
    if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
    r = cudaFuncSetAttribute(prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (r != cudaSuccess) return r;
    int n = 0;
    r = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (r == cudaSuccess && dev < 64) sm_count[dev].store(n);
    return r;
  });
  if (e != cudaSuccess) return e;
  // persistent grid: one CTA per SM (the kernel holds an SM's whole TMEM),
  // each walking its share of the item list
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64) sms = sm_count[dev].load();
  if (sms == 0) {
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
  }
  if (a.max_ctas > 0 && a.max_ctas < sms) sms = a.max_ctas;
  const int grid = a.n_items < sms ? a.n_items : sms;
  prefill_kernel<D><<<grid, kThreads, smem, s>>>(p, *a.q_map, *a.k_map, *a.v_map);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t s) {
  if (a.n_items <= 0) return cudaSuccess;
  return a.head_dim == 128 ? launch_d<128>(a, s) : launch_d<64>(a, s);
}

}  // namespace mb
