// The fused projection: the base projection and the delta in one accumulator.
//
//   y[t][c] = sum_j x[t][j] * W[c][j]  +  sum_l [c in lane l] scale[k][l] * (B[k][l] @ (A[k][l] @ x[t]))[c - off_l]
//
// with k = slot[t] (no delta for slot 0).  The delta is added to the fp32
// partial sum of the projection (TensorFold PR #47, the paragraph on the
// delta), and the base's own output carries it, so the delta costs no pass of
// its own over y (xLLM PR #2014, New subsystems, the LoRARowParallelLinear
// item's fused mode).  y is written once; it is never read.
//
// Before this kernel the two shrinks run in their row mode and leave
// u'[t][l] = scale[k][l] * (A[k][l] @ x[t]) in fp32 for every row with an
// adapter.  This kernel is then a tcgen05 GEMM over tiles of 128 rows x 256
// columns of y in row order:
//   1. K loop over d_in: TMA brings a 128 x 64 tile of x and a 256 x 64 tile of
//      W (128-byte swizzle) per stage; one thread issues
//      tcgen05.mma.kind::f16 (M = 128, N = 256, K = 16) into a 256-column fp32
//      accumulator in tensor memory.  On batches of long prompts the CTAs work
//      in pairs (a cluster of two) on 256 x 256 tiles with tcgen05's pair MMA
//      (cta_group::2, M = 256): each CTA loads its own 128 rows of x and 128
//      of the tile's 256 W rows, so each SM moves a third fewer bytes through
//      shared memory per flop and six 32 KB stages replace four of 48 KB.
//   2. Expand steps, into the same accumulator: for every slot present among
//      the tile's rows, every lane of that slot the tile's columns touch, and
//      every pair of 16-rank groups of its rank, an MMA of M = 128 rows and
//      N = the lane's columns in the tile: A = that slot's rows of u' (rows of
//      other slots are zero), split into bf16 hi = bf16(u') and
//      lo = bf16(u' - hi), both multiplied by the (exact) bf16 B.  The rows of
//      u' are gathered and split by four warps into the stage, in the MMA's
//      K-major core-matrix layout; B comes from the pool's K-major groups by TMA.
//   3. Epilogue: the four warps read the accumulator (tcgen05.ld, one row per
//      thread) and store the tile's rows of y.
// A row's bits depend only on its own x row, W and its own u': every output
// element sums its own products in an order fixed by d_in and its slot's
// rank, and the expand steps of other slots add exact zeros to it.
//
// Warp roles: warp 0 lane 0 issues TMA, warp 1 lane 0 issues MMAs, warps 2-5
// find the tile's slots, build the u' operands and write y.  Every mbarrier
// wait is bounded; a wait that gives up records LORA_ERR_TIMEOUT in the status
// word, the CTA writes nothing and unwinds.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>
#include <vector>

#include "device.cuh"
#include "internal.h"

namespace lora {
namespace {

constexpr int kFpM = 128;                                     // tile rows per CTA (MMA M per CTA)
constexpr int kFpN = 256;                                     // tile columns (MMA N)
constexpr int kFpK = 64;                                      // d_in per stage: one 128-byte swizzle row
constexpr int kFpXBytes = kFpM * kFpK * 2;                    // 16 KB
constexpr int kFpUGroupBytes = kFpM * 32;                     // u' of 128 rows x 16 ranks
constexpr int kFpThreads = 320;                               // TMA, MMA, 4 operand warps, 4 epilogue warps
constexpr int kFpBandTiles = 16;                              // row tiles per band of the tile order
constexpr int kFpSlotWords = LORA_MAX_SLOTS / 32;
constexpr int kFpMaxStages = 6;
constexpr int kFpMaxUBufs = 2;
// Batches of long prompts (at least this many rows per sequence on average)
// run in CTA pairs; the others, whose tiles hold more slots, in single CTAs,
// whose expand steps are cheaper (a pair's steps follow the slots of both of
// its tiles and wait on both CTAs' operand builders).  Both forms give every
// row the same bits.
constexpr int kFpPairMinRowsPerSeq = 256;

// The two forms of the kernel: one CTA per 128 x 256 tile (kCta = 1), or a
// CTA pair per 256 x 256 tile with tcgen05's pair MMA (kCta = 2): each CTA
// then holds its own 128 rows of x and 128 of the tile's 256 W rows, so a
// stage is 32 KB instead of 48 and six fit where four did, and the tensor
// cores read a third less from each SM's shared memory per flop.
template <int kCta>
struct FpShape {
  static constexpr int kWRows = kFpN / kCta;                   // W rows (tile columns) per CTA and stage
  static constexpr int kStageBytes = kFpXBytes + kWRows * kFpK * 2;
  static constexpr int kStages = kCta == 2 ? 6 : 4;
  // 16-rank groups per expand step: the same in both forms, so that a row's
  // expand MMAs add in the same order whichever form runs its tile
  static constexpr int kGroups = 2;
  static constexpr int kUBufs = 2;                             // u' operand buffers (hi then lo halves)
  static constexpr int kUBufBytes = 2 * kGroups * kFpUGroupBytes;
  static constexpr int kBkCols = kFpN / kCta;                  // B columns of an expand group per CTA
  static constexpr int kBkGroupBytes = kBkCols * 32;
  static constexpr int kAccBufs = 2;                           // TMEM accumulators of 256 columns
  static constexpr int kSmem = kStages * kStageBytes + kUBufs * kUBufBytes + 1024;
};
static_assert(FpShape<1>::kSmem == FpShape<2>::kSmem, "both forms take the same shared memory");
static_assert(FpShape<2>::kStages <= kFpMaxStages && FpShape<2>::kUBufs <= kFpMaxUBufs, "barrier arrays");
static_assert(FpShape<1>::kGroups * FpShape<1>::kBkGroupBytes <= FpShape<1>::kStageBytes, "a step's B fits a stage");
static_assert(FpShape<2>::kGroups * FpShape<2>::kBkGroupBytes <= FpShape<2>::kStageBytes, "a step's B fits a stage");

struct FpParams {
  const int32_t* slot;  // [T] per-token slot (segment builder)
  const int32_t* rank_tab;
  const float* u_rows;  // [T][L][R16] scale * u
  float* y;
  int32_t* status;
  int64_t ldy;
  int T, D, nkb, L, R16, N, ntm, ntn;
  int ntg, nunits;  // row groups (kCta row tiles each), units = row groups x column tiles
  int d_out[LORA_MAX_LANES], off[LORA_MAX_LANES];
};

// The expand steps of a unit, in a fixed order (slot list order, lane,
// group), handed to f(k, l, q0, ng, c_lo, c_w, lc0): slot k, lane l, first
// 16-rank group q0 and group count ng, tile columns [c_lo, c_lo + c_w) =
// lane columns [lc0, lc0 + c_w).  f returns false to stop.  Every role (of
// both CTAs of a pair) runs its own walk over the same list and tables, so
// all agree.
template <int kGroups, typename F>
__device__ __forceinline__ bool for_each_step(const FpParams& p, const uint16_t* slots, int nslots, int n0, F&& f) {
  for (int j = 0; j < nslots; ++j) {
    const int k = slots[j];
#pragma unroll
    for (int l = 0; l < LORA_MAX_LANES; ++l) {
      if (l >= p.L) continue;
      const int lo = max(n0, p.off[l]), hi = min(n0 + kFpN, p.off[l] + p.d_out[l]);
      if (lo >= hi) continue;
      const int r = p.rank_tab[k * p.L + l];
      if (r <= 0) continue;
      const int nk = (r + 15) / 16;
      for (int q0 = 0; q0 < nk; q0 += kGroups)
        if (!f(k, l, q0, min(kGroups, nk - q0), lo - n0, hi - lo, lo - p.off[l])) return false;
    }
  }
  return true;
}

// Unit u of the order: bands of kFpBandTiles row tiles, column tiles in order
// inside a band (CTAs working at the same time share W and x tiles in L2).  A
// unit is kCta row tiles from row mp on, by one column tile from n0.
template <int kCta>
__device__ __forceinline__ void unit_origin(const FpParams& p, int u, int& mp, int& n0) {
  constexpr int band_groups = kFpBandTiles / kCta;
  const int band_size = band_groups * p.ntn;
  const int band = u / band_size, in_band = u - band * band_size;
  const int groups_in_band = min(band_groups, p.ntg - band * band_groups);
  mp = (band * band_groups + in_band % groups_in_band) * kCta * kFpM;
  n0 = (in_band / groups_in_band) * kFpN;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Persistent: CTA (or pair) b takes units b, b + G, b + 2G, ... (G = the
// number of CTAs or pairs).  Two accumulators of 256 TMEM columns alternate
// between units, so the epilogue of one unit runs while the next one's K loop
// does.  A pair: CTA 0's thread issues every MMA, each CTA's producer loads
// its own halves and counts them on CTA 0's full barrier, every commit arrives
// in both CTAs, and both CTAs' operand builders and epilogue warps arrive on
// CTA 0's barriers.  The expand steps of a pair follow one slot list made from
// the rows of both tiles (a slot held by one tile only adds zeros to the
// other's rows).  Every barrier a role waits on is waited on phase by phase,
// in order, by that role.
template <int kCta>
__global__ void __launch_bounds__(kFpThreads, 1)
    fused_proj_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                      const __grid_constant__ TmapSized tm_bk, FpParams p) {
  using S = FpShape<kCta>;
  constexpr bool kPair = kCta == 2;
  constexpr int kStages = S::kStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kFpMaxStages], empty_bar[kFpMaxStages];
  __shared__ __align__(8) uint64_t ufull_bar[kFpMaxUBufs], uempty_bar[kFpMaxUBufs];
  __shared__ __align__(8) uint64_t plan_full[2], plan_empty[2], acc_full[2], acc_empty[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int fail_sh;
  __shared__ int bad_sh[2];   // a pair: the status word as each CTA read it
  __shared__ int nslots_sh[2];
  __shared__ int stop_sh[2];  // per plan buffer: a warp of warps 2-5 saw a failure (they stop together)
  __shared__ uint16_t slots_sh[2][kCta * kFpM];
  __shared__ uint32_t bits_sh[kFpSlotWords];

  pdl_wait();  // the shrinks' u' (and the builder's slots) are visible from here on
  const int rank = kPair ? (int)cluster_ctarank() : 0;
  // A routing error or an earlier timeout: y is not written.  Both CTAs of a
  // pair take the same decision, from the two readings they exchange below.
  if (!kPair && *p.status != 0) return;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ubuf = smem + kStages * S::kStageBytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int q = 0; q < S::kUBufs; ++q) {
      mbar_init(&ufull_bar[q], 4 * kCta);
      mbar_init(&uempty_bar[q], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&plan_full[b], 1);
      mbar_init(&plan_empty[b], rank == 0 ? 2 : 1);  // the producer and (in CTA 0) the MMA thread
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4 * kCta);
    }
    fail_sh = 0;
    stop_sh[0] = stop_sh[1] = 0;
    fence_mbar_init();
  }
  if (kPair) {
    // Both CTAs run and their barriers exist before either touches the
    // other's shared memory; then each sends its reading of the status word.
    cluster_sync_all();
    if (threadIdx.x == 0) {
      const int bad = *p.status != 0 ? 1 : 0;
      bad_sh[rank] = bad;
      st_dsmem_u32(mapa_shared(smem_u32(&bad_sh[rank]), (uint32_t)(rank ^ 1)), (uint32_t)bad);
    }
    cluster_sync_all();
    if (bad_sh[0] | bad_sh[1]) return;
  }
  if (warp == 0) {
    if constexpr (kPair) {
      tmem_alloc_pair(&tmem_base_sh, S::kAccBufs * kFpN);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&tmem_base_sh, S::kAccBufs * kFpN);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if (kPair)
    cluster_sync_all();  // both CTAs' accumulators exist before CTA 0's first MMA
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const int u_first = kPair ? (int)cluster_id_x() : (int)blockIdx.x;
  const int u_step = kPair ? (int)num_clusters_x() : (int)gridDim.x;
  // CTA 0's barriers as the pair's other CTA addresses them
  auto lead = [&](uint64_t* bar) -> uint32_t { return mapa_shared(smem_u32(bar), 0u); };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (in each CTA: its own rows and halves)
      uint32_t i = 0;
      bool ok = true;
      auto take = [&](uint32_t bytes) -> uint8_t* {
        const int s = (int)(i % kStages);
        if (i >= kStages && !mbar_wait_or_fail(&empty_bar[s], ((i / kStages) - 1) & 1, &fail_sh)) {
          fail_sh = 1;
          ok = false;
          return nullptr;
        }
        if (rank == 0) mbar_expect_tx(&full_bar[s], bytes * kCta);  // the pair's bytes land on CTA 0's count
        return smem + (size_t)s * S::kStageBytes;
      };
      int jj = 0;
      for (int u = u_first; u < p.nunits && ok; u += u_step, ++jj) {
        int mp, n0;
        unit_origin<kCta>(p, u, mp, n0);
        for (int kb = 0; kb < p.nkb && ok; ++kb) {
          uint8_t* st = take((uint32_t)S::kStageBytes);
          if (!st) break;
          uint64_t* fb = &full_bar[i % kStages];
          if constexpr (kPair) {
            const uint32_t lb = lead(fb);
            tma_load_2d_pair(st, &tm_x, kb * kFpK, mp + rank * kFpM, lb);
            tma_load_2d_pair(st + kFpXBytes, &tm_w, kb * kFpK, n0 + rank * S::kWRows, lb);
          } else {
            tma_load_2d(st, &tm_x, kb * kFpK, mp, fb);
            tma_load_2d(st + kFpXBytes, &tm_w, kb * kFpK, n0, fb);
          }
          ++i;
        }
        const int b = jj & 1;
        if (ok && !mbar_wait_or_fail(&plan_full[b], (jj >> 1) & 1, &fail_sh)) {
          fail_sh = 1;
          ok = false;
        }
        if (!ok) break;
        for_each_step<S::kGroups>(p, slots_sh[b], nslots_sh[b], n0, [&](int k, int l, int q0, int ng, int, int c_w, int lc0) {
          // a pair: this CTA's half of the columns, one box of 128; one CTA:
          // boxes of 128 columns per group
          const int nb = kPair ? 1 : (c_w + 127) / 128;
          uint8_t* st = take((uint32_t)(ng * nb * 4096));
          if (!st) return false;
          uint64_t* fb = &full_bar[i % kStages];
          for (int g = 0; g < ng; ++g)
            for (int h = 0; h < nb; ++h) {
              uint8_t* dst = st + g * S::kBkGroupBytes + h * 4096;
              const int c1 = lc0 + (kPair ? rank * (c_w / 2) : 128 * h), c2 = k * (p.R16 / 16) + q0 + g;
              if constexpr (kPair)
                tma_load_3d_pair(dst, &tm_bk.m[0][l], 0, c1, c2, lead(fb));
              else
                tma_load_3d(dst, &tm_bk.m[0][l], 0, c1, c2, fb);
            }
          ++i;
          return true;
        });
        if (ok) mbar_arrive(&plan_empty[b]);
      }
      if (!kPair || !ok || fail_sh) {
        // Copies already issued land before the CTA may leave (after a
        // failure the MMA thread may not have waited for them).  A pair's
        // copies are counted on CTA 0: there each latest fill of a stage is
        // waited for; in CTA 1 the bounded delay at the end covers them.
        if (rank == 0)
          for (uint32_t f = i > (uint32_t)kStages ? i - kStages : 0; f < i; ++f)
            if (!mbar_wait_bounded(&full_bar[f % kStages], (f / kStages) & 1)) fail_sh = 1;
      } else {
        // The MMAs are done with the latest fill of every stage: every copy
        // into this CTA has landed and every commit to its empty barriers
        // has arrived.
        for (uint32_t f = i > (uint32_t)kStages ? i - kStages : 0; f < i; ++f)
          if (!mbar_wait_bounded(&empty_bar[f % kStages], (f / kStages) & 1)) fail_sh = 1;
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------- MMA issuer (CTA 0 of a pair issues for both)
      uint32_t i = 0, n = 0;  // ring stage uses, u' buffer uses
      bool ok = true;
      const uint32_t idesc_main = idesc_bf16(kFpM * kCta, kFpN);
      auto mma = [&](uint32_t d, uint64_t a, uint64_t bdesc, uint32_t idesc, uint32_t acc_in) {
        if constexpr (kPair)
          mma_bf16_pair(d, a, bdesc, idesc, acc_in);
        else
          mma_bf16(d, a, bdesc, idesc, acc_in);
      };
      auto commit = [&](uint64_t* bar) {
        if constexpr (kPair)
          mma_commit_pair(bar, (uint16_t)3);
        else
          mma_commit(bar);
      };
      auto wait_peer_arrivals = [&](uint64_t* bar, uint32_t parity) {  // barriers the other CTA arrives on
        return kPair ? mbar_wait_cluster_or_fail(bar, parity, &fail_sh) : mbar_wait_or_fail(bar, parity, &fail_sh);
      };
      int jj = 0;
      for (int u = u_first; u < p.nunits && ok; u += u_step, ++jj) {
        int mp, n0;
        unit_origin<kCta>(p, u, mp, n0);
        const int b = jj & 1;
        const int ab = jj % S::kAccBufs, au = jj / S::kAccBufs;  // accumulator and its use count
        const uint32_t acc = tmem + (uint32_t)(ab * kFpN);
        if (au >= 1 && !wait_peer_arrivals(&acc_empty[ab], (au - 1) & 1)) {
          fail_sh = 1;
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < p.nkb; ++kb, ++i) {
          const int s = (int)(i % kStages);
          if (!mbar_wait_or_fail(&full_bar[s], (i / kStages) & 1, &fail_sh)) {
            fail_sh = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t xa = smem_u32(smem + (size_t)s * S::kStageBytes), wa = xa + kFpXBytes;
#pragma unroll
          for (int kk = 0; kk < kFpK / 16; ++kk)
            mma(acc, smem_desc(xa + 32 * kk, 16, 1024, kSwz128), smem_desc(wa + 32 * kk, 16, 1024, kSwz128),
                idesc_main, (kb | kk) != 0 ? 1u : 0u);
          commit(&empty_bar[s]);
        }
        if (ok && !mbar_wait_or_fail(&plan_full[b], (jj >> 1) & 1, &fail_sh)) {
          fail_sh = 1;
          ok = false;
        }
        if (!ok) break;
        ok = for_each_step<S::kGroups>(p, slots_sh[b], nslots_sh[b], n0, [&](int, int, int, int ng, int c_lo, int c_w, int) {
          const int s = (int)(i % kStages), q = (int)(n % S::kUBufs);
          if (!mbar_wait_or_fail(&full_bar[s], (i / kStages) & 1, &fail_sh) ||
              !wait_peer_arrivals(&ufull_bar[q], (n / S::kUBufs) & 1)) {
            fail_sh = 1;
            return false;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + (size_t)s * S::kStageBytes);
          const uint32_t ua = smem_u32(ubuf + (size_t)q * S::kUBufBytes);
          const uint32_t idesc = idesc_bf16(kFpM * kCta, c_w);
          for (int half = 0; half < 2; ++half)
            for (int g = 0; g < ng; ++g)
              mma(acc + (uint32_t)c_lo, smem_desc(ua + (half * S::kGroups + g) * kFpUGroupBytes, 128, 256, kSwzNone),
                  smem_desc(sa + g * S::kBkGroupBytes, 16, 256, kSwz32), idesc, 1u);
          commit(&empty_bar[s]);
          commit(&uempty_bar[q]);
          ++i;
          ++n;
          return true;
        });
        if (!ok) break;
        commit(&acc_full[ab]);
        mbar_arrive(&plan_empty[b]);
      }
    }
  } else if (warp < 6) {
    // ---------------- warps 2-5: each unit's slots, then the u' operands of
    // its expand steps: row m of this CTA's tile, zero for rows of other
    // slots, as bf16 hi and lo in the K-major core-matrix layout (8 rows x 16
    // bytes per core matrix; 16 ranks = two of them)
    const int m = (warp & 3) * 32 + lane;
    const int bt = threadIdx.x - 64;  // 0..127
    const uint32_t row_off = (uint32_t)((m >> 3) * 256 + (m & 7) * 16);
    // These four warps meet at named barriers, so they leave the unit loop
    // together: a failure any of them sees goes into stop_sh[b] between the
    // first and the third barrier of a unit, and all read it after the third.
    uint32_t n = 0;
    bool ok = true;
    int jj = 0;
    for (int u = u_first; u < p.nunits; u += u_step, ++jj) {
      int mp, n0;
      unit_origin<kCta>(p, u, mp, n0);
      const int b = jj & 1;
      const int tr = mp + rank * kFpM + m;
      const int myslot = tr < p.T ? p.slot[tr] : 0;
      if (ok && jj >= 2) {  // the plan buffer is free once the producer and the MMA thread are done with it
        int got = 1;
        if (lane == 0) got = mbar_wait_or_fail(&plan_empty[b], ((jj >> 1) - 1) & 1, &fail_sh) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, got, 0)) {
          fail_sh = 1;
          ok = false;
        }
      }
      if (bt == 0) stop_sh[b] = 0;  // every warp read it two units ago, before the barriers of the last unit
      for (int w = bt; w < kFpSlotWords; w += 128) bits_sh[w] = 0u;
      named_bar_sync(1, 128);
      if (lane == 0 && (!ok || fail_sh)) atomicOr(&stop_sh[b], 1);
#pragma unroll
      for (int h = 0; h < kCta; ++h) {  // the slots of every row tile of the unit
        const int rr = mp + h * kFpM + m;
        const int sl = h == rank ? myslot : rr < p.T ? p.slot[rr] : 0;
        if (sl > 0) atomicOr(&bits_sh[sl >> 5], 1u << (sl & 31));
      }
      named_bar_sync(1, 128);
      if (warp == 2) {
        // distinct slots of the unit in ascending order
        const int nw = (p.N + 31) / 32;
        uint32_t w0 = 2 * lane < nw ? bits_sh[2 * lane] : 0u, w1 = 2 * lane + 1 < nw ? bits_sh[2 * lane + 1] : 0u;
        const int c = __popc(w0) + __popc(w1);
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += v;
        }
        int pos = incl - c;
        while (w0) {
          slots_sh[b][pos++] = (uint16_t)(64 * lane + __ffs(w0) - 1);
          w0 &= w0 - 1;
        }
        while (w1) {
          slots_sh[b][pos++] = (uint16_t)(64 * lane + 32 + __ffs(w1) - 1);
          w1 &= w1 - 1;
        }
        if (lane == 31) nslots_sh[b] = incl;
      }
      named_bar_sync(1, 128);
      if (stop_sh[b]) break;
      if (warp == 2 && lane == 0) mbar_arrive(&plan_full[b]);
      ok = for_each_step<S::kGroups>(p, slots_sh[b], nslots_sh[b], n0, [&](int k, int l, int q0, int ng, int, int, int) {
        const int q = (int)(n % S::kUBufs);
        const bool mine = myslot == k;
        // this row's u' first, so the loads are in flight during the wait
        const float4* src =
            reinterpret_cast<const float4*>(p.u_rows + ((size_t)(mine ? tr : 0) * p.L + l) * p.R16 + 16 * q0);
        float4 v[4 * S::kGroups];
#pragma unroll
        for (int g = 0; g < S::kGroups; ++g)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            v[4 * g + e] = mine && g < ng ? __ldcg(src + 4 * g + e) : make_float4(0.f, 0.f, 0.f, 0.f);
        if (n >= S::kUBufs) {  // one lane waits for the buffer to be free; the warp follows it
          int got = 1;
          if (lane == 0) got = mbar_wait_or_fail(&uempty_bar[q], ((n / S::kUBufs) - 1) & 1, &fail_sh) ? 1 : 0;
          if (!__shfl_sync(0xffffffffu, got, 0)) {
            fail_sh = 1;
            return false;
          }
        }
        uint8_t* ub = ubuf + (size_t)q * S::kUBufBytes;
#pragma unroll
        for (int g = 0; g < S::kGroups; ++g) {
          if (g >= ng) break;
#pragma unroll
          for (int kc = 0; kc < 2; ++kc) {
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float4 f4 = v[4 * g + 2 * kc + (e >> 1)];
              const float u0 = (e & 1) ? f4.z : f4.x, u1 = (e & 1) ? f4.w : f4.y;
              const __nv_bfloat16 h0 = __float2bfloat16_rn(u0), h1 = __float2bfloat16_rn(u1);
              const __nv_bfloat16 l0 = __float2bfloat16_rn(u0 - __bfloat162float(h0));
              const __nv_bfloat16 l1 = __float2bfloat16_rn(u1 - __bfloat162float(h1));
              hw[e] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
              lw[e] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
            }
            const uint32_t o = (uint32_t)(g * kFpUGroupBytes + kc * 128) + row_off;
            *reinterpret_cast<uint4*>(ub + o) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4*>(ub + S::kGroups * kFpUGroupBytes + o) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          }
        }
        fence_proxy_async_smem();  // the MMA reads these through the async proxy
        __syncwarp();
        if (lane == 0) {
          if (rank == 0)
            mbar_arrive(&ufull_bar[q]);
          else
            mbar_arrive_cluster(lead(&ufull_bar[q]));
        }
        ++n;
        return true;
      });
    }
  } else {
    // ---------------- warps 6-9: epilogue, one tile row per thread, 32
    // columns at a time; the accumulator goes back to the MMA thread after
    const int quad = warp & 3;
    const int m = quad * 32 + lane;
    const uint32_t trow = (uint32_t)(quad * 32) << 16;
    int jj = 0;
    for (int u = u_first; u < p.nunits; u += u_step, ++jj) {
      int mp, n0;
      unit_origin<kCta>(p, u, mp, n0);
      const int ab = jj % S::kAccBufs, au = jj / S::kAccBufs;
      int got = 1;  // uniform over the warp: the tcgen05.ld below is warp-collective
      if (lane == 0) got = mbar_wait_or_fail(&acc_full[ab], au & 1, &fail_sh) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, got, 0)) {
        fail_sh = 1;
        break;
      }
      tc_fence_after();
      const int tr = mp + rank * kFpM + m;
      float* yr = p.y + (size_t)tr * p.ldy + n0;
#pragma unroll 1
      for (int j = 0; j < kFpN / 32; ++j) {
        float v[32];
        tmem_ld32(tmem + trow + (uint32_t)(ab * kFpN + 32 * j), v);
        if (tr < p.T && n0 + 32 * j < p.D) {
          float4* dst = reinterpret_cast<float4*>(yr + 32 * j);
#pragma unroll
          for (int e = 0; e < 8; ++e) dst[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0)
          mbar_arrive(&acc_empty[ab]);
        else
          mbar_arrive_cluster(lead(&acc_empty[ab]));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (kPair) {
    // Neither CTA of the pair leaves while the other may still send it
    // copies, commits or arrivals.  After a failure some may still be on
    // their way (nothing here counts them): give them 100 microseconds.
    cluster_sync_all();
    if (fail_sh) {
      const unsigned long long t0 = globaltimer();
      while (globaltimer() - t0 < 100000ull) {
      }
    }
  }
  if (warp == 0) {
    tc_fence_after();
    if constexpr (kPair)
      tmem_dealloc_pair(tmem, S::kAccBufs * kFpN);
    else
      tmem_dealloc(tmem, S::kAccBufs * kFpN);
  }
  if (threadIdx.x == 0 && fail_sh) set_error(p.status, LORA_ERR_TIMEOUT);
}

// Pairs of the fused kernel that fit on the device at once.
int fp_max_pairs(int device) {
  struct Entry {
    int device, n;
  };
  static std::mutex mu;
  static std::vector<Entry> cache;
  std::lock_guard<std::mutex> lock(mu);
  for (const Entry& e : cache)
    if (e.device == device) return e.n;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * 64);
  cfg.blockDim = dim3(kFpThreads);
  cfg.dynamicSmemBytes = FpShape<2>::kSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(fused_proj_kernel<2>), &cfg) != cudaSuccess ||
      n <= 0) {
    cudaGetLastError();  // the query failed: clear its error and assume one pair per two SMs
    n = sm_count(device) / 2;
  }
  cache.push_back({device, n});
  return n;
}

}  // namespace

int launch_fused_projection(const PoolView& pool, const lora_segments* seg, const uint16_t* W, int64_t ldw,
                            const uint16_t* x, int64_t ldx, float* y, int64_t ldy, cudaStream_t st) {
  const int T = seg->T;
  if (T <= 0) return LORA_OK;
  const int ntm = ceil_div(T, kFpM);
  // A CTA pair per 256 rows for batches of long prompts with two row tiles
  // to pair (one row tile would leave every second CTA without rows).
  const int cta = ntm >= 2 && (long long)T >= (long long)kFpPairMinRowsPerSeq * seg->S ? 2 : 1;
  CUtensorMap tm_x, tm_w;
  {
    const uint64_t dims[2] = {(uint64_t)pool.d_in, (uint64_t)T};
    const uint64_t strides[1] = {2ull * (uint64_t)ldx};
    const uint32_t box[2] = {(uint32_t)kFpK, (uint32_t)kFpM};
    if (!encode_tmap(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B))
      return LORA_ERR_CUDA;
  }
  {
    const uint64_t dims[2] = {(uint64_t)pool.d_in, (uint64_t)pool.D};
    const uint64_t strides[1] = {2ull * (uint64_t)ldw};
    const uint32_t box[2] = {(uint32_t)kFpK, (uint32_t)(kFpN / cta)};  // a pair's CTA loads half of a tile's W
    if (!encode_tmap(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(W), dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B))
      return LORA_ERR_CUDA;
  }
  FpParams p{};
  p.slot = seg->slot;
  p.rank_tab = pool.rank_tab;
  p.u_rows = pool.u_rows;
  p.y = y;
  p.status = seg->status;
  p.ldy = ldy;
  p.T = T;
  p.D = pool.D;
  p.nkb = pool.d_in / kFpK;
  p.L = pool.L;
  p.R16 = pool.R16;
  p.N = pool.N;
  p.ntm = ntm;
  p.ntn = ceil_div(pool.D, kFpN);
  p.ntg = ceil_div(ntm, cta);
  if ((long long)p.ntg * p.ntn > 0x7fffffffLL) return LORA_ERR_SHAPE;
  p.nunits = p.ntg * p.ntn;
  for (int l = 0; l < LORA_MAX_LANES; ++l) {
    p.d_out[l] = pool.d_out[l];
    p.off[l] = pool.off[l];
  }
  const int smem = FpShape<1>::kSmem;
  cudaError_t e;
  if (cta == 1) {
    if (!set_smem_limit(reinterpret_cast<const void*>(fused_proj_kernel<1>), pool.device, smem)) return LORA_ERR_CUDA;
    const int grid = p.nunits < sm_count(pool.device) ? p.nunits : sm_count(pool.device);  // one CTA per SM
    e = launch_pdl(fused_proj_kernel<1>, dim3((unsigned)grid), dim3(kFpThreads), smem, st, tm_x, tm_w, pool.tm_bk, p);
  } else {
    if (!set_smem_limit(reinterpret_cast<const void*>(fused_proj_kernel<2>), pool.device, smem)) return LORA_ERR_CUDA;
    const int cap = fp_max_pairs(pool.device);
    const int pairs = p.nunits < cap ? p.nunits : cap;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * pairs));
    cfg.blockDim = dim3(kFpThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, fused_proj_kernel<2>, tm_x, tm_w, pool.tm_bk, p);
  }
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cuda_status(e != cudaSuccess ? e : cudaGetLastError(), "fused_proj_kernel launch");
}

}  // namespace lora
