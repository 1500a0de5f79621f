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
//      accumulator in tensor memory.
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

#include "device.cuh"
#include "internal.h"

namespace lora {
namespace {

constexpr int kFpM = 128;                                     // tile rows (MMA M)
constexpr int kFpN = 256;                                     // tile columns (MMA N)
constexpr int kFpK = 64;                                      // d_in per stage: one 128-byte swizzle row
constexpr int kFpStages = 4;
constexpr int kFpXBytes = kFpM * kFpK * 2;                    // 16 KB
constexpr int kFpStageBytes = kFpXBytes + kFpN * kFpK * 2;    // 48 KB
constexpr int kFpGroups = 2;                                  // 16-rank groups per expand step
constexpr int kFpBkGroupBytes = kFpN * 32;                    // B of 256 columns x 16 ranks
constexpr int kFpUGroupBytes = kFpM * 32;                     // u' of 128 rows x 16 ranks
constexpr int kFpUBufs = 2;                                   // u' operand buffers (hi then lo halves)
constexpr int kFpUBufBytes = 2 * kFpGroups * kFpUGroupBytes;  // 16 KB
constexpr int kFpThreads = 320;                               // TMA, MMA, 4 operand warps, 4 epilogue warps
constexpr int kFpBandTiles = 16;                              // row tiles per band of the tile order
constexpr int kFpSlotWords = LORA_MAX_SLOTS / 32;
constexpr int kFpSmem = kFpStages * kFpStageBytes + kFpUBufs * kFpUBufBytes + 1024;
static_assert(kFpGroups * kFpBkGroupBytes <= kFpStageBytes, "an expand step's B fits a stage");

struct FpParams {
  const int32_t* slot;  // [T] per-token slot (segment builder)
  const int32_t* rank_tab;
  const float* u_rows;  // [T][L][R16] scale * u
  float* y;
  int32_t* status;
  int64_t ldy;
  int T, D, nkb, L, R16, N, ntm, ntn, ntiles;
  int d_out[LORA_MAX_LANES], off[LORA_MAX_LANES];
};

// The expand steps of a tile, in a fixed order (slot list order, lane,
// group), handed to f(k, l, q0, ng, c_lo, c_w, lc0): slot k, lane l, first
// 16-rank group q0 and group count ng, tile columns [c_lo, c_lo + c_w) =
// lane columns [lc0, lc0 + c_w).  f returns false to stop.  Every role runs
// its own walk over the same shared list and tables, so all agree.
template <typename F>
__device__ __forceinline__ bool for_each_step(const FpParams& p, const int* slots, int nslots, int n0, F&& f) {
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
      for (int q0 = 0; q0 < nk; q0 += kFpGroups)
        if (!f(k, l, q0, min(kFpGroups, nk - q0), lo - n0, hi - lo, lo - p.off[l])) return false;
    }
  }
  return true;
}

// Tile t of the order: bands of kFpBandTiles row tiles, column tiles in order
// inside a band (CTAs working at the same time share W and x tiles in L2).
__device__ __forceinline__ void tile_origin(const FpParams& p, int t, int& m0, int& n0) {
  const int band_size = kFpBandTiles * p.ntn;
  const int band = t / band_size, in_band = t - band * band_size;
  const int rows_in_band = min(kFpBandTiles, p.ntm - band * kFpBandTiles);
  m0 = (band * kFpBandTiles + in_band % rows_in_band) * kFpM;
  n0 = (in_band / rows_in_band) * kFpN;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Persistent: CTA b takes tiles b, b + G, b + 2G, ... (G = the grid).  Two
// accumulators of 256 TMEM columns alternate between tiles, so the epilogue of
// one tile runs while the next one's K loop does.  Every barrier a role waits
// on is waited on phase by phase, in order, by that role.
__global__ void __launch_bounds__(kFpThreads, 1)
    fused_proj_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                      const __grid_constant__ TmapSized tm_bk, FpParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kFpStages], empty_bar[kFpStages];
  __shared__ __align__(8) uint64_t ufull_bar[kFpUBufs], uempty_bar[kFpUBufs];
  __shared__ __align__(8) uint64_t plan_full[2], plan_empty[2], acc_full[2], acc_empty[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int fail_sh;
  __shared__ int nslots_sh[2];
  __shared__ int stop_sh[2];  // per plan buffer: a warp of warps 2-5 saw a failure (they stop together)
  __shared__ int slots_sh[2][kFpM];
  __shared__ uint32_t bits_sh[kFpSlotWords];

  pdl_wait();  // the shrinks' u' (and the builder's slots) are visible from here on
  if (*p.status != 0) return;  // a routing error or an earlier timeout: y is not written

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ubuf = smem + kFpStages * kFpStageBytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kFpStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int q = 0; q < kFpUBufs; ++q) {
      mbar_init(&ufull_bar[q], 4);
      mbar_init(&uempty_bar[q], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&plan_full[b], 1);
      mbar_init(&plan_empty[b], 2);
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    fail_sh = 0;
    stop_sh[0] = stop_sh[1] = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base_sh, 2 * kFpN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      uint32_t i = 0;
      bool ok = true;
      auto take = [&](uint32_t bytes) -> uint8_t* {
        const int s = (int)(i % kFpStages);
        if (i >= kFpStages && !mbar_wait_or_fail(&empty_bar[s], ((i / kFpStages) - 1) & 1, &fail_sh)) {
          fail_sh = 1;
          ok = false;
          return nullptr;
        }
        mbar_expect_tx(&full_bar[s], bytes);
        return smem + (size_t)s * kFpStageBytes;
      };
      int jj = 0;
      for (int t = blockIdx.x; t < p.ntiles && ok; t += gridDim.x, ++jj) {
        int m0, n0;
        tile_origin(p, t, m0, n0);
        for (int kb = 0; kb < p.nkb && ok; ++kb) {
          uint8_t* st = take((uint32_t)kFpStageBytes);
          if (!st) break;
          uint64_t* fb = &full_bar[i % kFpStages];
          tma_load_2d(st, &tm_x, kb * kFpK, m0, fb);
          tma_load_2d(st + kFpXBytes, &tm_w, kb * kFpK, n0, fb);
          ++i;
        }
        const int b = jj & 1;
        if (ok && !mbar_wait_or_fail(&plan_full[b], (jj >> 1) & 1, &fail_sh)) {
          fail_sh = 1;
          ok = false;
        }
        if (!ok) break;
        for_each_step(p, slots_sh[b], nslots_sh[b], n0, [&](int k, int l, int q0, int ng, int, int c_w, int lc0) {
          const int nb = (c_w + 127) / 128;  // boxes of 128 columns per group
          uint8_t* st = take((uint32_t)(ng * nb * 4096));
          if (!st) return false;
          uint64_t* fb = &full_bar[i % kFpStages];
          for (int g = 0; g < ng; ++g)
            for (int h = 0; h < nb; ++h)
              tma_load_3d(st + g * kFpBkGroupBytes + h * 4096, &tm_bk.m[0][l], 0, lc0 + 128 * h,
                          k * (p.R16 / 16) + q0 + g, fb);
          ++i;
          return true;
        });
        if (ok) mbar_arrive(&plan_empty[b]);
      }
      // Copies already issued land before the CTA may leave (after a failure
      // the MMA thread may not have waited for them): the latest fill of
      // every stage, each a bounded wait.
      for (uint32_t f = i > kFpStages ? i - kFpStages : 0; f < i; ++f)
        if (!mbar_wait_bounded(&full_bar[f % kFpStages], (f / kFpStages) & 1)) fail_sh = 1;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      uint32_t i = 0, n = 0;  // ring stage uses, u' buffer uses
      bool ok = true;
      const uint32_t idesc_main = idesc_bf16(kFpM, kFpN);
      int jj = 0;
      for (int t = blockIdx.x; t < p.ntiles && ok; t += gridDim.x, ++jj) {
        int m0, n0;
        tile_origin(p, t, m0, n0);
        const int b = jj & 1;
        const uint32_t acc = tmem + (uint32_t)(b * kFpN);
        if (jj >= 2 && !mbar_wait_or_fail(&acc_empty[b], ((jj >> 1) - 1) & 1, &fail_sh)) {
          fail_sh = 1;
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < p.nkb; ++kb, ++i) {
          const int s = (int)(i % kFpStages);
          if (!mbar_wait_or_fail(&full_bar[s], (i / kFpStages) & 1, &fail_sh)) {
            fail_sh = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t xa = smem_u32(smem + (size_t)s * kFpStageBytes), wa = xa + kFpXBytes;
#pragma unroll
          for (int kk = 0; kk < kFpK / 16; ++kk)
            mma_bf16(acc, smem_desc(xa + 32 * kk, 16, 1024, kSwz128), smem_desc(wa + 32 * kk, 16, 1024, kSwz128),
                     idesc_main, (kb | kk) != 0 ? 1u : 0u);
          mma_commit(&empty_bar[s]);
        }
        if (ok && !mbar_wait_or_fail(&plan_full[b], (jj >> 1) & 1, &fail_sh)) {
          fail_sh = 1;
          ok = false;
        }
        if (!ok) break;
        ok = for_each_step(p, slots_sh[b], nslots_sh[b], n0, [&](int, int, int, int ng, int c_lo, int c_w, int) {
          const int s = (int)(i % kFpStages), q = (int)(n % kFpUBufs);
          if (!mbar_wait_or_fail(&full_bar[s], (i / kFpStages) & 1, &fail_sh) ||
              !mbar_wait_or_fail(&ufull_bar[q], (n / kFpUBufs) & 1, &fail_sh)) {
            fail_sh = 1;
            return false;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + (size_t)s * kFpStageBytes);
          const uint32_t ua = smem_u32(ubuf + (size_t)q * kFpUBufBytes);
          const uint32_t idesc = idesc_bf16(kFpM, c_w);
          for (int half = 0; half < 2; ++half)
            for (int g = 0; g < ng; ++g)
              mma_bf16(acc + (uint32_t)c_lo,
                       smem_desc(ua + (half * kFpGroups + g) * kFpUGroupBytes, 128, 256, kSwzNone),
                       smem_desc(sa + g * kFpBkGroupBytes, 16, 256, kSwz32), idesc, 1u);
          mma_commit(&empty_bar[s]);
          mma_commit(&uempty_bar[q]);
          ++i;
          ++n;
          return true;
        });
        if (!ok) break;
        mma_commit(&acc_full[b]);
        mbar_arrive(&plan_empty[b]);
      }
    }
  } else if (warp < 6) {
    // ---------------- warps 2-5: each tile's slots, then the u' operands of
    // its expand steps: row m of the slot's rows, zero for rows of other
    // slots, as bf16 hi and lo in the K-major core-matrix layout (8 rows x 16
    // bytes per core matrix; 16 ranks = two of them)
    const int m = (warp & 3) * 32 + lane;
    const int bt = threadIdx.x - 64;  // 0..127
    const uint32_t row_off = (uint32_t)((m >> 3) * 256 + (m & 7) * 16);
    // These four warps meet at named barriers, so they leave the tile loop
    // together: a failure any of them sees goes into stop_sh[b] between the
    // first and the third barrier of a tile, and all read it after the third.
    uint32_t n = 0;
    bool ok = true;
    int jj = 0;
    for (int t = blockIdx.x; t < p.ntiles; t += gridDim.x, ++jj) {
      int m0, n0;
      tile_origin(p, t, m0, n0);
      const int b = jj & 1;
      const int tr = m0 + m;
      const int myslot = tr < p.T ? p.slot[tr] : 0;
      if (ok && jj >= 2) {  // the plan buffer is free once the producer and the MMA thread are done with it
        int got = 1;
        if (lane == 0) got = mbar_wait_or_fail(&plan_empty[b], ((jj >> 1) - 1) & 1, &fail_sh) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, got, 0)) {
          fail_sh = 1;
          ok = false;
        }
      }
      if (bt == 0) stop_sh[b] = 0;  // every warp read it two tiles ago, before the barriers of the last tile
      for (int w = bt; w < kFpSlotWords; w += 128) bits_sh[w] = 0u;
      named_bar_sync(1, 128);
      if (lane == 0 && (!ok || fail_sh)) atomicOr(&stop_sh[b], 1);
      if (myslot > 0) atomicOr(&bits_sh[myslot >> 5], 1u << (myslot & 31));
      named_bar_sync(1, 128);
      if (warp == 2) {
        // distinct slots of the tile in ascending order
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
          slots_sh[b][pos++] = 64 * lane + __ffs(w0) - 1;
          w0 &= w0 - 1;
        }
        while (w1) {
          slots_sh[b][pos++] = 64 * lane + 32 + __ffs(w1) - 1;
          w1 &= w1 - 1;
        }
        if (lane == 31) nslots_sh[b] = incl;
      }
      named_bar_sync(1, 128);
      if (stop_sh[b]) break;
      if (warp == 2 && lane == 0) mbar_arrive(&plan_full[b]);
      ok = for_each_step(p, slots_sh[b], nslots_sh[b], n0, [&](int k, int l, int q0, int ng, int, int, int) {
        const int q = (int)(n % kFpUBufs);
        const bool mine = myslot == k;
        // this row's u' first, so the loads are in flight during the wait
        const float4* src =
            reinterpret_cast<const float4*>(p.u_rows + ((size_t)(mine ? tr : 0) * p.L + l) * p.R16 + 16 * q0);
        float4 v[4 * kFpGroups];
#pragma unroll
        for (int g = 0; g < kFpGroups; ++g)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            v[4 * g + e] = mine && g < ng ? __ldcg(src + 4 * g + e) : make_float4(0.f, 0.f, 0.f, 0.f);
        if (n >= kFpUBufs) {  // one lane waits for the buffer to be free; the warp follows it
          int got = 1;
          if (lane == 0) got = mbar_wait_or_fail(&uempty_bar[q], ((n / kFpUBufs) - 1) & 1, &fail_sh) ? 1 : 0;
          if (!__shfl_sync(0xffffffffu, got, 0)) {
            fail_sh = 1;
            return false;
          }
        }
        uint8_t* ub = ubuf + (size_t)q * kFpUBufBytes;
#pragma unroll
        for (int g = 0; g < kFpGroups; ++g) {
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
            *reinterpret_cast<uint4*>(ub + kFpGroups * kFpUGroupBytes + o) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          }
        }
        fence_proxy_async_smem();  // the MMA reads these through the async proxy
        __syncwarp();
        if (lane == 0) mbar_arrive(&ufull_bar[q]);
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
    for (int t = blockIdx.x; t < p.ntiles; t += gridDim.x, ++jj) {
      int m0, n0;
      tile_origin(p, t, m0, n0);
      const int b = jj & 1;
      int got = 1;  // uniform over the warp: the tcgen05.ld below is warp-collective
      if (lane == 0) got = mbar_wait_or_fail(&acc_full[b], (jj >> 1) & 1, &fail_sh) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, got, 0)) {
        fail_sh = 1;
        break;
      }
      tc_fence_after();
      const int tr = m0 + m;
      float* yr = p.y + (size_t)tr * p.ldy + n0;
#pragma unroll 1
      for (int j = 0; j < kFpN / 32; ++j) {
        float v[32];
        tmem_ld32(tmem + trow + (uint32_t)(b * kFpN + 32 * j), v);
        if (tr < p.T && n0 + 32 * j < p.D) {
          float4* dst = reinterpret_cast<float4*>(yr + 32 * j);
#pragma unroll
          for (int e = 0; e < 8; ++e) dst[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[b]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * kFpN);
  }
  if (threadIdx.x == 0 && fail_sh) set_error(p.status, LORA_ERR_TIMEOUT);
}

}  // namespace

int launch_fused_projection(const PoolView& pool, const lora_segments* seg, const uint16_t* W, int64_t ldw,
                            const uint16_t* x, int64_t ldx, float* y, int64_t ldy, cudaStream_t st) {
  const int T = seg->T;
  if (T <= 0) return LORA_OK;
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
    const uint32_t box[2] = {(uint32_t)kFpK, (uint32_t)kFpN};
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
  p.ntm = ceil_div(T, kFpM);
  p.ntn = ceil_div(pool.D, kFpN);
  p.ntiles = p.ntm * p.ntn;
  for (int l = 0; l < LORA_MAX_LANES; ++l) {
    p.d_out[l] = pool.d_out[l];
    p.off[l] = pool.off[l];
  }
  if ((long long)p.ntm * p.ntn > 0x7fffffffLL) return LORA_ERR_SHAPE;
  const int grid = p.ntiles < sm_count(pool.device) ? p.ntiles : sm_count(pool.device);  // one CTA per SM
  const int smem = kFpSmem;
  if (!set_smem_limit(reinterpret_cast<const void*>(fused_proj_kernel), pool.device, smem)) return LORA_ERR_CUDA;
  const cudaError_t e =
      launch_pdl(fused_proj_kernel, dim3((unsigned)grid), dim3(kFpThreads), smem, st, tm_x, tm_w, pool.tm_bk, p);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cuda_status(e != cudaSuccess ? e : cudaGetLastError(), "fused_proj_kernel launch");
}

}  // namespace lora
