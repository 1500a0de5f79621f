// Decode path: rows whose own sequence is shorter than LORA_TC_MIN_QLEN
// (single-token decode rows, short chunks).  The segment builder groups them
// by slot, up to LORA_DEC_GROUP_ROWS rows of one slot per group, so a slot's
// factors are streamed once per group and shared by the group's rows.
//
//   shrink  u[row][i] = sum_j A[k][l][i][j] * x[row][j]     (TensorFold PR #47,
//   expand  y[row][o] += scale[k][l] * sum_i B[k][l][o][i] * u[row][i]   the delta
//           scale * B @ (A @ x); xLLM PR #2014, shrink then expand)
//
// One kernel does both halves.  A work unit is (decode group, lane) and runs
// on one thread-block cluster of CL CTAs (CL from the pool's shape only):
//   1. CTA c of the cluster shrinks its fixed range of d_in (K blocks of 64,
//      [c * nkb / CL, (c + 1) * nkb / CL)) for the group's rows: a partial
//      rank-space vector of 8 rows x r16 ranks, in its shared memory.
//   2. Every CTA tells every CTA of the cluster that its partial is ready
//      (remote mbarrier arrivals), then sums the CL partials in CTA order
//      straight out of the other CTAs' shared memory (distributed shared
//      memory).  So u never leaves the chip, and every CTA holds the same u.
//   3. CTA c expands its own slice of the lane's output columns
//      ([c * ncb / CL, (c + 1) * ncb / CL) in blocks of 64) and updates y.
// A producer warp streams, in the order the compute warps use them, the
// group's x rows of the K range (into an x buffer) and the slot's A rows
// (TMA tiles, 128-byte swizzle) and then, per 512-column chunk, the group's y
// rows and the slot's B^T rank rows (bulk copies) through a ring of 16 KB
// pages, so the expand's first loads are in flight while the shrink and the
// cluster exchange run.
//
// Fixed summation order, independent of the group a row lands in (so a row's
// bits depend only on its own x, its adapter and d_in):
//  * shrink: in each A page a compute thread takes two 8-element K chunks
//    (its K split s and s + nks); per (row, rank) it keeps an even-element and
//    an odd-element fma chain over its chunks in K order, adds them, and the
//    nks K splits of a rank tile are combined by a fixed xor butterfly inside
//    one warp; the cluster's CL partials are then added in CTA order.
//  * expand: v[o] accumulates B[o][i] * u[i] for i = 0..r-1 in order with fma;
//    y = fma(scale, v, y).
// The fmas are issued two at a time (packed f32x2), each exactly an fmaf in
// the order above.  Every wait is bounded; a wait that gives up records
// LORA_ERR_TIMEOUT and the CTA stops its work, still meeting its cluster
// barriers, so no CTA leaves while another may read its shared memory.
#include <cuda_runtime.h>

#include <mutex>
#include <vector>

#include "device.cuh"
#include "internal.h"

namespace lora {
namespace {

constexpr int kDfComputeWarps = 4;
constexpr int kDfCompute = kDfComputeWarps * 32;  // compute threads
constexpr int kDfThreads = kDfCompute + 32;       // + the producer warp
constexpr int kDfPageBytes = 16384;               // ring page
constexpr int kDfPages = 4;
constexpr int kDfCols = 512;                      // expand columns per chunk, 4 per compute thread
constexpr int kDfColsPerThread = kDfCols / kDfCompute;
constexpr int kDfRanksPerPage = kDfPageBytes / (kDfCols * 2);  // B^T rank rows per page
constexpr int kDfYPitch = kDfCols * 4;                         // bytes per y row of a page
constexpr int kDfMaxCluster = 8;
constexpr int kDfPartFloats = 128 * kDecGroup;  // a partial: [rank][row], ranks up to 128
static_assert(kDfColsPerThread == 4, "expand thread tile: 4 columns x 8 rows");
static_assert(kDecGroup * kDfYPitch == kDfPageBytes, "a y page holds the group's rows of one chunk");
static_assert(kDfRanksPerPage == 16, "16 B^T rank rows per page");

struct DfParams {
  const int32_t* counts;
  const int4* work;
  const int4* dec_rows;  // [group][2]: the group's 8 row indexes (entries past its row count unused)
  const int32_t* rank_tab;
  const float* scale_tab;
  int32_t* status;
  const uint16_t* Bt[LORA_MAX_LANES];
  const uint16_t* x;
  int64_t ldx;
  float* y;
  int64_t ldy;
  int L, R16, nkb, kc_max;
  int d_out[LORA_MAX_LANES], off[LORA_MAX_LANES];
};

// Element l of a per-lane parameter array, read with constant indexes (a
// run-time index would copy the array to local memory).
template <typename V>
__device__ __forceinline__ V lane_param(const V (&a)[LORA_MAX_LANES], int l) {
  V v = a[0];
#pragma unroll
  for (int i = 1; i < LORA_MAX_LANES; ++i)
    if (l == i) v = a[i];
  return v;
}

// One work unit as this CTA sees it.  Producer and compute warps derive it
// from the same device data, so they agree on every size.
struct Unit {
  int k, l, r, r16, nrows;
  int row[kDecGroup];
  int kb0, kb1;    // this CTA's K blocks of 64
  int c0, c1;      // this CTA's output columns of the lane
  int dout, off;
  int nks, nkbp;   // K splits per rank tile; K blocks per A page
};

__device__ __forceinline__ bool load_unit(const DfParams& p, int u, int cta, int ncta, Unit& U) {
  const int w = u / p.L;
  U.l = u - w * p.L;
  const int4 g = p.work[w];
  const int4 r0 = p.dec_rows[2 * w], r1 = p.dec_rows[2 * w + 1];
  U.k = g.x;
  U.nrows = g.z - g.y;
  U.row[0] = r0.x; U.row[1] = r0.y; U.row[2] = r0.z; U.row[3] = r0.w;
  U.row[4] = r1.x; U.row[5] = r1.y; U.row[6] = r1.z; U.row[7] = r1.w;
  U.r = p.rank_tab[U.k * p.L + U.l];
  if (U.r <= 0) return false;  // this lane of the slot is not loaded: nothing to do
  U.r16 = (U.r + 15) & ~15;
  U.kb0 = cta * p.nkb / ncta;
  U.kb1 = (cta + 1) * p.nkb / ncta;
  U.dout = lane_param(p.d_out, U.l);
  U.off = lane_param(p.off, U.l);
  const int ncb = U.dout / 64;
  U.c0 = (cta * ncb / ncta) * 64;
  U.c1 = ((cta + 1) * ncb / ncta) * 64;
  // rank tiles of 4 ranks, their count rounded up to a power of two; the
  // compute threads are split evenly over them
  int nrt = 4;
  while (nrt * 4 < U.r16) nrt *= 2;
  U.nks = kDfCompute / nrt;
  U.nkbp = kDfPageBytes / (U.r16 * 128);  // = nks / 4: two 8-element chunks per thread per page
  return true;
}

// One step of a butterfly reduce-scatter: lanes exchange half of their values
// with lane ^ o and keep the sum of the half selected by bit o of their id.
template <int HALF>
__device__ __forceinline__ void rs_step(float* v, int lane, int o) {
  const bool upper = (lane & o) != 0;
#pragma unroll
  for (int j = 0; j < HALF; ++j) {
    const float send = upper ? v[j] : v[j + HALF];
    const float keep = upper ? v[j + HALF] : v[j];
    v[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
  }
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

__global__ void __launch_bounds__(kDfThreads, 1)
    dec_fused_kernel(const __grid_constant__ TmapSized tm_a, DfParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kDfPages], empty_bar[kDfPages], xfull, xempty, pready[2];
  __shared__ __align__(16) float part[2][kDfPartFloats];  // this CTA's partial u, [rank][row], per unit parity
  __shared__ __align__(16) float us[kDfPartFloats];       // the summed u of the current unit, [rank][row]
  __shared__ int fail_sh;
  __shared__ int stop_sh[2];

  uint8_t* smem = align1024(smem_raw);
  uint8_t* ring = smem;                                              // kDfPages x 16 KB, 1024-aligned
  uint16_t* xbuf = reinterpret_cast<uint16_t*>(smem + kDfPages * kDfPageBytes);  // [8][kc_max] bf16

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cta = (int)cluster_ctarank(), ncta = (int)cluster_nctarank();
  pdl_wait();  // the segment builder's results are visible from here on
  if (tid == 0) {
    for (int s = 0; s < kDfPages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kDfComputeWarps);
    }
    mbar_init(&xfull, 1);
    mbar_init(&xempty, kDfComputeWarps);
    // one arrival from every CTA of the cluster per unit; two barriers used by
    // unit parity, so a CTA already on the next unit can never arrive on the
    // barrier of a unit that a slower CTA has not yet signalled
    mbar_init(&pready[0], (uint32_t)ncta);
    mbar_init(&pready[1], (uint32_t)ncta);
    fail_sh = 0;
    fence_mbar_init();
  }
  // every CTA's barriers are initialised before any CTA arrives on them remotely
  cluster_sync_all();

  // Units (decode group, lane) are dealt to the clusters round-robin; every
  // CTA of a cluster walks the same list.  The counts are final before this
  // grid runs (the builder wrote them; a builder error leaves them at 0).
  const int n_units = p.counts[2] * p.L;
  const int first = (int)cluster_id_x(), stride = (int)num_clusters_x();

  if (warp == kDfComputeWarps) {
    // ---------------- producer: x rows and A tiles of the K range, then per
    // chunk the y rows and the B^T rank rows, in the order they are used
    if (lane == 0) {
      uint32_t fill = 0, xj = 0;
      bool ok = true;
      auto next_page = [&](uint32_t bytes) -> uint8_t* {
        const int s = (int)(fill % kDfPages);
        if (fill >= kDfPages && !mbar_wait_or_fail(&empty_bar[s], ((fill / kDfPages) - 1) & 1, &fail_sh)) {
          fail_sh = 1;
          ok = false;
          return nullptr;
        }
        mbar_expect_tx(&full_bar[s], bytes);
        return ring + (size_t)s * kDfPageBytes;
      };
      for (int u = first; u < n_units && ok; u += stride) {
        Unit U;
        if (!load_unit(p, u, cta, ncta, U)) continue;
        const int kc = (U.kb1 - U.kb0) * 64;
        if (kc > 0) {
          if (xj >= 1 && !mbar_wait_or_fail(&xempty, (xj - 1) & 1, &fail_sh)) {
            fail_sh = 1;
            break;
          }
          mbar_expect_tx(&xfull, (uint32_t)(U.nrows * kc * 2));
#pragma unroll
          for (int g = 0; g < kDecGroup; ++g)
            if (g < U.nrows)
              bulk_load(xbuf + (size_t)g * p.kc_max, p.x + (size_t)U.row[g] * p.ldx + (size_t)U.kb0 * 64,
                        (uint32_t)(kc * 2), &xfull);
          ++xj;
          // A pages: nkbp K blocks of the slot's r16 rank rows each, one TMA
          // tile per power-of-two part of r16 (rows past the rank are the
          // pool's zero padding)
          for (int kb = U.kb0; kb < U.kb1 && ok; kb += U.nkbp) {
            const int n = min(U.nkbp, U.kb1 - kb);
            uint8_t* pg = next_page((uint32_t)(n * U.r16 * 128));
            if (!pg) break;
            ++fill;
            for (int i = 0; i < n; ++i) {
              int row = 0;
              for (int sz = kTmapSizes - 1; sz >= 0; --sz) {
                const int rows = 16 << sz;
                while (U.r16 - row >= rows) {
                  tma_load_3d(pg + (size_t)(i * U.r16 + row) * 128, &tm_a.m[sz][U.l], (kb + i) * 64, row, U.k,
                              &full_bar[(fill - 1) % kDfPages]);
                  row += rows;
                }
              }
            }
          }
        }
        const uint16_t* Bb = lane_param(p.Bt, U.l) + (size_t)U.k * p.R16 * U.dout;
        for (int c0 = U.c0; c0 < U.c1 && ok; c0 += kDfCols) {
          const int ec = min(kDfCols, U.c1 - c0);
          uint8_t* yp = next_page((uint32_t)(U.nrows * ec * 4));
          if (!yp) break;
          ++fill;
#pragma unroll
          for (int g = 0; g < kDecGroup; ++g)
            if (g < U.nrows)
              bulk_load(yp + (size_t)g * kDfYPitch, p.y + (size_t)U.row[g] * p.ldy + U.off + c0, (uint32_t)(ec * 4),
                        &full_bar[(fill - 1) % kDfPages]);
          for (int rb = 0; rb < U.r && ok; rb += kDfRanksPerPage) {
            const int nr = min(kDfRanksPerPage, U.r - rb);
            uint8_t* bp = next_page((uint32_t)(nr * ec * 2));
            if (!bp) break;
            ++fill;
            for (int i = 0; i < nr; ++i)
              bulk_load(bp + (size_t)i * (kDfCols * 2), Bb + (size_t)(rb + i) * U.dout + c0, (uint32_t)(ec * 2),
                        &full_bar[(fill - 1) % kDfPages]);
          }
        }
      }
      // Copies already issued land before the CTA may leave (after a failure
      // the compute warps may not have waited for them): the latest fill of
      // every page and the latest x load, each a bounded wait.
      for (uint32_t f = fill > kDfPages ? fill - kDfPages : 0; f < fill; ++f)
        if (!mbar_wait_bounded(&full_bar[f % kDfPages], (f / kDfPages) & 1)) fail_sh = 1;
      if (xj >= 1 && !mbar_wait_bounded(&xfull, (xj - 1) & 1)) fail_sh = 1;
    }
  } else {
    // ---------------- compute warps
    const int t = tid;
    uint32_t use = 0, xj = 0, uj = 0, dj = 0;
    const uint32_t part_addr0 = smem_u32(&part[0][0]);
    for (int u = first; u < n_units; u += stride) {
      Unit U;
      if (!load_unit(p, u, cta, ncta, U)) continue;
      // one stop decision per unit for all compute threads
      named_bar_sync(1, kDfCompute);
      if (t == 0) stop_sh[dj & 1] = fail_sh;
      named_bar_sync(1, kDfCompute);
      if (stop_sh[dj & 1]) break;
      ++dj;
      bool ok = true;
      const int kc = (U.kb1 - U.kb0) * 64;
      // ---- shrink of this CTA's K range: thread tile 8 rows x 4 ranks
      const int rt = t / U.nks, ks = t - rt * U.nks;
      const bool active = rt * 4 < U.r16;
      float2 acc[kDecGroup][4];  // (even-K, odd-K) sums of A[4 rt + j] . x[row]
#pragma unroll
      for (int g = 0; g < kDecGroup; ++g)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[g][j] = make_float2(0.f, 0.f);
      if (kc > 0) {
        if (!mbar_wait_or_fail(&xfull, xj & 1, &fail_sh)) {
          ok = false;
          fail_sh = 1;
        }
        for (int kb = U.kb0; kb < U.kb1; kb += U.nkbp, ++use) {
          const int s = (int)(use % kDfPages);
          if (ok && !mbar_wait_or_fail(&full_bar[s], (use / kDfPages) & 1, &fail_sh)) {
            ok = false;
            fail_sh = 1;
          }
          const int nq = min(U.nkbp, U.kb1 - kb) * 8;  // 8-element K chunks in this page
          if (ok && active) {
            const uint8_t* pg = ring + (size_t)s * kDfPageBytes;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int q = ks + h * U.nks;
              if (q < nq) {
                const int kbi = q >> 3, j = q & 7;
                float2 a[4][4];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                  const int i = 4 * rt + jj;
                  const uint4 w = *reinterpret_cast<const uint4*>(pg + (size_t)(kbi * U.r16 + i) * 128 +
                                                                  ((j ^ (i & 7)) << 4));
                  a[jj][0] = make_float2(bf16lo(w.x), bf16hi(w.x));
                  a[jj][1] = make_float2(bf16lo(w.y), bf16hi(w.y));
                  a[jj][2] = make_float2(bf16lo(w.z), bf16hi(w.z));
                  a[jj][3] = make_float2(bf16lo(w.w), bf16hi(w.w));
                }
                const uint16_t* xq = xbuf + (size_t)(kb - U.kb0) * 64 + q * 8;
#pragma unroll
                for (int g = 0; g < kDecGroup; ++g) {
                  const uint4 w = *reinterpret_cast<const uint4*>(xq + (size_t)g * p.kc_max);
                  const float2 xp[4] = {make_float2(bf16lo(w.x), bf16hi(w.x)), make_float2(bf16lo(w.y), bf16hi(w.y)),
                                        make_float2(bf16lo(w.z), bf16hi(w.z)), make_float2(bf16lo(w.w), bf16hi(w.w))};
#pragma unroll
                  for (int e = 0; e < 4; ++e)
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) acc[g][jj] = ffma2(a[jj][e], xp[e], acc[g][jj]);
                }
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty_bar[s]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&xempty);  // this warp is done with the x rows
        ++xj;
      }
      // ---- the nks K splits of a rank tile: a fixed butterfly inside the warp
      {
        float v[32];  // index row * 4 + j
#pragma unroll
        for (int g = 0; g < kDecGroup; ++g)
#pragma unroll
          for (int j = 0; j < 4; ++j) v[g * 4 + j] = acc[g][j].x + acc[g][j].y;
        int out0, nout;  // this lane's outputs v[0 .. nout) are tile outputs out0, out0 + 1, ...
        if (U.nks == 32) {
          rs_step<16>(v, lane, 16);
          rs_step<8>(v, lane, 8);
          rs_step<4>(v, lane, 4);
          rs_step<2>(v, lane, 2);
          rs_step<1>(v, lane, 1);
          out0 = lane;
          nout = 1;
        } else if (U.nks == 16) {
          rs_step<16>(v, lane, 8);
          rs_step<8>(v, lane, 4);
          rs_step<4>(v, lane, 2);
          rs_step<2>(v, lane, 1);
          out0 = 2 * (lane & 15);
          nout = 2;
        } else if (U.nks == 8) {
          rs_step<16>(v, lane, 4);
          rs_step<8>(v, lane, 2);
          rs_step<4>(v, lane, 1);
          out0 = 4 * (lane & 7);
          nout = 4;
        } else {  // nks == 4
          rs_step<16>(v, lane, 2);
          rs_step<8>(v, lane, 1);
          out0 = 8 * (lane & 3);
          nout = 8;
        }
        float* pt = part[uj & 1];
        if (active) {
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            if (e < nout) {
              const int o = out0 + e, g = o >> 2, i = 4 * rt + (o & 3);
              pt[i * kDecGroup + g] = v[e];
            }
          }
        }
      }
      // ---- cluster exchange: every CTA's partial is ready, then u = the sum
      // of the CL partials in CTA order
      named_bar_sync(1, kDfCompute);  // this CTA's partial is complete
      uint64_t* pr = &pready[uj & 1];
      if (t == 0) {
        fence_acq_rel_cluster();
        for (int c = 0; c < ncta; ++c) mbar_arrive_cluster(mapa_shared(smem_u32(pr), (uint32_t)c));
      }
      if (!mbar_wait_cluster_or_fail(pr, (uj >> 1) & 1, &fail_sh)) {
        ok = false;
        fail_sh = 1;
      }
      if (ok) {
        const uint32_t pa = part_addr0 + (uj & 1) * (uint32_t)(kDfPartFloats * 4);
        for (int idx = t; idx < U.r16 * kDecGroup; idx += kDfCompute) {
          float vals[kDfMaxCluster];
#pragma unroll
          for (int c = 0; c < kDfMaxCluster; ++c)
            if (c < ncta) vals[c] = ld_dsmem_f32(mapa_shared(pa + 4u * (uint32_t)idx, (uint32_t)c));
          float sum = vals[0];
#pragma unroll
          for (int c = 1; c < kDfMaxCluster; ++c)
            if (c < ncta) sum += vals[c];
          us[idx] = sum;
        }
      }
      ++uj;
      named_bar_sync(1, kDfCompute);  // u complete
      // ---- expand of this CTA's columns: thread tile 8 rows x 4 columns
      const float sc = p.scale_tab[U.k * p.L + U.l];
      for (int c0 = U.c0; c0 < U.c1; c0 += kDfCols) {
        const int ec = min(kDfCols, U.c1 - c0);
        const bool has = kDfColsPerThread * t < ec;
        // the y page: read this thread's values, then release the page
        float4 yv[kDecGroup];
        {
          const int s = (int)(use % kDfPages);
          if (ok && !mbar_wait_or_fail(&full_bar[s], (use / kDfPages) & 1, &fail_sh)) {
            ok = false;
            fail_sh = 1;
          }
          const uint8_t* yp = ring + (size_t)s * kDfPageBytes + 16 * t;
#pragma unroll
          for (int g = 0; g < kDecGroup; ++g)
            if (ok && has && g < U.nrows) yv[g] = *reinterpret_cast<const float4*>(yp + (size_t)g * kDfYPitch);
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty_bar[s]);
          ++use;
        }
        float2 eacc[kDecGroup][2];  // columns (4t, 4t+1) and (4t+2, 4t+3) of each row
#pragma unroll
        for (int g = 0; g < kDecGroup; ++g) eacc[g][0] = eacc[g][1] = make_float2(0.f, 0.f);
        for (int rb = 0; rb < U.r; rb += kDfRanksPerPage, ++use) {
          const int s = (int)(use % kDfPages);
          if (ok && !mbar_wait_or_fail(&full_bar[s], (use / kDfPages) & 1, &fail_sh)) {
            ok = false;
            fail_sh = 1;
          }
          if (ok && has) {
            const uint8_t* bp = ring + (size_t)s * kDfPageBytes + 8 * t;
            const int nr = min(kDfRanksPerPage, U.r - rb);
#pragma unroll 4
            for (int ri = 0; ri < nr; ++ri) {
              const uint2 q2 = *reinterpret_cast<const uint2*>(bp + (size_t)ri * (kDfCols * 2));
              const float2 b01 = make_float2(bf16lo(q2.x), bf16hi(q2.x));
              const float2 b23 = make_float2(bf16lo(q2.y), bf16hi(q2.y));
              const float4 u0 = *reinterpret_cast<const float4*>(&us[(rb + ri) * kDecGroup]);
              const float4 u1 = *reinterpret_cast<const float4*>(&us[(rb + ri) * kDecGroup + 4]);
              const float ug[kDecGroup] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
              for (int g = 0; g < kDecGroup; ++g) {
                const float2 u2 = make_float2(ug[g], ug[g]);
                eacc[g][0] = ffma2(b01, u2, eacc[g][0]);
                eacc[g][1] = ffma2(b23, u2, eacc[g][1]);
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty_bar[s]);
        }
        if (ok && has) {
#pragma unroll
          for (int g = 0; g < kDecGroup; ++g) {
            if (g < U.nrows) {
              float4 a = yv[g];
              a.x = fmaf(sc, eacc[g][0].x, a.x);
              a.y = fmaf(sc, eacc[g][0].y, a.y);
              a.z = fmaf(sc, eacc[g][1].x, a.z);
              a.w = fmaf(sc, eacc[g][1].y, a.w);
              *reinterpret_cast<float4*>(p.y + (size_t)U.row[g] * p.ldy + U.off + c0 + kDfColsPerThread * t) = a;
            }
          }
        }
      }
    }
  }
  // no CTA leaves while another CTA of its cluster may still read its partials
  cluster_sync_all();
  if (tid == 0 && fail_sh) set_error(p.status, LORA_ERR_TIMEOUT);
}

// Upper bound of decode groups for the last build: sum_k ceil(cnt_k / G) <= T/G + min(N, T).
int dec_group_bound(const PoolView& pool, const lora_segments* seg) {
  const int T = seg->T;
  return ceil_div(T, kDecGroup) + (pool.N < T ? pool.N : T);
}

// CTAs per cluster: a function of the pool's shape only (d_in), so a row's
// K split, and with it its bits, never depends on the batch.
int cluster_size(const PoolView& pool) {
  const int nkb = pool.d_in / 64;
  return nkb >= kDfMaxCluster ? kDfMaxCluster : (nkb >= 4 ? 4 : (nkb >= 2 ? 2 : 1));
}

size_t dec_smem_bytes(const PoolView& pool, int ncta) {
  const int nkb = pool.d_in / 64;
  const int kc_max = ceil_div(nkb, ncta) * 64;
  return 1024 + (size_t)kDfPages * kDfPageBytes + (size_t)kDecGroup * kc_max * 2;
}

// Clusters that can be resident at once, per (device, cluster size, shared memory).
int max_active_clusters(int device, int ncta, size_t smem) {
  struct Entry {
    int device, ncta;
    size_t smem;
    int n;
  };
  static std::mutex mu;
  static std::vector<Entry> cache;
  std::lock_guard<std::mutex> lock(mu);
  for (const Entry& e : cache)
    if (e.device == device && e.ncta == ncta && e.smem == smem) return e.n;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ncta * 64);
  cfg.blockDim = dim3(kDfThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ncta;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(dec_fused_kernel), &cfg) != cudaSuccess ||
      n <= 0) {
    cudaGetLastError();  // the query failed: clear its error and assume one cluster per ncta SMs
    n = sm_count(device) / ncta;
  }
  cache.push_back({device, ncta, smem, n});
  return n;
}

}  // namespace

int launch_decode(const PoolView& pool, const lora_segments* seg, const uint16_t* x, int64_t ldx, float* y,
                  int64_t ldy, cudaStream_t st) {
  const long long units = (long long)dec_group_bound(pool, seg) * pool.L;
  if (units <= 0) return LORA_OK;
  const int ncta = cluster_size(pool);
  const size_t smem = dec_smem_bytes(pool, ncta);
  if (smem > 227 * 1024) return LORA_ERR_SHAPE;
  if (!set_smem_limit(reinterpret_cast<const void*>(dec_fused_kernel), pool.device, (int)smem)) return LORA_ERR_CUDA;
  // Two waves of resident clusters at most; a cluster takes units
  // round-robin, so a step with more units reuses the clusters.
  const long long cap = 2LL * max_active_clusters(pool.device, ncta, smem);
  const int clusters = (int)(units < cap ? units : cap);
  DfParams p{};
  p.counts = seg->counts;
  p.work = seg->dec_work;
  p.dec_rows = reinterpret_cast<const int4*>(seg->dec_rows);
  p.rank_tab = pool.rank_tab;
  p.scale_tab = pool.scale_tab;
  p.status = seg->status;
  for (int l = 0; l < LORA_MAX_LANES; ++l) {
    p.Bt[l] = pool.Bt[l];
    p.d_out[l] = pool.d_out[l];
    p.off[l] = pool.off[l];
  }
  p.x = x;
  p.ldx = ldx;
  p.y = y;
  p.ldy = ldy;
  p.L = pool.L;
  p.R16 = pool.R16;
  p.nkb = pool.d_in / 64;
  p.kc_max = ceil_div(p.nkb, ncta) * 64;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(clusters * ncta));
  cfg.blockDim = dim3(kDfThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ncta;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, dec_fused_kernel, pool.tm_a, p);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cuda_status(e != cudaSuccess ? e : cudaGetLastError(), "dec_fused_kernel launch");
}

}  // namespace lora
