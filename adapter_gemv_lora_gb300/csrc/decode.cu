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
// on one thread-block cluster of CL CTAs (CL from d_in only: 8 from d_in 8192
// on, else 4 for d_in >= 256):
//   1. CTA c of the cluster shrinks its fixed range of d_in (K blocks of 64,
//      [c * nkb / CL, (c + 1) * nkb / CL)) for the group's rows: a partial
//      rank-space vector of up to 8 rows x r16 ranks.
//   2. The partials are reduced on chip in two rounds of st.async stores,
//      each counted on the receiver's mbarrier (no fence, no global memory):
//      every CTA sends each 1 / CL slice of its ranks to the CTA that owns
//      the slice, which adds the CL partials in CTA order; then every owner
//      sends its summed slice to every CTA.  So u never leaves the chip, every
//      CTA of the cluster holds the same u, and the buffers hold R16 x 8
//      floats a round whatever CL is.
//   3. CTA c expands its own slice of the lane's output columns
//      ([c * ncb / CL, (c + 1) * ncb / CL) in blocks of 64) and updates y.
// The clusters are persistent (as many as fit on the GPU at once) and take
// the units longest first (by rank class), dealt in snake order, so the
// longest units start first and the clusters finish close together.
// A producer warp streams, in the order the compute warps use them, pages of
// the group's x rows with the slot's A rows for a few K blocks (bulk copies
// and TMA tiles with the 128-byte swizzle) and then, per 512-column chunk,
// the slot's B^T rank rows (TMA boxes of 16 ranks x up to 256 columns) and the
// group's y rows (bulk copies), through a
// ring of pages; the compute warps hold one page at a time, so the expand's
// first loads are in flight while the shrink and the exchange run.
//
// Fixed summation order, independent of the group a row lands in (so a row's
// bits depend only on its own x, its adapter and d_in):
//  * shrink: thread (rank tile of 4 ranks, K split ks) takes the 8-element K
//    chunks ks, ks + nks, ks + 2 nks, ... of its CTA's K range (nks from r16
//    only); per (row, rank) it keeps an even-element and an odd-element fma
//    chain over its chunks in K order and adds them; the nks K splits are
//    combined by a fixed xor butterfly inside one warp; the cluster's CL
//    partials are then added in CTA order.
//  * expand: v[o] accumulates B[o][i] * u[i] for i = 0..r-1 in order with fma;
//    y = fma(scale, v, y).
// The fmas are issued two at a time (packed f32x2), each exactly an fmaf in
// the order above; the thread tiles cover 1, 2, 4 or 8 rows (the group's row
// count rounded up), which changes no row's arithmetic.  Every wait is
// bounded; a wait that gives up records LORA_ERR_TIMEOUT and the CTA stops
// its work, still meeting its cluster barriers, so no CTA leaves while
// another may still write into its shared memory.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "device.cuh"
#include "internal.h"

namespace lora {
namespace {

constexpr int kDfComputeWarps = 4;
constexpr int kDfCompute = kDfComputeWarps * 32;  // compute threads
constexpr int kDfThreads = kDfCompute + 32;       // + the producer warp
constexpr int kDfPageBytes = 18432;               // ring page (1024-aligned size)
constexpr int kDfMaxPages = 12;                   // ring pages: as many as the shared memory left allows
constexpr int kDfCtasPerSm = 2;                   // resident CTAs per SM the launch is sized for
constexpr int kDfCols = 512;                      // expand columns per chunk, 4 per compute thread
constexpr int kDfColsPerThread = kDfCols / kDfCompute;
constexpr int kDfRanksPerPage = 16;               // B^T rank rows per page (16 x 512 bf16 = 16 KB)
constexpr int kDfYPitch = kDfCols * 4;            // bytes per y row of a page
constexpr int kDfClassCache = 2048;               // units whose rank class is kept in shared memory
static_assert(kDfColsPerThread == 4, "expand thread tile: 4 columns x 8 rows");
static_assert(kDecGroup * kDfYPitch <= kDfPageBytes, "a y page holds the group's rows of one chunk");
static_assert(kDfRanksPerPage * kDfCols * 2 <= kDfPageBytes, "a B page holds 16 rank rows of one chunk");
static_assert(kDfPageBytes % 1024 == 0, "pages keep the 1024-byte alignment of the A tiles");

struct DfParams {
  const int32_t* counts;
  const int4* work;
  const int4* dec_rows;  // [group][2]: the group's 8 row indexes (entries past its row count unused)
  const int32_t* rank_tab;
  const float* scale_tab;
  int32_t* status;
  const uint16_t* x;
  int64_t ldx;
  float* y;
  int64_t ldy;
  float* u_rows;  // row mode: scale * u of each row to [T][L][R16], no expand (y is not touched)
  int L, R16, nkb, npages;
  int n_tab;  // entries of the rank and scale tables (slots x lanes)
  int parts;  // column parts per (group, lane), each its own unit (set on the device per step)
  int d_out[LORA_MAX_LANES], off[LORA_MAX_LANES], bt_cols[LORA_MAX_LANES];
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
  int bi;          // columns per B^T TMA box of the lane (the page holds ceil(ec / bi) boxes of 16 x bi)
  int nks;         // K splits per rank tile
  int nkbp;        // K blocks per A page
  int cpt;         // 8-element K chunks per thread per A page (1 or 2)
};

__device__ __forceinline__ bool load_unit(const DfParams& p, int u, int cta, int ncta, Unit& U) {
  const int per_group = p.L * p.parts;
  const int w = u / per_group, rem = u - w * per_group;
  U.l = rem / p.parts;
  const int part = rem - U.l * p.parts;
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
  U.bi = lane_param(p.bt_cols, U.l);
  // this unit's column part, then this CTA's share of it (blocks of 64)
  const int ncb = U.dout / 64;
  const int pb0 = part * ncb / p.parts, pb1 = (part + 1) * ncb / p.parts;
  U.c0 = (pb0 + cta * (pb1 - pb0) / ncta) * 64;
  U.c1 = (pb0 + (cta + 1) * (pb1 - pb0) / ncta) * 64;
  // rank tiles of 4 ranks, their count rounded up to a power of two; the
  // compute threads are split evenly over them
  int nrt = 4;
  while (nrt * 4 < U.r16) nrt *= 2;
  U.nks = kDfCompute / nrt;  // 32, 16, 8 or 4
  // K blocks per A page: a power of two with the page within kDfPageBytes
  // (x rows and A rows) and at most two chunks per thread
  int nkbp = U.nks >= 8 ? U.nks / 4 : 1;
  while (nkbp > 1 && nkbp * (kDecGroup + U.r16) * 128 > kDfPageBytes) nkbp >>= 1;
  U.nkbp = nkbp;
  U.cpt = 8 * nkbp / U.nks;
  return true;
}

// The units of one cluster, longest first.  Units are ranked by the rank
// class of their (slot, lane), r16 / 16 (a unit's bytes and fmas grow with
// its rank), highest class first and in unit order inside a class, and dealt
// to the clusters in snake order (0, 1, .., nc-1, nc-1, .., 0, 0, ..), so the
// longest units start first and every cluster gets a similar share.  Every
// warp runs its own copy of the iterator (ballots over 32 units at a time),
// so all warps of all CTAs of a cluster walk the same sequence; which cluster
// runs a unit never changes its result.
struct UnitIter {
  int n_units, q, nc;
  int cls;        // rank class being scanned (7..0), -1 when done
  int u0;         // first unit of the next 32-unit chunk to scan
  int base;       // units ranked before that chunk
  int pbase;      // first unit of the chunk that pend refers to
  unsigned pend;  // units of that chunk dealt to this cluster and not yet returned
  unsigned present;
};

__device__ __forceinline__ int unit_class_global(const DfParams& p, int u) {
  const int per_group = p.L * p.parts;
  const int w = u / per_group, l = (u - w * per_group) / p.parts;
  const int r = p.rank_tab[p.work[w].x * p.L + l];
  return r > 0 ? (r + 15) / 16 - 1 : -1;
}

// A unit's rank class: from the shared-memory copy filled at kernel start
// (the first kDfClassCache units), else from global memory.
__device__ __forceinline__ int unit_class(const DfParams& p, const int8_t* cls_sh, int u) {
  return u < kDfClassCache ? (int)cls_sh[u] : unit_class_global(p, u);
}

__device__ __forceinline__ void unit_iter_init(UnitIter& it, const DfParams& p, const int8_t* cls_sh, int n_units,
                                               int n_clusters, int lane) {
  it.n_units = n_units;
  it.q = (int)cluster_id_x();
  it.nc = n_clusters;
  unsigned present = 0;
  for (int u0 = 0; u0 < n_units; u0 += 32) {
    const int c = u0 + lane < n_units ? unit_class(p, cls_sh, u0 + lane) : -1;
    present |= __reduce_or_sync(0xffffffffu, c >= 0 ? 1u << c : 0u);
  }
  it.present = present;
  it.cls = present ? 31 - __clz((int)present) : -1;
  it.u0 = 0;
  it.base = 0;
  it.pbase = 0;
  it.pend = 0;
}

// The next unit of this cluster (all 32 lanes call it together); false when done.
__device__ __forceinline__ bool next_unit(UnitIter& it, const DfParams& p, const int8_t* cls_sh, int lane, int& u) {
  for (;;) {
    if (it.pend) {  // units of the last scanned chunk dealt to this cluster, in order
      const int j = __ffs(it.pend) - 1;
      it.pend &= it.pend - 1;
      u = it.pbase + j;
      return true;
    }
    if (it.cls < 0) return false;
    if (it.u0 >= it.n_units) {  // this class is done: the next present one
      const unsigned lower = it.present & ((1u << it.cls) - 1u);
      it.cls = lower ? 31 - __clz((int)lower) : -1;
      it.u0 = 0;
      continue;
    }
    const int uu = it.u0 + lane;
    const bool in = uu < it.n_units && unit_class(p, cls_sh, uu) == it.cls;
    const unsigned m = __ballot_sync(0xffffffffu, in);
    const int pos = (it.base + __popc(m & ((1u << lane) - 1u))) % (2 * it.nc);
    const int owner = pos < it.nc ? pos : 2 * it.nc - 1 - pos;
    it.pend = __ballot_sync(0xffffffffu, in && owner == it.q);
    it.base += __popc(m);
    it.pbase = it.u0;
    it.u0 += 32;
  }
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

// The shrink's fmas over one A page for a tile of RT rows (RT = the group's
// row count rounded up to 1, 2, 4 or 8): thread (rank tile rt, K split ks)
// takes the page's 8-element K chunks ks (and ks + nks when cpt == 2).  A row's
// chains do not depend on RT, so neither do its bits.  The page holds the x
// rows [8][nkbp * 64] then the A rows [nkbp][r16][64] (128-byte swizzle).
template <int RT>
__device__ __forceinline__ void shrink_page(const uint8_t* pg, int nkbp, int r16, int rt, int ks, int nks, int cpt,
                                            int nq, float2 (&acc)[kDecGroup][4]) {
  const uint8_t* ap = pg + (size_t)kDecGroup * nkbp * 128;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int q = ks + h * nks;
    if (h < cpt && q < nq) {
      const int kbi = q >> 3, j = q & 7;
      float2 a[4][4];
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int i = 4 * rt + jj;
        const uint4 w = *reinterpret_cast<const uint4*>(ap + (size_t)(kbi * r16 + i) * 128 + ((j ^ (i & 7)) << 4));
        a[jj][0] = make_float2(bf16lo(w.x), bf16hi(w.x));
        a[jj][1] = make_float2(bf16lo(w.y), bf16hi(w.y));
        a[jj][2] = make_float2(bf16lo(w.z), bf16hi(w.z));
        a[jj][3] = make_float2(bf16lo(w.w), bf16hi(w.w));
      }
      const uint8_t* xq = pg + (size_t)q * 16;
#pragma unroll
      for (int g = 0; g < RT; ++g) {
        const uint4 w = *reinterpret_cast<const uint4*>(xq + (size_t)g * nkbp * 128);
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

// The expand's fmas over one B^T page (nr rank rows starting at rank rb) for
// a tile of RT rows: this thread's 4 columns (bp already offset to them in
// its TMA box; pitch = the box's row bytes).
template <int RT>
__device__ __forceinline__ void expand_page(const uint8_t* bp, int pitch, const float* us, int rb, int nr,
                                            float2 (&eacc)[kDecGroup][2]) {
#pragma unroll 4
  for (int ri = 0; ri < nr; ++ri) {
    const uint2 q2 = *reinterpret_cast<const uint2*>(bp + (size_t)ri * pitch);
    const float2 b01 = make_float2(bf16lo(q2.x), bf16hi(q2.x));
    const float2 b23 = make_float2(bf16lo(q2.y), bf16hi(q2.y));
    float ug[kDecGroup];
    const float4 u0 = *reinterpret_cast<const float4*>(&us[(rb + ri) * kDecGroup]);
    ug[0] = u0.x; ug[1] = u0.y; ug[2] = u0.z; ug[3] = u0.w;
    if (RT > 4) {
      const float4 u1 = *reinterpret_cast<const float4*>(&us[(rb + ri) * kDecGroup + 4]);
      ug[4] = u1.x; ug[5] = u1.y; ug[6] = u1.z; ug[7] = u1.w;
    }
#pragma unroll
    for (int g = 0; g < RT; ++g) {
      const float2 u2 = make_float2(ug[g], ug[g]);
      eacc[g][0] = ffma2(b01, u2, eacc[g][0]);
      eacc[g][1] = ffma2(b23, u2, eacc[g][1]);
    }
  }
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

__global__ void __launch_bounds__(kDfThreads, kDfCtasPerSm)
    dec_fused_kernel(const __grid_constant__ TmapSized tm_a, const __grid_constant__ TmapLanes tm_bt, DfParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kDfMaxPages], empty_bar[kDfMaxPages];
  __shared__ __align__(8) uint64_t prs[2], pag[2];  // per unit parity: reduce-scatter and all-gather bytes
  __shared__ int fail_sh;
  __shared__ int stop_sh[2];
  __shared__ int xok_sh[2];  // per unit parity: every partial of this CTA's rank slice arrived
  __shared__ int xag_sh[2];  // per unit parity: every slice of u arrived
  __shared__ int8_t cls_sh[kDfClassCache];  // rank class of each unit (-1: nothing to do)

  uint8_t* smem = align1024(smem_raw);
  const uint32_t npages = (uint32_t)p.npages;
  uint8_t* ring = smem;  // npages pages, 1024-aligned
  // exchange buffers after the ring, per unit parity: the partials of this
  // CTA's rank slice from every CTA ([source CTA][slice rank][row]), then the
  // whole summed u ([rank][row]); R16 x 8 floats each whatever the cluster size
  float* rsbuf = reinterpret_cast<float*>(smem + (size_t)npages * kDfPageBytes);
  float* agbuf = rsbuf + 2 * (size_t)p.R16 * kDecGroup;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cta = (int)cluster_ctarank(), ncta = (int)cluster_nctarank();
  const int part_floats = p.R16 * kDecGroup;
  // Barriers, the cluster's meeting and the pool's tables and TMA descriptors
  // do not depend on the previous kernel: they are set up and warmed while it
  // finishes (the tables were written when the adapters were loaded).
  if (tid == 0) {
    for (uint32_t s = 0; s < npages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kDfComputeWarps);
    }
    // per unit parity, for each exchange round: one local arrival (with the
    // expected bytes) and the st.async bytes the other CTAs send
    for (int q = 0; q < 2; ++q) {
      mbar_init(&prs[q], 1);
      mbar_init(&pag[q], 1);
    }
    fail_sh = 0;
    fence_mbar_init();
  }
  if (tid == kDfCompute) {  // the producer's lane 0, with constant indexes into the parameters
#pragma unroll
    for (int l = 0; l < LORA_MAX_LANES; ++l) {
      if (l < p.L) {
#pragma unroll
        for (int sz = 0; sz < kTmapSizes; ++sz) prefetch_tensormap(&tm_a.m[sz][l]);
        prefetch_tensormap(&tm_bt.m[l]);
      }
    }
  }
  for (int i = tid * 32; i < p.n_tab; i += kDfThreads * 32) {
    prefetch_l2(p.rank_tab + i);
    prefetch_l2(p.scale_tab + i);
  }
  // every CTA's barriers are initialised before any CTA stores into it
  cluster_sync_all();
  pdl_wait();  // the segment builder's results are visible from here on

  // Units (decode group, lane), longest first (UnitIter).  The counts are
  // final before this grid runs (the builder wrote them; a builder error
  // leaves them at 0).
  // Column parts: when the step has fewer (group, lane) pairs than there are
  // clusters, each pair's columns are split into up to 4 parts (a power of
  // two), each its own unit that redoes the pair's shrink, so more clusters
  // work.  Every CTA computes the same value from the same counts, and a
  // row's bits do not depend on it.
  // Clusters at work: all, unless the step's tensor tiles (whose kernels run
  // beside this one on another stream) outweigh its decode units (a tile of up
  // to 128 rows against a group of up to 8: four units to a tile); then the
  // tensor path bounds the step, and only as many clusters work as give each
  // about four units (no column parts), which leaves the SMs to the tensor
  // path while the decode units still finish within its time.  Idle clusters
  // leave at once.
  const int pairs = p.counts[2] * p.L;
  const bool beside_tensor = p.counts[3] > 0 && 4LL * p.counts[3] >= pairs;
  int n_clusters = (int)num_clusters_x();
  if (beside_tensor) n_clusters = min(n_clusters, max(1, (pairs + 3) / 4));
  if ((int)cluster_id_x() >= n_clusters) return;  // every CTA of the cluster alike
  {
    int parts = 1;
    while (!p.u_rows && !beside_tensor && parts < 4 && pairs * parts * 2 <= n_clusters) parts *= 2;
    p.parts = parts;
  }
  const int n_units = p.counts[2] * p.L * p.parts;
  for (int u = tid; u < n_units && u < kDfClassCache; u += kDfThreads) cls_sh[u] = (int8_t)unit_class_global(p, u);
  __syncthreads();
  UnitIter it;
  unit_iter_init(it, p, cls_sh, n_units, n_clusters, lane);

  if (warp == kDfComputeWarps) {
    // ---------------- producer: per A page the group's x rows and the slot's
    // A tiles, then per chunk the B^T rank rows and the y rows, in the order
    // they are used.  All 32 lanes walk the units (the iterator's ballots) and
    // issue a page's copies together (lane g the copy of row g, lane 8 + i the
    // A tiles of the page's K block i, lane b B box b): one thread issuing
    // them in turn took ~0.1 µs a copy.  Lane 0 waits for the free page and
    // posts its bytes (a copy may land first: the count then goes below zero
    // until the post).
    uint32_t fill = 0;
    bool ok = true;
    auto next_page = [&](uint32_t bytes) -> uint8_t* {
      const int s = (int)(fill % npages);
      int good = 1;
      if (lane == 0) {
        if (fill >= npages && !mbar_wait_or_fail(&empty_bar[s], ((fill / npages) - 1) & 1, &fail_sh)) {
          fail_sh = 1;
          good = 0;
        } else {
          mbar_expect_tx(&full_bar[s], bytes);
        }
      }
      if (!__shfl_sync(0xffffffffu, good, 0)) {
        ok = false;
        return nullptr;
      }
      return ring + (size_t)s * kDfPageBytes;
    };
    int u;
    while (next_unit(it, p, cls_sh, lane, u)) {
      Unit U;
      if (ok && load_unit(p, u, cta, ncta, U)) {
        // this lane's row of the group (constant indexes: U.row stays in registers)
        int my_row = 0;
#pragma unroll
        for (int g = 0; g < kDecGroup; ++g)
          if (g == lane) my_row = U.row[g];
        for (int kb = U.kb0; kb < U.kb1 && ok; kb += U.nkbp) {
          const int n = min(U.nkbp, U.kb1 - kb);
          uint8_t* pg = next_page((uint32_t)(n * (U.nrows + U.r16) * 128));
          if (!pg) break;
          uint64_t* fb = &full_bar[fill % npages];
          ++fill;
          if (lane < U.nrows)
            bulk_load(pg + (size_t)lane * U.nkbp * 128, p.x + (size_t)my_row * p.ldx + (size_t)kb * 64,
                      (uint32_t)(n * 128), fb);
          // A tiles of K block i: one per power-of-two part of r16 (rows past
          // the rank are the pool's zero padding)
          const int i = lane - kDecGroup;
          if (i >= 0 && i < n) {
            uint8_t* ap = pg + (size_t)kDecGroup * U.nkbp * 128;
            int row = 0;
            for (int sz = kTmapSizes - 1; sz >= 0; --sz) {
              const int rows = 16 << sz;
              while (U.r16 - row >= rows) {
                tma_load_3d(ap + (size_t)(i * U.r16 + row) * 128, &tm_a.m[sz][U.l], (kb + i) * 64, row, U.k, fb);
                row += rows;
              }
            }
          }
        }
        for (int c0 = U.c0; c0 < U.c1 && ok && !p.u_rows; c0 += kDfCols) {
          const int ec = min(kDfCols, U.c1 - c0);
          const int nbox = (ec + U.bi - 1) / U.bi;
          for (int rb = 0; rb < U.r && ok; rb += kDfRanksPerPage) {
            // 16 rank rows x bi columns per TMA box (rows past the rank are
            // the pool's zero padding, columns past d_out read as zeros)
            uint8_t* bp = next_page((uint32_t)(nbox * kDfRanksPerPage * U.bi * 2));
            if (!bp) break;
            uint64_t* fb = &full_bar[fill % npages];
            ++fill;
            if (lane < nbox)
              tma_load_3d(bp + (size_t)lane * kDfRanksPerPage * U.bi * 2, &tm_bt.m[U.l], c0 + lane * U.bi, rb, U.k,
                          fb);
          }
          uint8_t* yp = ok ? next_page((uint32_t)(U.nrows * ec * 4)) : nullptr;
          if (!yp) break;
          uint64_t* fb = &full_bar[fill % npages];
          ++fill;
          if (lane < U.nrows)
            bulk_load(yp + (size_t)lane * kDfYPitch, p.y + (size_t)my_row * p.ldy + U.off + c0, (uint32_t)(ec * 4),
                      fb);
        }
      }
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
    }
    if (lane == 0) {
      // Copies already issued land before the CTA may leave (after a failure
      // the compute warps may not have waited for them): the latest fill of
      // every page, each a bounded wait.
      for (uint32_t f = fill > npages ? fill - npages : 0; f < fill; ++f)
        if (!mbar_wait_bounded(&full_bar[f % npages], (f / npages) & 1)) fail_sh = 1;
    }
  } else {
    // ---------------- compute warps
    const int t = tid;
    uint32_t use = 0, uj = 0, dj = 0;
    int u;
    while (next_unit(it, p, cls_sh, lane, u)) {
      Unit U;
      if (!load_unit(p, u, cta, ncta, U)) continue;
      // one stop decision per unit for all compute threads
      named_bar_sync(1, kDfCompute);
      if (t == 0) stop_sh[dj & 1] = fail_sh;
      named_bar_sync(1, kDfCompute);
      if (stop_sh[dj & 1]) break;
      ++dj;
      bool ok = true;
      const int par = (int)(uj & 1);
      float* rs = rsbuf + (size_t)par * part_floats;
      float* ag = agbuf + (size_t)par * part_floats;
      // this CTA expects every CTA's partial of this unit (st.async bytes)
      if (t == 0) {  // this CTA receives r16 x 8 floats in each of the two rounds
        mbar_expect_tx(&prs[par], (uint32_t)(U.r16 * kDecGroup * 4));
        mbar_expect_tx(&pag[par], (uint32_t)(U.r16 * kDecGroup * 4));
      }
      // ---- shrink of this CTA's K range: thread tile rtile rows x 4 ranks
      const int rtile = U.nrows <= 1 ? 1 : U.nrows <= 2 ? 2 : U.nrows <= 4 ? 4 : 8;
      const int rt = t / U.nks, ks = t - rt * U.nks;
      const bool active = rt * 4 < U.r16;
      float2 acc[kDecGroup][4];  // (even-K, odd-K) sums of A[4 rt + j] . x[row]
#pragma unroll
      for (int g = 0; g < kDecGroup; ++g)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[g][j] = make_float2(0.f, 0.f);
      for (int kb = U.kb0; kb < U.kb1; kb += U.nkbp, ++use) {
        const int s = (int)(use % npages);
        if (ok && !mbar_wait_or_fail(&full_bar[s], (use / npages) & 1, &fail_sh)) {
          ok = false;
          fail_sh = 1;
        }
        const int nq = min(U.nkbp, U.kb1 - kb) * 8;  // 8-element K chunks in this page
        if (ok && active) {
          const uint8_t* pg = ring + (size_t)s * kDfPageBytes;
          if (rtile == 1) shrink_page<1>(pg, U.nkbp, U.r16, rt, ks, U.nks, U.cpt, nq, acc);
          else if (rtile == 2) shrink_page<2>(pg, U.nkbp, U.r16, rt, ks, U.nks, U.cpt, nq, acc);
          else if (rtile == 4) shrink_page<4>(pg, U.nkbp, U.r16, rt, ks, U.nks, U.cpt, nq, acc);
          else shrink_page<8>(pg, U.nkbp, U.r16, rt, ks, U.nks, U.cpt, nq, acc);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);
      }
      // ---- the nks K splits of a rank tile: a fixed butterfly inside the
      // warp; then this CTA's partial goes to every CTA of the cluster
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
        if (active) {
          // reduce-scatter: rank i goes to the CTA owning its slice of r16 /
          // CL ranks, into that CTA's row for this source CTA
          const int slice = U.r16 / ncta;
          const uint32_t rs_a = smem_u32(rs), bar = smem_u32(&prs[par]);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            if (e < nout) {
              const int o = out0 + e, g = o >> 2, i = 4 * rt + (o & 3);
              const int dest = i / slice, li = i - dest * slice;
              st_async_f32(mapa_shared(rs_a + 4u * (uint32_t)((cta * slice + li) * kDecGroup + g), (uint32_t)dest),
                           v[e], mapa_shared(bar, (uint32_t)dest));
            }
          }
        }
      }
      // ---- u of this CTA's rank slice = the sum of the CL partials in CTA
      // order (one thread waits for the bytes, then releases the others);
      // then all-gather: the slice to every CTA of the cluster
      if (t == 0) {
        const bool got = mbar_wait_or_fail(&prs[par], (uj >> 1) & 1, &fail_sh);
        if (!got) fail_sh = 1;
        xok_sh[par] = got ? 1 : 0;
      }
      named_bar_sync(1, kDfCompute);
      if (!xok_sh[par]) ok = false;
      if (ok) {
        const int n_el = (U.r16 / ncta) * kDecGroup;
        const uint32_t ag_a = smem_u32(ag) + 4u * (uint32_t)(cta * n_el), bar = smem_u32(&pag[par]);
        for (int idx = t; idx < n_el; idx += kDfCompute) {
          float sum = rs[idx];
          for (int c = 1; c < ncta; ++c) sum += rs[(size_t)c * n_el + idx];
          for (int c = 0; c < ncta; ++c)
            st_async_f32(mapa_shared(ag_a + 4u * (uint32_t)idx, (uint32_t)c), sum, mapa_shared(bar, (uint32_t)c));
        }
      }
      if (t == 0) {
        const bool got = ok && mbar_wait_or_fail(&pag[par], (uj >> 1) & 1, &fail_sh);
        if (ok && !got) fail_sh = 1;
        xag_sh[par] = got ? 1 : 0;
      }
      ++uj;
      named_bar_sync(1, kDfCompute);  // u complete
      if (!xag_sh[par]) ok = false;
      if (p.u_rows) {  // row mode: scale * u of the group's rows, written once (by CTA 0)
        if (ok && cta == 0) {
          const float sc = p.scale_tab[U.k * p.L + U.l];
#pragma unroll
          for (int g = 0; g < kDecGroup; ++g) {
            if (g < U.nrows) {
              float* dst = p.u_rows + ((size_t)U.row[g] * p.L + U.l) * p.R16;
              for (int i = t; i < U.r16; i += kDfCompute) dst[i] = sc * ag[i * kDecGroup + g];
            }
          }
        }
        continue;
      }
      // ---- expand of this CTA's columns: thread tile rtile rows x 4 columns
      const float sc = p.scale_tab[U.k * p.L + U.l];
      // this thread's columns 4t..4t+3 of a chunk sit in TMA box 4t / bi of a B page
      const int b_box = (kDfColsPerThread * t) / U.bi;
      const int b_off = b_box * kDfRanksPerPage * U.bi * 2 + ((kDfColsPerThread * t) - b_box * U.bi) * 2;
      for (int c0 = U.c0; c0 < U.c1; c0 += kDfCols) {
        const int ec = min(kDfCols, U.c1 - c0);
        const bool has = kDfColsPerThread * t < ec;
        float2 eacc[kDecGroup][2];  // columns (4t, 4t+1) and (4t+2, 4t+3) of each row
#pragma unroll
        for (int g = 0; g < kDecGroup; ++g) eacc[g][0] = eacc[g][1] = make_float2(0.f, 0.f);
        for (int rb = 0; rb < U.r; rb += kDfRanksPerPage, ++use) {
          const int s = (int)(use % npages);
          if (ok && !mbar_wait_or_fail(&full_bar[s], (use / npages) & 1, &fail_sh)) {
            ok = false;
            fail_sh = 1;
          }
          if (ok && has) {
            const uint8_t* bp = ring + (size_t)s * kDfPageBytes + b_off;
            const int nr = min(kDfRanksPerPage, U.r - rb);
            if (rtile == 1) expand_page<1>(bp, 2 * U.bi, ag, rb, nr, eacc);
            else if (rtile == 2) expand_page<2>(bp, 2 * U.bi, ag, rb, nr, eacc);
            else if (rtile == 4) expand_page<4>(bp, 2 * U.bi, ag, rb, nr, eacc);
            else expand_page<8>(bp, 2 * U.bi, ag, rb, nr, eacc);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty_bar[s]);
        }
        // the y page (streamed after the chunk's B pages): y = fma(scale, v, y)
        {
          const int s = (int)(use % npages);
          if (ok && !mbar_wait_or_fail(&full_bar[s], (use / npages) & 1, &fail_sh)) {
            ok = false;
            fail_sh = 1;
          }
          if (ok && has) {
            const uint8_t* yp = ring + (size_t)s * kDfPageBytes + 16 * t;
#pragma unroll
            for (int g = 0; g < kDecGroup; ++g) {
              if (g < U.nrows) {
                float4 a = *reinterpret_cast<const float4*>(yp + (size_t)g * kDfYPitch);
                a.x = fmaf(sc, eacc[g][0].x, a.x);
                a.y = fmaf(sc, eacc[g][0].y, a.y);
                a.z = fmaf(sc, eacc[g][1].x, a.z);
                a.w = fmaf(sc, eacc[g][1].y, a.w);
                *reinterpret_cast<float4*>(p.y + (size_t)U.row[g] * p.ldy + U.off + c0 + kDfColsPerThread * t) = a;
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty_bar[s]);
          ++use;
        }
      }
    }
  }
  // no CTA leaves while another CTA of its cluster may still store into it
  cluster_sync_all();
  if (tid == 0 && fail_sh) set_error(p.status, LORA_ERR_TIMEOUT);
}

// Upper bound of decode groups for the last build: sum_k ceil(cnt_k / G) <= T/G + min(N, T).
int dec_group_bound(const PoolView& pool, const lora_segments* seg) {
  const int T = seg->T;
  return ceil_div(T, kDecGroup) + (pool.N < T ? pool.N : T);
}

// CTAs per cluster: a function of d_in only, so a row's K split, and with it
// its bits, depends neither on the batch nor on the pool's rank padding.
int cluster_size(const PoolView& pool) {
  const int nkb = pool.d_in / 64;
  return nkb >= 128 ? 8 : nkb >= 4 ? 4 : (nkb >= 2 ? 2 : 1);
}

// Ring pages: as many 18 KB pages as the shared memory left to each of the
// kDfCtasPerSm CTAs of an SM holds after the receive buffers (deep rings keep
// more bytes in flight per CTA; a page round trip is a few microseconds).
int dec_pages(const PoolView& pool, int ncta) {
  static std::atomic<int> static_smem{-1};
  int st = static_smem.load(std::memory_order_relaxed);
  if (st < 0) {
    cudaFuncAttributes fa;
    st = cudaFuncGetAttributes(&fa, reinterpret_cast<const void*>(dec_fused_kernel)) == cudaSuccess
             ? (int)fa.sharedSizeBytes
             : 8192;
    static_smem.store(st, std::memory_order_relaxed);
  }
  // per-SM shared memory 228 KiB, 1 KiB of it reserved per resident CTA; at
  // most 227 KiB per CTA
  long long per_cta = 233472 / kDfCtasPerSm - 1024;
  if (per_cta > 232448) per_cta = 232448;
  const long long recv = 4LL * pool.R16 * kDecGroup * 4;  // exchange buffers: two rounds x two parities
  const long long pages = (per_cta - st - 1024 - recv) / kDfPageBytes;
  return (int)(pages < kDfMaxPages ? pages : kDfMaxPages);
}

size_t dec_smem_bytes(const PoolView& pool, int ncta, int npages) {
  return 1024 + (size_t)npages * kDfPageBytes + (size_t)4 * pool.R16 * kDecGroup * 4;
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

namespace {
int decode_impl(const PoolView& pool, const lora_segments* seg, const uint16_t* x, int64_t ldx, float* y,
                int64_t ldy, float* u_rows, cudaStream_t st) {
  // units: (group, lane) pairs, each in up to 4 column parts (one in row mode)
  const long long units = (long long)dec_group_bound(pool, seg) * pool.L * (u_rows ? 1 : 4);
  if (units <= 0) return LORA_OK;
  const int ncta = cluster_size(pool);
  const int npages = dec_pages(pool, ncta);
  if (npages < 3) return LORA_ERR_SHAPE;
  const size_t smem = dec_smem_bytes(pool, ncta, npages);
  if (!set_smem_limit(reinterpret_cast<const void*>(dec_fused_kernel), pool.device, (int)smem)) return LORA_ERR_CUDA;
  // Persistent clusters: as many as can be resident at once (each takes its
  // share of the units), never more than there can be units.
  const long long cap = max_active_clusters(pool.device, ncta, smem);
  const int clusters = (int)(units < cap ? units : cap);
  DfParams p{};
  p.counts = seg->counts;
  p.work = seg->dec_work;
  p.dec_rows = reinterpret_cast<const int4*>(seg->dec_rows);
  p.rank_tab = pool.rank_tab;
  p.scale_tab = pool.scale_tab;
  p.status = seg->status;
  for (int l = 0; l < LORA_MAX_LANES; ++l) {
    p.d_out[l] = pool.d_out[l];
    p.off[l] = pool.off[l];
    p.bt_cols[l] = bt_box_cols(pool.d_out[l] > 0 ? pool.d_out[l] : 64);
  }
  p.x = x;
  p.ldx = ldx;
  p.y = y;
  p.ldy = ldy;
  p.u_rows = u_rows;
  p.L = pool.L;
  p.R16 = pool.R16;
  p.nkb = pool.d_in / 64;
  p.npages = npages;
  p.n_tab = pool.N * pool.L;
  p.parts = 1;
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
  const cudaError_t e = cudaLaunchKernelEx(&cfg, dec_fused_kernel, pool.tm_a, pool.tm_bt, p);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cuda_status(e != cudaSuccess ? e : cudaGetLastError(), "dec_fused_kernel launch");
}
}  // namespace

int launch_decode(const PoolView& pool, const lora_segments* seg, const uint16_t* x, int64_t ldx, float* y,
                  int64_t ldy, cudaStream_t st) {
  return decode_impl(pool, seg, x, ldx, y, ldy, nullptr, st);
}

int launch_decode_rows(const PoolView& pool, const lora_segments* seg, const uint16_t* x, int64_t ldx,
                       cudaStream_t st) {
  return decode_impl(pool, seg, x, ldx, nullptr, 0, pool.u_rows, st);
}

}  // namespace lora
