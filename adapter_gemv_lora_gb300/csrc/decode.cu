// Decode path: rows whose own sequence is shorter than LORA_TC_MIN_QLEN
// (single-token decode rows, short chunks).  Rows are grouped by slot (up to
// LORA_DEC_GROUP_ROWS rows of one slot per group), so a slot's factors are
// streamed once per group and shared by the group's rows.
//
//   shrink  u[row][i] = sum_j A[k][l][i][j] * x[row][j]     (TensorFold PR #47,
//   expand  y[row][o] += scale[k][l] * sum_i B[k][l][o][i] * u[row][i]   the delta
//           scale * B @ (A @ x); xLLM PR #2014, shrink then expand)
//
// Both kernels are HBM streams of factor rows: a producer warp copies the
// slot's rank rows (A rows for the shrink, the true rank rounded up to 4;
// B^T rows for the expand, the true rank) with the TMA bulk-copy engine into
// a ring of shared-memory stages, and the compute warps consume them with
// 128-bit shared loads.  The group's x rows (shrink, converted once to fp32)
// and u vectors (expand) stay in shared memory for the whole stream.
//
// Fixed summation order, independent of the group a row lands in:
//  * shrink: d_in is cut into 1024-wide chunks (one work item each).  The
//    slot's rank rows are taken in blocks of up to 32, each block in groups
//    of 4 (nig groups, a power of two); the chunk's 8-element K blocks are
//    dealt to nks = 128 / nig K splits: split s takes blocks s, s + nks, ....
//    In each block the even and the odd elements feed two fma chains, added
//    when the chunk is done; the splits are then combined by a fixed xor
//    butterfly over the lanes of a warp and, where a group spans several
//    warps, the warps left to right.  The chunks' partial sums go to the
//    pool's scratch and the expand kernel adds them in chunk order.
//  * expand: u is the in-order sum of the chunk partials; v[o] accumulates
//    B[o][i] * u[i] for i = 0..r-1 in order with fma; y = fma(scale, v, y).
//    Each compute thread owns 4 consecutive output columns of the group's rows.
// The fmas are issued two at a time (packed f32x2), each exactly an fmaf in
// the order above; which CTA or work item handles a row never changes it.
#include <cuda_runtime.h>

#include "device.cuh"
#include "internal.h"

namespace lora {
namespace {

constexpr int kShWarps = 4;                      // shrink compute warps
constexpr int kShThreads = (kShWarps + 1) * 32;  // + 1 producer warp
constexpr int kShCompute = kShWarps * 32;        // compute threads: rank groups x K splits
constexpr int kShStageBytes = 32768;             // A rows of one ring stage
constexpr int kShStages = 2;
constexpr size_t kShRingBytes = (size_t)kShStages * kShStageBytes;          // 64 KB
constexpr size_t kShXBytes = (size_t)kDecGroup * kDecKChunk * 2;            // 16 KB, the item's x rows (bf16)
constexpr size_t kShXfBytes = (size_t)kDecGroup * kDecKChunk * 4;           // 32 KB, the same rows in fp32
constexpr int kShRankBlock = 32;                 // rank rows per thread-tile pass
static_assert(kShCompute == 128 && kDecKChunk / 8 == kShCompute, "thread tiles: 128 threads, one K block each");
static_assert(kShRankBlock * 512 * 2 <= kShStageBytes, "a 32-row block streams 512-element stages");

constexpr int kExWarps = 8;                      // expand compute warps (4 columns per thread)
constexpr int kExThreads = (kExWarps + 1) * 32;
constexpr int kExCols = 4;                       // output columns per compute thread
constexpr int kExRows = 16;                      // rank rows per ring stage
constexpr int kExStages = 3;
constexpr size_t kExRingBytes = (size_t)kExStages * kExRows * kDecNChunk * 2;  // 96 KB
static_assert(kExWarps * 32 * kExCols == kDecNChunk, "the compute threads cover a chunk");

struct DecParams {
  const int32_t* counts;
  const int4* work;
  const int4* dec_rows;  // [group][2]: the group's 8 row indexes (entries past its row count unused)
  const int32_t* perm;
  const int32_t* rank_tab;
  const float* scale_tab;
  int32_t* status;
  const uint16_t* A[LORA_MAX_LANES];
  const uint16_t* Bt[LORA_MAX_LANES];
  float* u_dec;
  int32_t* sched;  // [2] the shrink's next-item and finished-CTA counters
  const uint16_t* x;
  int64_t ldx;
  float* y;
  int64_t ldy;
  int L, R16, d_in, C, max_tokens;
  int d_out[LORA_MAX_LANES], off[LORA_MAX_LANES];
  int nc_base[LORA_MAX_LANES + 1];
};

// Element l of a per-lane parameter array, read with constant indexes.
template <typename V>
__device__ __forceinline__ V lane_param(const V (&a)[LORA_MAX_LANES], int l) {
  V v = a[0];
#pragma unroll
  for (int i = 1; i < LORA_MAX_LANES; ++i)
    if (l == i) v = a[i];
  return v;
}

// Work items of the shrink are handed out dynamically: every CTA starts with
// item blockIdx.x and then takes tickets gridDim.x, gridDim.x + 1, ... from a
// counter (item costs differ with the rank of their slot, so a fixed
// round-robin split leaves some CTAs with several times the work of others).
// The CTA that finishes last resets the counters to zero for the next launch;
// which CTA runs an item never changes its result.
__device__ __forceinline__ int next_item(int32_t* ctr) { return (int)gridDim.x + atomicAdd(ctr, 1); }

__device__ __forceinline__ void finish_items(int32_t* ctr, int participants) {
  __threadfence();  // this CTA's last ticket is taken before it counts itself out
  if (atomicAdd(ctr + 1, 1) == participants - 1) {
    ctr[0] = 0;
    ctr[1] = 0;
  }
}

// Expand items cover `ncb` consecutive 1024-column blocks of one lane, so the
// group's u (the sum of the shrink's chunk partials) is formed once per ncb
// blocks.  ncb is the largest of 1, 2, 4 that still leaves every CTA of the
// grid at least two items; it depends on the step's real number of decode
// groups, so every CTA computes the same value.  Results do not depend on it.
struct ExGeom {
  int ncb, total, base[LORA_MAX_LANES + 1];  // items per lane start at base[l]
};

__device__ __forceinline__ ExGeom ex_geom(const DecParams& p, int n_groups) {
  ExGeom g;
  g.ncb = 1;
  for (int cand = 2; cand <= 4; cand *= 2) {
    int per_group = 0;
#pragma unroll
    for (int l = 0; l < LORA_MAX_LANES; ++l)
      if (l < p.L) per_group += (p.nc_base[l + 1] - p.nc_base[l] + cand - 1) / cand;
    if ((long long)n_groups * per_group >= 2LL * gridDim.x) g.ncb = cand;
  }
  g.base[0] = 0;
#pragma unroll
  for (int l = 0; l < LORA_MAX_LANES; ++l)
    g.base[l + 1] = g.base[l] + (l < p.L ? (p.nc_base[l + 1] - p.nc_base[l] + g.ncb - 1) / g.ncb : 0);
  g.total = g.base[LORA_MAX_LANES];
  return g;
}

// Lane, first column, width and y offset of expand item column range q.
__device__ __forceinline__ void pick_item_lane(const DecParams& p, const ExGeom& g, int q, int& l, int& n0, int& dout,
                                               int& off) {
  l = 0;
  n0 = q * g.ncb * kDecNChunk;
  dout = p.d_out[0];
  off = p.off[0];
#pragma unroll
  for (int i = 1; i < LORA_MAX_LANES; ++i) {
    if (i < p.L && q >= g.base[i]) {
      l = i;
      n0 = (q - g.base[i]) * g.ncb * kDecNChunk;
      dout = p.d_out[i];
      off = p.off[i];
    }
  }
}

// Thread tiles of a shrink item.  Its rank rows are taken in blocks of up to
// 32 (rb_rows, a multiple of 4; rows past r read the pool's zero padding),
// each block streamed over the item's K chunk in ring stages of rb_rows x kst
// elements.  Inside a block the rows form nig groups of 4 (a power of two)
// and the chunk's 8-element K blocks are dealt to nks = 128 / nig K splits:
// compute thread t takes group t / nks and the K blocks t % nks, t % nks +
// nks, ... .  The nks splits of a group sit in one warp (nks <= 32) or in
// nks / 32 consecutive warps.
struct ShGeom {
  int rows, nig, nks, kst, kbps;
};

__device__ __forceinline__ ShGeom sh_geom(int r4, int rb) {
  ShGeom g;
  g.rows = min(kShRankBlock, r4 - rb * kShRankBlock);
  g.nig = 1;
  while (g.nig * 4 < g.rows) g.nig *= 2;
  g.nks = kShCompute / g.nig;
  g.kst = min(kDecKChunk, kShStageBytes / (8 * g.nig));  // rows x kst bf16 <= one stage
  g.kbps = (g.kst / 8) / g.nks;                          // K blocks per thread per stage
  return g;
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

__global__ void __launch_bounds__(kShThreads, 2) dec_shrink_kernel(DecParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint16_t* ring = reinterpret_cast<uint16_t*>(smem);                        // [stage][rows][kst]
  uint16_t* xbuf = reinterpret_cast<uint16_t*>(smem + kShRingBytes);         // [row][kDecKChunk] bf16
  const float4* xf = reinterpret_cast<const float4*>(smem + kShRingBytes + kShXBytes);  // [row][half][K block]
  float4* xfw = reinterpret_cast<float4*>(smem + kShRingBytes + kShXBytes);
  __shared__ __align__(8) uint64_t full_bar[kShStages], empty_bar[kShStages], xfull, xempty;
  __shared__ int4 sitem;  // {rank | rows << 8 | lane << 16 (0 = no more items), K chunk, first perm row, -}
  __shared__ float wsum[kShWarps][32];  // per-warp sums when a rank group spans several warps
  __shared__ int stop_sh[2];            // per item parity: the compute warps leave the loop
  __shared__ int fail_sh;

  pdl_wait();  // the previous kernel's results are visible from here on
  const int status = *p.status, n_groups = p.counts[2];  // both loads in flight together
  // a timeout is the only status another kernel can raise while this one runs;
  // every CTA of the grid takes part in the item counting whatever it reads
  if (status != 0 && status != LORA_ERR_TIMEOUT) return;
  const int per_group = p.L * p.C;
  const int n_items = n_groups * per_group;
  if ((int)blockIdx.x >= n_items) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int s = 0; s < kShStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kShWarps);
    }
    mbar_init(&xfull, 1);
    mbar_init(&xempty, 1);
    fail_sh = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kShWarps) {
    // ---------------- producer: per item, the group's x rows of its K chunk, then the slot's A rows
    if (lane == 0) {
      uint32_t fill = 0, xj = 0;
      int item = blockIdx.x;
      for (;;) {
        int r = 0, l = 0, c = 0;
        int4 g = make_int4(0, 0, 0, 0), rw0 = g, rw1 = g;
        for (; item < n_items; item = next_item(p.sched)) {  // items of a rank-0 lane do nothing
          const int w = item / per_group, rem = item - w * per_group;
          l = rem / p.C;
          c = rem - l * p.C;
          g = p.work[w];  // the group and its rows load together; the rank follows the group
          rw0 = p.dec_rows[2 * w];
          rw1 = p.dec_rows[2 * w + 1];
          r = p.rank_tab[g.x * p.L + l];
          if (r > 0) break;
        }
        if (xj >= 1 && !mbar_wait_or_fail(&xempty, (xj - 1) & 1, &fail_sh)) {
          fail_sh = 1;
          break;
        }
        if (item >= n_items) {  // no more items: an empty item tells the compute warps
          sitem = make_int4(0, 0, 0, 0);
          mbar_arrive(&xfull);
          break;
        }
        const int k0 = c * kDecKChunk, klen = min(kDecKChunk, p.d_in - k0);
        const int nrows = g.z - g.y;
        sitem = make_int4(r | (nrows << 8) | (l << 16), c, g.y, 0);
        const int row[kDecGroup] = {rw0.x, rw0.y, rw0.z, rw0.w, rw1.x, rw1.y, rw1.z, rw1.w};
        mbar_expect_tx(&xfull, (uint32_t)(nrows * klen * 2));
#pragma unroll
        for (int gg = 0; gg < kDecGroup; ++gg)
          if (gg < nrows)
            bulk_load(xbuf + (size_t)gg * kDecKChunk, p.x + (size_t)row[gg] * p.ldx + k0, (uint32_t)(klen * 2), &xfull);
        ++xj;
        const int r4 = (r + 3) & ~3;
        const uint16_t* Ab = lane_param(p.A, l) + (size_t)g.x * p.R16 * p.d_in + k0;
        bool ok = true;
        for (int rb = 0; rb * kShRankBlock < r4 && ok; ++rb) {
          const ShGeom sg = sh_geom(r4, rb);
          const uint16_t* Arb = Ab + (size_t)rb * kShRankBlock * p.d_in;
          for (int ks0 = 0; ks0 < klen; ks0 += sg.kst, ++fill) {
            const int s = fill % kShStages;
            if (fill >= kShStages && !mbar_wait_or_fail(&empty_bar[s], ((fill / kShStages) - 1) & 1, &fail_sh)) {
              ok = false;
              fail_sh = 1;
              break;
            }
            const int kl = min(sg.kst, klen - ks0);
            mbar_expect_tx(&full_bar[s], (uint32_t)(sg.rows * kl * 2));
            uint16_t* dst = ring + (size_t)s * (kShStageBytes / 2);
            for (int i = 0; i < sg.rows; ++i)
              bulk_load(dst + (size_t)i * sg.kst, Arb + (size_t)i * p.d_in + ks0, (uint32_t)(kl * 2), &full_bar[s]);
          }
        }
        if (!ok) break;
        item = next_item(p.sched);
      }
      finish_items(p.sched, min((int)gridDim.x, n_items));
    }
  } else {
    // ---------------- compute warps
    uint32_t use = 0, xj = 0;
    const int t = tid;
    for (;;) {
      if (!mbar_wait_or_fail(&xfull, xj & 1, &fail_sh)) fail_sh = 1;
      const int4 it = sitem;
      named_bar_sync(1, kShCompute);  // every compute thread has waited (failures recorded)
      if (t == 0) stop_sh[xj & 1] = fail_sh || (it.x & 0xff) == 0;  // a failure, or no more items
      named_bar_sync(1, kShCompute);  // one decision for all compute threads
      if (stop_sh[xj & 1]) break;
      const int r = it.x & 0xff, nrows = (it.x >> 8) & 0xff, l = it.x >> 16, c = it.y, p0 = it.z;
      const int klen = min(kDecKChunk, p.d_in - c * kDecKChunk);
      // x rows to fp32, split into the two halves of each 8-element K block so
      // that the fma loop reads consecutive 16-byte words across threads
#pragma unroll
      for (int gg = 0; gg < kDecGroup; ++gg) {
        float v[8];
        unpack8(*reinterpret_cast<const uint4*>(xbuf + (size_t)gg * kDecKChunk + 8 * t), v);
        xfw[(gg * 2 + 0) * (kDecKChunk / 8) + t] = make_float4(v[0], v[1], v[2], v[3]);
        xfw[(gg * 2 + 1) * (kDecKChunk / 8) + t] = make_float4(v[4], v[5], v[6], v[7]);
      }
      named_bar_sync(1, kShCompute);  // fp32 rows complete; the bf16 buffer may be refilled
      if (t == 0) mbar_arrive(&xempty);
      ++xj;
      const int r4 = (r + 3) & ~3;
      bool ok = true;
      for (int rb = 0; rb * kShRankBlock < r4; ++rb) {
        const ShGeom sg = sh_geom(r4, rb);
        const int ig = t / sg.nks, ks = t - ig * sg.nks;
        const bool active = ig * 4 < sg.rows;
        // acc[row][j] = (sum over even k, sum over odd k) of A[4 ig + j][k] * x[row][k]
        float2 acc[kDecGroup][4];
#pragma unroll
        for (int gg = 0; gg < kDecGroup; ++gg)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[gg][j] = make_float2(0.f, 0.f);
        for (int ks0 = 0; ks0 < klen; ks0 += sg.kst, ++use) {
          const int s = use % kShStages;
          if (!mbar_wait_or_fail(&full_bar[s], (use / kShStages) & 1, &fail_sh)) {
            ok = false;
            fail_sh = 1;
          }
          if (ok && active) {
            const int kl = min(sg.kst, klen - ks0);
            const uint16_t* As = ring + (size_t)s * (kShStageBytes / 2) + (size_t)(4 * ig) * sg.kst;
            for (int jb = 0; jb < sg.kbps; ++jb) {
              const int kloc = 8 * (ks + jb * sg.nks);
              if (kloc >= kl) break;
              float2 a[4][4];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const uint4 q = *reinterpret_cast<const uint4*>(As + (size_t)j * sg.kst + kloc);
                a[j][0] = make_float2(bf16lo(q.x), bf16hi(q.x));
                a[j][1] = make_float2(bf16lo(q.y), bf16hi(q.y));
                a[j][2] = make_float2(bf16lo(q.z), bf16hi(q.z));
                a[j][3] = make_float2(bf16lo(q.w), bf16hi(q.w));
              }
              const int kb = (ks0 + kloc) >> 3;
#pragma unroll
              for (int gg = 0; gg < kDecGroup; ++gg) {
                const float4 x0 = xf[(gg * 2 + 0) * (kDecKChunk / 8) + kb];
                const float4 x1 = xf[(gg * 2 + 1) * (kDecKChunk / 8) + kb];
                const float2 xp[4] = {make_float2(x0.x, x0.y), make_float2(x0.z, x0.w), make_float2(x1.x, x1.y),
                                      make_float2(x1.z, x1.w)};
#pragma unroll
                for (int e = 0; e < 4; ++e)
#pragma unroll
                  for (int j = 0; j < 4; ++j) acc[gg][j] = ffma2(a[j][e], xp[e], acc[gg][j]);
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty_bar[s]);
        }
        // the K splits' sums: a fixed butterfly over the lanes of a group, then
        // (groups spanning several warps) the warps in order
        float v[32];  // index row * 4 + j
#pragma unroll
        for (int gg = 0; gg < kDecGroup; ++gg)
#pragma unroll
          for (int j = 0; j < 4; ++j) v[gg * 4 + j] = acc[gg][j].x + acc[gg][j].y;
        int out0, nout;  // this lane's outputs: v[0 .. nout) are outputs out0, out0 + 1, ...
        if (sg.nks == 16) {
          rs_step<16>(v, lane, 8);
          rs_step<8>(v, lane, 4);
          rs_step<4>(v, lane, 2);
          rs_step<2>(v, lane, 1);
          out0 = 2 * (lane & 15);
          nout = 2;
        } else {
          rs_step<16>(v, lane, 16);
          rs_step<8>(v, lane, 8);
          rs_step<4>(v, lane, 4);
          rs_step<2>(v, lane, 2);
          rs_step<1>(v, lane, 1);
          out0 = lane;
          nout = 1;
        }
        bool writer = true;
        if (sg.nks > 32) {
          const int wpg = sg.nks / 32;  // warps per rank group
          wsum[warp][lane] = v[0];
          named_bar_sync(1, kShCompute);
          writer = warp % wpg == 0;
          if (writer) {
            float sum = wsum[warp][lane];
            for (int ww = 1; ww < wpg; ++ww) sum += wsum[warp + ww][lane];
            v[0] = sum;
          }
          named_bar_sync(1, kShCompute);  // wsum is read before the next block writes it
        }
        if (ok && writer) {
          for (int e = 0; e < nout; ++e) {
            const int o = out0 + e, gg = o >> 2, i = rb * kShRankBlock + 4 * ig + (o & 3);
            if (gg < nrows && i < r) p.u_dec[(((size_t)c * p.max_tokens + p0 + gg) * p.L + l) * p.R16 + i] = v[e];
          }
        }
      }
    }
  }
  __syncthreads();
  if (tid == 0 && fail_sh) set_error(p.status, LORA_ERR_TIMEOUT);
}

__global__ void __launch_bounds__(kExThreads, 2) dec_expand_kernel(DecParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint16_t* ring = reinterpret_cast<uint16_t*>(smem);  // [stage][row][kDecNChunk]
  __shared__ __align__(16) float us[128][kDecGroup];   // [rank][row]
  __shared__ __align__(8) uint64_t full_bar[kExStages], empty_bar[kExStages];
  __shared__ int fail_sh;

  pdl_wait();  // the previous kernel's results are visible from here on
  const int status = *p.status, n_groups = p.counts[2];  // both loads in flight together
  if (status != 0) return;
  const ExGeom geom = ex_geom(p, n_groups);
  const int total_nc = geom.total;
  const int n_items = n_groups * total_nc;
  if ((int)blockIdx.x >= n_items) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int s = 0; s < kExStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kExWarps);
    }
    fail_sh = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const size_t cstride = (size_t)p.max_tokens * p.L * p.R16;

  if (warp == kExWarps) {
    // ---------------- producer: stream the slot's B^T rows of this column chunk
    if (lane == 0) {
      uint32_t fill = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        const int w = item / total_nc, q = item - w * total_nc;
        int l, n0, dout, off;
        pick_item_lane(p, geom, q, l, n0, dout, off);
        const int k = p.work[w].x;
        const int r = p.rank_tab[k * p.L + l];
        if (r <= 0) continue;
        for (int nb = n0; nb < min(dout, n0 + geom.ncb * kDecNChunk) && ok; nb += kDecNChunk) {
          const int ncols = min(kDecNChunk, dout - nb);
          const uint16_t* Bb = lane_param(p.Bt, l) + (size_t)k * p.R16 * dout + nb;
          for (int rb = 0; rb < r; rb += kExRows, ++fill) {
            const int s = fill % kExStages;
            if (fill >= kExStages && !mbar_wait_or_fail(&empty_bar[s], ((fill / kExStages) - 1) & 1, &fail_sh)) {
              ok = false;
              fail_sh = 1;
              break;
            }
            const int rows = min(kExRows, r - rb);
            mbar_expect_tx(&full_bar[s], (uint32_t)(rows * ncols * 2));
            for (int i = 0; i < rows; ++i)
              bulk_load(ring + ((size_t)s * kExRows + i) * kDecNChunk, Bb + (size_t)(rb + i) * dout,
                        (uint32_t)(ncols * 2), &full_bar[s]);
          }
        }
      }
    }
  } else {
    // ---------------- compute warps: kExCols output columns per thread
    uint32_t use = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
      const int w = item / total_nc, q = item - w * total_nc;
      int l, n0, dout, off;
      pick_item_lane(p, geom, q, l, n0, dout, off);
      const int4 g = p.work[w];
      const int k = g.x, p0 = g.y, nrows = g.z - g.y;
      const int r = p.rank_tab[k * p.L + l];
      if (r <= 0) continue;
      named_bar_sync(1, kExWarps * 32);  // us of the previous item are no longer read
      for (int idx = tid; idx < r * kDecGroup; idx += kExWarps * 32) {
        const int i = idx >> 3, gg = idx & 7;
        float s = 0.f;
        if (gg < nrows) {
          const float* u = p.u_dec + ((size_t)(p0 + gg) * p.L + l) * p.R16 + i;
          s = u[0];
          int c = 1;
          for (; c + 8 <= p.C; c += 8) {  // eight loads in flight, added in chunk order
            float v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = u[(size_t)(c + j) * cstride];
#pragma unroll
            for (int j = 0; j < 8; ++j) s += v[j];
          }
          for (; c < p.C; ++c) s += u[(size_t)c * cstride];
        }
        us[i][gg] = s;
      }
      named_bar_sync(1, kExWarps * 32);
      const float sc = p.scale_tab[k * p.L + l];
      for (int nb = n0; nb < min(dout, n0 + geom.ncb * kDecNChunk) && ok; nb += kDecNChunk) {
        const int o = nb + kExCols * tid;
        const bool has = o < dout;
        float4 yv[kDecGroup];
        float* const ycol = p.y + off + o;
#pragma unroll
        for (int gg = 0; gg < kDecGroup; ++gg)
          if (has && gg < nrows) yv[gg] = *reinterpret_cast<const float4*>(ycol + (size_t)p.perm[p0 + gg] * p.ldy);
        float2 acc[kDecGroup][kExCols / 2];  // columns (2c, 2c+1) of row gg
#pragma unroll
        for (int gg = 0; gg < kDecGroup; ++gg)
#pragma unroll
          for (int e = 0; e < kExCols / 2; ++e) acc[gg][e] = make_float2(0.f, 0.f);
        const int nrb = (r + kExRows - 1) / kExRows;
        for (int rb = 0; rb < nrb; ++rb, ++use) {
          const int s = use % kExStages;
          if (ok && !mbar_wait_or_fail(&full_bar[s], (use / kExStages) & 1, &fail_sh)) {
            ok = false;
            fail_sh = 1;
          }
          if (ok && has) {
            const uint16_t* st = ring + (size_t)s * kExRows * kDecNChunk + kExCols * tid;
#pragma unroll 4
            for (int i = 0; i < kExRows; ++i) {
              const int ri = rb * kExRows + i;
              if (ri < r) {
                const uint2 q2 = *reinterpret_cast<const uint2*>(st + (size_t)i * kDecNChunk);
                const float2 b01 = make_float2(bf16lo(q2.x), bf16hi(q2.x));
                const float2 b23 = make_float2(bf16lo(q2.y), bf16hi(q2.y));
                const float4 u0 = *reinterpret_cast<const float4*>(&us[ri][0]);
                const float4 u1 = *reinterpret_cast<const float4*>(&us[ri][4]);
                const float ug[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
                for (int gg = 0; gg < kDecGroup; ++gg) {
                  const float2 u2 = make_float2(ug[gg], ug[gg]);
                  acc[gg][0] = ffma2(b01, u2, acc[gg][0]);
                  acc[gg][1] = ffma2(b23, u2, acc[gg][1]);
                }
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty_bar[s]);
        }
        if (!ok || !has) continue;
#pragma unroll
        for (int gg = 0; gg < kDecGroup; ++gg) {
          if (gg < nrows) {
            float4 a = yv[gg];
            a.x = fmaf(sc, acc[gg][0].x, a.x);
            a.y = fmaf(sc, acc[gg][0].y, a.y);
            a.z = fmaf(sc, acc[gg][1].x, a.z);
            a.w = fmaf(sc, acc[gg][1].y, a.w);
            *reinterpret_cast<float4*>(ycol + (size_t)p.perm[p0 + gg] * p.ldy) = a;
          }
        }
      }
    }
  }
  __syncthreads();
  if (tid == 0 && fail_sh) set_error(p.status, LORA_ERR_TIMEOUT);
}

DecParams make_params(const lora_pool* pool, const lora_segments* seg) {
  DecParams p{};
  p.counts = seg->counts;
  p.work = seg->dec_work;
  p.dec_rows = reinterpret_cast<const int4*>(seg->dec_rows);
  p.perm = seg->perm;
  p.status = seg->status;
  p.rank_tab = pool->rank_tab;
  p.scale_tab = pool->scale_tab;
  for (int l = 0; l < LORA_MAX_LANES; ++l) {
    p.A[l] = pool->A[l];
    p.Bt[l] = pool->Bt[l];
    p.d_out[l] = pool->d_out[l];
    p.off[l] = pool->off[l];
  }
  p.u_dec = pool->u_dec;
  p.sched = pool->dec_sched;
  p.L = pool->L;
  p.R16 = pool->R16;
  p.d_in = pool->d_in;
  p.C = pool->C_dec;
  p.max_tokens = pool->max_tokens;
  p.nc_base[0] = 0;
  for (int l = 0; l < pool->L; ++l) p.nc_base[l + 1] = p.nc_base[l] + ceil_div(pool->d_out[l], kDecNChunk);
  for (int l = pool->L; l < LORA_MAX_LANES; ++l) p.nc_base[l + 1] = p.nc_base[l];
  return p;
}

// Upper bound of decode groups for the last build: sum_k ceil(cnt_k / G) <= T/G + min(N, T).
int dec_group_bound(const lora_pool* pool, const lora_segments* seg) {
  const int T = seg->T;
  return ceil_div(T, kDecGroup) + (pool->N < T ? pool->N : T);
}

}  // namespace

int launch_dec_shrink(const lora_pool* pool, const lora_segments* seg, const uint16_t* x, int64_t ldx,
                      cudaStream_t st) {
  DecParams p = make_params(pool, seg);
  p.x = x;
  p.ldx = ldx;
  const long long items = (long long)dec_group_bound(pool, seg) * pool->L * pool->C_dec;
  const long long cap = 2LL * sm_count(pool->device);
  const int grid = (int)(items < cap ? items : cap);
  if (grid <= 0) return LORA_OK;
  const int smem = (int)(kShRingBytes + kShXBytes + kShXfBytes);
  if (!set_smem_limit(reinterpret_cast<const void*>(dec_shrink_kernel), pool->device, smem)) return LORA_ERR_CUDA;
  const cudaError_t e = launch_pdl(dec_shrink_kernel, dim3(grid), dim3(kShThreads), smem, st, p);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cuda_status(e != cudaSuccess ? e : cudaGetLastError(), "dec_shrink_kernel launch");
}

int launch_dec_expand(const lora_pool* pool, const lora_segments* seg, float* y, int64_t ldy, cudaStream_t st) {
  DecParams p = make_params(pool, seg);
  p.y = y;
  p.ldy = ldy;
  const long long items = (long long)dec_group_bound(pool, seg) * p.nc_base[pool->L];
  const long long cap = 2LL * sm_count(pool->device);
  const int grid = (int)(items < cap ? items : cap);
  if (grid <= 0) return LORA_OK;
  const int smem = (int)kExRingBytes;
  if (!set_smem_limit(reinterpret_cast<const void*>(dec_expand_kernel), pool->device, smem)) return LORA_ERR_CUDA;
  const cudaError_t e = launch_pdl(dec_expand_kernel, dim3(grid), dim3(kExThreads), smem, st, p);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cuda_status(e != cudaSuccess ? e : cudaGetLastError(), "dec_expand_kernel launch");
}

}  // namespace lora
