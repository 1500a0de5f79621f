// Decode path: rows whose own sequence is shorter than LORA_TC_MIN_QLEN
// (single-token decode rows, short chunks).  Rows are grouped by slot (up to
// LORA_DEC_GROUP_ROWS rows of one slot per group), so a slot's factors are
// streamed once per group and shared by the group's rows.
//
//   shrink  u[row][i] = sum_j A[k][l][i][j] * x[row][j]     (TensorFold PR #47,
//   expand  y[row][o] += scale[k][l] * sum_i B[k][l][o][i] * u[row][i]   the delta
//           scale * B @ (A @ x); xLLM PR #2014, shrink then expand)
//
// Fixed summation order, independent of the group a row lands in:
//  * shrink: d_in is cut into 2048-wide chunks (one work item each).  Inside a
//    chunk, lane `ln` of warp `w` owns the 8-element runs at
//    k = 256*s + 8*ln (s = w, w+4, ...), accumulated in that order with fma;
//    the 32 lanes are then combined by a fixed xor butterfly (16,8,4,2,1) and
//    the 4 warps left to right.  The chunks' partial sums go to the pool's
//    scratch and are added in chunk order by the expand kernel.
//  * expand: u is summed over chunks in order, then v[o] accumulates
//    B[o][i] * u[i] for i = 0..r-1 in order with fma, and y = fma(scale, v, y).
// Only true-rank rows of A and B^T are read; the padding never is.
#include <cuda_runtime.h>

#include "device.cuh"
#include "internal.h"

namespace lora {
namespace {

struct DecParams {
  const int32_t* status;
  const int32_t* counts;
  const int4* work;
  const int32_t* perm;
  const int32_t* rank_tab;
  const float* scale_tab;
  const uint16_t* A[LORA_MAX_LANES];
  const uint16_t* Bt[LORA_MAX_LANES];
  float* u_dec;
  const uint16_t* x;
  int64_t ldx;
  float* y;
  int64_t ldy;
  int L, R16, d_in, C, max_tokens;
  int d_out[LORA_MAX_LANES], off[LORA_MAX_LANES];
  int nc_base[LORA_MAX_LANES + 1];
};

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

__global__ void __launch_bounds__(kDecThreads) dec_shrink_kernel(DecParams p) {
  __shared__ __align__(16) uint16_t xs[kDecGroup][kDecKChunk];  // 32 KB
  __shared__ float red[4][64];
  if (*p.status != 0) return;
  const int per_group = p.L * p.C;
  const int n_items = p.counts[2] * per_group;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int w = item / per_group;
    const int rem = item - w * per_group;
    const int l = rem / p.C, c = rem - (rem / p.C) * p.C;
    const int4 g = p.work[w];
    const int k = g.x, p0 = g.y, nrows = g.z - g.y;
    const int r = p.rank_tab[k * p.L + l];
    if (r <= 0) continue;
    const int k0 = c * kDecKChunk;
    const int klen = min(kDecKChunk, p.d_in - k0);
    const int nvec = klen >> 3;
    __syncthreads();  // xs / red of the previous item are no longer read
    for (int idx = tid; idx < kDecGroup * nvec; idx += kDecThreads) {
      const int gg = idx / nvec, v = idx - gg * nvec;
      uint4 q = make_uint4(0u, 0u, 0u, 0u);
      if (gg < nrows) {
        const int t = p.perm[p0 + gg];
        q = ldg_nc_v4(p.x + (size_t)t * p.ldx + k0 + 8 * v);
      }
      *reinterpret_cast<uint4*>(&xs[gg][8 * v]) = q;
    }
    __syncthreads();
    const uint16_t* Ab = p.A[l] + (size_t)k * p.R16 * p.d_in + k0;
    const int nseg = (klen + 255) >> 8;
    for (int rb = 0; rb < r; rb += 8) {
      float acc[kDecGroup * 8];  // index gg*8 + i
#pragma unroll
      for (int j = 0; j < kDecGroup * 8; ++j) acc[j] = 0.f;
      for (int s = warp; s < nseg; s += 4) {
        const int kk = 256 * s + 8 * lane;
        if (kk < klen) {
          float xv[kDecGroup][8];
#pragma unroll
          for (int gg = 0; gg < kDecGroup; ++gg) {
            const uint4 q = *reinterpret_cast<const uint4*>(&xs[gg][kk]);
            unpack8(q, xv[gg]);
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (rb + i < r) {
              float av[8];
              unpack8(ldg_nc_v4(Ab + (size_t)(rb + i) * p.d_in + kk), av);
#pragma unroll
              for (int gg = 0; gg < kDecGroup; ++gg)
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[gg * 8 + i] = fmaf(av[e], xv[gg][e], acc[gg * 8 + i]);
            }
          }
        }
      }
      rs_step<32>(acc, lane, 16);
      rs_step<16>(acc, lane, 8);
      rs_step<8>(acc, lane, 4);
      rs_step<4>(acc, lane, 2);
      rs_step<2>(acc, lane, 1);
      // lane now holds the warp sums of values 2*lane and 2*lane+1
      red[warp][2 * lane] = acc[0];
      red[warp][2 * lane + 1] = acc[1];
      __syncthreads();
      if (tid < 64) {
        const int gg = tid >> 3, i = tid & 7;
        if (gg < nrows && rb + i < r) {
          float s = red[0][tid] + red[1][tid];
          s += red[2][tid];
          s += red[3][tid];
          p.u_dec[(((size_t)c * p.max_tokens + p0 + gg) * p.L + l) * p.R16 + rb + i] = s;
        }
      }
      __syncthreads();
    }
  }
}

__global__ void __launch_bounds__(kDecThreads) dec_expand_kernel(DecParams p) {
  __shared__ __align__(16) float us[128][kDecGroup];  // [rank][row]
  if (*p.status != 0) return;
  const int total_nc = p.nc_base[p.L];
  const int n_items = p.counts[2] * total_nc;
  const int tid = threadIdx.x;
  const size_t cstride = (size_t)p.max_tokens * p.L * p.R16;
  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int w = item / total_nc;
    const int q = item - w * total_nc;
    int l = 0;
    while (l + 1 < p.L && q >= p.nc_base[l + 1]) ++l;
    const int j = q - p.nc_base[l];
    const int4 g = p.work[w];
    const int k = g.x, p0 = g.y, nrows = g.z - g.y;
    const int r = p.rank_tab[k * p.L + l];
    if (r <= 0) continue;
    __syncthreads();  // us of the previous item are no longer read
    for (int idx = tid; idx < r * kDecGroup; idx += kDecThreads) {
      const int i = idx >> 3, gg = idx & 7;
      float s = 0.f;
      if (gg < nrows) {
        const float* u = p.u_dec + ((size_t)(p0 + gg) * p.L + l) * p.R16 + i;
        s = u[0];
        for (int c = 1; c < p.C; ++c) s += u[c * cstride];
      }
      us[i][gg] = s;
    }
    __syncthreads();
    const int dout = p.d_out[l];
    const int o = j * kDecNChunk + 8 * tid;
    if (o >= dout) continue;
    float4 yv[kDecGroup][2];
    float* yrow[kDecGroup];
#pragma unroll
    for (int gg = 0; gg < kDecGroup; ++gg) {
      yrow[gg] = nullptr;
      if (gg < nrows) {
        const int t = p.perm[p0 + gg];
        yrow[gg] = p.y + (size_t)t * p.ldy + p.off[l] + o;
        yv[gg][0] = *reinterpret_cast<const float4*>(yrow[gg]);
        yv[gg][1] = *reinterpret_cast<const float4*>(yrow[gg] + 4);
      }
    }
    float acc[kDecGroup][8];
#pragma unroll
    for (int gg = 0; gg < kDecGroup; ++gg)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[gg][e] = 0.f;
    const uint16_t* Bb = p.Bt[l] + (size_t)k * p.R16 * dout + o;
#pragma unroll 2
    for (int i = 0; i < r; ++i) {
      float bv[8];
      unpack8(ldg_nc_v4(Bb + (size_t)i * dout), bv);
      const float4 u0 = *reinterpret_cast<const float4*>(&us[i][0]);
      const float4 u1 = *reinterpret_cast<const float4*>(&us[i][4]);
      const float ug[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
      for (int gg = 0; gg < kDecGroup; ++gg)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[gg][e] = fmaf(bv[e], ug[gg], acc[gg][e]);
    }
    const float sc = p.scale_tab[k * p.L + l];
#pragma unroll
    for (int gg = 0; gg < kDecGroup; ++gg) {
      if (gg < nrows) {
        float4 a = yv[gg][0], b = yv[gg][1];
        a.x = fmaf(sc, acc[gg][0], a.x);
        a.y = fmaf(sc, acc[gg][1], a.y);
        a.z = fmaf(sc, acc[gg][2], a.z);
        a.w = fmaf(sc, acc[gg][3], a.w);
        b.x = fmaf(sc, acc[gg][4], b.x);
        b.y = fmaf(sc, acc[gg][5], b.y);
        b.z = fmaf(sc, acc[gg][6], b.z);
        b.w = fmaf(sc, acc[gg][7], b.w);
        *reinterpret_cast<float4*>(yrow[gg]) = a;
        *reinterpret_cast<float4*>(yrow[gg] + 4) = b;
      }
    }
  }
}

DecParams make_params(const lora_pool* pool, const lora_segments* seg) {
  DecParams p{};
  p.status = seg->status;
  p.counts = seg->counts;
  p.work = seg->dec_work;
  p.perm = seg->perm;
  p.rank_tab = pool->rank_tab;
  p.scale_tab = pool->scale_tab;
  for (int l = 0; l < LORA_MAX_LANES; ++l) {
    p.A[l] = pool->A[l];
    p.Bt[l] = pool->Bt[l];
    p.d_out[l] = pool->d_out[l];
    p.off[l] = pool->off[l];
  }
  p.u_dec = pool->u_dec;
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
  const long long cap = 3LL * sm_count(pool->device);
  const int grid = (int)(items < cap ? items : cap);
  if (grid <= 0) return LORA_OK;
  dec_shrink_kernel<<<grid, kDecThreads, 0, st>>>(p);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError() == cudaSuccess ? LORA_OK : LORA_ERR_CUDA;
}

int launch_dec_expand(const lora_pool* pool, const lora_segments* seg, float* y, int64_t ldy, cudaStream_t st) {
  DecParams p = make_params(pool, seg);
  p.y = y;
  p.ldy = ldy;
  const long long items = (long long)dec_group_bound(pool, seg) * p.nc_base[pool->L];
  const long long cap = 3LL * sm_count(pool->device);
  const int grid = (int)(items < cap ? items : cap);
  if (grid <= 0) return LORA_OK;
  dec_expand_kernel<<<grid, kDecThreads, 0, st>>>(p);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError() == cudaSuccess ? LORA_OK : LORA_ERR_CUDA;
}

}  // namespace lora
