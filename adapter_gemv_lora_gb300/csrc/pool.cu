// The adapter pool of one projection: a fixed number of slots, each holding
// per lane the bf16 factors of one adapter padded to R16 rows, plus per
// (slot, lane) rank and fp32 scale tables (xLLM PR #2014, LoRARuntime's
// per-projection device pool; tokenspeed PR #976, max_loras bounds the slot
// count; TensorFold PR #47, any rank and scale per module).
//
// Layout in the caller's device memory (every region 1024-byte aligned):
//   rank_tab  int32 [N][L]
//   scale_tab f32   [N][L]
//   A_l       bf16  [N][R16][d_in]      per lane; rows >= rank are zero
//   Bt_l      bf16  [N][R16][d_out_l]   per lane; B transposed, for the decode
//                                       expand (each rank row is a contiguous
//                                       run of output columns)
//   Bk_l      bf16  [N][R16/16][d_out_l][16]  per lane; B as given, cut into
//                                       groups of 16 rank columns (K-major), so
//                                       one TMA box loads several whole groups
//                                       for the tensor-core expand
//   u_tc      f32   [2][tiles][L][R16*128]   tensor-path partial sums, one per
//                                            half of d_in, per tile as
//                                            [column quad][row] float4
//   u_fmt     bf16  [tiles][L][2][128*R16]   per tensor tile the summed U as
//                                            bf16 hi and lo halves, in the
//                                            layout the expand's MMA reads
//   tile_cnt  int32 [tiles]                  per tile, K-range CTAs done
//   u_rows    f32   [max_tokens][L][R16]     per row scale * u, the input of
//                                            the fused projection's expand
// The decode path needs no scratch: its rank-space vector stays on chip.
// (tiles = max_tokens / 64 + 1, the most a build can make)
#include <cuda_runtime.h>

#include <cstring>

#include "device.cuh"
#include "internal.h"

namespace lora {
namespace {

__global__ void repack_kernel(const uint16_t* __restrict__ A, const uint16_t* __restrict__ B, int rank, int R16,
                              int d_in, int d_out, uint16_t* __restrict__ Ap, uint16_t* __restrict__ Bt,
                              uint16_t* __restrict__ Bk, int32_t* rank_entry, float* scale_entry, float scale) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t na = (size_t)R16 * d_in, nb = (size_t)R16 * d_out;
  for (size_t idx = tid; idx < na; idx += stride) {
    const int i = (int)(idx / d_in), j = (int)(idx % d_in);
    Ap[idx] = i < rank ? A[(size_t)i * d_in + j] : (uint16_t)0;
  }
  for (size_t idx = tid; idx < nb; idx += stride) {
    const int i = (int)(idx / d_out), o = (int)(idx % d_out);
    Bt[idx] = i < rank ? B[(size_t)o * rank + i] : (uint16_t)0;
  }
  for (size_t idx = tid; idx < nb; idx += stride) {
    const int q = (int)(idx / ((size_t)d_out * 16));
    const int rem = (int)(idx % ((size_t)d_out * 16));
    const int o = rem / 16, i = 16 * q + rem % 16;
    Bk[idx] = i < rank ? B[(size_t)o * rank + i] : (uint16_t)0;
  }
  if (tid == 0) {
    *rank_entry = rank;
    *scale_entry = scale;
  }
}

struct PoolLayout {
  size_t rank_tab, scale_tab, A[LORA_MAX_LANES], Bt[LORA_MAX_LANES], Bk[LORA_MAX_LANES], u_tc, u_fmt, tile_cnt,
      u_rows, total;
  int R16;
};

size_t align1k(size_t v) { return (v + 1023) & ~(size_t)1023; }

bool pool_layout(int N, int R, int d_in, int L, const int* d_out, int max_tokens, PoolLayout* P) {
  if (N < 2 || N > LORA_MAX_SLOTS || R < 1 || R > 128 || d_in < 64 || d_in > 65536 || (d_in % 64) || L < 1 ||
      L > LORA_MAX_LANES ||
      !d_out || max_tokens < 1)
    return false;
  const int R16 = round_up(R, 16);  // L * R16 <= 4 * 128 = 512 TMEM columns for the tensor shrink
  for (int l = 0; l < L; ++l)
    if (d_out[l] < 64 || (d_out[l] % 64)) return false;
  P->R16 = R16;
  size_t o = 0;
  P->rank_tab = o; o = align1k(o + 4 * (size_t)N * L);
  P->scale_tab = o; o = align1k(o + 4 * (size_t)N * L);
  for (int l = 0; l < LORA_MAX_LANES; ++l) P->A[l] = P->Bt[l] = P->Bk[l] = 0;
  for (int l = 0; l < L; ++l) {
    P->A[l] = o; o = align1k(o + 2 * (size_t)N * R16 * d_in);
  }
  for (int l = 0; l < L; ++l) {
    P->Bt[l] = o; o = align1k(o + 2 * (size_t)N * R16 * d_out[l]);
  }
  for (int l = 0; l < L; ++l) {
    P->Bk[l] = o; o = align1k(o + 2 * (size_t)N * d_out[l] * R16);
  }
  P->u_tc = o; o = align1k(o + 4 * (size_t)kTcKSplit * tc_tile_cap(max_tokens) * L * R16 * kTcTile);
  P->u_fmt = o; o = align1k(o + 2 * (size_t)tc_tile_cap(max_tokens) * L * 2 * kTcTile * R16);
  P->tile_cnt = o; o = align1k(o + 4 * (size_t)tc_tile_cap(max_tokens));
  P->u_rows = o; o = align1k(o + 4 * (size_t)max_tokens * L * R16);
  P->total = o;
  return true;
}

}  // namespace

int launch_repack(const PoolView& pool, int slot, int lane, int rank, float scale, const uint16_t* A,
                  const uint16_t* B, cudaStream_t st) {
  const int R16 = pool.R16, d_in = pool.d_in, d_out = pool.d_out[lane];
  uint16_t* Ap = pool.A[lane] + (size_t)slot * R16 * d_in;
  uint16_t* Bt = pool.Bt[lane] + (size_t)slot * R16 * d_out;
  uint16_t* Bk = pool.Bk[lane] + (size_t)slot * d_out * R16;
  const size_t n = (size_t)R16 * (d_in > d_out ? d_in : d_out);
  int blocks = (int)((n + 255) / 256);
  if (blocks > 4096) blocks = 4096;
  repack_kernel<<<blocks, 256, 0, st>>>(A, B, rank, R16, d_in, d_out, Ap, Bt, Bk,
                                         pool.rank_tab + slot * pool.L + lane, pool.scale_tab + slot * pool.L + lane,
                                         scale);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cuda_status(cudaGetLastError(), "repack_kernel launch");
}

}  // namespace lora

using namespace lora;

extern "C" {

size_t lora_pool_bytes(int num_slots, int max_rank, int d_in, int num_lanes, const int* lane_d_out,
                       int max_tokens) {
  PoolLayout P;
  return pool_layout(num_slots, max_rank, d_in, num_lanes, lane_d_out, max_tokens, &P) ? P.total : 0;
}

int lora_pool_create(lora_pool** out, void* dev_mem, size_t bytes, int num_slots, int max_rank, int d_in,
                     int num_lanes, const int* lane_d_out, int max_tokens, lora_stream_t stream) {
  if (!out || !dev_mem || !lane_d_out || (reinterpret_cast<uintptr_t>(dev_mem) & 255)) return LORA_ERR_ARG;
  PoolLayout P;
  if (!pool_layout(num_slots, max_rank, d_in, num_lanes, lane_d_out, max_tokens, &P)) return LORA_ERR_SHAPE;
  if (bytes < P.total) return LORA_ERR_SHAPE;
  ensure_side_stream();  // now, not inside a caller's stream capture (the apply works without it)
  lora_pool* pp = new lora_pool();
  PoolView* p = &pp->v;
  if (cudaGetDevice(&p->device) != cudaSuccess) {
    delete pp;
    return LORA_ERR_CUDA;
  }
  char* b = static_cast<char*>(dev_mem);
  p->N = num_slots;
  p->R = max_rank;
  p->R16 = P.R16;
  p->d_in = d_in;
  p->L = num_lanes;
  p->max_tokens = max_tokens;
  p->base = b;
  p->bytes = bytes;
  p->D = 0;
  for (int l = 0; l < num_lanes; ++l) {
    p->d_out[l] = lane_d_out[l];
    p->off[l] = p->D;
    p->D += lane_d_out[l];
    p->A[l] = reinterpret_cast<uint16_t*>(b + P.A[l]);
    p->Bt[l] = reinterpret_cast<uint16_t*>(b + P.Bt[l]);
    p->Bk[l] = reinterpret_cast<uint16_t*>(b + P.Bk[l]);
  }
  p->rank_tab = reinterpret_cast<int32_t*>(b + P.rank_tab);
  p->scale_tab = reinterpret_cast<float*>(b + P.scale_tab);
  p->u_tc = reinterpret_cast<float*>(b + P.u_tc);
  p->u_fmt = reinterpret_cast<uint16_t*>(b + P.u_fmt);
  p->tile_cnt = reinterpret_cast<int32_t*>(b + P.tile_cnt);
  p->u_rows = reinterpret_cast<float*>(b + P.u_rows);
  pp->h_rank.assign((size_t)num_slots * num_lanes, 0);
  std::memset(&p->tm_a, 0, sizeof(p->tm_a));
  std::memset(&p->tm_bk, 0, sizeof(p->tm_bk));
  std::memset(&p->tm_bt, 0, sizeof(p->tm_bt));
  for (int l = 0; l < num_lanes; ++l) {
    const uint64_t R16 = (uint64_t)P.R16;
    {
      // Bt as 16 rank rows x up to 256 columns per box (decode expand pages)
      const uint64_t dims[3] = {(uint64_t)lane_d_out[l], R16, (uint64_t)num_slots};
      const uint64_t strides[2] = {2ull * lane_d_out[l], 2ull * lane_d_out[l] * R16};
      const uint32_t box[3] = {(uint32_t)bt_box_cols(lane_d_out[l]), 16u, 1u};
      if (!encode_tmap(&p->tm_bt.m[l], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p->Bt[l], dims, strides, box,
                       CU_TENSOR_MAP_SWIZZLE_NONE)) {
        delete pp;
        return LORA_ERR_CUDA;
      }
    }
    for (int sz = 0; sz < kTmapSizes; ++sz) {
      if ((16u << sz) <= R16) {
        const uint64_t dims[3] = {(uint64_t)d_in, R16, (uint64_t)num_slots};
        const uint64_t strides[2] = {2ull * d_in, 2ull * d_in * R16};
        const uint32_t box[3] = {(uint32_t)kTcKBlock, 16u << sz, 1u};
        if (!encode_tmap(&p->tm_a.m[sz][l], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p->A[l], dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_128B)) {
          delete pp;
          return LORA_ERR_CUDA;
        }
      }
      if ((1u << sz) <= R16 / 16) {
        const uint64_t dims[3] = {16ull, (uint64_t)lane_d_out[l], (R16 / 16) * (uint64_t)num_slots};
        const uint64_t strides[2] = {32ull, 32ull * lane_d_out[l]};
        const uint32_t box[3] = {16u, (uint32_t)kTcNT, 1u << sz};
        if (!encode_tmap(&p->tm_bk.m[sz][l], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p->Bk[l], dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_32B)) {
          delete pp;
          return LORA_ERR_CUDA;
        }
      }
    }
  }
  if (cudaMemsetAsync(dev_mem, 0, P.total, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    delete pp;
    return LORA_ERR_CUDA;
  }
  *out = pp;
  return LORA_OK;
}

int lora_pool_load(lora_pool* pool, int slot, int lane, int rank, float scale, const void* A, const void* B,
                   lora_stream_t stream) {
  if (!pool) return LORA_ERR_ARG;
  const PoolView& v = pool->v;
  if (slot < 1 || slot >= v.N) return LORA_ERR_SLOT;
  if (lane < 0 || lane >= v.L) return LORA_ERR_ARG;
  if (rank < 0 || rank > v.R) return LORA_ERR_RANK;
  if (rank > 0 && (!A || !B)) return LORA_ERR_ARG;
  if (rank > 0 && (reinterpret_cast<uintptr_t>(A) & 1 || reinterpret_cast<uintptr_t>(B) & 1)) return LORA_ERR_ARG;
  int dev = -1;  // the repack runs on the current device, where the pool must live
  if (cudaGetDevice(&dev) != cudaSuccess) return LORA_ERR_CUDA;
  if (dev != v.device) return LORA_ERR_ARG;
  const int st = launch_repack(v, slot, lane, rank, rank > 0 ? scale : 0.0f, static_cast<const uint16_t*>(A),
                               static_cast<const uint16_t*>(B), reinterpret_cast<cudaStream_t>(stream));
  if (st == LORA_OK) pool->h_rank[(size_t)slot * v.L + lane] = rank;
  return st;
}

int lora_pool_destroy(lora_pool* pool) {
  delete pool;
  return LORA_OK;
}

}  // extern "C"
