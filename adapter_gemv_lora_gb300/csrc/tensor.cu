// Tensor path: rows whose own sequence has q_len >= LORA_TC_MIN_QLEN (prompt
// chunks).  A chunk uses one slot for all its rows (TensorFold PR #47), so a
// 128-row tile of one sequence is a dense contraction against one adapter:
//
//   shrink  U[128][r] = X_tile[128][d_in] . A[k][l]^T       tcgen05, fp32 in TMEM
//   expand  y_tile[128][n] += scale * (U . B[k][l]^T)        tcgen05, fp32 in TMEM
//
// (the delta scale * B @ (A @ x) of TensorFold PR #47; shrink then expand as in
// xLLM PR #2014).  The shrink sums d_in in two fixed K ranges (one CTA each,
// fp32 partials); the CTA of a tile that finishes second adds them in K order
// and splits U into two bf16 halves, u_hi = bf16(u) and u_lo = bf16(u - u_hi),
// stored in the layout the expand's MMA reads.  Both halves are multiplied by
// the (exact) bf16 B and accumulated in fp32, so the rank-space vector keeps
// about 16 significant bits.
//
// Shrink CTA (6 warps): warp 0 lane 0 issues TMA loads into a ring of
// shared-memory stages, warp 1 lane 0 issues tcgen05.mma and tcgen05.commit,
// warps 2-5 are the epilogue (tcgen05.ld of their 32 TMEM lanes = tile rows).
// Expand CTA: described above tc_expand_kernel.
// Operands: X and A tiles are K-major with the 128-byte swizzle (TMA boxes of
// 64 bf16); B tiles are K-major with the 32-byte swizzle (boxes of 16 bf16);
// the U halves are in the plain K-major core matrix layout (8 rows x 16 bytes
// per core matrix), bulk-copied into shared memory by the expand.
// Each row's arithmetic is independent of every other row of its tile, and the
// tile of a row is fixed by its own sequence, so a row's bits do not depend on
// its batch neighbours.  Every mbarrier wait is bounded; a wait that gives up
// records LORA_ERR_TIMEOUT in the status word and the CTA unwinds.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "device.cuh"
#include "internal.h"

namespace lora {
namespace {

constexpr int kXBoxRows = 32;                          // TMA box rows of X
constexpr int kXStageBytes = kTcTile * kTcKBlock * 2;  // 16 KB
constexpr int kMaxStages = 8;

struct TcShrinkParams {
  const int32_t* counts;
  const int4* work;
  const int32_t* rank_tab;
  const float* scale_tab;
  float* u_tc;
  uint16_t* u_fmt;
  float* u_rows;  // row mode: scale * u per row [T][L][R16] instead of u_fmt
  int32_t* tile_cnt;
  int32_t* status;
  int L, R16, num_kb, ring_bytes, tmem_cols, tiles_cap;
  size_t u_split_stride;  // floats between the K-range partials of u_tc
};

struct TcExpandParams {
  const int32_t* counts;
  const int4* work;
  const int32_t* rank_tab;
  const float* scale_tab;
  const uint16_t* u_fmt;
  float* y;
  int32_t* status;
  int64_t ldy;
  int L, R16, total_ng, tail_items;
  int d_out[LORA_MAX_LANES], off[LORA_MAX_LANES], ng_base[LORA_MAX_LANES + 1];
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

__global__ void __launch_bounds__(kTcThreads, 2)
    tc_shrink_kernel(const __grid_constant__ CUtensorMap tm_x128, const __grid_constant__ CUtensorMap tm_x32,
                     const __grid_constant__ TmapSized tm_a, TcShrinkParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ __align__(8) uint64_t done_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int fail_sh, last_sh;

  pdl_wait();  // the previous kernel's results are visible from here on
  // A timeout is the only status a kernel of this step can raise while this
  // one runs; every other error is set before the launch and seen by all CTAs
  // alike, which keeps the per-tile arrival counts consistent.
  {
    const int st0 = *p.status;
    if (st0 != 0 && st0 != LORA_ERR_TIMEOUT) return;
  }
  // CTA = (tile, K range): the k-blocks of d_in are cut into kTcKSplit fixed
  // ranges; each CTA sums one range, and the last CTA of the tile to finish
  // adds the partials in K order and writes U for the expand.
  const int tile = blockIdx.x / kTcKSplit;
  const int ksplit = blockIdx.x - tile * kTcKSplit;
  if (tile >= p.counts[3]) return;
  const int kb_lo = ksplit * p.num_kb / kTcKSplit, kb_hi = (ksplit + 1) * p.num_kb / kTcKSplit;
  const int nkb = kb_hi - kb_lo;
  const int4 wk = p.work[tile];
  const int k = wk.x, rb = wk.y, re = wk.z;
  int r16[LORA_MAX_LANES], a_off[LORA_MAX_LANES];
  int r16_sum = 0;
#pragma unroll
  for (int l = 0; l < LORA_MAX_LANES; ++l) {
    const int r = l < p.L ? p.rank_tab[k * p.L + l] : 0;
    r16[l] = r > 0 ? (r + 15) & ~15 : 0;
    a_off[l] = r16_sum;
    r16_sum += r16[l];
  }
  if (r16_sum == 0) return;
  // Each stage holds one X block and the A blocks of the loaded lanes at
  // their own ranks, so low-rank tiles keep more stages in flight.
  const int stage_bytes = kXStageBytes + r16_sum * kTcKBlock * 2;
  int stages = p.ring_bytes / stage_bytes;
  if (stages > kMaxStages) stages = kMaxStages;

  uint8_t* smem = align1024(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(&done_bar, 1);
    fail_sh = 0;
    last_sh = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base_sh, (uint32_t)p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  // A full tile takes one 128-row X box per stage; the ragged last tile of a
  // sequence takes 32-row boxes up to its end.
  const bool full_tile = (re - rb) == kTcTile;
  const int nbox = (re - rb + kXBoxRows - 1) / kXBoxRows;
  const uint32_t tx_bytes =
      (uint32_t)(full_tile ? kTcTile : nbox * kXBoxRows) * kTcKBlock * 2 + (uint32_t)r16_sum * kTcKBlock * 2;

  if (warp == 0) {
    if (lane == 0) {
      for (int kj = 0; kj < nkb; ++kj) {
        const int kb = kb_lo + kj;
        const int s = kj % stages;
        if (kj >= stages) {
          if (!mbar_wait_or_fail(&empty_bar[s], ((kj / stages) - 1) & 1, &fail_sh)) {
            fail_sh = 1;
            break;
          }
        }
        uint8_t* xs = smem + (size_t)s * stage_bytes;
        uint8_t* as = xs + kXStageBytes;
        mbar_expect_tx(&full_bar[s], tx_bytes);
        if (full_tile) {
          tma_load_2d(xs, &tm_x128, kb * kTcKBlock, rb, &full_bar[s]);
        } else {
          for (int b = 0; b < nbox; ++b)
            tma_load_2d(xs + b * kXBoxRows * kTcKBlock * 2, &tm_x32, kb * kTcKBlock, rb + kXBoxRows * b,
                        &full_bar[s]);
        }
#pragma unroll
        for (int l = 0; l < LORA_MAX_LANES; ++l) {
          int row = 0;
          for (int sz = kTmapSizes - 1; sz >= 0; --sz) {
            const int rows = 16 << sz;
            while (r16[l] - row >= rows) {
              tma_load_3d(as + (size_t)(a_off[l] + row) * kTcKBlock * 2, &tm_a.m[sz][l], kb * kTcKBlock, row, k,
                          &full_bar[s]);
              row += rows;
            }
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      bool ok = true;
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % stages;
        if (!mbar_wait_or_fail(&full_bar[s], (kb / stages) & 1, &fail_sh)) {
          fail_sh = 1;
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t xa = smem_u32(smem + (size_t)s * stage_bytes);
        const uint32_t aa = xa + kXStageBytes;
#pragma unroll
        for (int l = 0; l < LORA_MAX_LANES; ++l) {
          if (r16[l] == 0) continue;
          const uint32_t idesc = idesc_bf16(kTcTile, r16[l]);
#pragma unroll
          for (int kk = 0; kk < kTcKBlock / 16; ++kk) {
            const uint64_t ad = smem_desc(xa + 32 * kk, 16, 1024, kSwz128);
            const uint64_t bd = smem_desc(aa + a_off[l] * kTcKBlock * 2 + 32 * kk, 16, 1024, kSwz128);
            mma_bf16(tmem + (uint32_t)(l * p.R16), ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
        }
        mma_commit(&empty_bar[s]);
      }
      if (ok) mma_commit(&done_bar);
    }
  } else {
    // ---------------- epilogue, one tile row per thread
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const int t = rb + row;
    const bool valid = t < re;
    bool ok = true;
    if (nkb > 0) {  // an empty K range (d_in of one k-block) contributes zeros
      ok = mbar_wait_or_fail(&done_bar, 0, &fail_sh);
      if (!ok) fail_sh = 1;
      else tc_fence_after();
    }
    // This K range's partial of the tile goes to u_tc, laid out per tile as
    // [lane][column quad][row] float4 so that a warp's stores (and the last
    // CTA's loads) cover 512 contiguous bytes.
    const uint32_t trow = (uint32_t)(quad * 32) << 16;
    auto part = [&](int ks, int l) {
      return reinterpret_cast<float4*>(p.u_tc + ks * p.u_split_stride) +
             ((size_t)tile * p.L + l) * (p.R16 / 4) * kTcTile + row;
    };
    if (ok) {
#pragma unroll
      for (int l = 0; l < LORA_MAX_LANES; ++l) {
        float4* dst = part(ksplit, l);
        for (int c0 = 0; c0 < r16[l]; c0 += 64) {
          const int ncol = min(64, r16[l] - c0);  // a multiple of 16
          uint32_t v[4][16];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (16 * q < ncol) {
              if (nkb > 0) {
                tmem_ld16_nowait(tmem + trow + (uint32_t)(l * p.R16 + c0 + 16 * q), v[q]);
              } else {
#pragma unroll
                for (int e = 0; e < 16; ++e) v[q][e] = 0u;
              }
            }
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (16 * q < ncol) {
              if (nkb > 0) tmem_wait_ld16(v[q]);
#pragma unroll
              for (int e = 0; e < 4; ++e)
                dst[(size_t)((c0 + 16 * q) / 4 + e) * kTcTile] =
                    make_float4(__uint_as_float(v[q][4 * e]), __uint_as_float(v[q][4 * e + 1]),
                                __uint_as_float(v[q][4 * e + 2]), __uint_as_float(v[q][4 * e + 3]));
            }
          }
        }
      }
    }
    // Every CTA that got this far counts itself in, failed or not, so the
    // counts stay whole; the one that completes the count resets it.
    __threadfence();
    named_bar_sync(1, 4 * 32);
    if (warp == 2 && lane == 0) {
      const int before = atomicAdd(&p.tile_cnt[tile], 1);
      last_sh = before == kTcKSplit - 1;
      if (last_sh) p.tile_cnt[tile] = 0;
    }
    named_bar_sync(1, 4 * 32);
    if (last_sh) {
      __threadfence();
      // U = partial 0 + partial 1 + ... (K order; this CTA's own partial
      // comes from TMEM, the others from L2), split into bf16 hi and lo and
      // stored in the expand's K-major core-matrix layout: row m, rank
      // columns 8g..8g+7 at (m / 8) * (r16 * 16) + g * 128 + (m % 8) * 16.
#pragma unroll
      for (int l = 0; l < LORA_MAX_LANES; ++l) {
        if (r16[l] == 0) continue;
        uint8_t* hi = reinterpret_cast<uint8_t*>(p.u_fmt + ((size_t)tile * p.L + l) * 2 * kTcTile * p.R16);
        uint8_t* lo = hi + (size_t)kTcTile * r16[l] * 2;
        const size_t sbo = (size_t)r16[l] * 16;
        for (int c0 = 0; c0 < r16[l]; c0 += 64) {
          const int ncol = min(64, r16[l] - c0);  // a multiple of 16
          float4 oth[kTcKSplit - 1][16];         // every load of this batch is issued before the sums
#pragma unroll
          for (int j = 0; j < kTcKSplit - 1; ++j) {
            const float4* src = part(j < ksplit ? j : j + 1, l) + (size_t)(c0 / 4) * kTcTile;
#pragma unroll
            for (int v = 0; v < 16; ++v)
              oth[j][v] = 4 * v < ncol ? __ldcg(src + (size_t)v * kTcTile) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
          uint32_t own[4][16];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (16 * q < ncol) {
              if (nkb > 0) {
                tmem_ld16_nowait(tmem + trow + (uint32_t)(l * p.R16 + c0 + 16 * q), own[q]);
              } else {
#pragma unroll
                for (int e = 0; e < 16; ++e) own[q][e] = 0u;
              }
            }
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (16 * q < ncol) {
              if (nkb > 0) tmem_wait_ld16(own[q]);
              float u[16];
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                float acc = 0.f;
#pragma unroll
                for (int ks = 0; ks < kTcKSplit; ++ks) {
                  float val;
                  if (ks == ksplit) {
                    val = __uint_as_float(own[q][e]);
                  } else {
                    const float4 w = oth[ks < ksplit ? ks : ks - 1][4 * q + e / 4];
                    val = (e & 3) == 0 ? w.x : (e & 3) == 1 ? w.y : (e & 3) == 2 ? w.z : w.w;
                  }
                  acc = ks == 0 ? val : acc + val;
                }
                u[e] = valid ? acc : 0.f;
              }
              if (p.u_rows) {  // row mode: scale * u of this row, fp32
                if (valid) {
                  const float sc = p.scale_tab[k * p.L + l];
                  float4* dst = reinterpret_cast<float4*>(p.u_rows + ((size_t)t * p.L + l) * p.R16 + c0 + 16 * q);
#pragma unroll
                  for (int e = 0; e < 4; ++e)
                    dst[e] = make_float4(sc * u[4 * e], sc * u[4 * e + 1], sc * u[4 * e + 2], sc * u[4 * e + 3]);
                }
                continue;
              }
#pragma unroll
              for (int g = 0; g < 2; ++g) {
                uint32_t hw[4], lw[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const float u0 = u[8 * g + 2 * e], u1 = u[8 * g + 2 * e + 1];
                  const __nv_bfloat16 h0 = __float2bfloat16_rn(u0);
                  const __nv_bfloat16 h1 = __float2bfloat16_rn(u1);
                  const __nv_bfloat16 l0 = __float2bfloat16_rn(u0 - __bfloat162float(h0));
                  const __nv_bfloat16 l1 = __float2bfloat16_rn(u1 - __bfloat162float(h1));
                  hw[e] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
                  lw[e] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
                }
                const int kg = (c0 + 16 * q) / 8 + g;
                const size_t o = (size_t)(row >> 3) * sbo + (size_t)kg * 128 + (size_t)(row & 7) * 16;
                *reinterpret_cast<uint4*>(hi + o) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                *reinterpret_cast<uint4*>(lo + o) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
              }
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, (uint32_t)p.tmem_cols);
  }
  if (threadIdx.x == 0 && fail_sh) set_error(p.status, LORA_ERR_TIMEOUT);
}

// Expand CTA: warp 0 TMA, warp 1 MMA, warps 2-5 read TMEM (one lane quadrant
// each) and stage scale * acc in shared memory, warps 6-21 do the y update with
// coalesced 128-bit loads and stores (two 256-byte row segments per warp
// instruction, the next half-chunk's y loads in flight while the current one
// is added).  Rows past the end of the tile's sequence are skipped.
constexpr int kExpTmemWarps = 4;
constexpr int kExpRmwWarps = 16;
constexpr int kExpThreads = (2 + kExpTmemWarps + kExpRmwWarps) * 32;
constexpr int kHalfCols = 64;                          // columns per staged half chunk
constexpr int kHalfBytes = kTcTile * kHalfCols * 4;    // 32 KB
constexpr int kRmwRowsPerWarp = kTcTile / kExpRmwWarps;  // 8

__global__ void __launch_bounds__(kExpThreads, 1)
    tc_expand_kernel(const __grid_constant__ TmapSized tm_b, TcExpandParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bfull[2], bempty[2], afull[2], aempty[2], sfull[2], sempty[2], ufull;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int fail_sh;

  pdl_wait();  // the previous kernel's results are visible from here on
  if (*p.status != 0) return;
  // The last `tail_items` items of the step (the last wave) run as two CTAs of
  // half the columns each, so the SMs finish closer together.
  const int n_items = p.counts[3] * p.total_ng;
  const int tail_start = max(0, n_items - p.tail_items);
  int item = blockIdx.x, half = -1;
  if (item >= tail_start) {
    item = tail_start + (blockIdx.x - tail_start) / 2;
    half = (blockIdx.x - tail_start) & 1;
  }
  if (item >= n_items) return;
  const int tile = item / p.total_ng;
  const int q = item - tile * p.total_ng;
  int l = 0;
  // lane of this item, and its column range, picked with constant indexes
  // (a parameter array indexed at run time would be copied to local memory)
  int ng = q, d_out_l = p.d_out[0], off_l = p.off[0];
#pragma unroll
  for (int i = 1; i < LORA_MAX_LANES; ++i) {
    if (i < p.L && q >= p.ng_base[i]) {
      l = i;
      ng = q - p.ng_base[i];
      d_out_l = p.d_out[i];
      off_l = p.off[i];
    }
  }
  const int4 wk = p.work[tile];
  const int k = wk.x, rb = wk.y, re = wk.z;
  const int r = p.rank_tab[k * p.L + l];
  if (r <= 0) return;
  const int r16 = (r + 15) & ~15;
  const int nk = r16 / 16;
  const int n_begin = ng * kTcNGroup + (half > 0 ? kTcNGroup / 2 : 0);
  const int n_end = min(d_out_l, ng * kTcNGroup + (half == 0 ? kTcNGroup / 2 : kTcNGroup));
  if (n_begin >= n_end) return;  // the second half of a narrow lane's last group
  const int nchunks = (n_end - n_begin + kTcNT - 1) / kTcNT;
  const float sc = p.scale_tab[k * p.L + l];

  // shared memory: [y staging 2 x 32 KB][B stages 2 x R16*256][U hi 128*R16*2][U lo]
  uint8_t* smem = align1024(smem_raw);
  uint8_t* ystage = smem;
  uint8_t* bst = smem + 2 * kHalfBytes;
  const size_t bstage_bytes = (size_t)p.R16 * kTcNT * 2;
  uint8_t* uhi = bst + 2 * bstage_bytes;
  uint8_t* ulo = uhi + (size_t)kTcTile * r16 * 2;  // the shrink stores hi and lo back to back
  const uint32_t u_sbo = (uint32_t)(r16 / 8) * 128;  // bytes between 8-row groups of U

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bfull[s], 1);
      mbar_init(&bempty[s], 1);
      mbar_init(&afull[s], 1);
      mbar_init(&aempty[s], kExpTmemWarps);
      mbar_init(&sfull[s], kExpTmemWarps);
      mbar_init(&sempty[s], kExpRmwWarps);
    }
    mbar_init(&ufull, 1);
    fail_sh = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base_sh, 2 * kTcNT);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();  // barriers initialised, TMEM allocated
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  if (warp == 0) {
    if (lane == 0) {
      // U of this tile and lane (bf16 hi and lo, written by the shrink) in one bulk copy
      const uint32_t u_bytes = (uint32_t)kTcTile * r16 * 2 * 2;
      mbar_expect_tx(&ufull, u_bytes);
      bulk_load(uhi, p.u_fmt + ((size_t)tile * p.L + l) * 2 * kTcTile * p.R16, u_bytes, &ufull);
      for (int c = 0; c < nchunks; ++c) {
        const int s = c & 1;
        if (c >= 2) {
          if (!mbar_wait_or_fail(&bempty[s], ((c >> 1) - 1) & 1, &fail_sh)) {
            fail_sh = 1;
            break;
          }
        }
        mbar_expect_tx(&bfull[s], (uint32_t)nk * kTcNT * 32);
        uint8_t* bs = bst + (size_t)s * bstage_bytes;
        // groups of 16 rank columns, several per copy: [group][128 rows][16]
        int qq = 0;
        for (int sz = kTmapSizes - 1; sz >= 0; --sz) {
          const int groups = 1 << sz;
          while (nk - qq >= groups) {
            tma_load_3d(bs + (size_t)qq * kTcNT * 32, &tm_b.m[sz][l], 0, n_begin + c * kTcNT,
                        k * (p.R16 / 16) + qq, &bfull[s]);
            qq += groups;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t uh = smem_u32(uhi), ul = smem_u32(ulo);
      const bool u_ok = mbar_wait_or_fail(&ufull, 0, &fail_sh);
      if (!u_ok) fail_sh = 1;
      for (int c = 0; c < nchunks && u_ok; ++c) {
        const int s = c & 1;
        if (!mbar_wait_or_fail(&bfull[s], (c >> 1) & 1, &fail_sh)) {
          fail_sh = 1;
          break;
        }
        if (c >= 2 && !mbar_wait_or_fail(&aempty[s], ((c >> 1) - 1) & 1, &fail_sh)) {
          fail_sh = 1;
          break;
        }
        tc_fence_after();
        const int nt = min(kTcNT, n_end - (n_begin + c * kTcNT));
        const uint32_t idesc = idesc_bf16(kTcTile, nt);
        const uint32_t d = tmem + (uint32_t)(s * kTcNT);
        const uint32_t bsa = smem_u32(bst + (size_t)s * bstage_bytes);
        for (int qq = 0; qq < nk; ++qq) {
          const uint64_t ad = smem_desc(uh + 256 * qq, 128, u_sbo, kSwzNone);
          const uint64_t bd = smem_desc(bsa + qq * kTcNT * 32, 16, 256, kSwz32);
          mma_bf16(d, ad, bd, idesc, qq > 0 ? 1u : 0u);
        }
        for (int qq = 0; qq < nk; ++qq) {
          const uint64_t ad = smem_desc(ul + 256 * qq, 128, u_sbo, kSwzNone);
          const uint64_t bd = smem_desc(bsa + qq * kTcNT * 32, 16, 256, kSwz32);
          mma_bf16(d, ad, bd, idesc, 1u);
        }
        mma_commit(&bempty[s]);
        mma_commit(&afull[s]);
      }
    }
  } else if (warp < 2 + kExpTmemWarps) {
    // ---------------- TMEM readers: acc * scale -> staging (row m, 16-byte chunk j at j ^ (m & 15))
    const int quad = warp & 3;
    const int m = quad * 32 + lane;
    int hh = 0;
    bool ok = true;
    for (int c = 0; c < nchunks && ok; ++c) {
      const int s = c & 1;
      if (!mbar_wait_or_fail(&afull[s], (c >> 1) & 1, &fail_sh)) {
        fail_sh = 1;
        ok = false;
        break;
      }
      tc_fence_after();
      const int nhalf = min(kTcNT, n_end - (n_begin + c * kTcNT)) / kHalfCols;
      for (int h = 0; h < nhalf; ++h, ++hh) {
        const int sb = hh & 1;
        if (hh >= 2 && !mbar_wait_or_fail(&sempty[sb], ((hh >> 1) - 1) & 1, &fail_sh)) {
          fail_sh = 1;
          ok = false;
          break;
        }
        uint8_t* row = ystage + (size_t)sb * kHalfBytes + (size_t)m * (kHalfCols * 4);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          float v[32];
          tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(s * kTcNT + h * kHalfCols + 32 * j), v);
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            const int cj = 8 * j + ch;
            *reinterpret_cast<float4*>(row + ((cj ^ (m & 15)) * 16)) =
                make_float4(v[4 * ch] * sc, v[4 * ch + 1] * sc, v[4 * ch + 2] * sc, v[4 * ch + 3] * sc);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfull[sb]);
      }
      tc_fence_before();
      __syncwarp();
      if (ok && lane == 0) mbar_arrive(&aempty[s]);
    }
  } else {
    // ---------------- y update: kRmwRowsPerWarp rows per warp; lanes 0-15 / 16-31 cover two rows of 64 columns
    const int rw = warp - 2 - kExpTmemWarps;
    const int chunk = lane & 15;
    int total_h = 0;
    for (int c = 0; c < nchunks; ++c) total_h += min(kTcNT, n_end - (n_begin + c * kTcNT)) / kHalfCols;
    auto col_of = [&](int hidx) {  // first column of half chunk hidx (halves never straddle chunks)
      return off_l + n_begin + hidx * kHalfCols + 4 * chunk;
    };
    // Two half chunks of y in flight per warp: the one being added and the
    // next; a half's buffer is refilled with the half two ahead as soon as it
    // has been added (two named arrays, so they stay in registers).
    float4 ya[kRmwRowsPerWarp / 2], yb[kRmwRowsPerWarp / 2];
    auto load_half = [&](int hidx, float4 (&dst)[kRmwRowsPerWarp / 2]) {
      const int col = col_of(hidx);
#pragma unroll
      for (int it = 0; it < kRmwRowsPerWarp / 2; ++it) {
        const int row = 2 * kExpRmwWarps * it + 2 * rw + (lane >> 4);
        const int t = rb + row;
        if (t < re) dst[it] = *reinterpret_cast<const float4*>(p.y + (size_t)t * p.ldy + col);
      }
    };
    auto add_half = [&](int hh, float4 (&yc)[kRmwRowsPerWarp / 2]) -> bool {
      const int sb = hh & 1;
      if (!mbar_wait_or_fail(&sfull[sb], (hh >> 1) & 1, &fail_sh)) {
        fail_sh = 1;
        return false;
      }
      const uint8_t* st = ystage + (size_t)sb * kHalfBytes;
      const int col = col_of(hh);
#pragma unroll
      for (int it = 0; it < kRmwRowsPerWarp / 2; ++it) {
        const int row = 2 * kExpRmwWarps * it + 2 * rw + (lane >> 4);
        const int t = rb + row;
        if (t < re) {
          const float4 d = *reinterpret_cast<const float4*>(st + (size_t)row * (kHalfCols * 4) +
                                                            ((chunk ^ (row & 15)) * 16));
          float4 a = yc[it];
          a.x += d.x;
          a.y += d.y;
          a.z += d.z;
          a.w += d.w;
          __stcs(reinterpret_cast<float4*>(p.y + (size_t)t * p.ldy + col), a);  // streaming: y is not read again
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sempty[sb]);
      if (hh + 2 < total_h) load_half(hh + 2, yc);
      return true;
    };
    if (total_h > 0) load_half(0, ya);
    if (total_h > 1) load_half(1, yb);
    for (int hh = 0; hh < total_h; hh += 2) {
      if (!add_half(hh, ya)) break;
      if (hh + 1 < total_h && !add_half(hh + 1, yb)) break;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * kTcNT);
  }
  if (threadIdx.x == 0 && fail_sh) set_error(p.status, LORA_ERR_TIMEOUT);
}

// Upper bound of tensor tiles for the last build: a sequence of q_len >= 64
// gives ceil(q_len / 128) <= q_len / 64 tiles, so there are at most
// min(T / 128 + S, T / 64) of them.
int tc_tile_bound(const lora_segments* seg) {
  const int a = ceil_div(seg->T, kTcTile) + seg->S, b = seg->T / LORA_TC_MIN_QLEN;
  return a < b ? a : b;
}

}  // namespace

namespace {
int tc_shrink_impl(const PoolView& pool, const lora_segments* seg, const uint16_t* x, int64_t ldx, float* u_rows,
                   cudaStream_t st) {
  const int grid = tc_tile_bound(seg) * kTcKSplit;
  if (grid <= 0) return LORA_OK;
  CUtensorMap tm_x128, tm_x32;
  {
    const uint64_t dims[2] = {(uint64_t)pool.d_in, (uint64_t)seg->T};
    const uint64_t strides[1] = {2ull * (uint64_t)ldx};
    const uint32_t box128[2] = {(uint32_t)kTcKBlock, (uint32_t)kTcTile};
    const uint32_t box32[2] = {(uint32_t)kTcKBlock, (uint32_t)kXBoxRows};
    if (!encode_tmap(&tm_x128, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box128,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tmap(&tm_x32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box32,
                     CU_TENSOR_MAP_SWIZZLE_128B))
      return LORA_ERR_CUDA;
  }
  TcShrinkParams p{};
  p.counts = seg->counts;
  p.work = seg->tc_work;
  p.rank_tab = pool.rank_tab;
  p.scale_tab = pool.scale_tab;
  p.u_rows = u_rows;
  p.u_tc = pool.u_tc;
  p.u_fmt = pool.u_fmt;
  p.tile_cnt = pool.tile_cnt;
  p.status = seg->status;
  p.L = pool.L;
  p.R16 = pool.R16;
  p.num_kb = pool.d_in / kTcKBlock;
  p.tiles_cap = tc_tile_cap(pool.max_tokens);
  p.u_split_stride = (size_t)p.tiles_cap * pool.L * pool.R16 * kTcTile;
  // Two CTAs per SM: each keeps its ring within ~100 KB of shared memory (at
  // least two stages of the largest kind: every lane at R16).
  const int max_stage = kXStageBytes + pool.L * pool.R16 * kTcKBlock * 2;
  p.ring_bytes = 100 * 1024 > 2 * max_stage ? 100 * 1024 : 2 * max_stage;
  int cols = 32;
  while (cols < pool.L * pool.R16) cols <<= 1;
  p.tmem_cols = cols;
  // Above 256 TMEM columns a CTA needs more than half of the SM's 512: ask for
  // enough shared memory that only one CTA fits on an SM, so no CTA's
  // allocation waits for another's to be released.
  if (cols > 256 && p.ring_bytes < 120 * 1024) p.ring_bytes = 120 * 1024;
  const int smem = p.ring_bytes + 1024;
  if (!set_smem_limit(reinterpret_cast<const void*>(tc_shrink_kernel), pool.device, smem)) return LORA_ERR_CUDA;
  const cudaError_t e = launch_pdl(tc_shrink_kernel, dim3(grid), dim3(kTcThreads), smem, st, tm_x128, tm_x32, pool.tm_a, p);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cuda_status(e != cudaSuccess ? e : cudaGetLastError(), "tc_shrink_kernel launch");
}
}  // namespace

int launch_tc_shrink(const PoolView& pool, const lora_segments* seg, const uint16_t* x, int64_t ldx,
                     cudaStream_t st) {
  return tc_shrink_impl(pool, seg, x, ldx, nullptr, st);
}

int launch_tc_shrink_rows(const PoolView& pool, const lora_segments* seg, const uint16_t* x, int64_t ldx,
                          cudaStream_t st) {
  return tc_shrink_impl(pool, seg, x, ldx, pool.u_rows, st);
}

int launch_tc_expand(const PoolView& pool, const lora_segments* seg, float* y, int64_t ldy, cudaStream_t st) {
  TcExpandParams p{};
  p.ng_base[0] = 0;
  for (int l = 0; l < LORA_MAX_LANES; ++l) {
    p.d_out[l] = pool.d_out[l];
    p.off[l] = pool.off[l];
    p.ng_base[l + 1] = p.ng_base[l] + (l < pool.L ? ceil_div(pool.d_out[l], kTcNGroup) : 0);
  }
  p.total_ng = p.ng_base[pool.L];
  p.tail_items = sm_count(pool.device) / 2;  // half an SM wave: measured best of 0.5, 1 and 2 waves
  const long long items = (long long)tc_tile_bound(seg) * p.total_ng;
  if (items <= 0) return LORA_OK;
  const long long grid = items + p.tail_items;  // the tail's items take two CTAs each
  p.counts = seg->counts;
  p.work = seg->tc_work;
  p.rank_tab = pool.rank_tab;
  p.scale_tab = pool.scale_tab;
  p.u_fmt = pool.u_fmt;
  p.y = y;
  p.ldy = ldy;
  p.status = seg->status;
  p.L = pool.L;
  p.R16 = pool.R16;
  const int smem = 2 * kHalfBytes + 4 * kTcTile * pool.R16 * 2 + 1024;  // staging + 2 B stages + U hi/lo
  if (!set_smem_limit(reinterpret_cast<const void*>(tc_expand_kernel), pool.device, smem)) return LORA_ERR_CUDA;
  const cudaError_t e = launch_pdl(tc_expand_kernel, dim3((unsigned)grid), dim3(kExpThreads), smem, st, pool.tm_bk, p);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cuda_status(e != cudaSuccess ? e : cudaGetLastError(), "tc_expand_kernel launch");
}

}  // namespace lora
