// Host-side descriptors and kernel parameter blocks shared by the library's
// translation units.  Not part of the public ABI (see include/lora_delta.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <vector>

#include "lora_delta.h"

namespace lora {

// Decode path tiling.
constexpr int kDecGroup = LORA_DEC_GROUP_ROWS;  // rows of one slot per decode group

// Tensor path tiling.
constexpr int kTcTile = LORA_TC_TILE_ROWS;  // MMA M
constexpr int kTcKBlock = 64;               // d_in elements per TMA stage (128 B of bf16)
constexpr int kTcNT = 128;                  // expand MMA N per accumulator buffer
constexpr int kTcNGroup = 1024;             // output columns per expand item
constexpr int kTcThreads = 192;             // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kTcKSplit = 2;                // shrink K ranges per tile (fixed: sums stay row-local)

inline int round_up(int v, int m) { return (v + m - 1) / m * m; }
inline int ceil_div(int v, int m) { return (v + m - 1) / m; }

// Tensor maps of one operand per lane in four box sizes: index s has a box of
// 16 << s rank rows (A) or 1 << s groups of 16 rank columns (B), so a rank is
// loaded with one TMA copy per set bit of r16 / 16.  Sizes above the pool's
// R16 are left zeroed and never used.
constexpr int kTmapSizes = 4;
// Tensor tiles a build can make: a sequence of q_len >= 64 gives at most
// q_len / 64 tiles, so T rows give at most T / 64.
inline int tc_tile_cap(int max_tokens) { return max_tokens / LORA_TC_MIN_QLEN + 1; }
struct TmapLanes {
  CUtensorMap m[LORA_MAX_LANES];
};
// Inner box width (columns) of the Bt maps of a lane of d_out columns.
inline int bt_box_cols(int d_out) { return d_out < 256 ? d_out : 256; }
struct TmapSized {
  CUtensorMap m[kTmapSizes][LORA_MAX_LANES];
};

}  // namespace lora

namespace lora {

// Everything the kernels' launchers read from a pool, as plain data: the
// shape, the factor regions, the tables, the tensor maps and the tensor
// path's scratch.  An apply that runs on another scratch region copies the
// view and replaces the three scratch pointers (and max_tokens, which sizes
// the scratch), so the two can never read different fields.
struct PoolView {
  int device = 0;
  int N = 0, R = 0, R16 = 0, d_in = 0, L = 0, D = 0, max_tokens = 0;
  int d_out[LORA_MAX_LANES] = {0, 0, 0, 0};
  int off[LORA_MAX_LANES] = {0, 0, 0, 0};
  char* base = nullptr;
  size_t bytes = 0;
  int32_t* rank_tab = nullptr;        // [N][L]
  float* scale_tab = nullptr;         // [N][L]
  uint16_t* A[LORA_MAX_LANES] = {};   // per lane [N][R16][d_in]
  uint16_t* Bt[LORA_MAX_LANES] = {};  // per lane [N][R16][d_out]   (decode expand)
  uint16_t* Bk[LORA_MAX_LANES] = {};  // per lane [N][R16/16][d_out][16] (tensor expand: K-major
                                      // groups of 16 rank columns, each group contiguous)
  // tensor-path scratch (tiles = tc_tile_cap(max_tokens))
  float* u_tc = nullptr;              // [kTcKSplit][tiles][L][R16/4][128] float4 partial sums over K ranges
  uint16_t* u_fmt = nullptr;          // [tiles][L][2][128*R16] per tensor tile: U as bf16 hi then lo,
                                      // K-major core-matrix layout of the tile's own rank, ready for the expand
  int32_t* tile_cnt = nullptr;        // [tiles] K-range CTAs of a tile that finished (0 between calls)
  float* u_rows = nullptr;            // [max_tokens][L][R16] per row scale * u (the fused projection's
                                      // rank-space input; written by the shrinks run in their row mode)
  TmapSized tm_a;                     // A, 3-D {d_in, R16, N}, box {64, 16<<s, 1}, 128-byte swizzle
  TmapSized tm_bk;                    // Bk, 3-D {16, d_out, R16/16*N}, box {16, 128, 1<<s}, 32-byte swizzle
  TmapLanes tm_bt;                    // Bt, 3-D {d_out, R16, N}, box {min(256, d_out), 16, 1}, no swizzle
};

}  // namespace lora

struct lora_pool {
  lora::PoolView v;
  std::vector<int> h_rank;  // host mirror of rank_tab
};

struct lora_segments {
  int device = 0;
  char* ws = nullptr;
  size_t bytes = 0;
  int max_seqs = 0, max_tokens = 0, N = 0;
  int S = 0, T = 0;  // of the last build
  int cap_dec = 0, cap_tc = 0;
  int32_t* status = nullptr;
  int32_t* counts = nullptr;
  int32_t* seq_start = nullptr;
  int32_t* slot = nullptr;
  int32_t* perm = nullptr;
  int32_t* seg_off = nullptr;
  int4* dec_work = nullptr;
  int32_t* dec_rows = nullptr;  // [cap_dec][kDecGroup] the rows of each decode group (its perm entries)
  int4* tc_work = nullptr;
  int32_t* run_ids = nullptr;   // [max_seqs] per-run slots of a dispatched-row (MoE) build
  int32_t* run_lens = nullptr;  // [max_seqs] per-run lengths; the run count is counts[8]
  int32_t* seq_scratch = nullptr;  // [6][max_seqs] the builder's per-sequence arrays when they do not
                                   // fit in its shared memory (else unused)
};

namespace lora {

extern std::atomic<uint64_t> g_launches;
int sm_count(int device);
// Record a failed CUDA call (its text is kept per thread for lora_last_error_string)
// and map it to LORA_ERR_CUDA; cudaSuccess maps to LORA_OK.
int cuda_status(cudaError_t e, const char* where);
// cudaFuncSetAttribute(max dynamic shared memory) once per (kernel, device, size).
bool set_smem_limit(const void* kernel, int device, int bytes);
bool encode_tmap(CUtensorMap* map, CUtensorMapDataType dt, int rank, void* addr, const uint64_t* dims,
                 const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swz);

// Host-side checks of an apply call: pointers, alignment, leading dimensions,
// shapes, and that the current device is the pool's and the segments' device.
int check_apply(const lora_pool* pool, const lora_segments* seg, const void* x, const float* y, int64_t ldx,
                int64_t ldy);

// True if some (slot, lane) of the pool holds an adapter (host mirror).
bool pool_has_adapter(const lora_pool* pool);
// One kernel of the apply: 1 = decode (fused shrink -> expand), 2 = tensor
// shrink, 3 = tensor expand.
int run_stage(const PoolView& pool, const lora_segments* seg, const void* x, float* y, int64_t ldx, int64_t ldy,
              int stage, cudaStream_t st);

// The apply's side stream for the current device, created on first use.
bool ensure_side_stream();

// Launchers (return a LORA_* status).
// S_dev: if set, the builder reads the sequence count there (at most S, the
// capacity its shared memory is laid out for).
int launch_seg_build(lora_segments* seg, const int32_t* ids, const int32_t* lens, int S, int T,
                     cudaStream_t st, const int32_t* S_dev = nullptr);
int launch_moe_runs(lora_segments* seg, const int32_t* row_expert, const int32_t* row_adapter,
                    const int32_t* row_seq, int T, int E, int A, cudaStream_t st);
int launch_repack(const PoolView& pool, int slot, int lane, int rank, float scale, const uint16_t* A,
                  const uint16_t* B, cudaStream_t st);
// Launch `kernel` allowing programmatic dependent launch on `st` (the kernel
// itself waits for its predecessor's results with griddepcontrol.wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// The decode path: one fused shrink -> expand kernel (u stays on chip).
int launch_decode(const PoolView& pool, const lora_segments* seg, const uint16_t* x, int64_t ldx, float* y,
                  int64_t ldy, cudaStream_t st);
int launch_tc_shrink(const PoolView& pool, const lora_segments* seg, const uint16_t* x, int64_t ldx,
                     cudaStream_t st);
// Row mode of the two shrinks: scale * u of every active row goes to
// pool.u_rows (fp32) and nothing else is written (no expand, no y access).
int launch_decode_rows(const PoolView& pool, const lora_segments* seg, const uint16_t* x, int64_t ldx,
                       cudaStream_t st);
int launch_tc_shrink_rows(const PoolView& pool, const lora_segments* seg, const uint16_t* x, int64_t ldx,
                          cudaStream_t st);
// The fused projection y = x W^T + delta (one tcgen05 GEMM whose accumulator
// also takes the expand), after the row-mode shrinks.
int launch_fused_projection(const PoolView& pool, const lora_segments* seg, const uint16_t* W, int64_t ldw,
                            const uint16_t* x, int64_t ldx, float* y, int64_t ldy, cudaStream_t st);
int launch_tc_expand(const PoolView& pool, const lora_segments* seg, float* y, int64_t ldy, cudaStream_t st);

}  // namespace lora
