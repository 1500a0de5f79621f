// lora_apply_shrink_expand_noalloc: the apply step for callers that cannot
// allocate device memory at call time.
//
// Some callers of this library never get to allocate: a plugin or custom-op
// host that hands the op only its input and output buffers, a serving loop
// whose memory plan is frozen after start-up (any cudaMalloc would stall the
// device and break the plan), or code that runs where an allocation is not
// allowed.  The normal apply keeps the tensor path's rank-space intermediate
// (the partial sums over K ranges, the U tiles and the per-tile counters) in
// a scratch region that the caller sized into the pool.  This variant runs the
// same kernels, but points them at a fixed scratch array compiled into the
// library instead, so the call itself allocates nothing.  (The decode kernel
// keeps its rank-space vector on chip and uses no scratch.)
//
// The array is a file-scope __device__ variable of LORA_NOALLOC_SCRATCH_BYTES;
// every GPU that loads the library holds it until the process exits.  In host
// code its name is only a stand-in, so its device address is looked up once
// per device with cudaGetSymbolAddress, with that device current, on the first
// call made on that device.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kScratchFloats = (size_t)LORA_NOALLOC_SCRATCH_BYTES / sizeof(float);
// The tensor shrink's per-tile arrival counters sit at the start of the
// array, where they keep their between-calls value of zero (the array is
// zero when the library loads, and each call leaves the counts it used at
// zero).
constexpr size_t kTileCounters = 16384;

static __device__ __align__(256) float g_noalloc_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on `device` (which must be current).
int scratch_address(int device, float** out) {
  if (device < 0 || device >= kMaxDevices) return LORA_ERR_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[device]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return LORA_ERR_CUDA;
    g_scratch_ptr[device] = static_cast<float*>(p);
  }
  *out = g_scratch_ptr[device];
  return LORA_OK;
}

}  // namespace

extern "C" int lora_apply_shrink_expand_noalloc(const lora_pool* pool, const lora_segments* seg, const void* x,
                                                float* y, int64_t ldx, int64_t ldy, lora_stream_t stream) {
  // the same host checks as the normal entry point (including that the pool
  // and the segments live on the current device)
  const int chk = lora::check_apply(pool, seg, x, y, ldx, ldy);
  if (chk != LORA_OK) return chk;
  const int T = seg->T;
  if (T == 0 || !lora::pool_has_adapter(pool)) return LORA_OK;  // nothing to do: nothing is launched

  // Rank-space scratch this step needs after the counters: tensor-path
  // partial tiles [kTcKSplit][tiles][L][R16*128] (fp32), then the tensor
  // tiles' U blocks [tiles][L][2][128*R16] (bf16).  The decode path keeps its
  // rank-space vector on chip and needs none.  The tensor kernels size the
  // tile regions from the view's max_tokens, set to T.
  const lora::PoolView& pv = pool->v;
  const size_t per_row = (size_t)pv.L * pv.R16;
  const size_t tiles = (size_t)lora::tc_tile_cap(T);
  const size_t tc_floats = (size_t)lora::kTcKSplit * tiles * per_row * lora::kTcTile;
  const size_t fmt_floats = tiles * per_row * lora::kTcTile;  // 2 bf16 halves = 1 float per element
  const size_t need = kTileCounters + tc_floats + fmt_floats;
  if (tiles > kTileCounters || need > kScratchFloats) return LORA_ERR_SHAPE;

  float* scratch = nullptr;
  const int st_addr = scratch_address(pv.device, &scratch);
  if (st_addr != LORA_OK) return st_addr;

  // The pool's view with the static array as its scratch (a plain copy: no
  // host or device allocation).
  lora::PoolView view = pv;
  view.max_tokens = T;  // sizes the scratch regions below
  view.tile_cnt = reinterpret_cast<int32_t*>(scratch);
  view.u_tc = scratch + kTileCounters;
  view.u_fmt = reinterpret_cast<uint16_t*>(view.u_tc + tc_floats);

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int r = LORA_OK;
  for (int stage = 1; stage <= 3 && r == LORA_OK; ++stage) r = lora::run_stage(view, seg, x, y, ldx, ldy, stage, st);
  return r;
}
