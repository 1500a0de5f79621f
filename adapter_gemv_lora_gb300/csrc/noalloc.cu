// lora_apply_shrink_expand_noalloc: the apply step for callers that cannot
// allocate device memory at call time.
//
// Some callers of this library never get to allocate: a plugin or custom-op
// host that hands the op only its input and output buffers, a serving loop
// whose memory plan is frozen after start-up (any cudaMalloc would stall the
// device and break the plan), or code that runs where an allocation is not
// allowed.  The normal apply keeps the rank-space intermediate (the decode
// split-K partial sums and the tensor-path rank rows) in a scratch region that
// the caller sized into the pool.  This variant runs the same four kernels,
// but points them at a fixed scratch array compiled into the library instead,
// so the call itself allocates nothing.
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
// The tensor shrink's per-tile arrival counters and the decode kernels' item
// counters sit at the start of the array, where they keep their between-calls
// value of zero (the array is zero when the library loads, and each call
// leaves the counts it used at zero).
constexpr size_t kTileCounters = 16384;
constexpr size_t kCounterWords = kTileCounters + 64;  // + the decode kernels' item counters

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
  if (!pool || !seg || !x || !y) return LORA_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(y) & 15)) return LORA_ERR_ARG;
  if (ldx < pool->d_in || ldy < pool->D || (ldx % 8) || (ldy % 4)) return LORA_ERR_ARG;
  if (seg->N != pool->N || seg->T > pool->max_tokens) return LORA_ERR_SHAPE;
  const int T = seg->T;
  bool loaded = false;
  for (int v : pool->h_rank) loaded |= v > 0;
  if (T == 0 || !loaded) return LORA_OK;  // nothing to do: nothing is launched

  // Rank-space scratch this step needs after the counters: decode partials
  // [C][T][L][R16] and tensor-path partial tiles [kTcKSplit][tiles][L][R16*128]
  // (fp32), then the tensor tiles' U blocks [tiles][L][2][128*R16] (bf16).
  // The kernels size the tile regions from the view's max_tokens, set to T.
  const size_t per_row = (size_t)pool->L * pool->R16;
  const size_t tiles = (size_t)lora::tc_tile_cap(T);
  const size_t dec_floats = (size_t)pool->C_dec * T * per_row;
  const size_t tc_floats = (size_t)lora::kTcKSplit * tiles * per_row * lora::kTcTile;
  const size_t fmt_floats = tiles * per_row * lora::kTcTile;  // 2 bf16 halves = 1 float per element
  const size_t need = kCounterWords + dec_floats + tc_floats + fmt_floats;
  if (tiles > kTileCounters || need > kScratchFloats) return LORA_ERR_SHAPE;

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return LORA_ERR_CUDA;
  if (dev != pool->device) return LORA_ERR_ARG;
  float* scratch = nullptr;
  const int st_addr = scratch_address(dev, &scratch);
  if (st_addr != LORA_OK) return st_addr;

  // A view of the pool whose scratch is the static array (no host or device
  // allocation: the host-side rank mirror is not copied, the kernels never read it).
  lora_pool view;
  view.device = pool->device;
  view.N = pool->N;
  view.R = pool->R;
  view.R16 = pool->R16;
  view.d_in = pool->d_in;
  view.L = pool->L;
  view.D = pool->D;
  view.C_dec = pool->C_dec;
  view.max_tokens = T;  // stride of the partial sums in the scratch
  for (int l = 0; l < LORA_MAX_LANES; ++l) {
    view.d_out[l] = pool->d_out[l];
    view.off[l] = pool->off[l];
    view.A[l] = pool->A[l];
    view.Bt[l] = pool->Bt[l];
    view.Bk[l] = pool->Bk[l];
  }
  view.base = pool->base;
  view.bytes = pool->bytes;
  view.rank_tab = pool->rank_tab;
  view.scale_tab = pool->scale_tab;
  view.tm_a = pool->tm_a;
  view.tm_bk = pool->tm_bk;
  view.tile_cnt = reinterpret_cast<int32_t*>(scratch);
  view.dec_sched = reinterpret_cast<int32_t*>(scratch) + kTileCounters;
  view.u_dec = scratch + kCounterWords;
  view.u_tc = view.u_dec + dec_floats;
  view.u_fmt = reinterpret_cast<uint16_t*>(view.u_tc + tc_floats);

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const uint16_t* xb = static_cast<const uint16_t*>(x);
  int r = lora::launch_dec_shrink(&view, seg, xb, ldx, st);
  if (r == LORA_OK) r = lora::launch_dec_expand(&view, seg, y, ldy, st);
  if (r == LORA_OK) r = lora::launch_tc_shrink(&view, seg, xb, ldx, st);
  if (r == LORA_OK) r = lora::launch_tc_expand(&view, seg, y, ldy, st);
  return r;
}
