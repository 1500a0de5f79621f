// Entry points that tie the pool, the segments and the kernels together, plus
// the small host utilities the kernels' launchers share.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdio>
#include <mutex>
#include <vector>

#include "internal.h"

namespace lora {

std::atomic<uint64_t> g_launches{0};

namespace {
thread_local char t_last_error[256] = "";
}

int cuda_status(cudaError_t e, const char* where) {
  if (e == cudaSuccess) return LORA_OK;
  snprintf(t_last_error, sizeof(t_last_error), "%s: %s (%d)", where, cudaGetErrorString(e), (int)e);
  return LORA_ERR_CUDA;
}

int sm_count(int device) {
  static std::atomic<int> cache[64];  // zero-initialised; 0 = not read yet
  if (device < 0 || device >= 64) return 148;
  int v = cache[device].load(std::memory_order_relaxed);
  if (v == 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || v <= 0) v = 148;
    cache[device].store(v, std::memory_order_relaxed);
  }
  return v;
}

bool set_smem_limit(const void* kernel, int device, int bytes) {
  struct Entry {
    const void* kernel;
    int device, bytes;
  };
  static std::mutex mu;
  static std::vector<Entry> done;
  std::lock_guard<std::mutex> lock(mu);
  for (const Entry& e : done)
    if (e.kernel == kernel && e.device == device && e.bytes >= bytes) return true;
  if (cuda_status(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes),
                  "cudaFuncSetAttribute(max dynamic shared memory)") != LORA_OK)
    return false;
  for (Entry& e : done)
    if (e.kernel == kernel && e.device == device) {
      e.bytes = bytes;
      return true;
    }
  done.push_back({kernel, device, bytes});
  return true;
}

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}
}  // namespace

bool encode_tmap(CUtensorMap* map, CUtensorMapDataType dt, int rank, void* addr, const uint64_t* dims,
                 const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swz) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t gd[5], gs[4];
  cuuint32_t bd[5], es[5];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bd[i] = box[i];
    es[i] = 1;
  }
  for (int i = 0; i + 1 < rank; ++i) gs[i] = strides_bytes[i];
  const CUresult r = fn(map, dt, (cuuint32_t)rank, addr, gd, gs, bd, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Host checks shared by every apply entry point (no GPU work).
int check_apply(const lora_pool* pool, const lora_segments* seg, const void* x, const float* y, int64_t ldx,
                int64_t ldy) {
  if (!pool || !seg || !x || !y) return LORA_ERR_ARG;
  const PoolView& v = pool->v;
  if ((reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(y) & 15)) return LORA_ERR_ARG;
  if (ldx < v.d_in || ldy < v.D || (ldx % 8) || (ldy % 4)) return LORA_ERR_ARG;
  if (seg->N != v.N) return LORA_ERR_SHAPE;
  if (seg->T > v.max_tokens) return LORA_ERR_SHAPE;
  // the kernels run on the current device: the pool and the segments must live there
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return LORA_ERR_CUDA;
  if (dev != v.device || dev != seg->device) return LORA_ERR_ARG;
  return LORA_OK;
}

bool pool_has_adapter(const lora_pool* pool) {
  for (int r : pool->h_rank)
    if (r > 0) return true;
  return false;
}

int run_stage(const PoolView& pool, const lora_segments* seg, const void* x, float* y, int64_t ldx, int64_t ldy,
              int stage, cudaStream_t st) {
  const uint16_t* xb = static_cast<const uint16_t*>(x);
  switch (stage) {
    case 1:
      return launch_decode(pool, seg, xb, ldx, y, ldy, st);
    case 2:
      return launch_tc_shrink(pool, seg, xb, ldx, st);
    case 3:
      return launch_tc_expand(pool, seg, y, ldy, st);
    default:
      return LORA_ERR_ARG;
  }
}

}  // namespace lora

using namespace lora;

namespace {

// A non-blocking side stream and two events per device, created on first use
// (no device memory is allocated).
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  std::mutex mu;
};

SideStream* side_stream() {
  static SideStream sides[64];
  static bool ready[64] = {};
  static std::mutex init_mu;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(init_mu);
  SideStream& s = sides[dev];
  if (!ready[dev]) {
    if (cudaStreamCreateWithFlags(&s.stream, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
    if (cudaEventCreateWithFlags(&s.fork, cudaEventDisableTiming) != cudaSuccess) return nullptr;
    if (cudaEventCreateWithFlags(&s.join, cudaEventDisableTiming) != cudaSuccess) return nullptr;
    ready[dev] = true;
  }
  return &s;
}

}  // namespace

// Creates the current device's side stream and events if they do not exist
// yet (outside any stream capture, from pool creation).
bool lora::ensure_side_stream() { return side_stream() != nullptr; }

extern "C" {

int lora_apply_shrink_expand(const lora_pool* pool, const lora_segments* seg, const void* x, float* y, int64_t ldx,
                             int64_t ldy, lora_stream_t stream) {
  const int chk = check_apply(pool, seg, x, y, ldx, ldy);
  if (chk != LORA_OK) return chk;
  if (seg->T == 0 || !pool_has_adapter(pool)) return LORA_OK;  // a layer no adapter edits launches nothing
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const PoolView& v = pool->v;
  SideStream* side = side_stream();
  if (!side) {
    for (int stage = 1; stage <= 3; ++stage) {
      const int r = run_stage(v, seg, x, y, ldx, ldy, stage, st);
      if (r != LORA_OK) return r;
    }
    return LORA_OK;
  }
  // The decode-path kernel (latency-bound, few bytes) runs on a side stream
  // while the tensor-path kernels (bandwidth-bound) run on the caller's
  // stream; the two touch disjoint rows of y and share only the metadata the
  // segment builder wrote before this call.  Fork and join are events, so the
  // call stays ordered on the caller's stream and can be stream-captured.
  std::lock_guard<std::mutex> lock(side->mu);
  int r = cuda_status(cudaEventRecord(side->fork, st), "cudaEventRecord(fork)");
  if (r == LORA_OK) r = cuda_status(cudaStreamWaitEvent(side->stream, side->fork, 0), "cudaStreamWaitEvent(fork)");
  if (r != LORA_OK) return r;
  const int rd = run_stage(v, seg, x, y, ldx, ldy, 1, side->stream);
  int rt = run_stage(v, seg, x, y, ldx, ldy, 2, st);
  if (rt == LORA_OK) rt = run_stage(v, seg, x, y, ldx, ldy, 3, st);
  // join even after a failed launch, so the caller's stream never runs ahead
  r = cuda_status(cudaEventRecord(side->join, side->stream), "cudaEventRecord(join)");
  if (r == LORA_OK) r = cuda_status(cudaStreamWaitEvent(st, side->join, 0), "cudaStreamWaitEvent(join)");
  if (rd != LORA_OK) return rd;
  if (rt != LORA_OK) return rt;
  return r;
}

int lora_apply_stage(const lora_pool* pool, const lora_segments* seg, const void* x, float* y, int64_t ldx,
                     int64_t ldy, int stage, lora_stream_t stream) {
  const int chk = check_apply(pool, seg, x, y, ldx, ldy);
  if (chk != LORA_OK) return chk;
  if (stage < 1 || stage > 3) return LORA_ERR_ARG;
  if (seg->T == 0 || !pool_has_adapter(pool)) return LORA_OK;
  return run_stage(pool->v, seg, x, y, ldx, ldy, stage, reinterpret_cast<cudaStream_t>(stream));
}

namespace {
int check_fused(const lora_pool* pool, const lora_segments* seg, const void* W, int64_t ldw, const void* x,
                const float* y, int64_t ldx, int64_t ldy) {
  const int chk = check_apply(pool, seg, x, y, ldx, ldy);
  if (chk != LORA_OK) return chk;
  if (!W || (reinterpret_cast<uintptr_t>(W) & 15)) return LORA_ERR_ARG;
  if (ldw < pool->v.d_in || (ldw % 8)) return LORA_ERR_ARG;
  return LORA_OK;
}

int run_fused_stage(const lora_pool* pool, const lora_segments* seg, const void* W, int64_t ldw, const void* x,
                    float* y, int64_t ldx, int64_t ldy, int stage, cudaStream_t st) {
  const uint16_t* xb = static_cast<const uint16_t*>(x);
  switch (stage) {
    case 1:
      return pool_has_adapter(pool) ? launch_decode_rows(pool->v, seg, xb, ldx, st) : LORA_OK;
    case 2:
      return pool_has_adapter(pool) ? launch_tc_shrink_rows(pool->v, seg, xb, ldx, st) : LORA_OK;
    case 3:
      return launch_fused_projection(pool->v, seg, static_cast<const uint16_t*>(W), ldw, xb, ldx, y, ldy, st);
    default:
      return LORA_ERR_ARG;
  }
}
}  // namespace

int lora_apply_fused_projection(const lora_pool* pool, const lora_segments* seg, const void* W, int64_t ldw,
                                const void* x, float* y, int64_t ldx, int64_t ldy, lora_stream_t stream) {
  const int chk = check_fused(pool, seg, W, ldw, x, y, ldx, ldy);
  if (chk != LORA_OK) return chk;
  if (seg->T == 0) return LORA_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  SideStream* side = pool_has_adapter(pool) ? side_stream() : nullptr;
  if (!side) {
    for (int stage = 1; stage <= 3; ++stage) {
      const int r = run_fused_stage(pool, seg, W, ldw, x, y, ldx, ldy, stage, st);
      if (r != LORA_OK) return r;
    }
    return LORA_OK;
  }
  // the decode shrink on the side stream, the tensor shrink on `stream`, joined
  // before the GEMM (the two write disjoint rows of the per-row scratch)
  std::lock_guard<std::mutex> lock(side->mu);
  int r = cuda_status(cudaEventRecord(side->fork, st), "cudaEventRecord(fork)");
  if (r == LORA_OK) r = cuda_status(cudaStreamWaitEvent(side->stream, side->fork, 0), "cudaStreamWaitEvent(fork)");
  if (r != LORA_OK) return r;
  const int rd = run_fused_stage(pool, seg, W, ldw, x, y, ldx, ldy, 1, side->stream);
  const int rt = run_fused_stage(pool, seg, W, ldw, x, y, ldx, ldy, 2, st);
  r = cuda_status(cudaEventRecord(side->join, side->stream), "cudaEventRecord(join)");
  if (r == LORA_OK) r = cuda_status(cudaStreamWaitEvent(st, side->join, 0), "cudaStreamWaitEvent(join)");
  if (rd != LORA_OK) return rd;
  if (rt != LORA_OK) return rt;
  if (r != LORA_OK) return r;
  return run_fused_stage(pool, seg, W, ldw, x, y, ldx, ldy, 3, st);
}

int lora_fused_projection_stage(const lora_pool* pool, const lora_segments* seg, const void* W, int64_t ldw,
                                const void* x, float* y, int64_t ldx, int64_t ldy, int stage,
                                lora_stream_t stream) {
  const int chk = check_fused(pool, seg, W, ldw, x, y, ldx, ldy);
  if (chk != LORA_OK) return chk;
  if (stage < 1 || stage > 3) return LORA_ERR_ARG;
  if (seg->T == 0) return LORA_OK;
  return run_fused_stage(pool, seg, W, ldw, x, y, ldx, ldy, stage, reinterpret_cast<cudaStream_t>(stream));
}

const char* lora_status_string(int status) {
  switch (status) {
    case LORA_OK: return "ok";
    case LORA_ERR_ARG: return "invalid argument (null or misaligned pointer, bad leading dimension)";
    case LORA_ERR_SHAPE: return "unsupported or inconsistent shape";
    case LORA_ERR_SLOT: return "adapter slot id out of range";
    case LORA_ERR_RANK: return "rank out of range";
    case LORA_ERR_CUDA: return "CUDA runtime error";
    case LORA_ERR_META: return "routing metadata inconsistent (negative length or lengths != num_tokens)";
    case LORA_ERR_TIMEOUT: return "a bounded in-kernel wait gave up";
    default: return "unknown status";
  }
}

uint64_t lora_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char* lora_last_error_string(void) { return t_last_error; }

}  // extern "C"
