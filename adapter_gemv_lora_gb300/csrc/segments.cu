// Segment builder: per-sequence adapter ids and query lengths -> per-token
// slots, slot-sorted active rows and the decode / tensor work lists.
//
// Source of the routing rule: xLLM PR #2014 ("multi-tenant LoRA framework",
// Wire-up: adapter_ids holds one entry per sequence, index-aligned with
// q_seq_lens; adapter_ids_per_token is their repeat_interleave; an empty list
// is a no-op).  Slot 0 = base model (tokenspeed PR #976, RequestSpec::lora_id);
// base rows enter no segment (TensorFold PR #47: a row of slot 0 is not read
// or written).  A prompt chunk keeps one slot for all its rows and tiles stay
// inside a sequence (TensorFold PR #47).
//
// One CTA of 512 threads does all of it; every ordering decision is made by
// prefix sums or by a warp-ordered pass, never by atomics, so the output is a
// pure function of the inputs.  Atomics are used only for order-free counts.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>

#include "device.cuh"
#include "internal.h"

namespace lora {
namespace {

constexpr int kSegThreads = 512;  // fewer threads, cheaper barriers: measured faster than 256 or 1024
static_assert(kSegThreads >= 128 && kSegThreads <= 1024 && kSegThreads % 32 == 0, "block scans use 3 warps");
constexpr int kShortSeq = 16;     // sequences up to this length are written by one thread
// Dynamic shared memory the builder may use (227 KB per block, less its static part).
constexpr size_t kSegSmemLimit = 227 * 1024 - 2048;

struct SegParams {
  const int32_t* ids;
  const int32_t* lens;
  int S, T, N;
  const int32_t* S_dev;  // if set, the sequence count is read here (at most S, the layout's capacity)
  int32_t* status;
  int32_t* counts;
  int32_t* seq_start;
  int32_t* slot;
  int32_t* perm;
  int32_t* seg_off;
  int4* dec_work;
  int32_t* dec_rows;
  int4* tc_work;
  int32_t* seq_scratch;  // [6][S] per-sequence arrays when they do not fit in shared memory
  int tables;            // 1: per-warp rank tables in shared memory
};

// Exclusive prefix sum over the block (all threads call it).  `sums` is a
// shared array of >= 33 ints.  Returns the prefix and sets `total`.  Without
// `reuse_sync` the caller must pass a barrier before `sums` is written again.
__device__ int block_exclusive_scan(int v, int* sums, int& total, bool reuse_sync) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < (int)(blockDim.x >> 5) ? sums[lane] : 0;
    int s = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    sums[lane] = s - w;
    if (lane == 31) sums[32] = s;
  }
  __syncthreads();
  const int ex = sums[warp] + x - v;
  total = sums[32];
  if (reuse_sync) __syncthreads();
  return ex;
}

// The three exclusive scans of the offsets at once, in shared memory: rows
// per (class, slot) r[n0] -> o0, decode groups per slot ceil(r[k] / group)
// (k < n1) -> o1, tiles per slot c[n2] -> o2 (each output entry the sum of
// the entries before it).  Each thread takes `per` consecutive entries; the
// totals are returned.  All threads call it; two barriers, and a barrier must
// separate the sources' last writes from the call.
__device__ void block_scan3(const int* r, int* o0, int n0, int* o1, int n1, const int* c, int* o2, int n2, int per,
                            int (*sums)[33], int& t0, int& t1, int& t2) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int lo = threadIdx.x * per;
  auto e0 = [&](int i) { return r[i]; };
  auto e1 = [&](int i) { return (r[i] + kDecGroup - 1) / kDecGroup; };
  auto e2 = [&](int i) { return c[i]; };
  int v0 = 0, v1 = 0, v2 = 0;
  for (int i = 0; i < per; ++i) {
    if (lo + i < n0) v0 += e0(lo + i);
    if (lo + i < n1) v1 += e1(lo + i);
    if (lo + i < n2) v2 += e2(lo + i);
  }
  int x0 = v0, x1 = v1, x2 = v2;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y0 = __shfl_up_sync(0xffffffffu, x0, o);
    const int y1 = __shfl_up_sync(0xffffffffu, x1, o);
    const int y2 = __shfl_up_sync(0xffffffffu, x2, o);
    if (lane >= o) {
      x0 += y0;
      x1 += y1;
      x2 += y2;
    }
  }
  if (lane == 31) {
    sums[0][warp] = x0;
    sums[1][warp] = x1;
    sums[2][warp] = x2;
  }
  __syncthreads();
  if (warp < 3) {
    const int w = lane < (int)(blockDim.x >> 5) ? sums[warp][lane] : 0;
    int x = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    sums[warp][lane] = x - w;
    if (lane == 31) sums[warp][32] = x;
  }
  __syncthreads();
  int c0 = sums[0][warp] + x0 - v0, c1 = sums[1][warp] + x1 - v1, c2 = sums[2][warp] + x2 - v2;
  for (int i = 0; i < per; ++i) {
    if (lo + i < n0) {
      o0[lo + i] = c0;
      c0 += e0(lo + i);
    }
    if (lo + i < n1) {
      o1[lo + i] = c1;
      c1 += e1(lo + i);
    }
    if (lo + i < n2) {
      o2[lo + i] = c2;
      c2 += e2(lo + i);
    }
  }
  t0 = sums[0][32];
  t1 = sums[1][32];
  t2 = sums[2][32];
}

// One warp writes dst[j] = v0 + j * step for j < n, with 16-byte stores
// wherever the destination is aligned.
__device__ __forceinline__ void warp_fill(int32_t* dst, int n, int v0, int step, int lane) {
  const int head = min(n, (int)((4 - ((reinterpret_cast<uintptr_t>(dst) >> 2) & 3)) & 3));
  if (lane < head) dst[lane] = v0 + lane * step;
  int4* d4 = reinterpret_cast<int4*>(dst + head);
  const int n4 = (n - head) >> 2;
  for (int i = lane; i < n4; i += 32) {
    const int b = v0 + (head + 4 * i) * step;
    d4[i] = make_int4(b, b + step, b + 2 * step, b + 3 * step);
  }
  for (int j = head + 4 * n4 + lane; j < n; j += 32) dst[j] = v0 + j * step;
}

// Shared memory of the builder, in ints: the per-key tables
// (2N + 2N + N + (N + 1) + (N + 1)), then, when they fit, six per-sequence
// arrays of S (else those live in the workspace's sequence scratch).
size_t seg_key_ints(int N) { return 7 * (size_t)N + 2; }
bool seq_arrays_in_smem(int N, int S) { return sizeof(int) * (seg_key_ints(N) + 6 * (size_t)S) <= kSegSmemLimit; }
// Per-warp rank tables ([warps][2N] rows and [warps][N] tiles of one chunk of
// sequences), used when they fit after the arrays above: every warp then
// ranks its sequences against the earlier warps at once instead of one warp
// walking the chunk.
constexpr int kSegWarps = kSegThreads / 32;
size_t seg_table_ints(int N) { return (size_t)kSegWarps * 3 * N; }

// SEQ_SMEM: the per-sequence arrays are in shared memory (the compiler then
// knows every access to them is a shared one), else in the workspace.
template <bool SEQ_SMEM>
__global__ void __launch_bounds__(kSegThreads, 1) seg_build_kernel(SegParams p) {
  extern __shared__ int smem_dyn[];
  __shared__ int scan_sums[3][33];
  __shared__ int bad_sh, long_sh;
  __shared__ unsigned long long len_sh;
  const int N = p.N, Scap = p.S, T = p.T;
  int* cnt_tok = smem_dyn;         // [2N] rows per (class, slot), then their first perm position
  int* run_tok = cnt_tok + 2 * N;  // [2N] running position while ranking sequences
  int* cnt_tile = run_tok + 2 * N; // [N]  class-1 tiles per slot, then the first tile index
  int* dec_cnt = cnt_tile + N;     // [N+1] decode groups per slot, then the first group index
  int* tc_cnt = dec_cnt + N + 1;   // [N+1] class-1 tiles per slot (scan input), then the first tile
  int* seqa = SEQ_SMEM ? tc_cnt + N + 1 : p.seq_scratch;
  int* s_len = seqa;                // [S] q_len
  int* s_id = s_len + Scap;         // [S] slot
  int* s_start = s_id + Scap;       // [S] first row
  int* s_pos = s_start + Scap;      // [S] rank of the first row inside its (class, slot) bin
  int* s_tile = s_pos + Scap;       // [S] rank of the first tile inside its slot's tiles
  int* s_key = s_tile + Scap;       // [S] (class, slot) key, -1 if the sequence is inactive; bits 24..28:
                                    //     the last lane of its warp with the same key
  int* tab_rows = tc_cnt + N + 1 + (SEQ_SMEM ? 6 * Scap : 0);  // [warps][2N] (when p.tables)
  int* tab_tiles = tab_rows + kSegWarps * 2 * N;               // [warps][N]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kLeadShift = 24, kKeyMask = (1 << kLeadShift) - 1;  // keys < 2N <= 4096

  // Shared state first: it does not depend on the previous kernel, so it is
  // set while that kernel finishes.  The rank tables start at zero; each
  // chunk's last pass over them sets them back to zero.
  for (int i = tid; i < 2 * N; i += kSegThreads) run_tok[i] = 0;
  for (int i = tid; i < N; i += kSegThreads) cnt_tile[i] = 0;
  if (p.tables)
    for (int i = tid; i < kSegWarps * 3 * N; i += kSegThreads) tab_rows[i] = 0;
  if (tid == 0) {
    bad_sh = 0;
    long_sh = 0;
    len_sh = 0ull;
  }
  pdl_launch_next();  // the apply kernels may be scheduled now; they wait for this grid
  pdl_wait();         // the previous kernel's results are visible from here on
  // the sequence count (from the device when a run-length pass wrote it)
  const int S = p.S_dev ? min(max(*p.S_dev, 0), Scap) : Scap;

  // ---- per sequence, 512 at a time: length, slot, key, first row (block
  // scan), and its rank among the earlier lanes of its warp with the same
  // key (rows and tiles; lanes of one key found with one match)
  int carry = 0;
  for (int b = 0; b < S; b += kSegThreads) {
    const int s = b + tid;
    int key = -1, len = 0, nt = 0;
    int bad = 0;  // bit 0: a negative length, bit 1: an id out of range
    if (s < S) {
      len = p.lens[s];
      const int id = p.ids[s];
      bad = (len < 0 ? 1 : 0) | ((id < 0 || id >= N) ? 2 : 0);
      s_len[s] = len;
      s_id[s] = id;
      if (id > 0 && id < N && len > 0) {
        const int cls = len >= LORA_TC_MIN_QLEN ? 1 : 0;
        key = cls * N + id;
        nt = cls ? (len + kTcTile - 1) / kTcTile : 0;
      }
    }
    const unsigned m = __match_any_sync(0xffffffffu, key);
    const unsigned below = m & ((1u << lane) - 1u);
    const int lead = 31 - __clz(m);
    int pl, pt;
    // when every lane of a key has the same length the rank is a count
    const unsigned m_len = __match_any_sync(0xffffffffu, ((unsigned long long)(unsigned)key << 32) | (unsigned)len);
    if (__all_sync(0xffffffffu, m_len == m)) {
      pl = __popc(below) * len;
      pt = __popc(below) * nt;
    } else {
      pl = pt = 0;
      unsigned rem = below;
      while (__any_sync(0xffffffffu, rem != 0)) {
        const int j = rem ? __ffs(rem) - 1 : lane;
        const int lj = __shfl_sync(0xffffffffu, len, j), tj = __shfl_sync(0xffffffffu, nt, j);
        if (rem) {
          pl += lj;
          pt += tj;
          rem &= rem - 1u;
        }
      }
    }
    int tot;
    // (with the tables, their two barriers below come before the sums are reused)
    const int ex = block_exclusive_scan(s < S ? len : 0, scan_sums[0], tot, !p.tables);
    {
      // validation: order-free reductions, one shared atomic per warp and chunk
      // (after the scan's barriers, so after thread 0 cleared the sums)
      long long wl = len;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) wl += __shfl_xor_sync(0xffffffffu, wl, o);
      const int wb = (int)__reduce_or_sync(0xffffffffu, (unsigned)bad);
      const bool wlong = __any_sync(0xffffffffu, len > kShortSeq);
      if (lane == 0) {
        if (wb) atomicOr(&bad_sh, wb);
        if (wl) atomicAdd(&len_sh, (unsigned long long)wl);
        if (wlong) long_sh = 1;
      }
    }
    if (s < S) {
      s_start[s] = carry + ex;
      p.seq_start[s] = carry + ex;
      s_pos[s] = pl;
      s_tile[s] = pt;
      s_key[s] = key < 0 ? -1 : (key | (lead << kLeadShift));
    }
    carry += tot;
    if (p.tables) {
      // stable ranks of this chunk: each warp's per-key totals go to its row
      // of the tables; a sequence adds the rows of the earlier warps and the
      // running counts of the earlier chunks; then the counts advance
      const bool tc = key >= N;
      const int id = tc ? key - N : key;
      // (the tables are zero: cleared before the first chunk, and by the
      // previous chunk's last pass, both ordered by the scan's barriers)
      if (key >= 0 && lead == lane) {
        tab_rows[warp * 2 * N + key] = pl + len;
        if (tc) tab_tiles[warp * N + id] = pt + nt;
      }
      __syncthreads();
      if (key >= 0) {
        int br = run_tok[key], bt = tc ? cnt_tile[id] : 0;
        for (int w = 0; w < warp; ++w) {
          br += tab_rows[w * 2 * N + key];
          if (tc) bt += tab_tiles[w * N + id];
        }
        s_pos[s] = br + pl;
        if (tc) s_tile[s] = bt + pt;
      }
      __syncthreads();  // every read of the running counts and of the tables is done
      for (int k = tid; k < 2 * N; k += kSegThreads) {
        int add = 0;
#pragma unroll
        for (int w = 0; w < kSegWarps; ++w) {
          add += tab_rows[w * 2 * N + k];
          tab_rows[w * 2 * N + k] = 0;
        }
        run_tok[k] += add;
      }
      for (int k = tid; k < N; k += kSegThreads) {
        int add = 0;
#pragma unroll
        for (int w = 0; w < kSegWarps; ++w) {
          add += tab_tiles[w * N + k];
          tab_tiles[w * N + k] = 0;
        }
        cnt_tile[k] += add;
      }
      // the next chunk's block scan has barriers before its tables are cleared
    }
  }
  // the validation sums are complete: with the tables, barriers in the loop
  // follow every chunk's atomics; without them, this one
  if (!p.tables || S == 0) __syncthreads();
  {
    const int bb = bad_sh;
    if ((bb & 1) || len_sh != (unsigned long long)(long long)T || (bb & 2)) {
      if (tid < 4) p.counts[tid] = 0;
      if (tid == 0) *p.status = ((bb & 1) || len_sh != (unsigned long long)(long long)T) ? LORA_ERR_META
                                                                                        : LORA_ERR_SLOT;
      return;
    }
  }
  if (tid == 0) p.seq_start[S] = T;

  // ---- stable ranks (without the tables): one warp walks the sequences 32
  // at a time in index order; the per-key running counts end as the rows per
  // (class, slot) and the tiles per slot
  if (!p.tables && warp == 0) {
    for (int b = 0; b < S; b += 32) {
      const int s = b + lane, sc = min(s, S - 1);
      const int kk = s_key[sc], pl = s_pos[sc], pt = s_tile[sc], len = s_len[sc];
      const bool act = s < S && kk >= 0;
      const int key = act ? (kk & kKeyMask) : 0;
      const int lead = act ? (kk >> kLeadShift) : lane;
      const bool tc = key >= N, last = act && lead == lane;
      const int id = tc ? key - N : key;
      // the last lane of each key reads and advances the running counts; the
      // other lanes of the key take the base from it
      int rt = 0, ct = 0;
      if (last) {
        rt = run_tok[key];
        ct = cnt_tile[id];
      }
      const int base_tok = __shfl_sync(0xffffffffu, rt, lead);
      const int base_tile = __shfl_sync(0xffffffffu, ct, lead);
      if (act) {
        s_pos[s] = base_tok + pl;
        if (tc) s_tile[s] = base_tile + pt;
      }
      if (last) {
        run_tok[key] = base_tok + pl + len;
        if (tc) cnt_tile[id] = base_tile + pt + (len + kTcTile - 1) / kTcTile;
      }
      __syncwarp();  // this chunk's counts are visible to the next chunk's reads
    }
  }
  __syncthreads();

  // ---- offsets: rows (class-major), decode groups per slot, tiles per slot
  int n_active, n_dec_work, n_tc;
  block_scan3(run_tok, cnt_tok, 2 * N, dec_cnt, N, cnt_tile, tc_cnt, N, (2 * N + kSegThreads - 1) / kSegThreads,
              scan_sums, n_active, n_dec_work, n_tc);
  if (tid == 0) {
    dec_cnt[N] = n_dec_work;
    tc_cnt[N] = n_tc;
  }
  __syncthreads();
  // cnt_tok = first perm position of each (class, slot); run_tok = its rows
  for (int i = tid; i < 2 * (N + 1); i += kSegThreads) {
    const int c = i / (N + 1), k = i % (N + 1);
    p.seg_off[i] = (k < N) ? cnt_tok[c * N + k] : (c == 0 ? cnt_tok[N] : n_active);
  }

  // ---- per-token slot and perm, and the tensor tiles.  A thread writes the
  // rows of each short sequence it owns (decode rows); the longer ones are
  // dealt out to the warps in index order (the k-th long sequence to warp
  // k mod warps), one warp to a sequence.
  for (int s = tid; s < S; s += kSegThreads) {
    const int kk = s_key[s], len = s_len[s], id = s_id[s], st = s_start[s];
    if (len <= kShortSeq) {
      const int pos = kk < 0 ? 0 : cnt_tok[kk & kKeyMask] + s_pos[s];
      const bool dec = kk >= 0 && (kk & kKeyMask) < N;  // decode rows also go to their group's row list
      const int g0 = dec ? dec_cnt[kk & kKeyMask] * kDecGroup + s_pos[s] : 0;
      for (int j = 0; j < len; ++j) {
        p.slot[st + j] = id;
        if (kk >= 0) p.perm[pos + j] = st + j;
        if (dec) p.dec_rows[g0 + j] = st + j;
      }
    }
    // each class-1 sequence cut into tiles of <= kTcTile rows
    if (kk >= 0 && (kk & kKeyMask) >= N) {
      const int base = tc_cnt[id] + s_tile[s];
      for (int i = 0, rb = st; rb < st + len; ++i, rb += kTcTile)
        p.tc_work[base + i] = make_int4(id, rb, min(rb + kTcTile, st + len), s);
    }
  }
  if (long_sh) {  // a step of decode rows only has none
    int n_long = 0;  // long sequences before this chunk
    for (int b = 0; b < S; b += 32) {
      const int s = b + lane;
      const unsigned lm = __ballot_sync(0xffffffffu, s < S && s_len[s] > kShortSeq);
      for (unsigned r = lm; r; r &= r - 1u, ++n_long) {
        if (n_long % (kSegThreads / 32) != warp) continue;
        const int sq = b + __ffs(r) - 1;
        const int id = s_id[sq], st = s_start[sq], len = s_len[sq], kk = s_key[sq];
        warp_fill(p.slot + st, len, id, 0, lane);
        if (kk >= 0) warp_fill(p.perm + cnt_tok[kk & kKeyMask] + s_pos[sq], len, st, 1, lane);
        if (kk >= 0 && (kk & kKeyMask) < N)  // decode rows (a sequence shorter than the tensor threshold)
          warp_fill(p.dec_rows + dec_cnt[kk & kKeyMask] * kDecGroup + s_pos[sq], len, st, 1, lane);
      }
    }
  }

  // ---- decode groups: slot k's class-0 run cut into runs of <= kDecGroup
  for (int w = tid; w < n_dec_work; w += kSegThreads) {
    int lo = 0, hi = N - 1;  // last k with dec_cnt[k] <= w
    while (lo < hi) {
      int mid = (lo + hi + 1) >> 1;
      if (dec_cnt[mid] <= w) lo = mid; else hi = mid - 1;
    }
    const int k = lo;
    const int gi = w - dec_cnt[k];
    const int pb = cnt_tok[k] + gi * kDecGroup;
    const int pe = min(pb + kDecGroup, cnt_tok[k] + run_tok[k]);
    p.dec_work[w] = make_int4(k, pb, pe, 0);
  }

  if (tid == 0) {
    p.counts[0] = n_active;
    p.counts[1] = cnt_tok[N];
    p.counts[2] = n_dec_work;
    p.counts[3] = n_tc;
    *p.status = LORA_OK;
  }
}

// Dispatched rows of an MoE layer -> the builder's sequences.  After routing,
// the rows of each expert are contiguous and, inside an expert, the rows of
// one sequence are contiguous; a maximal run of rows with the same (expert,
// sequence, adapter) becomes one sequence whose slot is the expert's copy of
// the adapter (1 + e * A + (a - 1); adapter 0 is the base model) and whose
// length is the run's length (xLLM PR #2014, "Not in this PR": the fused MoE
// expert LoRA delta by a grouped GEMM).  So a run of a prompt chunk's tokens
// routed to one expert is a dense tile on the tensor path exactly when enough
// of the chunk's own tokens chose that expert; other sequences never change
// it.  One CTA: a block scan of the run-start flags.  An expert or adapter id
// out of range gives the run slot N, which the builder reports as
// LORA_ERR_SLOT; more runs than the capacity give no runs, which the builder
// reports as LORA_ERR_META.
struct MoeRunParams {
  const int32_t* row_expert;
  const int32_t* row_adapter;
  const int32_t* row_seq;
  int T, E, A, N, cap;
  int32_t* run_ids;
  int32_t* run_lens;
  int32_t* run_starts;  // scratch (the builder rewrites this array as its seq_start)
  int32_t* run_count;
};

constexpr int kRunThreads = 1024;

__global__ void __launch_bounds__(kRunThreads, 1) moe_runs_kernel(MoeRunParams p) {
  __shared__ int sums[33];
  pdl_wait();  // the previous kernel's results are visible from here on
  int carry = 0;
  for (int b = 0; b < p.T; b += kRunThreads) {
    const int r = b + threadIdx.x;
    int flag = 0, slot = 0;
    if (r < p.T) {
      const int e = p.row_expert[r], sq = p.row_seq[r], a = p.row_adapter[r];
      flag = r == 0 || e != p.row_expert[r - 1] || sq != p.row_seq[r - 1] || a != p.row_adapter[r - 1];
      slot = (e < 0 || e >= p.E || a < 0 || a > p.A) ? p.N : (a == 0 ? 0 : 1 + e * p.A + (a - 1));
    }
    int tot;
    const int idx = carry + block_exclusive_scan(flag, sums, tot, true);
    if (flag && idx < p.cap) {
      p.run_ids[idx] = slot;
      p.run_starts[idx] = r;
    }
    carry += tot;
  }
  __syncthreads();  // every run start is written (and visible to the block)
  const int n = carry <= p.cap ? carry : 0;
  for (int i = threadIdx.x; i < n; i += kRunThreads)
    p.run_lens[i] = (i + 1 < n ? p.run_starts[i + 1] : p.T) - p.run_starts[i];
  if (threadIdx.x == 0) *p.run_count = n;
  pdl_launch_next();  // the builder may be scheduled; it waits for this grid
}

}  // namespace

int launch_moe_runs(lora_segments* seg, const int32_t* row_expert, const int32_t* row_adapter,
                    const int32_t* row_seq, int T, int E, int A, cudaStream_t st) {
  MoeRunParams p;
  p.row_expert = row_expert;
  p.row_adapter = row_adapter;
  p.row_seq = row_seq;
  p.T = T;
  p.E = E;
  p.A = A;
  p.N = seg->N;
  p.cap = T < seg->max_seqs ? T : seg->max_seqs;
  p.run_ids = seg->run_ids;
  p.run_lens = seg->run_lens;
  p.run_starts = seg->seq_start;
  p.run_count = seg->counts + 8;
  const cudaError_t e = launch_pdl(moe_runs_kernel, dim3(1), dim3(kRunThreads), 0, st, p);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cuda_status(e != cudaSuccess ? e : cudaGetLastError(), "moe_runs_kernel launch");
}

int launch_seg_build(lora_segments* seg, const int32_t* ids, const int32_t* lens, int S, int T,
                     cudaStream_t st, const int32_t* S_dev) {
  SegParams p;
  p.ids = ids;
  p.lens = lens;
  p.S = S;
  p.S_dev = S_dev;
  p.T = T;
  p.N = seg->N;
  p.status = seg->status;
  p.counts = seg->counts;
  p.seq_start = seg->seq_start;
  p.slot = seg->slot;
  p.perm = seg->perm;
  p.seg_off = seg->seg_off;
  p.dec_work = seg->dec_work;
  p.dec_rows = seg->dec_rows;
  p.tc_work = seg->tc_work;
  p.seq_scratch = seg->seq_scratch;
  const bool in_smem = seq_arrays_in_smem(seg->N, S);
  size_t sm = sizeof(int) * (seg_key_ints(seg->N) + (in_smem ? 6 * (size_t)S : 0));
  p.tables = sm + sizeof(int) * seg_table_ints(seg->N) <= kSegSmemLimit ? 1 : 0;
  if (p.tables) sm += sizeof(int) * seg_table_ints(seg->N);
  auto kern = in_smem ? seg_build_kernel<true> : seg_build_kernel<false>;
  if (sm > 48 * 1024 && !set_smem_limit(reinterpret_cast<const void*>(kern), seg->device, (int)sm))
    return LORA_ERR_CUDA;
  const cudaError_t e = launch_pdl(kern, dim3(1), dim3(kSegThreads), sm, st, p);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cuda_status(e != cudaSuccess ? e : cudaGetLastError(), "seg_build_kernel launch");
}

}  // namespace lora

using namespace lora;

namespace {

struct SegLayout {
  size_t status, counts, seq_start, slot, perm, seg_off, dec_work, dec_rows, tc_work, run_ids, run_lens, seq_scratch,
      total;
  int cap_dec, cap_tc;
};

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

bool seg_layout(int max_seqs, int max_tokens, int N, SegLayout* L) {
  if (max_seqs < 1 || max_tokens < 1 || N < 2 || N > LORA_MAX_SLOTS) return false;
  // the builder keeps every slot's counters in shared memory
  if (sizeof(int) * seg_key_ints(N) > kSegSmemLimit) return false;
  L->cap_dec = ceil_div(max_tokens, kDecGroup) + N;
  L->cap_tc = ceil_div(max_tokens, kTcTile) + max_seqs;
  size_t o = 0;
  L->status = o; o += 64;
  L->counts = o; o = align256(o + 64);
  L->seq_start = o; o = align256(o + 4 * (size_t)(max_seqs + 1));
  L->slot = o; o = align256(o + 4 * (size_t)max_tokens);
  L->perm = o; o = align256(o + 4 * (size_t)max_tokens);
  L->seg_off = o; o = align256(o + 4 * (size_t)(2 * (N + 1)));
  L->dec_work = o; o = align256(o + 16 * (size_t)L->cap_dec);
  L->dec_rows = o; o = align256(o + 4 * (size_t)kDecGroup * L->cap_dec);
  L->tc_work = o; o = align256(o + 16 * (size_t)L->cap_tc);
  L->run_ids = o; o = align256(o + 4 * (size_t)max_seqs);
  L->run_lens = o; o = align256(o + 4 * (size_t)max_seqs);
  // per-sequence arrays of the builder for steps whose sequences do not fit in shared memory
  L->seq_scratch = o;
  if (!seq_arrays_in_smem(N, max_seqs)) o = align256(o + 4 * 6 * (size_t)max_seqs);
  L->total = o;
  return true;
}

}  // namespace

extern "C" {

size_t lora_segments_bytes(int max_seqs, int max_tokens, int num_slots) {
  SegLayout L;
  return seg_layout(max_seqs, max_tokens, num_slots, &L) ? L.total : 0;
}

int lora_segments_create(lora_segments** out, void* dev_ws, size_t ws_bytes, int max_seqs, int max_tokens,
                         int num_slots) {
  if (!out || !dev_ws || (reinterpret_cast<uintptr_t>(dev_ws) & 255)) return LORA_ERR_ARG;
  SegLayout L;
  if (!seg_layout(max_seqs, max_tokens, num_slots, &L)) return LORA_ERR_SHAPE;
  if (ws_bytes < L.total) return LORA_ERR_SHAPE;
  lora_segments* s = new lora_segments();
  if (cudaGetDevice(&s->device) != cudaSuccess) {
    delete s;
    return LORA_ERR_CUDA;
  }
  char* b = static_cast<char*>(dev_ws);
  s->ws = b;
  s->bytes = ws_bytes;
  s->max_seqs = max_seqs;
  s->max_tokens = max_tokens;
  s->N = num_slots;
  s->cap_dec = L.cap_dec;
  s->cap_tc = L.cap_tc;
  s->status = reinterpret_cast<int32_t*>(b + L.status);
  s->counts = reinterpret_cast<int32_t*>(b + L.counts);
  s->seq_start = reinterpret_cast<int32_t*>(b + L.seq_start);
  s->slot = reinterpret_cast<int32_t*>(b + L.slot);
  s->perm = reinterpret_cast<int32_t*>(b + L.perm);
  s->seg_off = reinterpret_cast<int32_t*>(b + L.seg_off);
  s->dec_work = reinterpret_cast<int4*>(b + L.dec_work);
  s->dec_rows = reinterpret_cast<int32_t*>(b + L.dec_rows);
  s->tc_work = reinterpret_cast<int4*>(b + L.tc_work);
  s->run_ids = reinterpret_cast<int32_t*>(b + L.run_ids);
  s->run_lens = reinterpret_cast<int32_t*>(b + L.run_lens);
  s->seq_scratch = reinterpret_cast<int32_t*>(b + L.seq_scratch);
  *out = s;
  return LORA_OK;
}

int lora_build_segments(lora_segments* seg, const int32_t* adapter_ids, const int32_t* q_seq_lens, int num_seqs,
                        int num_tokens, lora_stream_t stream) {
  if (!seg) return LORA_ERR_ARG;
  if (num_seqs < 0 || num_tokens < 0) return LORA_ERR_SHAPE;
  if (num_seqs > seg->max_seqs || num_tokens > seg->max_tokens) return LORA_ERR_SHAPE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (num_seqs == 0) {
    // Empty step (an empty adapter id list): nothing to route, no kernel.
    if (num_tokens != 0) return LORA_ERR_SHAPE;
    seg->S = 0;
    seg->T = 0;
    if (cudaMemsetAsync(seg->counts, 0, 16, st) != cudaSuccess) return LORA_ERR_CUDA;
    return cudaMemsetAsync(seg->status, 0, 4, st) == cudaSuccess ? LORA_OK : LORA_ERR_CUDA;
  }
  if (!adapter_ids || !q_seq_lens) return LORA_ERR_ARG;
  int dev = -1;  // the builder runs on the current device, where the workspace must live
  if (cudaGetDevice(&dev) != cudaSuccess) return LORA_ERR_CUDA;
  if (dev != seg->device) return LORA_ERR_ARG;
  seg->S = num_seqs;
  seg->T = num_tokens;
  return launch_seg_build(seg, adapter_ids, q_seq_lens, num_seqs, num_tokens, st);
}

int lora_moe_slot(int expert, int adapter, int num_adapters) {
  return adapter == 0 ? 0 : 1 + expert * num_adapters + (adapter - 1);
}

int lora_build_segments_moe(lora_segments* seg, const int32_t* row_expert, const int32_t* row_adapter,
                            const int32_t* row_seq, int num_rows, int num_experts, int num_adapters,
                            lora_stream_t stream) {
  if (!seg) return LORA_ERR_ARG;
  if (num_rows < 0 || num_experts < 1 || num_adapters < 1) return LORA_ERR_SHAPE;
  if ((long long)num_experts * num_adapters + 1 != seg->N) return LORA_ERR_SHAPE;
  if (num_rows > seg->max_tokens) return LORA_ERR_SHAPE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (num_rows == 0) {  // no dispatched rows: nothing to route, no kernel
    seg->S = 0;
    seg->T = 0;
    if (cudaMemsetAsync(seg->counts, 0, 16, st) != cudaSuccess) return LORA_ERR_CUDA;
    return cudaMemsetAsync(seg->status, 0, 4, st) == cudaSuccess ? LORA_OK : LORA_ERR_CUDA;
  }
  if (!row_expert || !row_adapter || !row_seq) return LORA_ERR_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return LORA_ERR_CUDA;
  if (dev != seg->device) return LORA_ERR_ARG;
  // the runs are at most the rows and at most the capacity (more runs than
  // max_seqs is a device-detected LORA_ERR_META): the builder's layout and
  // the launchers' bounds take that many sequences
  const int cap = num_rows < seg->max_seqs ? num_rows : seg->max_seqs;
  seg->S = cap;
  seg->T = num_rows;
  const int r = launch_moe_runs(seg, row_expert, row_adapter, row_seq, num_rows, num_experts, num_adapters, st);
  if (r != LORA_OK) return r;
  return launch_seg_build(seg, seg->run_ids, seg->run_lens, cap, num_rows, st, seg->counts + 8);
}

int lora_segments_capacity(const lora_segments* seg, int* dec_work_cap, int* tc_work_cap) {
  if (!seg) return LORA_ERR_ARG;
  if (dec_work_cap) *dec_work_cap = seg->cap_dec;
  if (tc_work_cap) *tc_work_cap = seg->cap_tc;
  return LORA_OK;
}

int lora_segments_read(const lora_segments* seg, int32_t* host_slot, int32_t* host_perm, int32_t* host_seg_off,
                       int32_t* host_counts, int32_t* host_dec_work, int32_t* host_tc_work, lora_stream_t stream) {
  if (!seg) return LORA_ERR_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int32_t counts[4];
  if (cudaMemcpyAsync(counts, seg->counts, 16, cudaMemcpyDeviceToHost, st) != cudaSuccess) return LORA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return LORA_ERR_CUDA;
  const int T = seg->T;
  auto cp = [&](void* dst, const void* src, size_t n) {
    return n == 0 || cudaMemcpyAsync(dst, src, n, cudaMemcpyDeviceToHost, st) == cudaSuccess;
  };
  bool ok = true;
  if (host_counts) std::memcpy(host_counts, counts, 16);
  if (host_slot && T > 0) ok &= cp(host_slot, seg->slot, 4 * (size_t)T);
  if (host_perm) ok &= cp(host_perm, seg->perm, 4 * (size_t)std::max(0, counts[0]));
  if (host_seg_off) ok &= cp(host_seg_off, seg->seg_off, 4 * (size_t)(2 * (seg->N + 1)));
  if (host_dec_work) ok &= cp(host_dec_work, seg->dec_work, 16 * (size_t)std::max(0, counts[2]));
  if (host_tc_work) ok &= cp(host_tc_work, seg->tc_work, 16 * (size_t)std::max(0, counts[3]));
  if (!ok) return LORA_ERR_CUDA;
  return cudaStreamSynchronize(st) == cudaSuccess ? LORA_OK : LORA_ERR_CUDA;
}

int lora_segments_read_dec_rows(const lora_segments* seg, int32_t* host_rows, lora_stream_t stream) {
  if (!seg || !host_rows) return LORA_ERR_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int32_t counts[4];
  if (cudaMemcpyAsync(counts, seg->counts, 16, cudaMemcpyDeviceToHost, st) != cudaSuccess) return LORA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return LORA_ERR_CUDA;
  const size_t n = (size_t)std::max(0, counts[2]) * kDecGroup;
  if (n > 0 && cudaMemcpyAsync(host_rows, seg->dec_rows, 4 * n, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return LORA_ERR_CUDA;
  return cudaStreamSynchronize(st) == cudaSuccess ? LORA_OK : LORA_ERR_CUDA;
}

int lora_get_status(const lora_segments* seg, int32_t* host_status, lora_stream_t stream) {
  if (!seg || !host_status) return LORA_ERR_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(host_status, seg->status, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return LORA_ERR_CUDA;
  return cudaStreamSynchronize(st) == cudaSuccess ? LORA_OK : LORA_ERR_CUDA;
}

int lora_clear_status(lora_segments* seg, lora_stream_t stream) {
  if (!seg) return LORA_ERR_ARG;
  return cudaMemsetAsync(seg->status, 0, 4, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? LORA_OK
             : LORA_ERR_CUDA;
}

int lora_segments_destroy(lora_segments* seg) {
  delete seg;
  return LORA_OK;
}

}  // extern "C"
