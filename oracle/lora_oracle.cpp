// Plain CPU oracle for the mixed-adapter batched LoRA delta.
//
// TEST INFRASTRUCTURE ONLY.  Only the test suite, the package's smoke check
// and the benchmark's CPU-baseline leg may load this library.  It shares no
// code, header, table or constant with the CUDA path: every layout parameter
// (tile rows, group rows, tensor-path threshold) is passed in as an argument.
//
// What it computes, and where the pages state it:
//
//  * Routing metadata.  One adapter id per sequence, index-aligned with the
//    query lengths; the per-token id is the per-sequence id repeated over the
//    sequence's tokens (xLLM PR #2014, "Wire-up", ModelInputParams::adapter_ids
//    and adapter_ids_per_token built with repeat_interleave).  Id 0 is the base
//    model (tokenspeed PR #976, RequestSpec::lora_id).  Rows of id 0 are not
//    part of any segment (TensorFold PR #47, "a row of slot 0 is not read or
//    written").  A prompt chunk uses one slot for all its rows (TensorFold PR
//    #47), so row tiles never cross a sequence.
//
//  * The delta.  For a row t with slot k != 0 and every lane l whose rank
//    r = rank[k][l] > 0:
//        u_i  = sum_j A[k][l][i][j] * x[t][j]          (i < r, j ascending)
//        v_o  = sum_i B[k][l][o][i] * u_i              (i ascending)
//        y[t][off_l + o] = y0[t][off_l + o] + scale[k][l] * v_o
//    i.e. y += scale * B @ (A @ x) (TensorFold PR #47, "the delta scale * B @
//    (A @ x) is added to the fp32 partial sum"), with A stored [r, d_in] and B
//    stored [d_out, r] (xLLM PR #2014, LoRAQKVParallelLinear: B.size(0) is the
//    lane's output width).  Lanes are laid side by side in y in lane order
//    (fused q,k,v or gate,up outputs; xLLM PR #2014 LoRAQKVParallelLinear and
//    LoRAColumnParallelLinear).  Rows of slot 0, and lanes of rank 0, keep y0.
//    Everything is evaluated in double precision from the bf16 / fp32 inputs.
//
// Readings where the pages are silent are listed with the tests that pin them.

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <numeric>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

// bf16 bit pattern -> double.  A bf16 value is the upper half of an IEEE
// binary32 word; widening is a 16-bit shift, exact.
double bf16_to_double(uint16_t h) {
  uint32_t w = static_cast<uint32_t>(h) << 16;
  float f;
  std::memcpy(&f, &w, sizeof(f));
  return static_cast<double>(f);
}

enum { ST_OK = 0, ST_SLOT = -3, ST_META = -6 };

}  // namespace

extern "C" {

// Routing metadata of one step.
//
//   adapter_ids[S], q_seq_lens[S]  per-sequence slot and query length
//   T                              number of token rows the caller declares
//   N                              number of slots, slot 0 = base
//   tc_min_qlen                    a row whose own sequence has q_len >= this
//                                  takes the tensor path (class 1), else the
//                                  decode path (class 0)
//   tile_rows                      rows per tensor-path tile (tiles stay inside
//                                  one sequence)
//   group_rows                     rows per decode work group (groups stay
//                                  inside one slot's decode segment)
//
// Outputs (caller-sized):
//   slot[T]        per-token slot
//   seq_start[S+1] exclusive prefix of q_seq_lens
//   perm[T]        active rows (slot != 0) ordered by (class, slot, row);
//                  only the first counts[0] entries are defined
//   seg_off[2*(N+1)]  seg_off[c*(N+1)+k] = first perm position of (class c,
//                  slot k); seg_off[c*(N+1)+N] = end of class c
//   dec_work[..][4]   {slot, perm_begin, perm_end, 0}: class-0 rows of one slot
//                  cut into consecutive runs of <= group_rows, in perm order
//   tc_work[..][4]    {slot, row_begin, row_end, seq}: each class-1 sequence
//                  cut into consecutive tiles of <= tile_rows rows, in the order
//                  of the sequences' perm positions
//   counts[4]      {active rows, class-0 rows, #dec_work, #tc_work}
// Returns the status: 0, -6 (a negative length or lengths not summing to T),
// -3 (an id outside [0, N)).  -6 takes precedence.  On error every count is 0.
int oracle_segments(int S, int T, int N, int tc_min_qlen, int tile_rows, int group_rows,
                    const int32_t* adapter_ids, const int32_t* q_seq_lens,
                    int32_t* slot, int32_t* seq_start, int32_t* perm, int32_t* seg_off,
                    int32_t* dec_work, int32_t* tc_work, int32_t* counts) {
  for (int i = 0; i < 4; ++i) counts[i] = 0;
  // Validation.
  bool bad_len = false, bad_id = false;
  long long total = 0;
  for (int s = 0; s < S; ++s) {
    if (q_seq_lens[s] < 0) bad_len = true;
    total += q_seq_lens[s];
    if (adapter_ids[s] < 0 || adapter_ids[s] >= N) bad_id = true;
  }
  if (total != T) bad_len = true;
  if (bad_len) return ST_META;
  if (bad_id) return ST_SLOT;

  // seq_start: exclusive prefix sum of the lengths.
  seq_start[0] = 0;
  for (int s = 0; s < S; ++s) seq_start[s + 1] = seq_start[s] + q_seq_lens[s];

  // Per-token slot (repeat_interleave) and the owning sequence of each row.
  std::vector<int> row_seq(T);
  for (int s = 0; s < S; ++s)
    for (int t = seq_start[s]; t < seq_start[s + 1]; ++t) {
      slot[t] = adapter_ids[s];
      row_seq[t] = s;
    }

  // Class of a row: decided by its own sequence's length only.
  auto row_class = [&](int t) { return q_seq_lens[row_seq[t]] >= tc_min_qlen ? 1 : 0; };

  // Active rows sorted by (class, slot); stable, so ties keep row order.
  std::vector<int> active;
  for (int t = 0; t < T; ++t)
    if (slot[t] != 0) active.push_back(t);
  std::stable_sort(active.begin(), active.end(), [&](int a, int b) {
    int ca = row_class(a), cb = row_class(b);
    if (ca != cb) return ca < cb;
    return slot[a] < slot[b];
  });
  const int n_active = static_cast<int>(active.size());
  for (int p = 0; p < n_active; ++p) perm[p] = active[p];

  // Segment offsets: count rows per (class, slot), then prefix over class-major order.
  std::vector<int> cnt(2 * N, 0);
  for (int t : active) cnt[row_class(t) * N + slot[t]]++;
  int acc = 0;
  for (int c = 0; c < 2; ++c) {
    for (int k = 0; k < N; ++k) {
      seg_off[c * (N + 1) + k] = acc;
      acc += cnt[c * N + k];
    }
    seg_off[c * (N + 1) + N] = acc;
  }
  const int n_dec_rows = seg_off[0 * (N + 1) + N];

  // Decode groups: each class-0 slot run cut into runs of <= group_rows.
  int nd = 0;
  for (int k = 0; k < N; ++k) {
    int b = seg_off[k], e = seg_off[k + 1];
    for (int p = b; p < e; p += group_rows) {
      dec_work[4 * nd + 0] = k;
      dec_work[4 * nd + 1] = p;
      dec_work[4 * nd + 2] = std::min(p + group_rows, e);
      dec_work[4 * nd + 3] = 0;
      ++nd;
    }
  }

  // Tensor tiles: class-1 sequences visited in the order their rows appear in
  // perm; each cut into consecutive tiles of <= tile_rows rows.
  int nt = 0;
  int last_seq = -1;
  for (int p = n_dec_rows; p < n_active; ++p) {
    int s = row_seq[perm[p]];
    if (s == last_seq) continue;
    last_seq = s;
    for (int b = seq_start[s]; b < seq_start[s + 1]; b += tile_rows) {
      tc_work[4 * nt + 0] = adapter_ids[s];
      tc_work[4 * nt + 1] = b;
      tc_work[4 * nt + 2] = std::min(b + tile_rows, seq_start[s + 1]);
      tc_work[4 * nt + 3] = s;
      ++nt;
    }
  }
  counts[0] = n_active;
  counts[1] = n_dec_rows;
  counts[2] = nd;
  counts[3] = nt;
  return ST_OK;
}

// The delta, in double precision, for the rows listed in rows[n_rows].
//
//   d_in, L, d_out[L]     projection shape; lane l occupies columns
//                         [off_l, off_l + d_out[l]) of a y row, off_l the sum
//                         of the earlier lanes' widths
//   N, rank[N*L], scale[N*L]   per (slot, lane) rank and scale (float32)
//   A_flat, a_off[N*L]    A of (k,l) is [rank][d_in] bf16 at A_flat + a_off
//   B_flat, b_off[N*L]    B of (k,l) is [d_out[l]][rank] bf16 at B_flat + b_off
//   x[T][ldx] bf16, slot[T], y0[T][ldy] float32
//   y_ref[n_rows][D], delta[n_rows][D]   double outputs, D = sum d_out
void oracle_delta(int d_in, int L, const int32_t* d_out, int N,
                  const int32_t* rank, const float* scale,
                  const uint16_t* A_flat, const int64_t* a_off,
                  const uint16_t* B_flat, const int64_t* b_off,
                  const uint16_t* x, int64_t ldx, const int32_t* slot,
                  const float* y0, int64_t ldy,
                  const int64_t* rows, int64_t n_rows,
                  double* y_ref, double* delta, int num_threads) {
  int D = 0;
  std::vector<int> off(L);
  for (int l = 0; l < L; ++l) {
    off[l] = D;
    D += d_out[l];
  }
#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int64_t q = 0; q < n_rows; ++q) {
    const int64_t t = rows[q];
    const int k = slot[t];
    double* yr = y_ref + q * D;
    double* dl = delta + q * D;
    for (int c = 0; c < D; ++c) {
      yr[c] = static_cast<double>(y0[t * ldy + c]);
      dl[c] = 0.0;
    }
    if (k == 0) continue;  // base row: not read, not written
    std::vector<double> u;
    for (int l = 0; l < L; ++l) {
      const int r = rank[k * L + l];
      if (r <= 0) continue;
      const uint16_t* A = A_flat + a_off[k * L + l];
      const uint16_t* B = B_flat + b_off[k * L + l];
      const double s = static_cast<double>(scale[k * L + l]);
      // shrink: u = A x
      u.assign(r, 0.0);
      for (int i = 0; i < r; ++i) {
        double acc = 0.0;
        for (int j = 0; j < d_in; ++j)
          acc += bf16_to_double(A[static_cast<int64_t>(i) * d_in + j]) * bf16_to_double(x[t * ldx + j]);
        u[i] = acc;
      }
      // expand: v = B u, then y += scale * v
      for (int o = 0; o < d_out[l]; ++o) {
        double v = 0.0;
        for (int i = 0; i < r; ++i) v += bf16_to_double(B[static_cast<int64_t>(o) * r + i]) * u[i];
        dl[off[l] + o] = s * v;
        yr[off[l] + o] = static_cast<double>(y0[t * ldy + off[l] + o]) + s * v;
      }
    }
  }
}

// The base projection the delta is added to, in double precision, for the
// rows listed in rows[n_rows]:
//     base[q][c]     = sum_j W[c][j] * x[t][j]      (j ascending), t = rows[q]
//     abs_base[q][c] = sum_j |W[c][j] * x[t][j]|
// W is the projection's weight as a linear layer stores it, [D][ldw] bf16
// (output feature c, input feature j; the fused lanes stacked in lane order),
// x is [T][ldx] bf16.  The delta "is added to the fp32 partial sum" of this
// product (TensorFold PR #47, the paragraph on the delta); in the fused form a
// row's output is base + delta, and a slot-0 row's output is the base alone
// (xLLM PR #2014, the LoRARowParallelLinear item: the base's own output
// carries the delta partial sum).  abs_base is the magnitude that bounds the
// rounding error of any float32 evaluation of the same sum.
void oracle_base_product(int d_in, int D, const uint16_t* W, int64_t ldw,
                         const uint16_t* x, int64_t ldx,
                         const int64_t* rows, int64_t n_rows,
                         double* base, double* abs_base, int num_threads) {
#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int64_t q = 0; q < n_rows; ++q) {
    const int64_t t = rows[q];
    std::vector<double> xt(d_in);
    for (int j = 0; j < d_in; ++j) xt[j] = bf16_to_double(x[t * ldx + j]);
    for (int c = 0; c < D; ++c) {
      const uint16_t* w = W + static_cast<int64_t>(c) * ldw;
      double acc = 0.0, mag = 0.0;
      for (int j = 0; j < d_in; ++j) {
        const double p = bf16_to_double(w[j]) * xt[j];
        acc += p;
        mag += p < 0 ? -p : p;
      }
      base[q * D + c] = acc;
      abs_base[q * D + c] = mag;
    }
  }
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

}  // extern "C"
