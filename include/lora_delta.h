/*
 * lora_delta.h — C ABI of the GB300 (sm_103a) mixed-adapter LoRA delta.
 *
 * One step of multi-tenant LoRA serving adds, for every token row t whose
 * adapter slot k = slot[t] is not 0,
 *
 *     y[t][off_l : off_l + d_out_l] += scale[k][l] * B[k][l] @ (A[k][l] @ x[t])
 *
 * for every lane l of the projection (one lane for o_proj / down_proj, three
 * for fused q,k,v, two for fused gate,up).  The formula, the fp32 partial sum
 * it is added to, the per-row slot with slot 0 = base (a slot-0 row is neither
 * read nor written), and per-row determinism come from TensorFold PR #47
 * ("Add native per-request LoRA adapters to the DeepSeek-V4.1 CUDA engine",
 * the kernels-and-ranks paragraph).  The shrink / expand split and the lane
 * shapes (B.size(0) = the lane's output width, GQA k/v lanes narrower than q)
 * come from xLLM PR #2014 ("multi-tenant LoRA framework", the
 * LoRAQKVParallelLinear / LoRAColumnParallelLinear / LoRARowParallelLinear
 * items).  The routing input (one adapter id per sequence, index-aligned with
 * the query lengths; per-token ids by repeat_interleave; an empty id list is a
 * no-op) comes from xLLM PR #2014, "Wire-up".  The fixed slot pool sized by
 * the largest number of distinct adapters in a batch comes from tokenspeed
 * PR #976 (max_loras).
 *
 * Conventions shared by every entry point
 *  - All device memory is allocated and freed by the caller.  The library
 *    never allocates device memory and keeps only small host descriptors.
 *  - Every GPU action is enqueued on the caller's stream (a cudaStream_t; 0 is
 *    the legacy default stream).  Entry points on the hot path never
 *    synchronise with the host.
 *  - Matrices are row-major.  Leading dimensions (ldx, ldy) are in elements.
 *  - bf16 data is passed as raw 16-bit words (bf16 bit patterns).
 *  - Host-checkable errors are returned before anything is enqueued.
 *    Errors found on the device (bad routing metadata, a kernel wait that
 *    gave up) are written to the segments' status word; read it with
 *    lora_get_status().  No kernel traps or asserts.
 *  - Entry points are thread-compatible: calls on distinct objects may run
 *    concurrently; calls on one object must be serialised by the caller.
 */
#ifndef LORA_DELTA_H
#define LORA_DELTA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* lora_stream_t; /* identical to cudaStream_t */

/* Status codes. */
enum {
  LORA_OK = 0,
  LORA_ERR_ARG = -1,     /* null pointer, misaligned pointer, bad leading dimension, or
                            a call made while another device than the object's is current */
  LORA_ERR_SHAPE = -2,   /* unsupported or inconsistent sizes                          */
  LORA_ERR_SLOT = -3,    /* a slot id outside [0, num_slots) (host or device detected) */
  LORA_ERR_RANK = -4,    /* rank outside [0, max_rank]                                 */
  LORA_ERR_CUDA = -5,    /* a CUDA runtime call failed                                 */
  LORA_ERR_META = -6,    /* device-detected: a negative q_seq_len or sum != num_tokens */
  LORA_ERR_TIMEOUT = -7  /* device-detected: a bounded in-kernel wait gave up          */
};

/* Layout constants of the work lists (part of the ABI). */
#define LORA_MAX_LANES 4         /* lanes per projection                               */
#define LORA_MAX_SLOTS 2048      /* slots per pool, slot 0 included                    */
#define LORA_DEC_GROUP_ROWS 8    /* rows per decode work group                         */
#define LORA_TC_TILE_ROWS 128    /* rows per tensor-path tile                          */
#define LORA_TC_MIN_QLEN 64      /* a row takes the tensor path iff its own sequence's */
                                 /* q_seq_len >= this; otherwise the decode path       */

typedef struct lora_pool lora_pool;
typedef struct lora_segments lora_segments;

/* ------------------------------------------------------------------ pool --
 * The adapter pool of one projection (xLLM PR #2014, LoRARuntime "per-proj
 * device pool"; the pool has a fixed number of slots, tokenspeed PR #976;
 * ranks and scales may differ per slot and per module, TensorFold PR #47).
 *
 * Slot 0 is the base model and holds nothing.  Slots 1..num_slots-1 hold, per
 * lane, bf16 factors of a rank r <= max_rank padded with zeros to
 * R16 = max_rank rounded up to a multiple of 16, a rank and an fp32 scale
 * (the caller computes scale = lora_alpha / r * strength).  The pool also
 * holds the tensor path's rank-space scratch for up to max_tokens rows, used
 * between its shrink and expand kernels (fp32 partial sums, bf16 U tiles, and
 * per-tile counters that the zero fill starts at zero and every apply leaves
 * at zero), so two applies on one pool must be ordered on one stream.
 *
 * Shapes: d_in (<= 65536) and every lane_d_out[l] must be positive multiples of 64;
 * 1 <= num_lanes <= LORA_MAX_LANES; 2 <= num_slots <= LORA_MAX_SLOTS;
 * 1 <= max_rank <= 128; max_tokens >= 1.  (The tensor path keeps a tile's
 * num_lanes * R16 <= 512 rank columns of fp32 accumulators in tensor memory.)
 */

/* Bytes of device memory a pool of this shape needs (0 if the shape is invalid). */
size_t lora_pool_bytes(int num_slots, int max_rank, int d_in, int num_lanes,
                       const int* lane_d_out /* host [num_lanes] */, int max_tokens);

/* Create a pool descriptor over caller memory dev_mem (>= lora_pool_bytes,
 * 256-byte aligned).  Enqueues a zero fill of dev_mem on `stream`, so every
 * slot starts unloaded (rank 0).  The descriptor records the current CUDA
 * device; the first pool of a device also creates the library's side stream
 * and events for that device (see lora_apply_shrink_expand).  Errors:
 * LORA_ERR_ARG, LORA_ERR_SHAPE, LORA_ERR_CUDA. */
int lora_pool_create(lora_pool** out, void* dev_mem, size_t bytes, int num_slots, int max_rank,
                     int d_in, int num_lanes, const int* lane_d_out /* host */, int max_tokens,
                     lora_stream_t stream);

/* Load (or replace) lane `lane` of slot `slot` (1..num_slots-1):
 *   A: device bf16 [rank][d_in] row-major (PEFT lora_A layout),
 *   B: device bf16 [lane_d_out[lane]][rank] row-major (PEFT lora_B layout).
 * rank = 0 unloads the lane (A and B may then be NULL).  The copy/repack is
 * enqueued on `stream`; A and B must stay valid until it has run.  The caller
 * must not run this concurrently with an apply that reads the slot.
 * Errors: LORA_ERR_ARG, LORA_ERR_SLOT, LORA_ERR_RANK, LORA_ERR_CUDA. */
int lora_pool_load(lora_pool* pool, int slot, int lane, int rank, float scale,
                   const void* A, const void* B, lora_stream_t stream);

/* Free the host descriptor only (device memory stays the caller's). */
int lora_pool_destroy(lora_pool* pool);

/* -------------------------------------------------------------- segments --
 * Routing metadata of one step, shared by every layer and projection of that
 * step.  Built on the device from per-sequence adapter ids and query lengths
 * (xLLM PR #2014, Wire-up: adapter_ids index-aligned with q_seq_lens,
 * adapter_ids_per_token by repeat_interleave).  Contents after a build:
 *   slot[T]       per-token slot
 *   perm[]        active rows (slot != 0) ordered by (class, slot, row), class
 *                 0 = decode path (own q_seq_len < LORA_TC_MIN_QLEN), 1 = tensor
 *   seg_off[2*(N+1)]  first perm position of each (class, slot); [c*(N+1)+N] is
 *                 the end of class c
 *   dec_work[][4] {slot, perm_begin, perm_end, 0}: each class-0 slot run cut
 *                 into runs of <= LORA_DEC_GROUP_ROWS rows
 *   tc_work[][4]  {slot, row_begin, row_end, seq}: each class-1 sequence cut
 *                 into tiles of <= LORA_TC_TILE_ROWS rows, sequences in perm order
 *   counts[4]     {active rows, class-0 rows, #dec_work, #tc_work}
 * A prompt chunk therefore uses one slot for all its rows, and a tile never
 * crosses a sequence (TensorFold PR #47).  On a device-detected error every
 * count is 0, so a following apply does nothing.
 */

/* Bytes of device workspace for up to max_seqs sequences, max_tokens rows and num_slots slots
 * (0 if the shape is invalid).  The builder keeps every slot's counters in one CTA's shared
 * memory, and its six per-sequence arrays there too when 4 * (6 * max_seqs + 7 * num_slots + 2)
 * fits in 227 KiB - 2 KiB; beyond that the workspace holds them (24 bytes per sequence more),
 * so max_seqs has no limit of its own. */
size_t lora_segments_bytes(int max_seqs, int max_tokens, int num_slots);

/* Create a segments descriptor over caller workspace dev_ws (256-byte aligned). */
int lora_segments_create(lora_segments** out, void* dev_ws, size_t ws_bytes, int max_seqs,
                         int max_tokens, int num_slots);

/* Build the metadata of one step on `stream` (one kernel, one CTA).
 *   adapter_ids[num_seqs], q_seq_lens[num_seqs]: device int32.
 * num_seqs = 0 (with num_tokens = 0) is a no-op step: no kernel is launched
 * and the counts read as 0; num_seqs = 0 with num_tokens > 0 is LORA_ERR_SHAPE.  Device-detected errors: LORA_ERR_META if a length is negative or
 * the lengths do not sum to num_tokens (checked first), LORA_ERR_SLOT if an id
 * is outside [0, num_slots).  Host errors: LORA_ERR_ARG, LORA_ERR_SHAPE. */
int lora_build_segments(lora_segments* seg, const int32_t* adapter_ids, const int32_t* q_seq_lens,
                        int num_seqs, int num_tokens, lora_stream_t stream);

/* ------------------------------------------------------- MoE expert LoRA --
 * The delta of an MoE layer's expert projections, where every expert has its
 * own LoRA factors per adapter (xLLM PR #2014, "Not in this PR": the fused MoE
 * expert LoRA delta by a grouped GEMM; TensorFold PR #47 also names the
 * shared expert's w2).  After routing, the layer's dispatched rows (one per
 * (token, chosen expert)) are grouped by expert, and inside an expert the rows
 * of one sequence are contiguous.  One pool holds every expert's copy of every
 * adapter: adapter k (1..A) of expert e (0..E-1) sits in slot
 * lora_moe_slot(e, k, A) = 1 + e * A + (k - 1), so num_slots = 1 + E * A
 * (<= LORA_MAX_SLOTS); adapter 0 is the base model.  lora_build_segments_moe
 * turns the dispatched rows into the builder's sequences: each maximal run of
 * rows with the same (expert, sequence, adapter) is one sequence of that
 * expert's adapter slot, so the run takes the tensor path when it has at least
 * LORA_TC_MIN_QLEN rows (a prompt chunk's tokens that chose one expert).  The
 * ordinary lora_apply_shrink_expand then adds the delta to the dispatched
 * rows' fp32 outputs (x, y: [num_rows] dispatched rows).
 *   row_expert[num_rows], row_adapter[num_rows], row_seq[num_rows]: device
 *     int32; row_seq only delimits runs (any id, equal for a sequence's rows).
 * The segments must have num_slots = 1 + E * A, max_tokens >= num_rows and
 * max_seqs >= the number of runs.  Two kernels (a run-length pass, then the
 * builder) on `stream`.  Device-detected errors: LORA_ERR_SLOT (an expert id
 * outside [0, E) or an adapter id outside [0, A]), LORA_ERR_META (more runs
 * than max_seqs); host errors: LORA_ERR_ARG, LORA_ERR_SHAPE.
 * num_rows = 0 is a no-op step (no kernel). */
int lora_moe_slot(int expert, int adapter, int num_adapters);
int lora_build_segments_moe(lora_segments* seg, const int32_t* row_expert, const int32_t* row_adapter,
                            const int32_t* row_seq, int num_rows, int num_experts, int num_adapters,
                            lora_stream_t stream);

/* Capacities of the work lists of this descriptor (host, no GPU work). */
int lora_segments_capacity(const lora_segments* seg, int* dec_work_cap, int* tc_work_cap);

/* Copy the metadata of the last build to host buffers (tests and tools; this
 * synchronises `stream`).  Sizes: host_slot[T], host_perm[T], host_seg_off[2*(N+1)],
 * host_counts[4], host_dec_work[4*dec_work_cap], host_tc_work[4*tc_work_cap]; any may be NULL. */
int lora_segments_read(const lora_segments* seg, int32_t* host_slot, int32_t* host_perm,
                       int32_t* host_seg_off, int32_t* host_counts, int32_t* host_dec_work,
                       int32_t* host_tc_work, lora_stream_t stream);

/* Copy the last build's decode-group row lists to host_rows[8 * n] (n = the
 * build's decode group count, counts[2]; tests and tools; synchronises
 * `stream`).  Group w's rows are perm[pb .. pe) of its work entry (k, pb, pe)
 * in order; the entries past pe - pb are unspecified. */
int lora_segments_read_dec_rows(const lora_segments* seg, int32_t* host_rows, lora_stream_t stream);

/* Read the status word (copies 4 bytes and synchronises `stream`). */
int lora_get_status(const lora_segments* seg, int32_t* host_status, lora_stream_t stream);

/* Reset the status word to LORA_OK on `stream`. */
int lora_clear_status(lora_segments* seg, lora_stream_t stream);

int lora_segments_destroy(lora_segments* seg);

/* ----------------------------------------------------------------- apply --
 * y += delta for every active row of the last lora_build_segments on `seg`:
 *   x: device bf16 [T][ldx] (ldx >= d_in, ldx % 8 == 0, 16-byte aligned)
 *   y: device fp32 [T][ldy] (ldy >= sum of lane_d_out, ldy % 4 == 0, 16-byte
 *      aligned), updated in place; lane l occupies columns
 *      [off_l, off_l + lane_d_out[l]), off_l = sum of the earlier lanes' widths.
 * Rows of slot 0, and lanes of rank 0, are neither read nor written.  Each
 * row's result depends only on its own x row, its adapter's factors and its
 * own sequence's length: sums run in fp32 in a fixed order that depends on
 * d_in and the lane's rank only (decode path: one fused kernel per call, a
 * thread-block cluster per (row group, lane) shrinks fixed K ranges of d_in,
 * adds the ranges' partial sums in order on chip, expands over the rank in
 * ascending order, y = fma(scale, v, y); tensor path: tcgen05 bf16 MMAs with
 * fp32 accumulation, the rank-space vector split into two bf16 halves for the
 * expand, y = y + scale * v).
 * The decode-path kernel runs on a side stream the library creates per device
 * (forked from and joined back to `stream` with events), concurrently with the
 * tensor-path kernels on `stream`; the call stays ordered on `stream` and can
 * be stream-captured.
 * If the step has no rows, or the pool has no loaded lane, nothing is
 * launched.  Errors: LORA_ERR_ARG, LORA_ERR_SHAPE, LORA_ERR_CUDA; device
 * timeouts set LORA_ERR_TIMEOUT in the segments' status word. */
int lora_apply_shrink_expand(const lora_pool* pool, const lora_segments* seg, const void* x,
                             float* y, int64_t ldx, int64_t ldy, lora_stream_t stream);

/* One kernel of lora_apply_shrink_expand, for per-kernel timing:
 * stage 1 = decode path (fused shrink -> expand), 2 = tensor shrink,
 * 3 = tensor expand.  Running stages 1..3 in order on one stream gives
 * exactly the result of lora_apply_shrink_expand. */
int lora_apply_stage(const lora_pool* pool, const lora_segments* seg, const void* x, float* y,
                     int64_t ldx, int64_t ldy, int stage, lora_stream_t stream);

/* The same step as lora_apply_shrink_expand for callers that cannot allocate
 * device memory when they run: a plugin or custom-op host that passes the op
 * only its input and output buffers, or a serving loop whose memory plan is
 * frozen after start-up.  No passage of the pages has a counterpart; this is a
 * property of the library, not of the method.
 *   - The tensor path's rank-space intermediate lives in a fixed array
 *     compiled into the library, of LORA_NOALLOC_SCRATCH_BYTES; every GPU
 *     that loads the library holds it until the process exits.  A step needs,
 *     in floats, 16384 (per-tile counters) + 3 * (T / 64 + 1) * num_lanes *
 *     R16 * 128 (the tensor tiles' partial sums and U tiles); one that needs
 *     more returns LORA_ERR_SHAPE before anything is enqueued.  (The decode
 *     path keeps its rank-space vector on chip and needs no scratch.)
 *   - The call allocates nothing.  Its first call on a device looks up the
 *     array's device address (cudaGetSymbolAddress) with that device current;
 *     make that first call before any stream capture.  The current device must
 *     be the pool's device (else LORA_ERR_ARG).
 *   - Every call shares the one array.  Each scratch word a call reads it has
 *     written earlier in the same call, except the per-tile counters, which
 *     start at zero and which every call leaves at zero; so nothing needs
 *     clearing, but calls whose GPU work overlaps (other streams, other
 *     threads) race on it: order them on one stream.
 * Arguments, results and other errors are those of lora_apply_shrink_expand. */
#define LORA_NOALLOC_SCRATCH_BYTES (64u << 20)
int lora_apply_shrink_expand_noalloc(const lora_pool* pool, const lora_segments* seg, const void* x,
                                     float* y, int64_t ldx, int64_t ldy, lora_stream_t stream);

/* ------------------------------------------------------ fused projection --
 * The projection with the delta in its own accumulator: for every row t of
 * the last build on `seg` (slot 0 rows included),
 *     y[t][c] = sum_j x[t][j] * W[c][j] + delta[t][c]
 * written once (y is not read).  The delta is added to the projection's fp32
 * partial sum (TensorFold PR #47, the paragraph on the delta), so it needs no
 * pass of its own over y (xLLM PR #2014, New subsystems, the
 * LoRARowParallelLinear item's fused mode, where the base's own output
 * carries the delta partial sum).  delta is 0 for slot-0 rows and rank-0 lanes.
 *   W: device bf16 [D][ldw], D = sum of lane_d_out (the lanes' weights
 *      stacked in lane order, as a linear layer stores [out][in]);
 *      ldw >= d_in, ldw % 8 == 0, 16-byte aligned.
 *   x, y, ldx, ldy: as for lora_apply_shrink_expand (y is written, not updated).
 * Arithmetic: one tcgen05 GEMM over tiles of 128 rows x 256 columns (on
 * batches of long prompts, 256 x 256 tiles on CTA pairs with the pair MMA;
 * both forms give a row the same bits), bf16 products summed in fp32 over
 * d_in in a fixed order; the expand of every slot
 * present in a tile goes into the same fp32 accumulator as MMAs whose
 * rank-space input is u' = scale * (A @ x) split into bf16 hi and lo halves
 * (u' from the two shrinks, run before it in a row mode that writes u' to the
 * pool's per-row scratch; rows of other slots take zeros).  A row's bits
 * depend only on its own x row, W and its own adapter.
 * Kernels: the decode shrink (side stream, as in lora_apply_shrink_expand) and
 * the tensor shrink when the pool has a loaded lane, then the GEMM.  If the
 * build found a routing error (or a kernel timed out), the GEMM writes nothing.
 * T = 0 launches nothing.  Errors: LORA_ERR_ARG, LORA_ERR_SHAPE,
 * LORA_ERR_CUDA; device timeouts set LORA_ERR_TIMEOUT in the status word. */
int lora_apply_fused_projection(const lora_pool* pool, const lora_segments* seg, const void* W,
                                int64_t ldw, const void* x, float* y, int64_t ldx, int64_t ldy,
                                lora_stream_t stream);

/* One kernel of lora_apply_fused_projection, for per-kernel timing: stage 1 =
 * decode shrink (row mode), 2 = tensor shrink (row mode), 3 = the GEMM.
 * Running stages 1..3 in order on one stream gives exactly its result. */
int lora_fused_projection_stage(const lora_pool* pool, const lora_segments* seg, const void* W,
                                int64_t ldw, const void* x, float* y, int64_t ldx, int64_t ldy,
                                int stage, lora_stream_t stream);

/* ----------------------------------------------------------------- misc -- */

/* Text of a status code. */
const char* lora_status_string(int status);

/* Text of the last failed CUDA call made by this library on the calling
 * thread (empty if none): what a LORA_ERR_CUDA came from. */
const char* lora_last_error_string(void);

/* Kernels this library has launched in this process (all entry points). */
uint64_t lora_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* LORA_DELTA_H */
