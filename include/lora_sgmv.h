/*
 * lora_sgmv.h -- C ABI of the B300 (sm_103a) multi-LoRA SGMV library
 * (liblora_sgmv.so).
 *
 * The operation.  Punica: Serving Multiple LoRA Finetuned LLM as One
 * (vecbase.com), "How It Works": a LoRA finetune adds two small matrices A and
 * B to a pretrained weight W, and the output is produced with Segmented Gather
 * Matrix-Vector multiplication (SGMV) in a CUDA kernel.  Punica: Multi-Tenant
 * LoRA Serving (research.elamur.ai summary), "Summary": one batch mixes
 * requests of many adapters; the backbone runs as an ordinary GEMM and the
 * per-adapter low-rank additions are computed together, requests of the same
 * adapter grouped; "Interesting ideas" I2: sort the batch by adapter so that
 * same-adapter rows form dense segments.  For token i with adapter a_i:
 *
 *     y[i,:] += s * ((x[i,:] . A[a_i]) . B[a_i])
 *
 * computed as a shrink v = x.A (rank r, fp32) followed by an expand
 * y += s * v.B.
 *
 * Conventions shared by every call.
 *  - bf16 data is passed as raw 16-bit patterns (lora_bf16).
 *  - Every pointer argument named as device memory must be device memory of
 *    the current CUDA device; host memory is never read by a kernel.  The
 *    caller owns and allocates every buffer (including workspaces); the
 *    library allocates no device memory and keeps no per-call state.
 *  - Calls are ordered on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and never synchronise the host.
 *  - The return value reports errors found on the host before any launch
 *    (bad sizes, null or misaligned pointers, too small workspace) and launch
 *    failures (LORA_ERR_CUDA).  Nothing is launched when it is not LORA_OK.
 *  - Errors found on the device (an adapter id outside [0, n_adapters), a
 *    permutation entry outside [0, n_tokens), a wait that ran out of time) are
 *    recorded in *err_flag (device int32, may be NULL) with the first error's
 *    code winning (atomic compare-and-swap from 0); the offending token or
 *    segment is skipped and its output rows are left untouched.  The caller
 *    clears *err_flag and reads it after its own synchronisation.
 *  - Layouts (a reading: the pages give none): x is [n_tokens][ldx] row-major,
 *    y is [n_tokens][ldy] row-major, the adapter pools are contiguous slabs
 *    A_pool[n_adapters][h_in][r] and B_pool[n_adapters][r][h_out], row-major,
 *    so that the adapter id is the slab index.
 *  - Supported shapes: r in {8, 16, 32, 64}; h_in, h_out >= 8 and multiples
 *    of 8; ldx, ldy multiples of 8; x, y, A_pool, B_pool, v 16-byte aligned.
 *    Other shapes return LORA_ERR_UNSUPPORTED, other alignments
 *    LORA_ERR_MISALIGNED.
 */
#ifndef LORA_SGMV_H_
#define LORA_SGMV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LORA_SGMV_ABI_VERSION 2

#if defined(__GNUC__)
#define LORA_API __attribute__((visibility("default")))
#else
#define LORA_API
#endif

typedef uint16_t lora_bf16;                /* bfloat16 bit pattern */
typedef struct CUstream_st* lora_stream_t; /* same type as cudaStream_t */

typedef enum {
  LORA_OK = 0,
  LORA_ERR_INVALID_ARG = -1,    /* null pointer, negative size, ld < width ... */
  LORA_ERR_MISALIGNED = -2,     /* pointer or leading dimension not 16-byte aligned */
  LORA_ERR_UNSUPPORTED = -3,    /* rank or width outside the supported set */
  LORA_ERR_BAD_ADAPTER_ID = -4, /* device: adapter id, permutation entry, slot or rank out of range */
  LORA_ERR_WORKSPACE = -5,      /* workspace missing or smaller than required */
  LORA_ERR_CUDA = -6,           /* a CUDA runtime call or launch failed */
  LORA_ERR_TIMEOUT = -7         /* device: a bounded wait inside a kernel ran out */
} lora_status;

/* Static string naming a status code (unknown codes give "unknown status"). */
LORA_API const char* lora_status_str(int status);

/* LORA_SGMV_ABI_VERSION of the loaded library. */
LORA_API int lora_abi_version(void);

/*
 * Segmentation record produced by lora_segment and read by every SGMV call
 * (all pointers device memory, owned by the caller).
 *   perm[n_tokens]             perm[k] = original index of the k-th token in
 *                              adapter order (stable: ties in token order).
 *   seg_offsets[max_segments+1]  segment s covers perm[seg_offsets[s] ..
 *                              seg_offsets[s+1]); entries past the last segment
 *                              hold the number of valid tokens.
 *   seg_adapter[max_segments]  adapter id of segment s, ascending; -1 past the
 *                              last segment.
 *   num_segments               device scalar: number of non-empty segments.
 *   max_segments               min(n_tokens, n_adapters) (capacity of the arrays).
 * A record built by the caller must keep perm ascending within each segment,
 * as lora_segment's does: the tensor-tile kernel takes a 128-token tile
 * whose first and last rows are 127 apart as contiguous rows.
 */
typedef struct {
  const int32_t* perm;
  const int32_t* seg_offsets;
  const int32_t* seg_adapter;
  const int32_t* num_segments;
  int32_t n_tokens;
  int32_t max_segments;
} lora_segments;

/*
 * Bytes of device workspace lora_segment needs for (n_tokens, n_adapters).
 * 0 for batches of at most 256 tokens (ranked without a histogram over the
 * pool) and when the per-warp histograms fit in shared memory (pools of up to
 * ~25k adapters); otherwise the histograms live in the workspace.
 */
LORA_API size_t lora_segment_workspace_bytes(int32_t n_tokens, int32_t n_adapters);

/*
 * Group tokens by adapter: Punica: Multi-Tenant LoRA Serving, "Interesting
 * ideas" I2 (sort the batch by adapter) and "Summary" (requests of the same
 * adapter grouped).  A stable counting sort: histogram of ids over
 * [0, n_adapters), exclusive scan into segment offsets, compaction of the
 * non-empty adapters (ascending id), stable scatter of token indices; a batch
 * of at most 256 tokens is ranked directly (one thread per token counts the
 * tokens that sort before it), with the same result.
 *   ids[n_tokens]      device int32 adapter ids.
 *   perm, seg_offsets, seg_adapter, num_segments: outputs as described for
 *                      lora_segments, sized with max_segments =
 *                      min(n_tokens, n_adapters).
 *   workspace          device memory of lora_segment_workspace_bytes() bytes
 *                      (may be NULL when that is 0); contents on entry are
 *                      ignored, contents on exit are unspecified.
 * Ids outside [0, n_adapters) join no segment: they are counted out of
 * seg_offsets[num_segments] and listed in perm after every valid token, in
 * token order; *err_flag gets LORA_ERR_BAD_ADAPTER_ID.
 * n_tokens == 0 writes num_segments = 0 and seg_offsets[0] = 0.
 */
LORA_API lora_status lora_segment(const int32_t* ids, int32_t n_tokens, int32_t n_adapters,
                         int32_t* perm, int32_t* seg_offsets, int32_t* seg_adapter,
                         int32_t* num_segments, void* workspace, size_t workspace_bytes,
                         int32_t* err_flag, lora_stream_t stream);

/*
 * lora_segment for callers that cannot allocate device memory (no cudaMalloc
 * and no allocator of their own at hand: code running under a framework that
 * owns the allocator, a real-time loop whose memory was planned up front, a
 * plugin handed only its input and output buffers).  The paper has no
 * counterpart; this is a packaging variant of lora_segment.
 *
 * Same arguments, outputs and device-side errors as lora_segment, without the
 * workspace: when the pool is too large for shared-memory histograms the
 * scratch comes from a library-owned device array of
 * LORA_SEGMENT_NOALLOC_SCRATCH_BYTES (8 MiB) that every GPU which loads the
 * library holds until the process exits (under CUDA's lazy module loading the
 * array is reserved when the first call in a context loads the module that
 * holds it).  Batches of more than 256 tokens over pools needing more scratch
 * than that (more than about 63,500 adapters) return LORA_ERR_WORKSPACE
 * without a launch.
 * The call allocates nothing.
 *  - The first call in each CUDA context (with its device current) looks up
 *    the array's device address and caches it for that context; make that
 *    first call before any stream capture.  A context created later (after
 *    cudaDeviceReset, or another context made current through the driver API)
 *    gets its own lookup on its first call: a cached address is never reused
 *    in another context.
 *  - All calls share the array and it keeps the last call's contents (each
 *    kernel clears the part it uses), so calls whose kernels overlap on the
 *    GPU (different streams, or concurrent graphs) race on it: order them.
 */
#define LORA_SEGMENT_NOALLOC_SCRATCH_BYTES (8u << 20)
LORA_API lora_status lora_segment_noalloc(const int32_t* ids, int32_t n_tokens, int32_t n_adapters,
                                          int32_t* perm, int32_t* seg_offsets, int32_t* seg_adapter,
                                          int32_t* num_segments, int32_t* err_flag, lora_stream_t stream);

/*
 * Shrink: v[i,:] = x[i,:] . A[a_i]  (fp32 accumulate, fp32 output).
 * Punica: Multi-Tenant LoRA Serving, "Summary" (the low-rank part of the
 * per-adapter addition).  x [n][ldx] bf16; A_pool [n_adapters][h_in][r] bf16;
 * v [n][r] fp32 in original token order (rows of skipped tokens untouched).
 */
LORA_API lora_status sgmv_shrink(const lora_bf16* x, int64_t ldx, const lora_bf16* A_pool,
                        int32_t n_adapters, int32_t h_in, int32_t r, const lora_segments* seg,
                        float* v, int32_t* err_flag, lora_stream_t stream);

/*
 * Expand: y[i,:] += s * v[i,:] . B[a_i]  (fp32 accumulate, one round-to-
 * nearest-even to bf16 at the store).  v [n][r] fp32; B_pool
 * [n_adapters][r][h_out] bf16; y [n][ldy] bf16, updated in place.
 */
LORA_API lora_status sgmv_expand(const float* v, const lora_bf16* B_pool, int32_t n_adapters, int32_t r,
                        int32_t h_out, float scale, const lora_segments* seg, lora_bf16* y,
                        int64_t ldy, int32_t* err_flag, lora_stream_t stream);

/*
 * Shrink and expand in one launch, v kept on chip (never written to device
 * memory): y[i,:] += s * ((x[i,:] . A[a_i]) . B[a_i]).  Arguments as for
 * sgmv_shrink / sgmv_expand.  v is accumulated in fp32; the expand product
 * takes it as two bf16 operands, v = hi + lo with hi = bf16(v) and
 * lo = bf16(v - hi), which keep 16 bits of its mantissa (relative error about
 * 2^-17, far inside the parity tolerance).
 */
LORA_API lora_status sgmv_fused(const lora_bf16* x, int64_t ldx, const lora_bf16* A_pool,
                       const lora_bf16* B_pool, int32_t n_adapters, int32_t h_in, int32_t h_out,
                       int32_t r, float scale, const lora_segments* seg, lora_bf16* y,
                       int64_t ldy, int32_t* err_flag, lora_stream_t stream);

/* One projection of a multi-projection call (device pointers, host struct). */
typedef struct {
  const lora_bf16* x;      /* [n][ldx] */
  const lora_bf16* A_pool; /* [n_adapters][h_in][r] */
  const lora_bf16* B_pool; /* [n_adapters][r][h_out] */
  lora_bf16* y;            /* [n][ldy], updated in place */
  int64_t ldx, ldy;
  int32_t h_in, h_out;
  float scale;
} lora_proj;

#define LORA_MAX_PROJ 8

/*
 * sgmv_fused for up to LORA_MAX_PROJ projections (e.g. q,k,v,o,gate,up,down
 * of one transformer layer) sharing one segmentation and one rank, in one
 * launch.  `projs` is a host array of n_proj descriptors (read during the
 * call only).  Projections may share x; their y must not overlap.
 */
LORA_API lora_status sgmv_multi(const lora_proj* projs, int32_t n_proj, int32_t n_adapters, int32_t r,
                       const lora_segments* seg, int32_t* err_flag, lora_stream_t stream);

/*
 * lora_segment followed by sgmv_multi on its result, as one call: the
 * segmentation is written to perm / seg_offsets / seg_adapter /
 * num_segments exactly as lora_segment writes it (for later calls of the
 * same batch) and the projections are updated as sgmv_multi updates them.
 * Small decode-like batches (n_tokens <= 128, n_adapters <= 1024, no
 * segment long enough for the tensor-tile kernel) are segmented inside the
 * SGMV launch itself, so the step is one kernel; other batches run
 * lora_segment's kernel first (with `workspace`, sized as
 * lora_segment_workspace_bytes says) and then the SGMV kernels.  Errors: as
 * lora_segment and sgmv_multi.
 * Ordering: a one-launch step reads `ids` and the adapter pools while the
 * preceding kernel in the stream may still be running (programmatic dependent
 * launch); it reads x and y, and writes anything, only after that kernel has
 * completed.  So ids and pools must not be written by a preceding kernel that
 * lets its dependents start early (griddepcontrol.launch_dependents) before
 * it writes them; copies and ordinary kernels are waited for in full.
 */
LORA_API lora_status sgmv_multi_segment(const lora_proj* projs, int32_t n_proj, int32_t n_adapters, int32_t r,
                                        const int32_t* ids, int32_t n_tokens, int32_t* perm, int32_t* seg_offsets,
                                        int32_t* seg_adapter, int32_t* num_segments, void* workspace,
                                        size_t workspace_bytes, int32_t* err_flag, lora_stream_t stream);

/*
 * The whole step from host memory: token ids, x and y0 rows in host memory
 * (pinned for an asynchronous call), adapter pools on the device.  Copies
 * every distinct x and every y to the device workspace, segments the ids and
 * runs sgmv_multi on them (one launch for small batches, as
 * sgmv_multi_segment) and copies every y back, all ordered on `stream` with
 * one cudaMemcpyAsync (contiguous rows) or cudaMemcpy2DAsync per buffer; the
 * ids of a batch segmented inside the launch travel in the launch's
 * parameters (read from ids_host when the call is made), larger batches copy
 * them to the workspace first.  The caller synchronises before reading y.  projs[i].x / .y are HOST pointers
 * here (x [n][ldx], y [n][ldy]); A_pool / B_pool are device pointers.
 * Projections that name the same host x share one device copy.  The
 * workspace (device, 256-byte aligned, caller-owned) must hold
 * sgmv_multi_host_workspace_bytes(...) bytes.  Errors: as lora_segment and
 * sgmv_multi, plus ids_host NULL (LORA_ERR_INVALID_ARG), workspace missing or
 * too small (LORA_ERR_WORKSPACE), a failed copy (LORA_ERR_CUDA).
 */
LORA_API size_t sgmv_multi_host_workspace_bytes(const lora_proj* projs, int32_t n_proj, int32_t n_tokens,
                                                int32_t n_adapters);
LORA_API lora_status sgmv_multi_host(const lora_proj* projs, int32_t n_proj, int32_t n_adapters, int32_t r,
                                     const int32_t* ids_host, int32_t n_tokens, void* workspace,
                                     size_t workspace_bytes, int32_t* err_flag, lora_stream_t stream);

/*
 * The backbone projection with the LoRA delta, y written once:
 *
 *     y[i,:] = x[i,:] . W + s * ((x[i,:] . A[a_i]) . B[a_i])
 *
 * Punica: Multi-Tenant LoRA Serving (research.elamur.ai summary), "Summary":
 * the backbone runs as one ordinary GEMM over the batch and the per-adapter
 * low-rank additions are computed together; "Interesting ideas" I1: the
 * shared and the per-tenant computation are split.  Here the expand of every
 * segment of at least 64 tokens joins the GEMM's accumulator (tensor cores,
 * fp32), so it adds no y read or write: a shrink launch writes v = x . A of
 * those tokens to the workspace, the GEMM launch computes x . W + s * v . B
 * for them and x . W for every other token and writes y, and the split-K
 * SGMV launch then adds the delta of the shorter segments to y in place.
 *   x [n][ldx], y [n][ldy] (written, not accumulated): as sgmv_fused.
 *   W [h_in][h_out] row-major bf16 (device), shared by every token,
 *     16-byte aligned.
 *   A_pool, B_pool, seg, r: as sgmv_fused.
 *   workspace: device memory of gemm_lora_workspace_bytes(n, r) bytes (v as
 *     up to four fp32 [n][r] slices of partial sums over parts of h_in,
 *     which the GEMM launch adds in slice order), 16-byte aligned; contents
 *     on exit unspecified.
 * A token whose adapter id is invalid (outside every segment) gets
 * y = x . W; err_flag as for lora_segment.  Errors: as sgmv_fused, plus W
 * NULL (LORA_ERR_INVALID_ARG) or misaligned, workspace missing or too small
 * (LORA_ERR_WORKSPACE).  The product x . W is accumulated in fp32 in tile
 * order (not the oracle's order); y is rounded to bf16 once.
 */
LORA_API size_t gemm_lora_workspace_bytes(int32_t n_tokens, int32_t r);
LORA_API lora_status gemm_lora(const lora_bf16* x, int64_t ldx, const lora_bf16* W, const lora_bf16* A_pool,
                               const lora_bf16* B_pool, int32_t n_adapters, int32_t h_in, int32_t h_out, int32_t r,
                               float scale, const lora_segments* seg, lora_bf16* y, int64_t ldy, void* workspace,
                               size_t workspace_bytes, int32_t* err_flag, lora_stream_t stream);

/*
 * Slot tables: adapter pools stored as arenas of fixed-size slots, so that
 * adapters are loaded into free slots and evicted while the pool is in use,
 * and adapters of different ranks share one launch.  Punica: Multi-Tenant
 * LoRA Serving (research.elamur.ai summary), "Summary": adapters are loaded
 * on demand, in milliseconds; "Key points": rank is far below the hidden
 * size (16 vs 4096).
 *
 * Per projection, the arenas are (lora_proj.A_pool / B_pool point to them):
 *   A arena [n_slots][h_in * r_max]: slot s holds its adapter's A, rank r,
 *           as [h_in][r] row-major at the slot start (the rest unused);
 *   B arena [n_slots][r_max * h_out]: B as [r][h_out] row-major at the start.
 * Adapter id a of the batch (0 <= a < n_adapters) lives in slot slot_of[a]
 * with rank rank_of[a]; one id names the same slot in every projection's
 * arenas.  Both tables are device int32 arrays of n_adapters entries, read
 * by the kernel after the segmentation it waits for.
 */
typedef struct {
  const int32_t* slot_of; /* device [n_adapters]: slot of adapter a */
  const int32_t* rank_of; /* device [n_adapters]: rank of adapter a, in {8,16,32,64}, <= r_max */
  int32_t n_adapters;     /* ids of the batch and of the segmentation index these tables */
  int32_t n_slots;        /* slots in every arena */
  int32_t r_max;          /* slot capacity in ranks: 8, 16, 32 or 64 */
  uint32_t rank_mask;     /* ranks that may occur: bit c for rank 8 << c; no bit above r_max */
} lora_slot_table;

/*
 * sgmv_multi over slot arenas: y_p[i,:] += s_p * ((x_p[i,:] . A_p[a_i]) .
 * B_p[a_i]) with A_p[a], B_p[a] the rank-rank_of[a] matrices in slot
 * slot_of[a] of projection p's arenas.  One rank in rank_mask: one launch
 * for all projections; several ranks: each launch takes the projections
 * whose (projection, rank) pairs fit 8, i.e. 8 / popcount(rank_mask)
 * projections.  Prefill-like batches also run the tensor-tile kernel once
 * per rank of the mask, for the segments of at least 64 tokens of that rank
 * (rows contiguous or gathered through perm).
 * Host errors as sgmv_multi, plus: table NULL, a table pointer NULL or not
 * 4-byte aligned, n_slots < 1, r_max or rank_mask invalid
 * (LORA_ERR_INVALID_ARG / LORA_ERR_UNSUPPORTED), n_slots*r_max*max(h_in,
 * h_out) >= 2^31 (LORA_ERR_UNSUPPORTED).  Device errors: an adapter id
 * outside [0, n_adapters), a slot outside [0, n_slots) or a rank not in
 * rank_mask: LORA_ERR_BAD_ADAPTER_ID in *err_flag, the segment skipped.
 */
LORA_API lora_status sgmv_multi_slots(const lora_proj* projs, int32_t n_proj, const lora_slot_table* table,
                                      const lora_segments* seg, int32_t* err_flag, lora_stream_t stream);

/*
 * Adapter loading into slot arenas.  Punica: Multi-Tenant LoRA Serving
 * (research.elamur.ai summary), "Summary": an adapter is loaded on demand and
 * the load takes milliseconds.  A load is a copy of the adapter's matrices
 * into a free slot of every arena (lora_slot_copy, e.g. on a loader stream
 * while SGMV runs on another), followed by the table entry that makes the
 * adapter id point at the slot (lora_slot_assign, ordered after the copies).
 * The caller orders the steps around the batches: a slot is reused only
 * after the last batch that reads its old adapter, and a batch names a new
 * adapter only after its lora_slot_assign.
 */
typedef struct {
  lora_bf16* A_arena;     /* device [n_slots][h_in * r_max] */
  lora_bf16* B_arena;     /* device [n_slots][r_max * h_out] */
  const lora_bf16* A_src; /* [h_in][rank] row-major: pinned host memory (asynchronous) or device memory */
  const lora_bf16* B_src; /* [rank][h_out] row-major */
  int32_t h_in, h_out;
} lora_slot_src;

/*
 * Copies adapter matrices into slot `slot` of each listed arena pair (any
 * number of pairs: all projections of all layers), packed at the slot start
 * as the slot layout requires, with one cudaMemcpyAsync per matrix on
 * `stream` (cudaMemcpyDefault: host or device sources; a pageable host source
 * makes the call wait for its copy).  Errors: srcs NULL or n_src < 1, a NULL
 * pointer, slot outside [0, n_slots), rank not in {8,16,32,64} or above r_max,
 * widths not multiples of 8 (LORA_ERR_INVALID_ARG / LORA_ERR_UNSUPPORTED),
 * arenas not 16-byte aligned (LORA_ERR_MISALIGNED), a failed copy
 * (LORA_ERR_CUDA; earlier copies of the call may have been issued).
 */
LORA_API lora_status lora_slot_copy(const lora_slot_src* srcs, int32_t n_src, int32_t n_slots, int32_t r_max,
                                    int32_t slot, int32_t rank, lora_stream_t stream);

/*
 * Table entry of adapter `adapter`: slot_of[adapter] = slot, rank_of[adapter]
 * = rank, written by a one-thread kernel on `stream`.  slot = -1 evicts the
 * adapter (rank is then stored as 0): later batches that name it get
 * LORA_ERR_BAD_ADAPTER_ID in their err_flag.  Errors: NULL or misaligned
 * tables, adapter outside [0, n_adapters), slot < -1, rank invalid for a
 * slot >= 0.
 */
LORA_API lora_status lora_slot_assign(int32_t* slot_of, int32_t* rank_of, int32_t n_adapters, int32_t adapter,
                                      int32_t slot, int32_t rank, lora_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* LORA_SGMV_H_ */
