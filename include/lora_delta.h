/*
 * lora_delta.h -- C ABI of the GB300 (sm_103a) routed multi-tenant LoRA delta.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensors are caller-owned DEVICE memory unless an argument says
 *    "host".  bf16 tensors are row-major with the stated leading dimension.
 *  - Launchers enqueue work on `stream` (a cudaStream_t; NULL is the legacy
 *    default stream): they allocate no device memory and never synchronize
 *    ("Module lora_delta", module invariants).  The one exception is
 *    lora_get_error, which waits on `stream` to read the error word back.
 *    A call whose slots split between the small-segment kernel and the
 *    tensor-core path (lora_delta_fused, lora_delta_segmented) runs the former
 *    on a second stream of the library's, forked from `stream` by an event
 *    and joined back by another: all of the call's work still comes before
 *    anything enqueued on `stream` after it, and inside a stream capture the
 *    fork and the join become part of the captured graph.  That stream and
 *    its two events are created once per device, on the first such call made
 *    outside a capture (a call made during a capture before then runs both
 *    parts on `stream`); calls from several host threads share them, under a
 *    lock.  LORA_FORK=0 in the environment keeps every call on `stream`.
 *  - Return value: LORA_OK (0) or a host-detected LORA_ERR_* status; an error
 *    status means nothing was enqueued.  Nothing is ever thrown.
 *  - Device-detected problems never trap: the offending row / pair is handled
 *    as stated per call and a LORA_DEV_ERR_* bit is OR-ed into the caller's
 *    `err_word` (a device uint32, may be NULL to ignore).  Read it with
 *    lora_get_error.
 *  - Alignment: k_in, every slice width, ld_out, offset_start and the pool
 *    rank R must be multiples of 8 elements (16 bytes of bf16), and x / out /
 *    h must be 16-byte aligned; otherwise LORA_ERR_ALIGN.  A pool address in a
 *    device table that is not 16-byte aligned is found on the device: that
 *    slice is skipped and LORA_DEV_ERR_ALIGN is set.
 *  - Limits: 1 <= S <= 8 slices, 8 <= R <= 128, S*R <= 512, max_loras <= 3071
 *    (LORA_ERR_UNSUPPORTED beyond).
 *
 * Pages the calls follow (cited per call below):
 *  [punica]     "vllm/lora/punica_wrapper/punica_base.py": add_shrink,
 *               add_expand, add_lora_linear "Semantics"; prefill_metadata;
 *               add_lora_w13 / add_lora_w2 (in-place MoE deltas).
 *  [sharded]    "vllm.lora.fully_sharded_layers": the float32 shrink buffer
 *               and the shrink-with-scale-1.0 then expand sequence.
 *  [metrale]    "Module lora_delta": LoraPair / LoraRoute layouts, the
 *               padded-rank invariant, apply_lora_bgmv, the scale rule.
 *  [flashinfer] "flashinfer.fused_moe.bgmv_moe_gemm1_lora_delta".
 */
#ifndef LORA_DELTA_H
#define LORA_DELTA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *lora_stream_t; /* == cudaStream_t */

/* host-detected status codes */
#define LORA_OK 0
#define LORA_ERR_ARG 1         /* NULL pointer, negative size, bad flag        */
#define LORA_ERR_SHAPE 2       /* inconsistent sizes                           */
#define LORA_ERR_ALIGN 3       /* a size or pointer breaks the 16-byte rule    */
#define LORA_ERR_CUDA 4        /* a CUDA launch or copy failed                 */
#define LORA_ERR_WORKSPACE 5   /* workspace missing or smaller than required   */
#define LORA_ERR_UNSUPPORTED 6 /* outside the limits stated above              */
#define LORA_ERR_TOO_LARGE 7   /* needs more scratch than the library's fixed
                                  no-allocation buffer holds                   */

/* device-detected bits, OR-ed into *err_word */
#define LORA_DEV_ERR_SLOT 1u    /* seq_slot >= max_loras: the row gets no delta        */
#define LORA_DEV_ERR_EXPERT 2u  /* MoE expert id outside [0, E): pair written as zeros */
#define LORA_DEV_ERR_LORA 4u    /* MoE adapter id >= num_loras: pair written as zeros  */
#define LORA_DEV_ERR_TIMEOUT 8u /* a bounded wait inside a kernel gave up              */
#define LORA_DEV_ERR_ALIGN 16u  /* a table address is not 16-byte aligned: slice skipped */
#define LORA_DEV_ERR_INTERNAL 32u /* a launch invariant of the library failed (a bug)   */
#define LORA_DEV_ERR_SEGMENT 64u  /* segment starts not nondecreasing in [0, n]: clamped  */

/* Human-readable name of a status code (static string). */
const char *lora_status_string(int status);

/* ABI version of this library (bumped on any signature change). */
int lora_abi_version(void);

/*
 * lora_set_wait_limit_ns -- set the limit, in nanoseconds of the GPU's global
 * timer, after which a bounded wait inside a kernel gives up; returns the
 * previous limit.  None of the pages has this: it is a guard of this
 * library's own kernels.  Every mbarrier wait of the tensor-core kernels is
 * bounded; one that runs out sets LORA_DEV_ERR_TIMEOUT in the call's error
 * word, and its CTA skips its stores, lets its issued MMAs finish, frees its
 * tensor memory and returns, so the context stays usable.  The default is
 * 2 s (2000000000), far above any legitimate wait.  0 makes a wait give up at
 * its first poll that finds the awaited phase incomplete, which lets a test
 * run the time-out path without a fault or a hang.  Process-wide; each
 * launch copies the value current when it is enqueued (a captured CUDA
 * graph keeps the value of its capture).  Thread-safe.
 */
uint64_t lora_set_wait_limit_ns(uint64_t ns);

/*
 * lora_scale -- the adapter scale ([metrale] LoraPair): alpha / r, or
 * alpha / sqrt(r) when use_rslora is nonzero.  Computed on the host; the
 * caller stores it in its scale table.  Applied in the fold (after the
 * expand's rank contraction), never folded into B.  r <= 0 gives 0.
 */
float lora_scale(float alpha, int r, int use_rslora);

/*
 * lora_pool_pack -- pack one PEFT adapter into one padded pool slot
 * ([metrale] module invariants + LoraPair).
 *   a_slot [R, k_in] bf16 (out): rows 0..r-1 = a_r, rows r..R-1 = 0.
 *   b_slot [w, R]    bf16 (out): columns 0..r-1 of each row = b_r, r..R-1 = 0.
 *   a_r    [r, k_in] bf16 (in) : PEFT lora_A, row-major.
 *   b_r    [w, r]    bf16 (in) : PEFT lora_B, row-major.
 * Every element of both slots is written (the zero padding is what lets both
 * stages contract at R).  The caller then stores a_slot / b_slot in its
 * a_table / b_table.  Errors: LORA_ERR_ARG (r < 0, r > R, NULL), ALIGN.
 */
int lora_pool_pack(void *a_slot, void *b_slot, const void *a_r, const void *b_r, int r, int R,
                   int k_in, int w, lora_stream_t stream);

/*
 * Routing tables shared by the linear calls ([metrale] LoraRoute):
 *   a_table, b_table [S * max_loras] uint64 (device): entry j*max_loras + s
 *     is the device address of slot s's A_j [R, k_in] (resp. B_j [w_j, R])
 *     pool region, 0 when slot s does not adapt slice j.
 *   scale_table [max_loras] float (device), or NULL for scale 1.
 *   seq_slot [n] int32 (device): the row's slot; negative = no delta
 *     ([metrale] apply_lora_bgmv); >= max_loras = no delta + LORA_DEV_ERR_SLOT.
 *   widths [S] int32 (HOST): the output slice widths; slice j's columns start
 *     at offset_start + widths[0] + ... + widths[j-1] ([punica] add_expand).
 *
 * Workspace: when n > 1024, or when a workspace is given and n >= 256, the
 * rows are first clustered by slot on the device (a stable counting sort,
 * [punica] prefill_metadata) into a caller-provided scratch buffer of
 * lora_workspace_size(n, S, R, max_loras) bytes, 256-byte aligned; the same
 * buffer holds the fp32 rank intermediate of the tensor-core path that
 * lora_delta_fused takes for slots with many rows.  For n <= 1024 with no
 * workspace each kernel clusters its own rows.
 */
size_t lora_workspace_size(int n, int S, int R, int max_loras);

/*
 * lora_workspace_min_size -- the smallest workspace the linear calls accept
 * for these sizes.  A workspace between this and lora_workspace_size works;
 * the tensor-core path then splits k_in over fewer CTAs.
 */
size_t lora_workspace_min_size(int n, int S, int R, int max_loras);

/*
 * lora_route -- the routing step on its own ([punica] prefill_metadata):
 * a stable clustering of the n rows by slot.
 *   perm      [n] int32 (out): perm[0 .. seg_start[max_loras]) are the rows
 *             with 0 <= slot < max_loras, by ascending slot, then ascending
 *             row index; entries past that are unspecified.
 *   seg_start [max_loras + 2] int32 (out): cluster s is
 *             perm[seg_start[s] .. seg_start[s+1]); the rows with no valid
 *             slot follow, up to seg_start[max_loras + 1] == n.
 * Rows with slot >= max_loras set LORA_DEV_ERR_SLOT.
 */
int lora_route(int32_t *perm, int32_t *seg_start, const int32_t *seq_slot, int n,
               int max_loras, uint32_t *err_word, lora_stream_t stream);

/*
 * lora_route_with_scratch -- lora_route for large batches: the same output
 * (bit for bit), but batches of 2048 rows or more are sorted by many CTAs in
 * chunks of 1024 rows, using a caller-provided scratch buffer of
 * lora_route_scratch_size(n, max_loras) bytes (16-byte aligned; one count per
 * (chunk, slot)).  Errors as lora_route, plus LORA_ERR_WORKSPACE when the
 * scratch is missing or too small.  ([punica] prefill_metadata.)
 */
size_t lora_route_scratch_size(int n, int max_loras);
int lora_route_with_scratch(int32_t *perm, int32_t *seg_start, const int32_t *seq_slot, int n,
                            int max_loras, void *scratch, size_t scratch_bytes,
                            uint32_t *err_word, lora_stream_t stream);

/*
 * lora_shrink -- [punica] add_shrink: for every slice j and routed row i
 *   h[j, i, q] += scale_s * sum_k x[i, k] * A_j,s[q, k],   q < R
 * ("y[i] += (x @ lora_a_stacked[i]) * scale" with A in the [R, k_in] pool
 * layout, so the product is x A^T).  h [S, n, R] float32 (in/out): the
 * [sharded] layers zero it and pass scale 1.0 (scale_table NULL).  Rows with
 * no slot and slices whose a_table entry is 0 are left untouched.
 */
int lora_shrink(float *h, const void *x, int n, int k_in, const int32_t *seq_slot,
                const uint64_t *a_table, const float *scale_table, int S, int R, int max_loras,
                void *workspace, size_t ws_bytes, uint32_t *err_word, lora_stream_t stream);

/*
 * lora_expand -- [punica] add_expand: for every slice j and routed row i
 *   v = scale_s * sum_q h[j, i, q] * B_j,s[c, q]
 *   out[i, off_j + c] = RN_bf16(out + v)   (add_inputs != 0)
 *                     = RN_bf16(v)         (add_inputs == 0)
 * out [n, ld_out] bf16 (in/out).  scale_table NULL means scale 1 (the
 * [punica] expand carries no scale; pass the table to fold it here as
 * [metrale] does).  Rows with no slot and slices whose b_table entry is 0
 * are left untouched bit for bit.  Accumulation is fp32; one rounding to bf16.
 */
int lora_expand(void *out, int64_t ld_out, const float *h, const int32_t *seq_slot,
                const uint64_t *b_table, const float *scale_table, const int32_t *widths, int S,
                int R, int n, int max_loras, int offset_start, int add_inputs, void *workspace,
                size_t ws_bytes, uint32_t *err_word, lora_stream_t stream);

/*
 * lora_expand_gathered -- lora_expand on h as the all-gather of rank-sharded
 * shrinks leaves it ([sharded] _mcp_apply, ColumnParallelLinearWithShardedLoRA
 * and MergedColumnParallelLinearWithShardedLoRA: A sliced along the rank,
 * each of `parts` tensor-parallel ranks shrinks its R / parts rows into an
 * fp32 buffer [S, n, R / parts], and the buffers are all-gathered).  h is
 * [parts][S][n][R / parts] fp32, rank-major: h[p][j][i][q] is rank
 * p * R / parts + q of slice j, row i.  The rest is lora_expand with R the
 * whole rank; each rank calls it with the B rows of its own output columns
 * (b_table, widths) and gets them bit for bit as the unsharded delta does.
 * parts = 1 is lora_expand.  Requires R % parts == 0 (else LORA_ERR_ARG).
 */
int lora_expand_gathered(void *out, int64_t ld_out, const float *h, int parts,
                         const int32_t *seq_slot, const uint64_t *b_table,
                         const float *scale_table, const int32_t *widths, int S, int R, int n,
                         int max_loras, int offset_start, int add_inputs, void *workspace,
                         size_t ws_bytes, uint32_t *err_word, lora_stream_t stream);

/*
 * lora_delta_fused -- the routed delta in one pass ([punica] add_lora_linear,
 * [metrale] apply_lora_bgmv): for every routed row i (s = seq_slot[i]) and
 * slice j whose A and B table entries are both nonzero,
 *   out[i, off_j : off_j + w_j] = RN_bf16(out + scale_s * (x[i] A_j,s^T) B_j,s^T)
 * (RN_bf16(scale_s * ...) when add_inputs == 0).  Both contractions run at
 * the padded rank R, and the rank-R intermediate is fp32.  For slots with
 * few rows it stays on chip; slots with many rows go to the tensor-core path,
 * whose intermediate passes through fp32 planes in the workspace.  x [n, k_in]
 * bf16, out [n, ld_out] bf16.
 */
int lora_delta_fused(void *out, int64_t ld_out, const void *x, int n, int k_in,
                     const int32_t *seq_slot, const uint64_t *a_table, const uint64_t *b_table,
                     const float *scale_table, const int32_t *widths, int S, int R,
                     int max_loras, int offset_start, int add_inputs, void *workspace,
                     size_t ws_bytes, uint32_t *err_word, lora_stream_t stream);

/*
 * lora_delta_segmented -- the delta on rows already grouped by adapter, such
 * as the expert-sorted rows of a grouped MoE GEMM ("expert_apply.rs",
 * apply_expert_lora_sorted / expert_delta_workitems, with the row blocks read
 * from device memory instead of a host copy).  Rows seg_start[s] ..
 * seg_start[s+1] - 1 take adapter s (table entries j * n_segs + s, as in
 * lora_delta_fused with max_loras = n_segs); rows from seg_start[n_segs] on
 * are untouched.  seg_start [n_segs + 1] int32 (device) must start at 0 and
 * be nondecreasing up to at most n; otherwise the starts are clamped into
 * that form (no row outside the batch is read or written) and
 * LORA_DEV_ERR_SEGMENT is set.  Arithmetic, layouts and the other arguments
 * as lora_delta_fused; a workspace of lora_workspace_size(n, S, R, n_segs)
 * bytes is required (no routing sort runs).
 */
int lora_delta_segmented(void *out, int64_t ld_out, const void *x, int n, int k_in,
                         const int32_t *seg_start, int n_segs, const uint64_t *a_table,
                         const uint64_t *b_table, const float *scale_table,
                         const int32_t *widths, int S, int R, int offset_start, int add_inputs,
                         void *workspace, size_t ws_bytes, uint32_t *err_word,
                         lora_stream_t stream);

/*
 * lora_moe_fc1_delta -- [flashinfer] bgmv_moe_gemm1_lora_delta.  For every
 * routed pair (token t, slot j): e = topk_ids[t, j], l = lora_ids[t];
 *   regular (shared_a == 0): w_ptr_a / w_ptr_b are [2, E] int64 tables of
 *     bank base addresses [A_gate, A_up] / [B_gate, B_up];
 *     out[t, j, 0:I]  = RN_bf16(scale * B_gate[l,e] (A_gate[l,e] x[t]))
 *     out[t, j, I:2I] = RN_bf16(scale * B_up[l,e]   (A_up[l,e]   x[t]))
 *   shared  (shared_a != 0): [E] tables, one shared A and a fused
 *     B [2I, rank] (gate rows 0:I, up rows I:2I);
 *     out[t, j, :] = RN_bf16(scale * B_fused[l,e] (A_shared[l,e] x[t]))
 * Adapter l of a bank starts l * stride elements after the bank base; A[l,e]
 * is [rank, H] row-major, B[l,e] is [I, rank] (or [2I, rank]) row-major.
 * out [T, top_k, 2I] bf16 is fully written: pairs with l < 0 are zeros (the
 * page skips them), pairs with l >= num_loras or e outside [0, E) are zeros
 * and set LORA_DEV_ERR_LORA / LORA_DEV_ERR_EXPERT.  The delta stays per
 * (token, slot): no routing weights, no sum over experts.
 * Requires H, I, rank multiples of 8, rank <= 128, E * num_loras <= 3071 and
 * a workspace of lora_moe_workspace_size(T, top_k, E, num_loras, rank,
 * shared_a) bytes.
 */
size_t lora_moe_workspace_size(int T, int top_k, int E, int num_loras, int rank, int shared_a);
int lora_moe_fc1_delta(void *out, const void *x, const int64_t *w_ptr_a, int64_t stride_a,
                       const int64_t *w_ptr_b, int64_t stride_b, int shared_a,
                       const int32_t *topk_ids, const int32_t *lora_ids, int T, int top_k, int E,
                       int H, int I, int rank, int num_loras, float scale, void *workspace,
                       size_t ws_bytes, uint32_t *err_word, lora_stream_t stream);

/*
 * lora_moe_w13_delta -- [punica] add_lora_w13: the gate/up delta of
 * lora_moe_fc1_delta added IN PLACE to y = intermediate_cache1
 * [T, top_k, 2I] bf16 (the expert gate/up GEMM's output, before the
 * activation):
 *   y[t, j, :] = RN_bf16(y[t, j, :] + delta[t, j, :])     (add_inputs != 0)
 *   y[t, j, :] = RN_bf16(delta[t, j, :])                   (add_inputs == 0)
 * with delta and the bank tables, strides and layouts exactly as
 * lora_moe_fc1_delta (regular or shared-A / fused-B mode).  Routing, per pair
 * (t, j): l = lora_ids[t] (the token-to-adapter mapping), e = topk_ids[t, j];
 *   - expert_map [n_global_experts] int32 (device, or NULL = identity):
 *     global expert id -> this rank's local id in [0, E), -1 = the expert
 *     is not on this rank (no delta).  A global id outside the map or a
 *     local id >= E sets LORA_DEV_ERR_EXPERT (no delta);
 *   - adapter_enabled [num_loras] int32 (device, or NULL): an adapter with
 *     entry 0 adds nothing;
 *   - l < 0: no delta; l >= num_loras: no delta + LORA_DEV_ERR_LORA.
 * A pair without a delta is left untouched (y belongs to the caller).
 * Requirements as lora_moe_fc1_delta, with E the local expert count; the
 * workspace is lora_moe_workspace_size(T, top_k, E, num_loras, rank,
 * shared_a) bytes.  Readings: the page gives the signature and docstring
 * only; routing weights are not applied before the activation.
 */
int lora_moe_w13_delta(void *y, const void *x, const int64_t *w_ptr_a, int64_t stride_a,
                       const int64_t *w_ptr_b, int64_t stride_b, int shared_a,
                       const int32_t *topk_ids, const int32_t *lora_ids,
                       const int32_t *expert_map, int n_global_experts,
                       const int32_t *adapter_enabled, int T, int top_k, int E, int H, int I,
                       int rank, int num_loras, float scale, int add_inputs, void *workspace,
                       size_t ws_bytes, uint32_t *err_word, lora_stream_t stream);

/*
 * lora_moe_w2_delta -- [punica] add_lora_w2: the down-projection delta added
 * IN PLACE to y = intermediate_cache3 [T, top_k, H] bf16 (the expert down
 * GEMM's per-pair output, before moe_sum), from x = intermediate_cache2
 * [T * top_k, I] bf16, one activation row per (token, slot) pair p = t *
 * top_k + j:
 *   v[c] = w_p * scale * sum_r B[l,e][c, r] * (A[l,e] x[p])[r]      (fp32)
 *   y[t, j, c] = RN_bf16(y[t, j, c] + v[c])  (add_inputs != 0), else RN_bf16(v[c])
 * w_ptr_a / w_ptr_b: [E] int64 tables of bank base addresses; adapter l of a
 * bank starts l * stride elements after its base; A[l,e] [rank, I] and
 * B[l,e] [H, rank] row-major bf16.  topk_weights [T, top_k] fp32 (device, or
 * NULL: w_p = 1) are the routing weights the down GEMM applied before
 * moe_sum.  Routing (expert_map, adapter_enabled, lora_ids, errors) and the
 * untouched pairs as lora_moe_w13_delta.  Requires H, I, rank multiples of 8,
 * rank <= 128, E * num_loras <= 3071 and a workspace of
 * lora_moe_workspace_size(T, top_k, E, num_loras, rank, 1) bytes (one slice).
 */
int lora_moe_w2_delta(void *y, const void *x, const int64_t *w_ptr_a, int64_t stride_a,
                      const int64_t *w_ptr_b, int64_t stride_b, const int32_t *topk_ids,
                      const int32_t *lora_ids, const int32_t *expert_map, int n_global_experts,
                      const int32_t *adapter_enabled, const float *topk_weights, int T,
                      int top_k, int E, int H, int I, int rank, int num_loras, float scale,
                      int add_inputs, void *workspace, size_t ws_bytes, uint32_t *err_word,
                      lora_stream_t stream);

/*
 * lora_moe_w2_delta_routed -- [punica] add_lora_w2 with the routing that the
 * preceding add_lora_w13 of the same layer handed over ("Reuses routing
 * tensors returned by add_lora_w13"): the same delta as lora_moe_w2_delta,
 * without sorting the pairs again.  `workspace` must be the workspace that a
 * preceding lora_moe_w13_delta call was given, on the same stream, with the
 * same T, top_k, E, num_loras and routing arrays (topk_ids, lora_ids,
 * expert_map, adapter_enabled), and left untouched since: that call wrote the
 * pairs' clustering by (adapter, local expert) at the front of it, and this
 * call reads it.  Every routing decision (no adapter, a switched-off adapter,
 * a non-local expert, a bad id) is taken from there, and its errors were
 * already reported by the w13 call.  x, the banks, topk_weights, y and the
 * arithmetic are as in lora_moe_w2_delta; ws_bytes must be at least
 * lora_moe_workspace_size(T, top_k, E, num_loras, rank, 1).  The workspace is
 * not written before the kernels read the routing, so a following call may
 * reuse it again.
 */
int lora_moe_w2_delta_routed(void *y, const void *x, const int64_t *w_ptr_a, int64_t stride_a,
                             const int64_t *w_ptr_b, int64_t stride_b, const float *topk_weights,
                             int T, int top_k, int E, int H, int I, int rank, int num_loras,
                             float scale, int add_inputs, void *workspace, size_t ws_bytes,
                             uint32_t *err_word, lora_stream_t stream);

/*
 * lora_delta_fused_floor -- a measurement aid, not part of the method (none of
 * the pages has it): moves the bytes that lora_delta_fused moves for a small
 * batch -- every routed slot's A and B (each CTA's share), the slot's x rows
 * and out rows, out written back -- with the same launch plan (grid, thread-
 * block cluster size, shared-memory plan, programmatic dependent launch), but
 * computes nothing: out is written back unchanged.  Timed next to
 * lora_delta_fused on the same inputs, it gives the data-movement floor of a
 * decode step in this launch shape.  Arguments as lora_delta_fused without
 * scale table, add_inputs, workspace and error word; LORA_ERR_UNSUPPORTED
 * unless n <= 1024 and the shape takes the fused small-segment kernel (one k
 * stage per CTA, R a multiple of 16 up to 64, S * R <= 256).
 */
int lora_delta_fused_floor(void *out, int64_t ld_out, const void *x, int n, int k_in,
                           const int32_t *seq_slot, const uint64_t *a_table,
                           const uint64_t *b_table, const int32_t *widths, int S, int R,
                           int max_loras, int offset_start, lora_stream_t stream);

/*
 * lora_delta_fused_noalloc -- lora_delta_fused for callers that cannot
 * allocate device memory.  The pages have no counterpart to this call: it
 * exists for callers whose memory is fixed up front (a budget set at start
 * up, an allocator that refuses allocations after warm-up, a runtime that
 * only lends this library the tensors it already owns) and who therefore
 * cannot provide lora_delta_fused's scratch workspace.
 * Same arguments and results as lora_delta_fused minus the workspace: the
 * scratch comes from a fixed buffer inside the library of
 * lora_noalloc_scratch_bytes() bytes (4 MiB).  The buffer sits in its own
 * CUDA module, which the runtime loads lazily by default: the first call on a
 * device (with that device current) looks the buffer up, and that is when the
 * driver reserves its 4 MiB on the device, which then holds it until the
 * process exits.  Make one warm-up call on every device before the memory
 * budget is fixed and before any stream capture; later calls reserve
 * nothing.  The looked-up address is cached per device and is stale after a
 * cudaDeviceReset.  A call whose smallest workspace
 * (lora_workspace_min_size(n, S, R, max_loras)) exceeds the buffer returns
 * LORA_ERR_TOO_LARGE and enqueues nothing.  Apart from that first reservation
 * the call never allocates (no cudaMalloc, no allocating library routine).
 * All calls share the one buffer: calls that
 * may overlap on the GPU (different streams) race and must be serialized by
 * the caller.  The buffer keeps the last call's contents; nothing in it needs
 * to start at zero.
 */
size_t lora_noalloc_scratch_bytes(void);
int lora_delta_fused_noalloc(void *out, int64_t ld_out, const void *x, int n, int k_in,
                             const int32_t *seq_slot, const uint64_t *a_table,
                             const uint64_t *b_table, const float *scale_table,
                             const int32_t *widths, int S, int R, int max_loras,
                             int offset_start, int add_inputs, uint32_t *err_word,
                             lora_stream_t stream);

/*
 * lora_get_error -- copy the device error word to *host_out after all work
 * queued on `stream` so far has finished (this call synchronizes `stream`),
 * then clear it on the device when `clear` is nonzero.
 */
int lora_get_error(uint32_t *err_word, uint32_t *host_out, int clear, lora_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* LORA_DELTA_H */
