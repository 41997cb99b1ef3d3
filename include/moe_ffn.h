/*
 * moe_ffn.h -- C ABI of the GB300 (sm_103a) routed-expert MoE FFN layer.
 *
 * The layer (GLM-5.3-Flash MoE FFN; "Add GLM-5.3-Flash (glm5next) support
 * with ROCmFP mix qtypes (105/106)", lucebox PR #1, sections "Architecture"
 * and "MoE FFN (REAL routed expert execution)"):
 *
 *   z[t][e]   = sum_h x[t][h] * Wr[e][h] + b[e]          router logits
 *   s[t][e]   = sigmoid(z[t][e])                          routing probability
 *   sel[t]    = the top_k experts by s (ties: lower e)    top-k selection
 *   w[t][j]   = s[t][sel_j] / sum_j' s[t][sel_j']         weight normalisation
 *   FFN_e(v)  = Wd_e . (silu(min(Wg_e v, 10)) * clamp(Wu_e v, -10, 10))
 *   out[t]    = sum_j w[t][j] FFN_{sel_j}(x_t) + FFN_shared(x_t)
 *
 * Int4 storage follows the grouped fmt=4 format with offset-binary decode,
 * value = (nibble - 8) * scale ("feat(glm53): add device-resident HIP backend
 * for MI350P", colibri PR #1448, section "Key changes").  Top-k is
 * deterministic: the lower expert index wins a tie (same section).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every pointer argument is a DEVICE pointer owned by the caller, except
 *   the moe_dims / moe_weights structs themselves, which are host structs
 *   read during the call.  The library allocates no device memory and keeps
 *   no per-call state between calls; scratch lives in the caller's
 *   workspace (see moe_workspace_size).
 * - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *   default stream).  Argument errors are reported synchronously, before
 *   anything is launched.  A failed launch returns MOE_ERR_CUDA.
 * - Device pointers must be 16-byte aligned.
 * - bf16 / fp16 values are IEEE bit patterns in uint16 storage.
 * - T == 0 is a no-op: the call returns MOE_OK and reads or writes nothing.
 * - Shapes: T >= 0 tokens with (top_k+1)*T <= 2^30; H hidden size, a
 *   multiple of 128 up to 12288; E routed experts, top_k <= E <= 512; I
 *   expert intermediate size, multiple of 64; I_shared == I;
 *   1 <= top_k <= 16.  Int4 weights also need H and I to be multiples of 256,
 *   and token values within fp16's range (|x| <= 65504) wherever the tokens
 *   enter as fp16 (moe_permute / moe_expert_ffn, moe_dense_ffn, and
 *   moe_ffn_forward above 64 tokens); larger values are not checked.
 *   Other shapes return MOE_ERR_UNSUPPORTED.  The device must be sm_103
 *   (GB300).
 * - There is no CPU fallback: without a suitable GPU every call fails.
 *
 * Matrix layouts ("nn.Linear", output-major, reduction dim contiguous):
 *   x        [T][H]    bf16          router weight Wr [E][H] bf16
 *   b_router [E]       fp32
 *   bf16 weights: gate, up [E][I][H]; down [E][H][I]; shared: leading dim 1.
 *   Int4 (fmt MOE_W_INT4_G32): codes uint8 [E][N][K/2] with element 2m of a
 *   row in the low nibble of byte m and 2m+1 in the high nibble; scales bf16
 *   [E][N][K/32], one per 32 consecutive reduction elements.  N x K is the
 *   matrix shape above (gate/up: N=I, K=H; down: N=H, K=I).
 */
#ifndef MOE_FFN_H_
#define MOE_FFN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_FFN_ABI_VERSION 6

/* A cudaStream_t, spelled without the CUDA headers. */
typedef struct CUstream_st* moe_stream_t;

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* null / misaligned pointer, negative size */
  MOE_ERR_UNSUPPORTED = 2,   /* shape, top_k, format or GPU not supported */
  MOE_ERR_WORKSPACE = 3,     /* workspace smaller than moe_workspace_size() */
  MOE_ERR_CUDA = 4,          /* a CUDA runtime / driver call failed */
  MOE_ERR_TIMEOUT = 5        /* a device-side wait ran out of time (device status) */
} moe_status;

typedef enum moe_wfmt {
  MOE_W_BF16 = 0,            /* bf16 weights */
  MOE_W_INT4_G32 = 1         /* offset-binary Int4, bf16 scale per 32 elements */
} moe_wfmt;

/* Behaviour flags (moe_dims.flags). */
#define MOE_FLAG_DETERMINISTIC 1  /* fixed-order combination: bitwise reproducible output */
#define MOE_FLAG_ACCUMULATE 2     /* out += layer(x) (out holds e.g. the residual on entry) */

typedef struct moe_dims {
  int32_t T, H, E, I, I_shared, top_k;
  int32_t fmt;               /* moe_wfmt */
  int32_t flags;             /* MOE_FLAG_* bits; 0 = defaults */
} moe_dims;

typedef struct moe_weights {
  const void* gate;          /* bf16 [E][I][H] or Int4 codes [E][I][H/2] */
  const void* up;            /* bf16 [E][I][H] or Int4 codes [E][I][H/2] */
  const void* down;          /* bf16 [E][H][I] or Int4 codes [E][H][I/2] */
  const void* gate_scale;    /* bf16 [E][I][H/32]; NULL for bf16 weights */
  const void* up_scale;      /* bf16 [E][I][H/32]; NULL for bf16 weights */
  const void* down_scale;    /* bf16 [E][H][I/32]; NULL for bf16 weights */
} moe_weights;

/* Library ABI version (MOE_FFN_ABI_VERSION). */
int moe_abi_version(void);

/* Human-readable name of a status code (static storage, never NULL). */
const char* moe_status_string(moe_status s);

/*
 * Bytes of device workspace the calls below need for these dims (0 if the
 * dims are invalid).  The same workspace may serve every entry point for the
 * same dims; calls on one workspace must be stream-ordered.  The first 256
 * bytes hold the device status word (see moe_workspace_status); the caller
 * zeroes the workspace once before first use.
 */
size_t moe_workspace_size(const moe_dims* d);

/*
 * Router + top-k: logits with fused bias, sigmoid, top_k selection (ties to
 * the lower expert index; slot j holds the j-th largest score) and
 * normalisation of the selected scores.
 *   x          [T][H] bf16         w_router [E][H] bf16      b_router [E] fp32
 *   topk_idx   [T][top_k] int32    topk_w   [T][top_k] fp32 (rows sum to 1)
 * Follows "MoE FFN (REAL routed expert execution)": sigmoid routing, top-8
 * selection, weight normalisation (lucebox PR #1).
 */
moe_status moe_router_topk(const moe_dims* d, const void* x, const void* w_router,
                           const float* b_router, int32_t* topk_idx, float* topk_w, void* ws,
                           size_t ws_bytes, moe_stream_t stream);

/*
 * Counting-sort permutation of the (token, slot) pairs by expert, with the
 * shared expert appended as group E holding every token in order:
 *   offsets  [E+2] int32: group g owns rows [offsets[g], offsets[g+1]);
 *            offsets[E] = top_k*T, offsets[E+1] = (top_k+1)*T
 *   gather   [(top_k+1)*T] int32: token of each row (ascending within a group)
 *   row_of   [T][top_k] int32: row holding (t, j)
 *   x_perm   [(top_k+1)*T][H]: x[gather[r]] -- bf16 for MOE_W_BF16; for
 *            MOE_W_INT4_G32 fp16 (the bf16 input converted: exact in fp16's
 *            normal range, within 2^-25 below it) in the
 *            Int4 kernels' operand order: within every aligned group of 8
 *            columns, position p holds column (0, 4, 1, 5, 2, 6, 3, 7)[p].
 *            The order is what lets the kernels expand packed codes with
 *            mask-and-or steps alone; the dot products are unchanged.
 * The grouping that feeds the per-expert matmuls ("ggml_mul_mat_id for
 * gate/up/down", lucebox PR #1, "MoE FFN" section).  Up to 128 tokens one
 * CTA builds all of it (the same code moe_ffn_forward runs at those sizes);
 * above, a count, a scan and a scatter kernel.  Both give the same arrays.
 * Precondition: every topk_idx entry lies in [0, E) and a token's top_k ids
 * are distinct, as moe_router_topk writes them.  The ids are on the device and no error is reported for
 * others: such a pair gets no row (row_of = -1, which moe_combine skips),
 * the other results are undefined, and nothing is written outside the
 * arrays passed in.
 */
moe_status moe_permute(const moe_dims* d, const int32_t* topk_idx, const void* x,
                       int32_t* offsets, int32_t* gather, int32_t* row_of, void* x_perm, void* ws,
                       size_t ws_bytes, moe_stream_t stream);

/*
 * Grouped expert FFN over permuted rows: for row r of group g,
 *   y_perm[r] = FFN_g(x_perm[r])   (g == E: the shared expert), fp32 [(top_k+1)T][H],
 * unweighted.  Gate/up and down run on tcgen05 tensor cores with fp32
 * accumulation; the clamped SwiGLU ("gate (-inf, 10] -> SiLU, up [-10, 10]",
 * lucebox PR #1, Architecture) is fused into the gate/up epilogue.
 * x_perm and offsets as produced by moe_permute.  Int4 weights run on fp16
 * operands here at every T (the 8-bit path of moe_ffn_forward needs the e4m3
 * planes that only the fused call prepares).
 */
moe_status moe_expert_ffn(const moe_dims* d, const void* x_perm, const int32_t* offsets,
                          const moe_weights* experts, const moe_weights* shared, float* y_perm,
                          void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Weighted combination in a fixed order ("Weighted combination of expert
 * outputs", lucebox PR #1, "What Executes vs. TODO" item 3):
 *   out[t] = sum_{j=0..top_k-1} topk_w[t][j] * y_perm[row_of[t][j]] + y_perm[top_k*T + t]
 * out fp32 [T][H] is overwritten, or, with MOE_FLAG_ACCUMULATE, added to
 * (its entry value first, then the slots in order).  Bitwise reproducible.
 * Precondition: row_of as moe_permute writes it.  A slot whose row lies
 * outside [0, (top_k+1)*T) (moe_permute writes -1 for an out-of-range
 * expert id) is skipped.
 */
moe_status moe_combine(const moe_dims* d, const float* y_perm, const int32_t* row_of,
                       const float* topk_w, float* out, moe_stream_t stream);

/*
 * The whole layer, fused: router/top-k, permutation, grouped gate/up with the
 * clamped SwiGLU epilogue, grouped down whose epilogue multiplies by the
 * routing weight and adds into out (fp32 [T][H]), with the shared expert run
 * as one more group of weight 1.  By default out is overwritten and the fp32
 * additions into it are atomic, so the last bits may differ run to run.
 * Int4 weights up to 32 tokens with H a multiple of 1024 up to 4096 and I a
 * multiple of 512 up to 2048 run on CUDA cores: 8-bit integer dot products of
 * the codes against x and h quantised to 16 bits under a power-of-two scale
 * per row and group of 32 (x exactly for entries within 2^-7 of their group's
 * largest |x|, within 2^-15 of it below; h within 2^-14 of its group's
 * largest |h|), exact integer group sums, each group's scale applied in fp32.
 * Other Int4 shapes up to 64 tokens (and these from 33 tokens) run on 8-bit
 * tensor-core operands: the codes
 * as e5m2 (n - 8, exact), x and h as e4m3 planes under power-of-two scales
 * (x exactly for entries at least 2^-9 of their row's largest |x|, within
 * 2^-17 of it below; h within 2^-12 relative near each 32-feature group's
 * largest |h| and 2^-17 of it absolute below), each group's scale applied to its
 * fp32 partial product; larger T expands the weights to fp16 operands.
 * Flags (moe_dims.flags):
 *   MOE_FLAG_DETERMINISTIC  the down GEMM stores unweighted rows into the
 *       workspace and a fixed-order combination (slot 0..top_k-1, then the
 *       shared expert) writes out: bitwise identical run to run; the
 *       workspace grows by (top_k+1)*T*H*4 bytes.
 *   MOE_FLAG_ACCUMULATE  out += layer(x): out's contents on entry (e.g. the
 *       residual stream, "Residual connections" around the FFN in "Add
 *       GLM-5.3-Flash (glm5next) support with ROCmFP mix qtypes (105/106)",
 *       "What Executes vs. TODO") are added to, not replaced.
 */
moe_status moe_ffn_forward(const moe_dims* d, const void* x, const void* w_router,
                           const float* b_router, const moe_weights* experts,
                           const moe_weights* shared, float* out, void* ws, size_t ws_bytes,
                           moe_stream_t stream);

/*
 * Stage boundaries of moe_ffn_forward_timed: ev[i] is recorded on `stream`
 * before stage i, ev[MOE_STAGE_COUNT] after the last one.  Stages:
 *   0 router logits + top-k (for T <= 16 also the permutation, run by the
 *     top-k kernel's last CTA)   1 permutation (one CTA for T <= 128; count,
 *     scan, scatter above) and the gather of x_perm (bf16 weights and T <= 8:
 *     none; the gate/up GEMM gathers its token rows from x itself; Int4
 *     weights and T <= 64: the split of each row into two e4m3 planes)
 *   2 grouped gate/up + SwiGLU   3 grouped down + weighted scatter-add
 * Each ev[i] is a cudaEvent_t created by the caller (NULL entries are skipped).
 * When `stream` is being captured into a CUDA graph the records are captured
 * as external event nodes, so each replay of the graph records them again.
 */
#define MOE_STAGE_COUNT 4
typedef struct moe_stage_events {
  void* ev[MOE_STAGE_COUNT + 1];
} moe_stage_events;

/*
 * moe_ffn_forward with CUDA events recorded between its stages, so that a
 * caller can time each kernel on the launching stream.  Same arguments and
 * results as moe_ffn_forward; `events` may be NULL.
 */
moe_status moe_ffn_forward_timed(const moe_dims* d, const void* x, const void* w_router,
                                 const float* b_router, const moe_weights* experts,
                                 const moe_weights* shared, float* out, void* ws,
                                 size_t ws_bytes, const moe_stage_events* events,
                                 moe_stream_t stream);

/*
 * Dense FFN (the first dense layers of the model, "Dense FFN for layers 0-2
 * (no experts)", lucebox PR #1, "MoE FFN" section) through the same grouped
 * tensor-core GEMMs, all T tokens as one group:
 *   out[t] = Wd . (silu(min(Wg x_t, 10)) * clamp(Wu x_t, -10, 10))
 * d->T, H, I (the dense intermediate size), fmt and flags are used; E, I_shared
 * and top_k are ignored.  weights: gate, up [1][I][H], down [1][H][I] in the
 * format d->fmt (Int4: with scales).  out fp32 [T][H] is overwritten, or
 * added to with MOE_FLAG_ACCUMULATE.  When few tiles would leave SMs idle the
 * down projection is split along K and its parts added atomically, so the
 * last bits may vary run to run; with MOE_FLAG_DETERMINISTIC it is not split
 * and every output element gets one contribution (bitwise reproducible).
 * ws: moe_dense_workspace_size(d).
 */
size_t moe_dense_workspace_size(const moe_dims* d);
moe_status moe_dense_ffn(const moe_dims* d, const void* x, const moe_weights* weights, float* out,
                         void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Where the fused call leaves the layer's routing.  After moe_ffn_forward or
 * moe_ffn_forward_timed has run on `ws` with these dims, the workspace holds
 * the router's selection and the permutation the grouped GEMMs consumed
 * (the top-k of "MoE FFN (REAL routed expert execution)", lucebox PR #1, and
 * the grouping that feeds its per-expert matmuls), in the layouts of
 * moe_router_topk and moe_permute:
 *   topk_idx [T][top_k] int32, topk_w [T][top_k] fp32,
 *   offsets [E+2] int32, gather [(top_k+1)*T] int32, row_of [T][top_k] int32.
 * This call only computes addresses inside `ws` (device pointers, read-only
 * for the caller); it launches and synchronises nothing.  The arrays are
 * valid once the forward call has completed on its stream and until the
 * next call that uses the same workspace.  d must be the dims of that
 * forward call.  T == 0 gives MOE_OK and null pointers.  Useful for
 * inspecting expert loads (e.g. offsets) and for checking the routing
 * against a reference.
 */
typedef struct moe_routing_view {
  const int32_t* topk_idx;
  const float* topk_w;
  const int32_t* offsets;
  const int32_t* gather;
  const int32_t* row_of;
} moe_routing_view;
moe_status moe_workspace_routing(const moe_dims* d, const void* ws, size_t ws_bytes,
                                 moe_routing_view* view);

/*
 * Tensor parallelism along the expert intermediate dimension: copies slice
 * `part` of `parts` of a stack's weights into caller-allocated buffers.
 * The pages' dual-GPU plan places experts on two GPUs ("GLM5next Production
 * Readiness: Optional Mix Qtypes + Cache Allocation", lucebox PR #2, section
 * "UNIT 2: Dual-GPU Placement"); this split is the compute form of it.  The
 * clamped SwiGLU is elementwise in I, so with Is = I / parts, slice p keeps
 * rows [p Is, (p+1) Is) of gate and up and the same columns of down, and
 *   layer(x) = sum over p of layer_p(x)
 * where layer_p is moe_ffn_forward with dims I = I_shared = Is on slice p of
 * both the routed and the shared stack (routing is computed identically by
 * every part).  A caller sums the parts' fp32 outputs: on one GPU by
 * running the parts with MOE_FLAG_ACCUMULATE into one output, across GPUs
 * with one reduce-scatter or all-reduce of out [T][H].
 *   d          dims of the FULL layer (I is the full intermediate size)
 *   n_experts  experts in the stack (d->E for the routed stack, 1 for the
 *              shared expert)
 *   full       the stack as moe_ffn_forward takes it
 *   slice      destination buffers (device, 16-byte aligned, written by the
 *              call; the const of the struct's fields is not honoured here):
 *              bf16: gate, up [n][Is][H], down [n][H][Is]; Int4: codes
 *              gate, up [n][Is][H/2], down [n][H][Is/2] and scales gate, up
 *              [n][Is][H/32], down [n][H][Is/32]
 * Copies run asynchronously on `stream` (copy engine, no kernel).  Returns
 * MOE_ERR_UNSUPPORTED unless I is a multiple of parts and Is a multiple of
 * 64 (bf16) or 256 (Int4); MOE_ERR_INVALID_ARG for a part outside
 * [0, parts), n_experts < 1 or null / misaligned pointers.
 */
moe_status moe_tp_slice_weights(const moe_dims* d, int32_t n_experts, int32_t part,
                                int32_t parts, const moe_weights* full, const moe_weights* slice,
                                moe_stream_t stream);

/*
 * How moe_ffn_forward runs the expert FFN for these dims: 1 when gate/up and
 * down are one kernel launch (bf16 weights, up to 64 tokens, H a multiple of
 * 256, I of 128, not MOE_FLAG_DETERMINISTIC: a persistent kernel in which
 * each down unit waits, through counters in the workspace, for the gate/up
 * tiles of its expert group), 0 when they are two launches, -1 for invalid
 * dims.  For profilers and benchmarks: with one launch the gate/up stage of
 * moe_ffn_forward_timed brackets both projections and the down stage is
 * empty.  Host-only; launches nothing.
 */
int moe_ffn_one_launch(const moe_dims* d);

/*
 * How moe_ffn_forward runs Int4 expert weights for these dims: 1 when gate/up
 * and down run on CUDA cores with 8-bit integer dot products (Int4 weights,
 * up to 32 tokens, H a multiple of 1024 up to 4096, I a multiple of 512 up to
 * 2048), 0 otherwise (tensor-core kernels), -1 for invalid dims.  For
 * profilers and benchmarks.  Host-only; launches nothing.
 */
int moe_ffn_int4_gemv(const moe_dims* d);

/*
 * Synchronises `stream`, returns the device status word that kernels using
 * this workspace have set (MOE_OK, or MOE_ERR_TIMEOUT when a bounded
 * device-side wait gave up), and clears it.
 */
moe_status moe_workspace_status(void* ws, moe_stream_t stream);

/*
 * Diagnostic: runs one device-side bounded wait on a barrier that nothing
 * completes, with a budget of `budget_ns`, so that the timeout path can be
 * exercised without a fault.  Sets the workspace status to MOE_ERR_TIMEOUT.
 * ws must hold at least 256 bytes.
 */
moe_status moe_debug_wait_timeout(void* ws, uint64_t budget_ns, moe_stream_t stream);

/*
 * Router + top-k for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this entry point; it exists for the
 * library's users.  Some callers cannot hand the library a workspace: a
 * plugin or operator interface that passes only input and output pointers,
 * code that must not call cudaMalloc while other work is in flight (the call
 * synchronises the device), or a runtime that owns all device memory through
 * its own pool and gives none out.  This variant takes only inputs and
 * outputs.  Its scratch (the [T][E] fp32 router logits) lives in a
 * fixed-size array inside the library, MOE_STATIC_ROUTER_LOGITS floats
 * (1 MiB), which every GPU that loads the library keeps until the process
 * exits.
 *
 * Arguments and results are those of moe_router_topk (same x, w_router,
 * b_router, topk_idx, topk_w), except that the logits are always computed on
 * the CUDA cores.  T * E above MOE_STATIC_ROUTER_LOGITS returns
 * MOE_ERR_WORKSPACE before anything is launched.
 *
 * The first call in each device context looks up the array's device
 * address (with that device current) and caches it under the context's
 * unique id, so a device reset, which ends the context, leads to a fresh
 * lookup; make the first call in a context before any stream capture.
 * All calls share the one array: calls that may overlap on the GPU (on
 * different streams, or from different threads, without ordering between
 * them) race on it and must be serialised by the caller.  The library
 * allocates nothing in this call.
 */
#define MOE_STATIC_ROUTER_LOGITS (1u << 18)
moe_status moe_router_topk_static_scratch(const moe_dims* d, const void* x, const void* w_router,
                                          const float* b_router, int32_t* topk_idx,
                                          float* topk_w, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_FFN_H_ */
