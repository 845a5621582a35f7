/*
 * moe_gb300.h -- C ABI of the DeepSeek-style MoE FFN forward on one GB300 (sm_103a).
 *
 * The layer: router linear -> sigmoid group-top-k gate with e_score_correction_bias ->
 * token-to-expert dispatch -> expert SwiGLU GEMMs over the gathered tokens -> weighted
 * combine plus the always-active shared expert.  Sources (page title, section):
 *   [gate]  "feat(engine): E1 DeepSeek-style MoE gate (sigmoid, group top-k, bias) (#108)",
 *           sections "API", "Algorithm (mlx-lm group_expert_select)", "Scope decisions",
 *           and the review sections "What looks solid", "Findings" and "Architecture and
 *           design";
 *   [epic]  "Epic: Engine Inference Core Stage E - MoE + hybrid families", first paragraph
 *           (expert dispatch through gather_mm / gather_qmm) and "Decision 5" (4-bit target
 *           checkpoint).
 *
 * Conventions shared by every entry point
 *   - Every tensor pointer is a DEVICE pointer on the current CUDA device, unless the
 *     argument says otherwise; the caller owns all memory (outputs and workspaces too).
 *     Row-major layouts throughout; bf16 is IEEE bfloat16, fp16 is IEEE binary16.
 *   - A call with zero tokens (T == 0 / rows == 0) launches nothing except moe_permute,
 *     which still writes counts and offsets; its token-sized arrays may then be NULL.
 *   - Every call is asynchronous on `stream` (NULL = the legacy default stream) and
 *     never synchronises the host, except moe_device_status().
 *   - Return value: MOE_OK (0) or a negative code.  All argument checks run on the host
 *     BEFORE the first launch, so on MOE_ERR_INVALID no output has been touched (the
 *     gate's contract: outputs unchanged on failure).  MOE_ERR_CUDA means a launch failed;
 *     outputs are then undefined.  moe_last_error() returns a thread-local message naming
 *     the failed check.
 *   - Device-side waits are bounded: a kernel whose wait exceeds its limit stops, leaves
 *     its outputs undefined and records MOE_ERR_TIMEOUT in a per-device status word read
 *     by moe_device_status().
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* identical to cudaStream_t */

enum {
    MOE_OK = 0,
    MOE_ERR_INVALID = -1, /* an argument check failed; nothing was launched            */
    MOE_ERR_CUDA = -2,    /* a CUDA call or launch failed                               */
    MOE_ERR_TIMEOUT = -3, /* a device-side wait gave up (reported by moe_device_status) */
    MOE_ERR_NODEVICE = -4 /* no usable sm_103 device is current                         */
};

typedef enum { MOE_DTYPE_F32 = 0, MOE_DTYPE_BF16 = 1 } moe_dtype_t;

/* Gate parameters ([gate] "API": the params struct of the DeepSeek route). */
typedef struct {
    int32_t top_k;                 /* K experts per token, 1 <= K <= min(E, 32)            */
    int32_t n_group;               /* G >= 1, E % G == 0, E/G >= 2 when G > 1, G <= 32      */
    int32_t topk_group;            /* 1 <= topk_group <= G                                  */
    int32_t norm_topk_prob;        /* renormalise the K weights (only when K > 1)           */
    float routed_scaling_factor;   /* multiplies the K weights last                         */
} moe_route_params_t;

/*
 * Expert weights, stacked on a leading expert axis of length NE (NE = E for the routed
 * experts, NE = 1 for the shared expert).
 *   bits == 16: gate, up: bf16 [NE, I, d]; down: bf16 [NE, d, I]; the scale/bias
 *               pointers are ignored.
 *   bits == 4 : affine 4-bit, one fp16 scale and bias per group_size (32, 64 or 128)
 *               consecutive inputs.  gate, up: uint32 [NE, I, d/8]; down: uint32
 *               [NE, d, I/8]; element j of a row is nibble j%8 (bits 4*(j%8)..+3, low
 *               nibble first) of word j/8; *_scale, *_bias: fp16 [NE, I, d/group_size]
 *               (gate, up) and [NE, d, I/group_size] (down); w = scale * q + bias.
 *   bits == 8 : affine 8-bit, the same groups; gate, up: uint32 [NE, I, d/4]; down: uint32
 *               [NE, d, I/4]; element j of a row is byte j%4 (bits 8*(j%4)..+7, low byte
 *               first) of word j/4.
 *   Quantised weights are dequantised to bf16 inside the expert GEMMs (4-bit: one bf16
 *   fused multiply-add; 8-bit: fp32 fused multiply-add, then one rounding to bf16).
 *   All pointers 16-byte aligned (the scales and biases: 2-byte).
 */
typedef struct {
    int32_t bits;
    int32_t group_size;
    const void* gate;
    const void* up;
    const void* down;
    const void* gate_scale;
    const void* gate_bias;
    const void* up_scale;
    const void* up_bias;
    const void* down_scale;
    const void* down_bias;
} moe_expert_weights_t;

/* Thread-local text of the last failed check or CUDA error ("" if none). */
const char* moe_last_error(void);

/* Library version, major*10000 + minor*100 + patch. */
int32_t moe_version(void);

/* Reads (and, if clear != 0, resets) the current device's status word: MOE_OK or
 * MOE_ERR_TIMEOUT.  Synchronises `stream` first. */
int moe_device_status(int32_t clear, moe_stream_t stream);

/*
 * moe_indexer_topk -- the DSA indexer's selection (SwiftLM issue #139, "What needs
 * building" items 1 and 3: argPartition(scores, kth: -index_topk); decode gathers the
 * selected positions, prefill ANDs them into the causal mask).
 *   scores [rows, ld] fp32 or bf16, n positions per row (ld >= n, in elements).
 *   lengths [rows] int32 or NULL: row r considers positions j < lengths[r] only (clamped to
 *     [0, n]; the causal length of a prefill query); NULL means n for every row.
 *   k = index_topk (1 <= k <= 2^20).
 *   Out: inds [rows, k] int32: the positions of the min(k, n_r) largest scores of the row,
 *     larger score first and equal scores by lower position (NaN lowest, -0 == +0),
 *     written in ASCENDING position order and padded with -1.  A row with n_r <= k selects
 *     all its positions (the inert regime: identical to dense attention).
 *   mask [rows, mask_ld] uint8 or NULL (mask_ld >= n): 1 at the selected positions, 0 at
 *     every other position j < n (the selection already excludes j >= n_r).
 *   Exact: positions are chosen by comparisons only, no arithmetic on the scores.
 */
int moe_indexer_topk(const void* scores, moe_dtype_t dtype, int64_t rows, int32_t n,
                     int64_t ld, const int32_t* lengths, int32_t k, int32_t* inds,
                     uint8_t* mask, int64_t mask_ld, moe_stream_t stream);

/* Exercises the device-side timeout path without a fault: one CTA waits on an mbarrier that
 * nothing completes, through the same bounded wait the GEMM kernels use, gives up after
 * limit_ns (1e3 <= limit_ns <= 1e9, else MOE_ERR_INVALID) and records MOE_ERR_TIMEOUT in the
 * status word.  A following moe_device_status() must then report MOE_ERR_TIMEOUT, and the
 * context stays usable.  Lets a deployment check the watchdog plumbing on its device. */
int moe_watchdog_selftest(int64_t limit_ns, moe_stream_t stream);

/*
 * moe_route_deepseek -- the DeepSeek gate ([gate] "API" and "Algorithm").
 *   logits [rows, E] (fp32 or bf16; any leading dims flattened to rows), bias [E] fp32
 *   (required; pass zeros when the checkpoint has none).
 *   Out: inds [rows, K] int32, scores [rows, K] fp32.
 * Per row: s = sigmoid(f32(logit)); selection runs on s + bias; for G > 1 the group score
 * is the sum of the group's two largest biased scores, and the experts of the
 * G - topk_group worst groups are set to 0.0 (skipped when that difference is 0); the K
 * largest biased scores are selected, in descending order with ties to the lower expert
 * index (lower group index for group ties); the weights are the pre-bias s of the
 * selected experts, divided by their sum only when K > 1 and norm_topk_prob (no zero-sum
 * guard), then multiplied by routed_scaling_factor.
 * Errors: MOE_ERR_INVALID for a NULL pointer, rows < 0, E < 1 or E > 1024, and every
 * parameter rule listed at moe_route_params_t.  rows == 0 is a no-op.
 */
int moe_route_deepseek(const void* logits, moe_dtype_t dtype, int64_t rows, int32_t E,
                       const float* bias, const moe_route_params_t* params, int32_t* inds,
                       float* scores, moe_stream_t stream);

/*
 * moe_route_softmax -- the softmax route of the generic MoE block ([gate] "Scope decisions"
 * and review "What looks solid" 1: the softmax route always renormalises its top-k, unlike
 * the DeepSeek gate).  logits [rows, E] fp32 or bf16.  Out: inds [rows, K] (the K largest
 * logits = the K most probable experts; descending, ties to the lower index), scores
 * [rows, K] = the selected softmax probabilities renormalised over the selection, computed
 * as exp(l_k - l_max) / sum_sel exp(l_j - l_max) in fp32 (K = 1 gives 1.0).
 * Errors: MOE_ERR_INVALID for NULL pointers, rows < 0, E < 1 or > 1024, top_k outside
 * [1, min(E, 32)], an unknown dtype.  rows == 0 is a no-op.
 */
int moe_route_softmax(const void* logits, moe_dtype_t dtype, int64_t rows, int32_t E,
                      int32_t top_k, int32_t* inds, float* scores, moe_stream_t stream);

/*
 * moe_permute -- token-to-expert dispatch ([epic] first paragraph: the grouping that
 * gather_mm / gather_qmm consume).  inds [T, K] int32 expert ids of the P = T*K pairs
 * p = t*K + k.
 * Out: counts [E] (pairs per expert), offsets [E+1] (exclusive scan, offsets[E] = number
 * of dispatched pairs), perm [P] (slot j -> pair id, sorted by (expert, p): stable),
 * inv_perm [P] (pair id -> slot).  A pair whose expert id is outside [0, E) is not
 * dispatched: its inv_perm entry is -1 and offsets[E] < P.
 * Errors: MOE_ERR_INVALID for NULL pointers, T < 0, K < 1, E < 1, E > 1024, T*K >= 2^31.
 */
int moe_permute(const int32_t* inds, int64_t T, int32_t K, int32_t E, int32_t* counts,
                int32_t* offsets, int32_t* perm, int32_t* inv_perm, moe_stream_t stream);

/*
 * moe_router_logits -- the router linear (the DeepSeek body's first call, [gate]
 * "Merge recommendation": linear(router) -> route -> switch_glu -> combine).
 *   x bf16 [T, d], w_router bf16 [E, d], logit_offset fp32 [E] or NULL (an additive
 *   per-expert term, the router linear's bias).  Out: logits fp32 [T, E] = x w_router^T
 *   (+ logit_offset), bf16 products accumulated in fp32.
 * Errors: MOE_ERR_INVALID for NULL pointers, T < 0, d % 64 != 0, E < 1, E > 1024.
 */
int moe_router_logits(const void* x, int64_t T, int32_t d, const void* w_router, int32_t E,
                      const float* logit_offset, float* logits, moe_stream_t stream);

/*
 * moe_grouped_swiglu -- expert SwiGLU over the dispatched tokens (switch_glu with
 * gather_mm / gather_qmm, [epic] first paragraph and [gate] "Architecture and design").
 * For each slot j of expert e (token t = perm[j] / K):
 *     out[j] = W_down[e] (silu(W_gate[e] x[t]) * (W_up[e] x[t])),  silu(a) = a/(1+e^-a),
 * with fp32 accumulation, h rounded to bf16 between the two GEMMs, out stored as bf16.
 * If shared != NULL the shared expert runs on every token in the same launches and its
 * rows follow: out[P + t] = FFN_shared(x[t]).
 *   x bf16 [T, d]; offsets [E+1] and perm [P] as produced by moe_permute; experts with
 *   NE = E; shared (NE = 1, bits 16) or NULL.  Out: out bf16 [P (+T), d].
 *   ws: device workspace of at least moe_grouped_swiglu_workspace_bytes() bytes,
 *   256-byte aligned; its contents need no initialisation and are clobbered.
 * Errors: MOE_ERR_INVALID for NULL pointers, T < 0, K < 1, E < 1 or > 1024, d or I not a
 * multiple of 128, T*K >= 2^31, bits not 16, 8 or 4, group_size not 32, 64 or 128 for
 * quantised weights, shared bits != 16, misaligned pointers, or a workspace that is too
 * small.
 */
int moe_grouped_swiglu(const void* x, int64_t T, int32_t d, int32_t I, int32_t E, int32_t K,
                       const int32_t* offsets, const int32_t* perm,
                       const moe_expert_weights_t* experts, const moe_expert_weights_t* shared,
                       void* out, void* ws, size_t ws_bytes, moe_stream_t stream);

size_t moe_grouped_swiglu_workspace_bytes(int64_t T, int32_t d, int32_t I, int32_t E,
                                          int32_t K, int32_t has_shared);

/*
 * moe_combine -- weighted combine plus the shared expert ([gate] "Architecture and
 * design": combine with an always-active, ungated shared expert):
 *     y[t] = sum_k scores[t,k] * expert_out[inv_perm[t*K+k]] (+ shared_out[t]),
 * summed in fp32 in k order, stored as bf16.  Pairs with inv_perm == -1 contribute 0.
 *   expert_out bf16 [P, d] (slot order), scores fp32 [T, K], inv_perm [P],
 *   shared_out bf16 [T, d] or NULL.  Out: y bf16 [T, d].
 * Errors: MOE_ERR_INVALID for NULL pointers, T < 0, K < 1, d % 8 != 0.
 */
int moe_combine(const void* expert_out, const float* scores, const int32_t* inv_perm,
                const void* shared_out, int64_t T, int32_t K, int32_t d, void* y,
                moe_stream_t stream);

/*
 * moe_shared_gate -- per-token weight of a gated shared expert ([gate] "Architecture and
 * design": the combine's has_shared_expert_gate option): gate[t] = sigmoid(x[t] . w_gate),
 * bf16 x [T, d] and w_gate [d], fp32 products and sum.  Out: gate fp32 [T].
 * Errors: MOE_ERR_INVALID for NULL pointers, T < 0, d % 8 != 0, misaligned x / w_gate.
 */
int moe_shared_gate(const void* x, int64_t T, int32_t d, const void* w_gate, float* gate,
                    moe_stream_t stream);

/*
 * moe_combine_gated -- moe_combine with the gated shared expert:
 *     y[t] = sum_k scores[t,k] * expert_out[inv_perm[t*K+k]] + shared_gate[t] * shared_out[t]
 * shared_gate fp32 [T] (e.g. from moe_shared_gate).  Other arguments and errors as
 * moe_combine; shared_out and shared_gate are required.
 */
int moe_combine_gated(const void* expert_out, const float* scores, const int32_t* inv_perm,
                      const void* shared_out, const float* shared_gate, int64_t T, int32_t K,
                      int32_t d, void* y, moe_stream_t stream);

/*
 * moe_forward -- the whole layer: router linear, gate, dispatch, expert SwiGLU (+ shared
 * expert), combine.  Arguments as in the calls above; y bf16 [T, d].  inds_out [T, K],
 * scores_out [T, K] and logits_out [T, E] are optional copies of the intermediate results
 * (NULL to skip).  ws: at least moe_forward_workspace_bytes() bytes, 256-byte aligned.
 * Errors: the union of the checks of the calls above.
 */
int moe_forward(const void* x, int64_t T, int32_t d, int32_t I, int32_t E,
                const void* w_router, const float* bias, const float* logit_offset,
                const moe_route_params_t* params, const moe_expert_weights_t* experts,
                const moe_expert_weights_t* shared, void* y, int32_t* inds_out,
                float* scores_out, float* logits_out, void* ws, size_t ws_bytes,
                moe_stream_t stream);

size_t moe_forward_workspace_bytes(int64_t T, int32_t d, int32_t I, int32_t E, int32_t top_k,
                                   int32_t has_shared);

/*
 * moe_forward_ex -- the layer with a choice of gate and an optional shared-expert gate:
 * route_kind MOE_ROUTE_DEEPSEEK (moe_route_deepseek; bias required) or MOE_ROUTE_SOFTMAX
 * (moe_route_softmax; bias, groups, norm and scale unused), and w_shared_gate bf16 [d]
 * (non-NULL: the shared expert's output is weighted by sigmoid(x . w_shared_gate), as in
 * moe_combine_gated; NULL: weight 1).  Every other field as in moe_forward.
 * ws: at least moe_forward_ex_workspace_bytes(args) bytes, 256-byte aligned.
 * Errors: those of moe_forward, an unknown route_kind, w_shared_gate without a shared
 * expert.
 */
typedef enum { MOE_ROUTE_DEEPSEEK = 0, MOE_ROUTE_SOFTMAX = 1 } moe_route_kind_t;

typedef struct {
    int32_t route_kind;
    const void* x;
    int64_t T;
    int32_t d;
    int32_t I;
    int32_t E;
    const void* w_router;
    const float* logit_offset;
    const float* bias;
    moe_route_params_t params;
    const moe_expert_weights_t* experts;
    const moe_expert_weights_t* shared;
    const void* w_shared_gate;
    void* y;
    int32_t* inds_out;
    float* scores_out;
    float* logits_out;
} moe_layer_args_t;

int moe_forward_ex(const moe_layer_args_t* args, void* ws, size_t ws_bytes, moe_stream_t stream);

size_t moe_forward_ex_workspace_bytes(const moe_layer_args_t* args);

/*
 * moe_forward_noalloc -- moe_forward without a caller workspace.  The pages have no
 * counterpart: it exists for callers that cannot allocate device memory — serving engines
 * that reserve nearly all of HBM for their own pools up front and hand out nothing else,
 * hosts whose device allocator belongs to another framework.  Arguments and results are
 * those of moe_forward minus ws / ws_bytes.
 *   - The workspace is a fixed array of MOE_NOALLOC_SCRATCH_BYTES (64 MiB) in the
 *     library's own device memory, held on every device that loads the library until the
 *     process exits; it fits decode batches (up to 227 tokens at d = 7168, E = 256,
 *     I = 2048, top_k = 8 with a shared expert).  A layer whose
 *     moe_forward_workspace_bytes() exceeds it is rejected with MOE_ERR_INVALID before
 *     anything runs.
 *   - The first call on a device resolves the array's address with that device current;
 *     make that first call before any stream capture.
 *   - All calls on a device share the array: calls that overlap on the GPU race, so keep
 *     them on one stream.  The array keeps the last call's contents; nothing in it needs
 *     to start at zero.
 *   - Allocates nothing: no cudaMalloc / cudaFree and no allocating library routine.
 */
#define MOE_NOALLOC_SCRATCH_BYTES (64ull << 20)
int moe_forward_noalloc(const void* x, int64_t T, int32_t d, int32_t I, int32_t E,
                        const void* w_router, const float* bias, const float* logit_offset,
                        const moe_route_params_t* params, const moe_expert_weights_t* experts,
                        const moe_expert_weights_t* shared, void* y, int32_t* inds_out,
                        float* scores_out, float* logits_out, moe_stream_t stream);

/*
 * moe_set_fault / moe_get_fault -- host-side fault injection, a test hook with no
 * counterpart in the pages (which fix only the contract it exercises: outputs unchanged on
 * a rejected call).  With kind MOE_FAULT_LAUNCH the at-th kernel launch (0-based) of every
 * following API call is not made: the call returns MOE_ERR_CUDA at that point, with
 * moe_last_error() naming the step and "injected launch fault".  Kernels launched before it
 * in the same call have run and written what they write; nothing after it runs.  In
 * moe_forward the launches are, in order: 0 router linear, 1 gate, 2 dispatch, 3 token
 * gather, 4 gate/up GEMM, 5 down GEMM, then (moe_forward_ex with a shared-expert gate) the
 * shared gate, then the combine, the only launch that writes y.  The gate is the first
 * launch that writes inds_out / scores_out / logits_out.  The count restarts at every entry
 * point and is kept per host thread.  MOE_FAULT_NONE turns the hook off.
 * The environment variable MOE_FAULT=launch or MOE_FAULT=launch:N sets the initial state
 * (read once, at the first call that needs it).
 * Errors: MOE_ERR_INVALID for an unknown kind, at < 0, NULL pointers.  Process-wide setting.
 */
enum { MOE_FAULT_NONE = 0, MOE_FAULT_LAUNCH = 1 };
int moe_set_fault(int32_t kind, int32_t at);
int moe_get_fault(int32_t* kind, int32_t* at);

/*
 * moe_set_phase_events -- a timing aid with no counterpart in the pages: while set,
 * moe_forward records events[i] on its stream at the boundaries of its steps:
 *   0 start, 1 after the router linear, 2 after the gate, 3 after the dispatch,
 *   4 after the token gather, 5 after the gate/up GEMM, 6 after the down GEMM,
 *   7 after the combine.
 * events: n (<= 8) cudaEvent_t handles owned by the caller, or NULL / n == 0 to stop.
 * Process-wide setting, not thread-safe; events of index >= n are not recorded.
 * Errors: MOE_ERR_INVALID for n < 0, n > 8, or events == NULL with n > 0.
 */
int moe_set_phase_events(void* const* events, int32_t n);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
