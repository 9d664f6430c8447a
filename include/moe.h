/*
 * moe.h -- C ABI of the GB300 (sm_103a) Mixture-of-Experts layer hot path.
 *
 * One MoE layer on one GPU: router scoring and top-k selection, dispatch
 * (per-expert histogram, scan, permute), the per-expert SwiGLU FFN as grouped
 * GEMMs, and the gate-weighted combine.  The layer is the DeepSeek-V3 MoE layer
 * that "CUCo: An Agentic Framework for Compute and Communication Co-design"
 * uses as a headline workload (abstract; Table 4, row "MoE Dispatch/Combine":
 * dispatch and combine around local expert compute).  The pages do not write
 * the arithmetic down; each entry point states the reading it implements.
 *
 * Conventions for every entry point
 *   - Every array argument is a DEVICE pointer unless stated otherwise; the
 *     caller allocates and owns all of them.  The library never allocates or
 *     frees memory.  Between calls it keeps only per-device launch settings
 *     (the grouped-GEMM kernels' shared-memory limit) and, for
 *     moe_dispatch_noalloc alone, a fixed scratch array described there.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued asynchronously; nothing synchronises.
 *   - Return value: a moe_status.  Invalid arguments are detected on the host
 *     before anything is enqueued (MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED /
 *     MOE_ERR_WORKSPACE).  MOE_ERR_CUDA means a launch failed.
 *   - Kernels never spin without bound.  A wait that runs out (about one
 *     second) or an inconsistent device-side input (e.g. non-monotone
 *     offsets) makes the kernel stop early and set the workspace's error word;
 *     moe_check_error() reports it.  Outputs of such a call are unspecified.
 *   - Row-major layouts throughout; T tokens, d hidden size, E routed experts,
 *     k experts per token, I expert intermediate size, S = T*k slots.
 *   - Pointers to bf16 / fp32 / int32 arrays must be 16-byte aligned; d and I
 *     must be multiples of 8 (16-byte rows for the bulk-copy engine).
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size or config   */
    MOE_ERR_UNSUPPORTED = 2,  /* valid but outside what the kernels handle     */
    MOE_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required    */
    MOE_ERR_CUDA = 4,         /* a CUDA launch or runtime call failed          */
    MOE_ERR_TIMEOUT = 5,      /* a bounded device wait ran out (error word)    */
    MOE_ERR_DEVICE_INPUT = 6  /* a kernel found inconsistent device-side input */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

typedef enum {
    MOE_SCORE_SOFTMAX = 0,  /* scores are the router logits; gates from softmax */
    MOE_SCORE_SIGMOID = 1   /* scores are sigmoid(logits); gates from scores     */
} moe_score_fn;

/* Routing configuration.
 *   num_experts  E (1..1024)
 *   top_k        k (1..32, k <= eligible experts)
 *   n_group      number of contiguous expert groups (1 = no group limit);
 *                E % n_group == 0, group size >= 2 when n_group > 1, n_group <= 32
 *   topk_group   groups kept per token (1..n_group)
 *   score_fn     moe_score_fn
 *   routed_scale gates are multiplied by this after normalisation (1.0, 2.5) */
typedef struct {
    int32_t num_experts;
    int32_t top_k;
    int32_t n_group;
    int32_t topk_group;
    int32_t score_fn;
    float routed_scale;
} moe_route_cfg;

/* Source: the pages have no counterpart (library support call).
 * Human-readable name of a status code (static string, never NULL). */
const char* moe_status_string(int status);

/* Source: the pages have no counterpart (library support call).
 * ABI version (major * 100 + minor). */
int moe_version(void);

/* ---------------------------------------------------------------- routing */

/* Source: the pages define no interface; this is the routing that decides
 * the dispatch of Table 4, row "MoE Dispatch/Combine", read as DeepSeek-V3 /
 * Mixtral top-k routing.
 * Top-k selection and gates from a given fp32 score tensor.
 *   scores   [T,E] fp32: logits (softmax) or sigmoid outputs (sigmoid)
 *   bias     [E] fp32 or NULL: added to the scores for SELECTION only
 *            (DeepSeek-V3 style); must be NULL for softmax
 *   topk_idx [T,k] int32 out: experts in selection order -- descending key
 *            (score + bias), equal keys by ascending expert index
 *   topk_w   [T,k] fp32 out: softmax: p_j / sum_sel p with p = softmax over
 *            all E; sigmoid: s_j / sum_sel s; both times routed_scale
 * With n_group > 1, each group's score is the sum of its two largest keys and
 * only the topk_group best groups (ties to the lower group) stay eligible.
 * Selection compares fp32 keys exactly; ties go to the lower index. */
int moe_route_from_scores(const float* scores, const float* bias, int T,
                          const moe_route_cfg* cfg, int32_t* topk_idx, float* topk_w,
                          void* stream);

/* Source: the pages have no counterpart (sizing query).
 * Workspace bytes moe_route needs (T tokens, E experts, hidden size d). */
size_t moe_route_workspace_size(int T, int E, int d, int dtype);

/* Source: the pages define no interface; the router of the DeepSeek-V3 MoE
 * layer named in the abstract and Table 4, row "MoE Dispatch/Combine".
 * Router GEMM then moe_route_from_scores.
 *   x        [T,d] bf16 or fp32 (dtype)
 *   w_router [E,d] fp32
 *   scores   [T,E] fp32 out (logits, or sigmoid(logits)); fp32 accumulate
 * bf16 x: tcgen05 tensor cores, with w_router split into three bf16 terms
 * (hi + mid + lo, each the bf16 rounding of what the previous leave) so that
 * every product is exact and only the fp32 accumulation rounds: each logit
 * is within (ceil(d/16) + 6) * 2^-23 * R of the exact dot product, R the
 * range of its running sum over steps of 16 products (a sigmoid score within
 * a quarter of that plus 2^-21); the K range may be cut into parts whose
 * partial sums are added (in order) before the sigmoid.  fp32 x: CUDA cores
 * in fp32.
 * ws: moe_route_workspace_size bytes (error word, split weight, partials). */
int moe_route(const void* x, int dtype, const float* w_router, const float* bias, int T, int d,
              const moe_route_cfg* cfg, float* scores, int32_t* topk_idx, float* topk_w, void* ws,
              size_t ws_bytes, void* stream);

/* --------------------------------------------------------------- dispatch */

/* Source: the pages have no counterpart (sizing query).
 * Workspace bytes moe_dispatch needs for T tokens, k slots, E experts. */
size_t moe_dispatch_workspace_size(int T, int k, int E);

/* Source: the pages define no interface; the dispatch half of Table 4, row
 * "MoE Dispatch/Combine", on one GPU a stable sort of the slots by expert
 * and a row gather into unpadded expert segments.
 * Stable counting sort of the S = T*k slots (s = t*k + j) by expert, then the
 * row gather.  Outputs (all int32 unless noted):
 *   counts[E]        slots routed to each expert
 *   offsets[E+1]     exclusive prefix of counts, offsets[E] = S
 *   slot_to_row[S]   row(s) = offsets[e] + #{s' < s : idx(s') = e}
 *   row_to_token[S]  t such that row lies in token t's slots
 *   x_perm [S,d]     x_perm[row(s)] = x[s / k]  (dtype of x; may be NULL to
 *                    compute the index maps only)
 * topk_idx entries must lie in [0,E); others set the error word and leave
 * the outputs unspecified.  With T = 0 only counts/offsets are written (zeros)
 * and the per-slot pointers may be NULL.  ws: moe_dispatch_workspace_size bytes, any
 * contents; its first 16 bytes hold the error word (see moe_check_error). */
int moe_dispatch(const int32_t* topk_idx, const void* x, int dtype, int T, int d, int k, int E,
                 int32_t* counts, int32_t* offsets, int32_t* slot_to_row, int32_t* row_to_token,
                 void* x_perm, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------ expert FFN */

/* Source: the pages have no counterpart (sizing query).
 * Workspace bytes moe_grouped_ffn needs for `rows` permuted rows. */
size_t moe_grouped_ffn_workspace_size(int rows, int d, int I, int dtype);

/* Source: the pages define no interface; the local expert compute between
 * dispatch and combine (Table 4, row "MoE Dispatch/Combine", whose padding
 * overhead on imbalanced loads the exact segments here avoid).
 * Per-expert SwiGLU FFN over permuted rows, as two grouped GEMMs:
 *   rows [offsets[e], offsets[e+1]) belong to expert e (offsets on device,
 *   E+1 int32, non-decreasing, offsets[E] <= rows);
 *   H[r]  = silu(x_perm[r] W1_e^T) * (x_perm[r] W3_e^T)   (bf16 for bf16)
 *   y[r]  = H[r] W2_e^T                                     (fp32)
 *   w13 [E,2I,d]: rows 0..I-1 are W1 (gate), rows I..2I-1 are W3 (up)
 *   w2  [E,d,I]   (row-major; the tile-major layouts are for moe_layer)
 *   x_perm [rows,d], y_perm [rows,d] fp32 (rows past offsets[E] untouched).
 * bf16 runs on the tcgen05 tensor cores with fp32 accumulation; fp32 runs on
 * the CUDA cores in fp32.  Experts with no rows read none of their weights.
 * ws: moe_grouped_ffn_workspace_size bytes (holds H and the error word). */
int moe_grouped_ffn(const void* x_perm, const int32_t* offsets, int E, int rows, int d, int I,
                    const void* w13, const void* w2, int dtype, float* y_perm, void* ws,
                    size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- combine */

/* Source: the pages define no interface; the combine half of Table 4, row
 * "MoE Dispatch/Combine": each token's expert results weighted and summed.
 * out[t,:] = sum_{j<k} topk_w[t,j] * y_perm[slot_to_row[t*k+j], :]  (+ shared[t,:])
 * summed in slot order in fp32.  y_perm [S,d] fp32, shared [T,d] fp32 or NULL,
 * out [T,d] fp32 (must not alias the inputs). */
int moe_combine(const float* y_perm, const int32_t* slot_to_row, const float* topk_w,
                const float* shared, int T, int k, int d, float* out, void* stream);

/* ---------------------------------------------------------- the whole layer */

/* Number of stage-boundary events moe_layer records when asked (see below). */
#define MOE_LAYER_EVENTS 7

/* Inputs of one MoE layer.  Expert weights and x share `dtype`; the router
 * weight and bias are fp32.  w13_sh/w2_sh (shared expert, [2I_sh,d] and
 * [d,I_sh], gate weight 1) may be NULL with I_sh = 0.  The optional outputs,
 * when non-NULL, receive the intermediate routing results.
 * stage_events, when non-NULL, points to MOE_LAYER_EVENTS cudaEvent_t handles
 * (host array, caller-created) that moe_layer records on `stream` at: start,
 * after routing (router GEMM, top-k and gates), once more at the same point
 * (kept so that stage indices stay fixed), after dispatch, after the routed
 * gate/up GEMM, after the routed down GEMM, and at the end (after combine).
 * They let a caller time each stage inside a run of the whole layer. */
typedef struct {
    const void* x;          /* [T,d]   */
    const float* w_router;  /* [E,d]   */
    const float* bias;      /* [E] or NULL */
    const void* w13;        /* [E,2I,d] */
    const void* w2;         /* [E,d,I]  */
    const void* w13_sh;     /* [2I_sh,d] or NULL */
    const void* w2_sh;      /* [d,I_sh]  or NULL */
    int32_t T, d, I, I_sh, dtype;
    moe_route_cfg route;
    float* scores_out;      /* [T,E]  or NULL */
    int32_t* topk_idx_out;  /* [T,k]  or NULL */
    float* topk_w_out;      /* [T,k]  or NULL */
    int32_t* offsets_out;   /* [E+1]  or NULL */
    void* const* stage_events; /* MOE_LAYER_EVENTS cudaEvent_t, or NULL */
    int32_t flags;          /* MOE_LAYER_* bits, 0 = defaults */
    /* bf16 only, optional: w_router already split by moe_split_router_weight
     * ([3,E,d] bf16), so that the call skips that step; NULL: split per call */
    const void* w_router_split;
    /* optional: MOE_LAYER_SYNC_EVENTS cudaEvent_t handles (host array,
     * caller-created, timing disabled is best) with which the call forks
     * stream2 from `stream` and joins it back (with MOE_LAYER_SPLIT_DISPATCH
     * it reads all four; otherwise only the first two).  NULL: the call
     * creates and destroys the events it needs itself, a host-side cost on
     * every call.  A caller that reuses them must not record them elsewhere
     * while a call that uses them is being enqueued. */
    void* const* sync_events;
} moe_layer_args;

/* Number of events in moe_layer_args.sync_events. */
#define MOE_LAYER_SYNC_EVENTS 4

/* moe_layer_args.flags: add the down projection's results straight into `out`
 * (16-byte fp32 vector reductions in the grouped GEMM's epilogue) instead of
 * writing the permuted fp32 rows and combining them in a separate pass.  bf16 with the
 * shared expert of the routed experts' size (or none) only.  The summation
 * order then varies from run to run (results agree to fp32 rounding). */
#define MOE_LAYER_FUSED_COMBINE 1

/* moe_layer_args.flags: w13 and w2 (and w13_sh, w2_sh) are in the tile-major
 * layouts written by moe_pack_expert_weights, which the grouped GEMMs stream
 * faster.  bf16 with I % 128 == 0, d % 256 == 0 and I_sh % 128 == 0 only
 * (else MOE_ERR_UNSUPPORTED).  Results are the same, bit for bit, as with
 * the row-major weights they were packed from. */
#define MOE_LAYER_PACKED_WEIGHTS 2

/* moe_layer_args.flags: the shared expert's work on stream2 starts once the
 * router GEMM has finished, rather than when it is launched.  A fixed order
 * for CUDA-graph capture: a replayed graph may otherwise start the shared
 * expert's first GEMM ahead of the router GEMM and delay it.  Results are
 * the same either way. */
#define MOE_LAYER_SHARED_AFTER_ROUTER 4

/* moe_layer_args.flags: dispatch overlapped with the routed gate/up (the
 * pages' two-stream dispatch overlap, CUCo, Table 4, row "MoE
 * Dispatch/Combine", on one GPU).  After the count and scan, stream2
 * permutes the tokens of experts [E/2, E) (then runs the shared expert, if
 * any) while `stream` permutes those of experts [0, E/2) and runs their
 * gate/up GEMM; the gate/up of the upper half follows once its permute is
 * done, then the down projection over all experts and the combine.  Needs
 * stream2, bf16 and no MOE_LAYER_FUSED_COMBINE (else MOE_ERR_UNSUPPORTED);
 * E = 1 runs unsplit.  Results are the same, bit for bit, as without it. */
#define MOE_LAYER_SPLIT_DISPATCH 8

/* Source: the pages have no counterpart (sizing query).
 * Workspace bytes moe_layer needs (0 for invalid sizes or configuration).
 * Only the sizes, dtype, routing configuration, I_sh (> 0: shared expert
 * present) and which optional outputs are non-NULL matter here; the input
 * pointers may still be NULL. */
size_t moe_layer_workspace_size(const moe_layer_args* a);

/* Source: the pages define no interface; the whole DeepSeek-V3 MoE layer of
 * the abstract and Table 4, row "MoE Dispatch/Combine" (with its two-stream
 * overlap, on one GPU: the shared expert on stream2).
 * out [T,d] fp32 = the layer: route, dispatch, grouped FFN, shared expert,
 * combine.  `stream2` (may be NULL) is a second stream of the same device.
 * Given stream2, the shared expert's two GEMMs run there, launched with the
 * router GEMM and concurrent with it, top-k and dispatch (with
 * MOE_LAYER_FUSED_COMBINE only its gate/up; its down tiles then ride in the
 * routed down launch).  Without stream2, bf16 with I_sh == I runs the shared
 * expert's tiles inside the routed launches; other shapes run it as launches
 * of its own on `stream`.  Streams are ordered by events; everything is
 * complete on `stream` when the call's work finishes there.  T = 0 is an
 * empty batch: x and out may be NULL, only offsets_out (if given) is written
 * (zeros). */
int moe_layer(const moe_layer_args* a, float* out, void* ws, size_t ws_bytes, void* stream,
              void* stream2);

/* Source: the pages have no counterpart (a one-time weight preparation).
 * Expert weights into the tile-major layouts of MOE_LAYER_PACKED_WEIGHTS, a
 * one-time preparation of a layer's weights.  Each 128-row x 64-column tile
 * (16 KB of bf16) is stored contiguously, so that the grouped GEMMs read it
 * from HBM in one piece rather than as 128 pieces one matrix row apart.
 *   w13 [E, 2I, d] -> w13_packed, tiles (row tile r, column block c) in the
 *     order r-major then c; w2 [E, d, I] -> w2_packed, the two row tiles
 *     2m, 2m+1 of each column block next to each other (the two feature tiles
 *     one down-projection unit reads per stage).  Same sizes as the inputs.
 *   The shared expert's w13_sh [2I_s, d] and w2_sh [d, I_s]: call with E = 1.
 *   Either pair (w13, w13_packed) or (w2, w2_packed) may be NULL (skipped).
 *   Requirements: I % 128 == 0, d % 256 == 0, E >= 1, 16-byte aligned device
 *   pointers (MOE_ERR_INVALID_ARG otherwise); outputs must not overlap the
 *   inputs.  Asynchronous on `stream`. */
int moe_pack_expert_weights(const void* w13, const void* w2, int E, int d, int I,
                            void* w13_packed, void* w2_packed, void* stream);

/* Source: the pages have no counterpart (a one-time weight preparation).
 * The fp32 router weight [E,d] as the three bf16 terms the tensor-core router
 * multiplies (out [3,E,d] bf16: hi, mid, lo, each term the bf16 rounding of
 * what the previous ones leave; w = hi + mid + lo exactly for |w| >= 2^-110,
 * to within 2^-134 below, where bf16's finest spacing ends), for
 * moe_layer_args.w_router_split: a one-time preparation instead of a split
 * on every call.  E >= 1, d >= 8 with d % 8 == 0, 16-byte aligned device
 * pointers (MOE_ERR_INVALID_ARG otherwise).  Asynchronous on `stream`. */
int moe_split_router_weight(const float* w_router, int E, int d, void* out, void* stream);

/* ------------------------------------------------- allocation-free dispatch */

/* Largest T*k that moe_dispatch_noalloc accepts (E up to 1024). */
#define MOE_DISPATCH_NOALLOC_MAX_SLOTS 131072

/* moe_dispatch for callers that cannot allocate device memory while they run
 * (a serving runtime whose memory pool is fixed at start-up, a plug-in inside
 * a framework that owns the allocator, code allowed to allocate only during
 * initialisation).  The pages have no counterpart; this is a library
 * convenience.  Same arguments and outputs as moe_dispatch, but no workspace:
 * the scratch lives in a fixed 1 MiB array in the library's device memory,
 * which every GPU that loads the library holds until the process exits.
 *   - T*k above MOE_DISPATCH_NOALLOC_MAX_SLOTS or E above 1024 is refused
 *     with MOE_ERR_UNSUPPORTED; nothing is enqueued.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it with the identity of the current
 *     CUDA context; a call in a different context (after cudaDeviceReset,
 *     say) looks it up again.  Make the first call on a device, and the
 *     first after such a reset, before any stream capture.
 *   - All calls share the one array, which keeps the last call's contents
 *     (each call clears what must start at zero).  Calls that may overlap on
 *     the GPU -- on different streams without ordering between them -- race
 *     on it and give wrong results; order them.
 *   - device_error: optional device pointer to one uint32 that receives, in
 *     stream order, this call's error word (0 = no error; otherwise the bits
 *     moe_check_error would report).  NULL skips it.
 *   - Calls no allocating function (no cudaMalloc/cudaFree or equivalent). */
int moe_dispatch_noalloc(const int32_t* topk_idx, const void* x, int dtype, int T, int d, int k,
                         int E, int32_t* counts, int32_t* offsets, int32_t* slot_to_row,
                         int32_t* row_to_token, void* x_perm, uint32_t* device_error,
                         void* stream);

/* Source: the pages have no counterpart (failure detection support).
 * Synchronises `stream`, reads and clears the error word of `ws` (a workspace
 * previously passed to moe_dispatch / moe_grouped_ffn / moe_layer).  Returns
 * MOE_OK, MOE_ERR_TIMEOUT, MOE_ERR_DEVICE_INPUT or MOE_ERR_CUDA.  `detail`
 * (host pointer, may be NULL) receives the raw error word. */
int moe_check_error(void* ws, void* stream, uint32_t* detail);

/* Source: the pages have no counterpart (failure detection support).
 * Self-test of the bounded device waits (failure detection without a fault).
 * Launches one tiny kernel that waits on something nothing will ever signal:
 * which = 0: an mbarrier, as in the grouped-GEMM pipeline; which = 1: a
 * predecessor's look-back flag, as in the dispatch scan; which = 2: an
 * mbarrier with cluster-scope acquire in each CTA of a two-CTA cluster, as
 * in the CTA-pair grouped GEMM's cross-CTA waits.  The wait gives up
 * after limit_us microseconds (1..1000000) and sets the error word of `ws`
 * (>= 512 bytes, any contents); moe_check_error(ws, ...) then returns
 * MOE_ERR_TIMEOUT.  The kernels of the layer use the same waits with a
 * one-second limit. */
int moe_selftest_bounded_wait(int which, uint32_t limit_us, void* ws, size_t ws_bytes,
                              void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
