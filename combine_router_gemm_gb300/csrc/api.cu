// api.cu -- the C entry points: argument checks, workspace layout, launches.
//
// Every check runs on the host before anything is enqueued; see moe.h for
// the contract of each call.
#include <math.h>

#include <climits>

#include "common.cuh"

namespace moe_f32 {
int grouped_ffn_f32(const float* x_perm, const int32_t* offsets, int E, int rows, int d, int I,
                    const float* w13, const float* w2, float* y, float* h, uint32_t* err,
                    cudaStream_t s);
}

namespace moe_host {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int launch_status() { return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

int num_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
        return 1;
    return n;
}

}  // namespace moe_host

namespace {

// Workspace header: the error word, then zeroed counters of the grouped
// GEMMs' dynamic unit schedule (one per launch that may be in flight).
constexpr size_t ERR_BYTES = 256;
constexpr int CTR_ROUTER = 1, CTR_FFN = 2 /* +1 */, CTR_SHARED = 4 /* +1 */, CTR_FFN_HI = 6;
constexpr size_t HDR_CLEAR = 64;  // bytes of the header cleared per call
unsigned* ctr(void* ws, int i) { return static_cast<unsigned*>(ws) + i; }

size_t al(size_t v) { return (v + 255) / 256 * 256; }

bool dtype_ok(int dt) { return dt == MOE_F32 || dt == MOE_BF16; }
size_t esize(int dt) { return dt == MOE_BF16 ? 2 : 4; }

int check_cfg(const moe_route_cfg* c) {
    if (!c) return MOE_ERR_INVALID_ARG;
    const int E = c->num_experts, k = c->top_k, g = c->n_group, tg = c->topk_group;
    if (E < 1 || k < 1 || g < 1 || tg < 1) return MOE_ERR_INVALID_ARG;
    if (c->score_fn != MOE_SCORE_SOFTMAX && c->score_fn != MOE_SCORE_SIGMOID)
        return MOE_ERR_INVALID_ARG;
    if (!isfinite(c->routed_scale)) return MOE_ERR_INVALID_ARG;
    if (E % g != 0 || tg > g) return MOE_ERR_INVALID_ARG;
    if (g > 1 && E / g < 2) return MOE_ERR_INVALID_ARG;
    const int eligible = g > 1 ? tg * (E / g) : E;
    if (k > eligible) return MOE_ERR_INVALID_ARG;
    if (E > 1024 || k > 32 || g > 32) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

int check_dims(long long T, int d, int k) {
    if (T < 0 || d < 8 || d % 8 != 0) return MOE_ERR_INVALID_ARG;
    if (T * (long long)k > INT_MAX / 2) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

size_t ffn_ws(int rows, int d, int I, int dtype) {
    (void)d;
    return ERR_BYTES + al((size_t)rows * I * esize(dtype));
}

int run_ffn(const void* x_perm, const int32_t* offsets, int E, int rows, int d, int I,
            const void* w13, const void* w2, int dtype, float* y, void* h, uint32_t* err,
            unsigned* work, cudaStream_t s, cudaEvent_t between = nullptr, bool packed = false) {
    if (rows == 0) {
        if (between && cudaEventRecord(between, s) != cudaSuccess) return MOE_ERR_CUDA;
        return MOE_OK;
    }
    if (dtype == MOE_BF16)
        return moe_tc::grouped_ffn_bf16(x_perm, offsets, E, rows, d, I, w13, w2, y, h, err, work,
                                        s, between, nullptr, nullptr, 3, nullptr, packed);
    int rc = moe_f32::grouped_ffn_f32(static_cast<const float*>(x_perm), offsets, E, rows, d, I,
                                      static_cast<const float*>(w13), static_cast<const float*>(w2),
                                      y, static_cast<float*>(h), err, s);
    if (rc == MOE_OK && between && cudaEventRecord(between, s) != cudaSuccess) rc = MOE_ERR_CUDA;
    return rc;
}

size_t route_ws(int T, int E, int d, int dtype) {
    return ERR_BYTES + (dtype == MOE_BF16 ? al(moe_tc::router_ws_bytes(T, E, d)) : 0);
}

// Scores, top-k and gates.  bf16 activations: tcgen05 GEMM against the fp32
// router weight split into three bf16 terms, writing partial logits of K
// parts that the top-k kernel sums (and passes through the sigmoid) into
// `scores`; fp32 activations: fp32 CUDA-core GEMM writing `scores`.
// side_start (optional) is recorded where work on another stream may begin:
// bf16, once the router weight is split (the router GEMM is one wave that
// leaves SMs idle, and the top-k and dispatch kernels share SMs with other
// work), or with side_after_gemm after the router GEMM; fp32, after the
// router GEMM.
int run_route(const void* x, int dtype, const float* w_router, const float* bias, int T, int d,
              const moe_route_cfg* cfg, float* scores, int32_t* idx, float* w, void* rws,
              uint32_t* err, unsigned* work, cudaStream_t s, cudaEvent_t side_start = nullptr,
              const void* presplit = nullptr, bool side_after_gemm = false) {
    const int E = cfg->num_experts;
    if (dtype == MOE_BF16) {
        float* partial = nullptr;
        int ks = 0;
        int rc = moe_tc::router_bf16(x, w_router, T, d, E, rws, err, work, &partial, &ks, s,
                                     side_after_gemm ? nullptr : side_start, presplit);
        if (rc != MOE_OK) return rc;
        if (side_after_gemm && side_start && cudaEventRecord(side_start, s) != cudaSuccess)
            return MOE_ERR_CUDA;
        return moe_launch::topk(nullptr, bias, T, cfg, idx, w, s, partial, ks, scores);
    }
    int rc = moe_launch::router_gemm(x, dtype, w_router, T, d, E, cfg->score_fn, scores, s);
    if (rc != MOE_OK) return rc;
    if (side_start && cudaEventRecord(side_start, s) != cudaSuccess) return MOE_ERR_CUDA;
    return moe_launch::topk(scores, bias, T, cfg, idx, w, s);
}

struct LayerWs {
    uint32_t* err;
    float* scores;
    int32_t* idx;
    float* w;
    int32_t* counts;
    int32_t* offsets;
    int32_t* s2r;
    int32_t* r2t;
    void* xp;
    float* yp;
    void* h;
    float* ysh;
    void* hsh;
    void* disp;
    void* wsplit;
    float* w_row;  // fused combine: gate weight of each permuted row
    size_t total;
};

LayerWs carve_layer(const moe_layer_args* a, void* base) {
    const int T = a->T, d = a->d, I = a->I, E = a->route.num_experts, k = a->route.top_k;
    const size_t S = (size_t)T * k, es = esize(a->dtype);
    char* p = static_cast<char*>(base);
    size_t off = 0;
    auto take = [&](size_t bytes) -> void* {
        void* r = p ? p + off : nullptr;
        off += al(bytes);
        return r;
    };
    LayerWs w;
    w.err = static_cast<uint32_t*>(take(ERR_BYTES));
    w.scores = a->scores_out ? a->scores_out : static_cast<float*>(take((size_t)T * E * 4));
    w.idx = a->topk_idx_out ? a->topk_idx_out : static_cast<int32_t*>(take(S * 4));
    w.w = a->topk_w_out ? a->topk_w_out : static_cast<float*>(take(S * 4));
    w.counts = static_cast<int32_t*>(take((size_t)E * 4));
    w.offsets = a->offsets_out ? a->offsets_out : static_cast<int32_t*>(take((size_t)(E + 1) * 4));
    w.s2r = static_cast<int32_t*>(take(S * 4));
    w.r2t = static_cast<int32_t*>(take(S * 4));
    w.xp = take(S * d * es);
    w.yp = static_cast<float*>(take(S * d * 4));
    w.h = take(S * I * es);
    const bool sh = a->I_sh > 0;  // a shared expert is present iff I_sh > 0
    w.ysh = sh ? static_cast<float*>(take((size_t)T * d * 4)) : nullptr;
    w.hsh = sh ? take((size_t)T * a->I_sh * es) : nullptr;
    w.disp = take(moe_launch::dispatch_ws_bytes(T, k, E));
    w.wsplit = a->dtype == MOE_BF16 ? take(moe_tc::router_ws_bytes(T, E, d)) : nullptr;
    w.w_row = (a->flags & MOE_LAYER_FUSED_COMBINE) ? static_cast<float*>(take(S * 4)) : nullptr;
    w.total = off;
    return w;
}

// Sizes and configuration only (what the workspace size depends on).
int check_layer_sizes(const moe_layer_args* a) {
    if (!a) return MOE_ERR_INVALID_ARG;
    int rc = check_cfg(&a->route);
    if (rc != MOE_OK) return rc;
    if ((rc = check_dims(a->T, a->d, a->route.top_k)) != MOE_OK) return rc;
    if (!dtype_ok(a->dtype) || a->I < 8 || a->I % 8 != 0) return MOE_ERR_INVALID_ARG;
    if (a->I_sh < 0 || (a->I_sh > 0 && a->I_sh % 8 != 0)) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

int check_layer(const moe_layer_args* a) {
    int rc = check_layer_sizes(a);
    if (rc != MOE_OK) return rc;
    // x may be NULL for an empty batch (T == 0)
    if ((a->T > 0 && !a->x) || !a->w_router || !a->w13 || !a->w2) return MOE_ERR_INVALID_ARG;
    if ((a->x && !moe_host::aligned16(a->x)) || !moe_host::aligned16(a->w_router) ||
        !moe_host::aligned16(a->w13) || !moe_host::aligned16(a->w2))
        return MOE_ERR_INVALID_ARG;
    if (a->bias && a->route.score_fn == MOE_SCORE_SOFTMAX) return MOE_ERR_INVALID_ARG;
    const bool sh = a->w13_sh || a->w2_sh || a->I_sh;
    if (sh) {
        if (!a->w13_sh || !a->w2_sh || a->I_sh < 8 || a->I_sh % 8 != 0) return MOE_ERR_INVALID_ARG;
        if (!moe_host::aligned16(a->w13_sh) || !moe_host::aligned16(a->w2_sh))
            return MOE_ERR_INVALID_ARG;
    }
    if (a->w_router_split &&
        (a->dtype != MOE_BF16 || !moe_host::aligned16(a->w_router_split)))
        return MOE_ERR_INVALID_ARG;
    const void* outs[] = {a->scores_out, a->topk_idx_out, a->topk_w_out, a->offsets_out};
    for (const void* o : outs)
        if (o && !moe_host::aligned16(o)) return MOE_ERR_INVALID_ARG;
    if (a->flags & ~(MOE_LAYER_FUSED_COMBINE | MOE_LAYER_PACKED_WEIGHTS |
                     MOE_LAYER_SHARED_AFTER_ROUTER | MOE_LAYER_SPLIT_DISPATCH))
        return MOE_ERR_INVALID_ARG;
    if ((a->flags & MOE_LAYER_SPLIT_DISPATCH) &&
        (a->dtype != MOE_BF16 || (a->flags & MOE_LAYER_FUSED_COMBINE)))
        return MOE_ERR_UNSUPPORTED;
    if ((a->flags & MOE_LAYER_PACKED_WEIGHTS) &&
        (a->dtype != MOE_BF16 || a->I % 128 != 0 || a->d % 256 != 0 || a->I_sh % 128 != 0))
        return MOE_ERR_UNSUPPORTED;
    if ((a->flags & MOE_LAYER_FUSED_COMBINE) &&
        (a->dtype != MOE_BF16 || (a->I_sh > 0 && a->I_sh != a->I)))
        return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

}  // namespace

extern "C" {

const char* moe_status_string(int status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
        case MOE_ERR_WORKSPACE: return "workspace missing or too small";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_TIMEOUT: return "a bounded device wait ran out";
        case MOE_ERR_DEVICE_INPUT: return "inconsistent device-side input";
        default: return "unknown status";
    }
}

int moe_version(void) { return 100; }

int moe_route_from_scores(const float* scores, const float* bias, int T, const moe_route_cfg* cfg,
                          int32_t* topk_idx, float* topk_w, void* stream) {
    int rc = check_cfg(cfg);
    if (rc != MOE_OK) return rc;
    if (T < 0 || !scores || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
    if (bias && cfg->score_fn == MOE_SCORE_SOFTMAX) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    return moe_launch::topk(scores, bias, T, cfg, topk_idx, topk_w,
                            static_cast<cudaStream_t>(stream));
}

size_t moe_route_workspace_size(int T, int E, int d, int dtype) {
    if (T < 0 || E < 1 || d < 1 || !dtype_ok(dtype)) return 0;
    return route_ws(T, E, d, dtype);
}

int moe_route(const void* x, int dtype, const float* w_router, const float* bias, int T, int d,
              const moe_route_cfg* cfg, float* scores, int32_t* topk_idx, float* topk_w, void* ws,
              size_t ws_bytes, void* stream) {
    int rc = check_cfg(cfg);
    if (rc != MOE_OK) return rc;
    if ((rc = check_dims(T, d, cfg->top_k)) != MOE_OK) return rc;
    if (!dtype_ok(dtype) || !x || !w_router || !scores || !topk_idx || !topk_w)
        return MOE_ERR_INVALID_ARG;
    if (!moe_host::aligned16(x) || !moe_host::aligned16(w_router)) return MOE_ERR_INVALID_ARG;
    if (bias && cfg->score_fn == MOE_SCORE_SOFTMAX) return MOE_ERR_INVALID_ARG;
    if (!ws || !moe_host::aligned16(ws) || ws_bytes < route_ws(T, cfg->num_experts, d, dtype))
        return MOE_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, HDR_CLEAR, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (T == 0) return MOE_OK;
    return run_route(x, dtype, w_router, bias, T, d, cfg, scores, topk_idx, topk_w,
                     static_cast<char*>(ws) + ERR_BYTES, static_cast<uint32_t*>(ws),
                     ctr(ws, CTR_ROUTER), s);
}

size_t moe_dispatch_workspace_size(int T, int k, int E) {
    if (T < 0 || k < 1 || E < 1) return 0;
    return ERR_BYTES + moe_launch::dispatch_ws_bytes(T, k, E);
}

int moe_dispatch(const int32_t* topk_idx, const void* x, int dtype, int T, int d, int k, int E,
                 int32_t* counts, int32_t* offsets, int32_t* slot_to_row, int32_t* row_to_token,
                 void* x_perm, void* ws, size_t ws_bytes, void* stream) {
    if (k < 1 || k > 32 || E < 1 || E > 1024) return E > 1024 ? MOE_ERR_UNSUPPORTED : MOE_ERR_INVALID_ARG;
    int rc = check_dims(T, d, k);
    if (rc != MOE_OK) return rc;
    if (!dtype_ok(dtype) || !counts || !offsets) return MOE_ERR_INVALID_ARG;
    // with no slots the per-slot arrays are empty and may be NULL
    if (T > 0 && (!topk_idx || !slot_to_row || !row_to_token)) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (x_perm != nullptr) != (x != nullptr)) return MOE_ERR_INVALID_ARG;
    if (x && (!moe_host::aligned16(x) || !moe_host::aligned16(x_perm))) return MOE_ERR_INVALID_ARG;
    if (!ws || ws_bytes < moe_dispatch_workspace_size(T, k, E)) return MOE_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t* err = static_cast<uint32_t*>(ws);
    if (cudaMemsetAsync(err, 0, sizeof(uint32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
    if (T == 0) {
        if (cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s) != cudaSuccess ||
            cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s) != cudaSuccess)
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    return moe_launch::dispatch(topk_idx, x, dtype, T, d, k, E, counts, offsets, slot_to_row,
                                row_to_token, x_perm, static_cast<char*>(ws) + ERR_BYTES, err, s);
}

size_t moe_grouped_ffn_workspace_size(int rows, int d, int I, int dtype) {
    if (rows < 0 || d < 1 || I < 1 || !dtype_ok(dtype)) return 0;
    return ffn_ws(rows, d, I, dtype);
}

int moe_grouped_ffn(const void* x_perm, const int32_t* offsets, int E, int rows, int d, int I,
                    const void* w13, const void* w2, int dtype, float* y_perm, void* ws,
                    size_t ws_bytes, void* stream) {
    if (E < 1 || rows < 0 || d < 8 || d % 8 || I < 8 || I % 8 || !dtype_ok(dtype))
        return MOE_ERR_INVALID_ARG;
    if (E > 1024) return MOE_ERR_UNSUPPORTED;
    if (!x_perm || !offsets || !w13 || !w2 || !y_perm) return MOE_ERR_INVALID_ARG;
    if (!moe_host::aligned16(x_perm) || !moe_host::aligned16(w13) || !moe_host::aligned16(w2) ||
        !moe_host::aligned16(y_perm))
        return MOE_ERR_INVALID_ARG;
    if (!ws || ws_bytes < ffn_ws(rows, d, I, dtype)) return MOE_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t* err = static_cast<uint32_t*>(ws);
    if (cudaMemsetAsync(ws, 0, HDR_CLEAR, s) != cudaSuccess) return MOE_ERR_CUDA;
    return run_ffn(x_perm, offsets, E, rows, d, I, w13, w2, dtype, y_perm,
                   static_cast<char*>(ws) + ERR_BYTES, err, ctr(ws, CTR_FFN), s);
}

int moe_combine(const float* y_perm, const int32_t* slot_to_row, const float* topk_w,
                const float* shared, int T, int k, int d, float* out, void* stream) {
    if (T < 0 || k < 1 || d < 4 || d % 4) return MOE_ERR_INVALID_ARG;
    // the kernel indexes rows of y_perm with int: T*k must stay well inside it
    if (k > 32 || (long long)T * k > INT_MAX / 2) return MOE_ERR_UNSUPPORTED;
    if (!y_perm || !slot_to_row || !topk_w || !out) return MOE_ERR_INVALID_ARG;
    if (!moe_host::aligned16(y_perm) || !moe_host::aligned16(out) ||
        (shared && !moe_host::aligned16(shared)))
        return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    return moe_launch::combine(y_perm, T * k, slot_to_row, topk_w, shared, T, k, d, out, nullptr,
                               static_cast<cudaStream_t>(stream));
}

size_t moe_layer_workspace_size(const moe_layer_args* a) {
    if (check_layer_sizes(a) != MOE_OK) return 0;
    return carve_layer(a, nullptr).total;
}

int moe_layer(const moe_layer_args* a, float* out, void* ws, size_t ws_bytes, void* stream,
              void* stream2) {
    int rc = check_layer(a);
    if (rc != MOE_OK) return rc;
    if ((a->T > 0 && !out) || (out && !moe_host::aligned16(out))) return MOE_ERR_INVALID_ARG;
    if (!ws || !moe_host::aligned16(ws) || ws_bytes < carve_layer(a, nullptr).total)
        return MOE_ERR_WORKSPACE;
    const LayerWs w = carve_layer(a, ws);
    const int T = a->T, d = a->d, I = a->I, E = a->route.num_experts, k = a->route.top_k;
    cudaStream_t s0 = static_cast<cudaStream_t>(stream);
    cudaStream_t s1 = static_cast<cudaStream_t>(stream2);
    const bool two_streams = s1 && s1 != s0;
    const bool fused = a->flags & MOE_LAYER_FUSED_COMBINE;
    if ((a->flags & MOE_LAYER_SPLIT_DISPATCH) && (!two_streams || a->dtype != MOE_BF16 || fused))
        return MOE_ERR_UNSUPPORTED;
    // dispatch overlapped with the gate/up of the lower half of the experts
    const bool split = (a->flags & MOE_LAYER_SPLIT_DISPATCH) && E >= 2;
    if (cudaMemsetAsync(w.err, 0, HDR_CLEAR, s0) != cudaSuccess) return MOE_ERR_CUDA;
    if (T == 0) {
        // an empty batch: every expert gets zero rows
        if (a->offsets_out &&
            cudaMemsetAsync(a->offsets_out, 0, sizeof(int32_t) * (size_t)(E + 1), s0) != cudaSuccess)
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    const bool sh = w.ysh != nullptr;
    cudaEvent_t stage[MOE_LAYER_EVENTS] = {};
    if (a->stage_events)
        for (int i = 0; i < MOE_LAYER_EVENTS; ++i) stage[i] = static_cast<cudaEvent_t>(a->stage_events[i]);
    auto mark = [&](int i) {
        if (rc == MOE_OK && stage[i] && cudaEventRecord(stage[i], s0) != cudaSuccess) rc = MOE_ERR_CUDA;
    };
    mark(0);
    // Where the shared expert runs.  Given stream2, both of its GEMMs run
    // there while the routing and dispatch kernels leave the tensor cores
    // idle, and the combine waits for them.  With the fused combine (bf16,
    // I_sh == I) its down tiles ride in the routed down launch instead,
    // which adds them into the output.  Without stream2, bf16 with I_sh == I
    // puts both of its halves into the routed launches; other shapes run it
    // as launches of its own on the main stream.
    const bool fits = sh && a->dtype == MOE_BF16 && a->I_sh == I;
    const bool merged = fits && (!two_streams || (a->flags & MOE_LAYER_FUSED_COMBINE));
    moe_tc::SharedExpert shx{a->x, T, a->w13_sh, a->w2_sh, w.hsh, w.ysh,
                             /*in_gate_up=*/!two_streams, /*in_down=*/true};
    const bool overlap = sh && two_streams;
    // fork/join events: the caller's, else made (and destroyed) here.  [0]
    // the shared expert's start, [1] its end, [2] counts and offsets done,
    // [3] the upper half's permute done.
    cudaEvent_t ev[MOE_LAYER_SYNC_EVENTS] = {};
    const int n_ev = split ? 4 : overlap ? 2 : 0;
    const bool own_events = n_ev > 0 && !a->sync_events;
    for (int i = 0; i < n_ev; ++i) {
        if (own_events) {
            if (cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming) != cudaSuccess) {
                for (int j = 0; j < i; ++j) cudaEventDestroy(ev[j]);
                return MOE_ERR_CUDA;
            }
        } else {
            ev[i] = static_cast<cudaEvent_t>(a->sync_events[i]);
            if (!ev[i]) return MOE_ERR_INVALID_ARG;
        }
    }
    cudaEvent_t ev_start = ev[0], ev_shared = ev[1], ev_count = ev[2], ev_upper = ev[3];
    // the shared expert on stream2 starts when the router GEMM is launched
    // (bf16): its CTAs take the SMs that the router's single wave of tiles
    // leaves idle, then continue beside the top-k and dispatch kernels.
    // Measured on DeepSeek-V3 prefill: 4.129 ms vs 4.157 ms when started
    // after the router GEMM, which in turn beat starting before the router
    // (its CTAs then delayed the router); both GEMMs there rather than its
    // down tiles in the routed down launch: 4.057 vs 4.110 ms.
    if (rc == MOE_OK)
        rc = run_route(a->x, a->dtype, a->w_router, a->bias, T, d, &a->route, w.scores, w.idx, w.w,
                       w.wsplit, w.err, ctr(w.err, CTR_ROUTER), s0, overlap ? ev_start : nullptr,
                       a->w_router_split, a->flags & MOE_LAYER_SHARED_AFTER_ROUTER);
    mark(1);
    mark(2);
    // fused combine: the output is accumulated into, so it starts at zero;
    // on stream2 (before the shared expert, which the down launch waits for)
    // when given, so that the main stream does not pay for it
    const bool zero_on_s1 = fused && merged && overlap;
    const bool packed = a->flags & MOE_LAYER_PACKED_WEIGHTS;
    const int Ea = E / 2;  // split: experts [0, Ea) on `stream` first
    if (split) {
        // counts and offsets, then the upper half's permute (and the shared
        // expert after it) on stream2 while the lower half's permute and
        // gate/up run here
        if (rc == MOE_OK)
            rc = moe_launch::dispatch(w.idx, a->x, a->dtype, T, d, k, E, w.counts, w.offsets,
                                      w.s2r, w.r2t, w.xp, w.disp, w.err, s0, nullptr, nullptr,
                                      /*parts=*/1);
        if (rc == MOE_OK && cudaEventRecord(ev_count, s0) != cudaSuccess) rc = MOE_ERR_CUDA;
        if (rc == MOE_OK && cudaStreamWaitEvent(s1, ev_count, 0) != cudaSuccess) rc = MOE_ERR_CUDA;
        if (rc == MOE_OK)
            rc = moe_launch::dispatch(w.idx, a->x, a->dtype, T, d, k, E, w.counts, w.offsets,
                                      w.s2r, w.r2t, w.xp, w.disp, w.err, s1, nullptr, nullptr,
                                      /*parts=*/2, Ea, E);
        if (rc == MOE_OK && cudaEventRecord(ev_upper, s1) != cudaSuccess) rc = MOE_ERR_CUDA;
        if (rc == MOE_OK && overlap)
            rc = run_ffn(a->x, nullptr, 1, T, d, a->I_sh, a->w13_sh, a->w2_sh, a->dtype, w.ysh,
                         w.hsh, w.err, ctr(w.err, CTR_SHARED), s1, nullptr, packed);
        if (rc == MOE_OK && overlap && cudaEventRecord(ev_shared, s1) != cudaSuccess)
            rc = MOE_ERR_CUDA;
        if (rc == MOE_OK)
            rc = moe_launch::dispatch(w.idx, a->x, a->dtype, T, d, k, E, w.counts, w.offsets,
                                      w.s2r, w.r2t, w.xp, w.disp, w.err, s0, nullptr, nullptr,
                                      /*parts=*/2, 0, Ea);
        mark(3);
        // gate/up of each half (experts' weights are contiguous per expert in
        // both layouts), the tile chosen as for all E experts; then the down
        // projection over all of them
        const size_t w13_e = (size_t)2 * I * d * 2, w2_e = (size_t)d * I * 2;
        const char* w13c = static_cast<const char*>(a->w13);
        const char* w2c = static_cast<const char*>(a->w2);
        if (rc == MOE_OK)
            rc = moe_tc::grouped_ffn_bf16(w.xp, w.offsets, Ea, T * k, d, I, a->w13, a->w2, w.yp,
                                          w.h, w.err, ctr(w.err, CTR_FFN), s0, nullptr, nullptr,
                                          nullptr, /*parts=*/1, nullptr, packed, E);
        if (rc == MOE_OK && cudaStreamWaitEvent(s0, ev_upper, 0) != cudaSuccess) rc = MOE_ERR_CUDA;
        if (rc == MOE_OK)
            rc = moe_tc::grouped_ffn_bf16(w.xp, w.offsets + Ea, E - Ea, T * k, d, I,
                                          w13c + (size_t)Ea * w13_e, w2c + (size_t)Ea * w2_e,
                                          w.yp, w.h, w.err, ctr(w.err, CTR_FFN_HI), s0, nullptr,
                                          nullptr, nullptr, /*parts=*/1, nullptr, packed, E);
        mark(4);
        if (rc == MOE_OK)
            rc = moe_tc::grouped_ffn_bf16(w.xp, w.offsets, E, T * k, d, I, a->w13, a->w2, w.yp,
                                          w.h, w.err, ctr(w.err, CTR_FFN), s0, nullptr, nullptr,
                                          nullptr, /*parts=*/2, nullptr, packed);
        mark(5);
        if (rc == MOE_OK && overlap && cudaStreamWaitEvent(s0, ev_shared, 0) != cudaSuccess)
            rc = MOE_ERR_CUDA;
        if (rc == MOE_OK)
            rc = moe_launch::combine(w.yp, T * k, w.s2r, w.w, w.ysh, T, k, d, out, w.err, s0);
        mark(6);
        if (own_events)
            for (int i = 0; i < n_ev; ++i) cudaEventDestroy(ev[i]);
        return rc;
    }
    if (overlap) {
        if (rc == MOE_OK && cudaStreamWaitEvent(s1, ev_start, 0) != cudaSuccess) rc = MOE_ERR_CUDA;
        if (rc == MOE_OK && zero_on_s1 &&
            cudaMemsetAsync(out, 0, sizeof(float) * (size_t)T * d, s1) != cudaSuccess)
            rc = MOE_ERR_CUDA;
        if (rc == MOE_OK) {
            if (merged)  // gate/up only; the down tiles ride in the routed launch
                rc = moe_tc::grouped_ffn_bf16(a->x, nullptr, 1, T, d, I, a->w13_sh, a->w2_sh, w.ysh,
                                              w.hsh, w.err, ctr(w.err, CTR_SHARED), s1, nullptr,
                                              nullptr, nullptr, /*parts=*/1, nullptr, packed);
            else
                rc = run_ffn(a->x, nullptr, 1, T, d, a->I_sh, a->w13_sh, a->w2_sh, a->dtype, w.ysh,
                             w.hsh, w.err, ctr(w.err, CTR_SHARED), s1, nullptr, packed);
        }
        if (rc == MOE_OK && cudaEventRecord(ev_shared, s1) != cudaSuccess) rc = MOE_ERR_CUDA;
    }
    if (rc == MOE_OK)
        rc = moe_launch::dispatch(w.idx, a->x, a->dtype, T, d, k, E, w.counts, w.offsets, w.s2r,
                                  w.r2t, w.xp, w.disp, w.err, s0, fused ? w.w : nullptr, w.w_row);
    mark(3);
    if (rc == MOE_OK && fused && !zero_on_s1 &&
        cudaMemsetAsync(out, 0, sizeof(float) * (size_t)T * d, s0) != cudaSuccess)
        rc = MOE_ERR_CUDA;
    const moe_tc::FusedCombine fc{out, w.r2t, w.w_row};
    if (rc == MOE_OK) {
        if (merged || fused)
            rc = moe_tc::grouped_ffn_bf16(w.xp, w.offsets, E, T * k, d, I, a->w13, a->w2, w.yp, w.h,
                                          w.err, ctr(w.err, CTR_FFN), s0, stage[4],
                                          merged ? &shx : nullptr, fused ? &fc : nullptr, 3,
                                          merged && overlap ? ev_shared : nullptr, packed);
        else
            rc = run_ffn(w.xp, w.offsets, E, T * k, d, I, a->w13, a->w2, a->dtype, w.yp, w.h,
                         w.err, ctr(w.err, CTR_FFN), s0, stage[4], packed);
    }
    mark(5);
    if (rc == MOE_OK && sh && !merged && !overlap)
        rc = run_ffn(a->x, nullptr, 1, T, d, a->I_sh, a->w13_sh, a->w2_sh, a->dtype, w.ysh, w.hsh,
                     w.err, ctr(w.err, CTR_SHARED), s0, nullptr, packed);
    if (rc == MOE_OK && overlap && !merged && cudaStreamWaitEvent(s0, ev_shared, 0) != cudaSuccess)
        rc = MOE_ERR_CUDA;
    if (rc == MOE_OK && !fused)
        rc = moe_launch::combine(w.yp, T * k, w.s2r, w.w, w.ysh, T, k, d, out, w.err, s0);
    mark(6);
    if (own_events)
        for (int i = 0; i < n_ev; ++i) cudaEventDestroy(ev[i]);
    return rc;
}

int moe_split_router_weight(const float* w_router, int E, int d, void* out, void* stream) {
    if (E < 1 || d < 8 || d % 8 != 0 || !w_router || !out) return MOE_ERR_INVALID_ARG;
    if (!moe_host::aligned16(w_router) || !moe_host::aligned16(out)) return MOE_ERR_INVALID_ARG;
    return moe_tc::split_router_weight(w_router, E, d, out, static_cast<cudaStream_t>(stream));
}

int moe_pack_expert_weights(const void* w13, const void* w2, int E, int d, int I,
                            void* w13_packed, void* w2_packed, void* stream) {
    if (E < 1 || d < 256 || d % 256 != 0 || I < 128 || I % 128 != 0) return MOE_ERR_INVALID_ARG;
    if (!w13 != !w13_packed || !w2 != !w2_packed) return MOE_ERR_INVALID_ARG;
    for (const void* p : {w13, w2, static_cast<const void*>(w13_packed),
                          static_cast<const void*>(w2_packed)})
        if (p && !moe_host::aligned16(p)) return MOE_ERR_INVALID_ARG;
    if ((long long)E * 2 * I * d > (1ll << 40)) return MOE_ERR_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int rc = MOE_OK;
    if (w13) rc = moe_tc::pack_weights(w13, E, 2 * I, d, /*pairs=*/false, w13_packed, s);
    if (rc == MOE_OK && w2) rc = moe_tc::pack_weights(w2, E, d, I, /*pairs=*/true, w2_packed, s);
    return rc;
}

int moe_selftest_bounded_wait(int which, uint32_t limit_us, void* ws, size_t ws_bytes,
                              void* stream) {
    if (which < 0 || which > 2 || limit_us < 1 || limit_us > 1000000) return MOE_ERR_INVALID_ARG;
    if (!ws || !moe_host::aligned16(ws) || ws_bytes < ERR_BYTES + 256) return MOE_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, ERR_BYTES + 256, s) != cudaSuccess) return MOE_ERR_CUDA;
    uint32_t* err = static_cast<uint32_t*>(ws);
    const uint64_t ns = 1000ull * limit_us;
    if (which == 0) return moe_tc::mbar_probe(ns, err, s);
    if (which == 2) return moe_tc::cluster_probe(ns, err, s);
    return moe_launch::lookback_probe(static_cast<char*>(ws) + ERR_BYTES, ns, err, s);
}

int moe_check_error(void* ws, void* stream, uint32_t* detail) {
    if (!ws) return MOE_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MOE_ERR_CUDA;
    uint32_t v = 0;
    if (cudaMemcpy(&v, ws, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    if (v && cudaMemset(ws, 0, sizeof v) != cudaSuccess) return MOE_ERR_CUDA;
    if (detail) *detail = v;
    if (v & moe::ERR_TIMEOUT_MASK) return MOE_ERR_TIMEOUT;
    if (v) return MOE_ERR_DEVICE_INPUT;
    return MOE_OK;
}

}  // extern "C"
