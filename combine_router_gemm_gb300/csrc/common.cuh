// common.cuh -- shared device helpers of the MoE CUDA library (sm_103a).
//
// Error word: a uint32 in device memory.  Kernels OR in a code when a bounded
// wait runs out or a device-side input is inconsistent, then stop early.
// Consumers of earlier stages read it on entry and skip their work if set.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// error-word bits
constexpr uint32_t ERR_TIMEOUT_SCAN = 1u << 0;
constexpr uint32_t ERR_TIMEOUT_PIPE = 1u << 1;
constexpr uint32_t ERR_BAD_INDEX = 1u << 8;
constexpr uint32_t ERR_BAD_OFFSETS = 1u << 9;
constexpr uint32_t ERR_TIMEOUT_MASK = 0xffu;

// a bounded wait gives up after this many nanoseconds of %globaltimer
constexpr uint64_t WAIT_LIMIT_NS = 1000ull * 1000ull * 1000ull;

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void raise_error(uint32_t* err, uint32_t code) {
    if (err) atomicOr(err, code);
}

__device__ __forceinline__ uint32_t read_error(const uint32_t* err) {
    return err ? *(volatile const uint32_t*)err : 0u;
}

__device__ __forceinline__ float bf16_to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

inline int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

}  // namespace moe

// ---- host-side helpers shared by the entry points (defined in api.cu) ------
namespace moe_host {
bool aligned16(const void* p);
int launch_status();  // MOE_OK or MOE_ERR_CUDA after a launch
int num_sms();
}  // namespace moe_host

// ---- tcgen05 kernels (grouped_gemm_tc.cu) ----------------------------------
namespace moe_tc {
// A second, dense problem run inside the same grouped-GEMM launches: the
// shared expert over all T tokens (same I as the routed experts).
struct SharedExpert {
    const void* x;    // [T,d] bf16
    int T;
    const void* w13;  // [2I,d]
    const void* w2;   // [d,I]
    void* h;          // [T,I] bf16 scratch
    float* y;         // [T,d] fp32 out
    bool in_gate_up;  // its gate/up tiles ride in the gate/up launch
    bool in_down;     // its down tiles ride in the down launch (h ready)
};
// work: two zeroed counters (gate/up launch, down launch) for the dynamic
// unit schedule
// The down projection's results added straight into the layer output:
// out[row_token[r]] += w_row[r] * y[r] (shared expert rows: weight 1).
struct FusedCombine {
    float* out;                // [T,d] fp32, zeroed before the launch
    const int32_t* row_token;  // [rows]
    const float* w_row;        // [rows]
};
// parts: 1 = gate/up launch, 2 = down launch, 3 = both.  before_down: an
// event the down launch waits for (e.g. the shared expert's gate/up on
// another stream).  heur_E: the expert count whose rows the launch's tile
// choice averages over (0: E); a launch over a range of a layer's experts
// passes the layer's, so that it takes the tile the whole layer would.
int grouped_ffn_bf16(const void* x_perm, const int32_t* offsets, int E, int rows, int d, int I,
                     const void* w13, const void* w2, float* y, void* h, uint32_t* err,
                     unsigned* work, cudaStream_t s, cudaEvent_t between = nullptr,
                     const SharedExpert* sh = nullptr, const FusedCombine* fc = nullptr,
                     int parts = 3, cudaEvent_t before_down = nullptr, bool packed = false,
                     int heur_E = 0);
// Expert weights [E, rows, K] bf16 into the tile-major layout (pairs: the
// down projection's), on stream s.  rows % 128 == 0 (pairs: % 256), K % 64 == 0.
int pack_weights(const void* w, int E, int rows, int K, bool pairs, void* out, cudaStream_t s);
size_t router_ws_bytes(int T, int E, int d);
int mbar_probe(uint64_t limit_ns, uint32_t* err, cudaStream_t s);
int cluster_probe(uint64_t limit_ns, uint32_t* err, cudaStream_t s);
// after_split: recorded once the weight split is done, before the GEMM.
// presplit: the weight already split ([3,E,d] bf16), or NULL to split it
// into the workspace first.
int router_bf16(const void* x, const float* w_router, int T, int d, int E, void* ws,
                uint32_t* err, unsigned* work, float** partial, int* ksplit, cudaStream_t s,
                cudaEvent_t after_split = nullptr, const void* presplit = nullptr);
// w_router [E,d] fp32 -> out [3,E,d] bf16 (hi, mid, lo), on stream s
int split_router_weight(const float* w_router, int E, int d, void* out, cudaStream_t s);
}  // namespace moe_tc

// ---- internal launchers (one per kernel family), used by api.cu -----------
namespace moe_launch {
int router_gemm(const void* x, int dtype, const float* w_router, int T, int d, int E, int score_fn,
                float* scores, cudaStream_t s);
// Top-k and gates.  With partial != NULL the scores are first finalised:
// logits = sum of the ksplit partial tensors (in order), scores = logits or
// sigmoid(logits), written to scores (which is then an output).
int topk(const float* scores, const float* bias, int T, const moe_route_cfg* cfg, int32_t* idx,
         float* w, cudaStream_t s, const float* partial = nullptr, int ksplit = 0,
         float* scores_out = nullptr);
size_t dispatch_ws_bytes(int T, int k, int E);
int lookback_probe(void* flags_zeroed, uint64_t limit_ns, uint32_t* err, cudaStream_t s);
// w_slot/w_row (both or neither): also write each permuted row's gate weight.
// parts: 1 = count and scan only, 2 = permute only (after a count launch of
// the same call, on the same workspace), 3 = both.  The permute moves only
// the slots routed to experts [e_lo, e_hi) (e_hi < 0: all).
int dispatch(const int32_t* idx, const void* x, int dtype, int T, int d, int k, int E, int32_t* counts,
             int32_t* offsets, int32_t* slot_to_row, int32_t* row_to_token, void* x_perm, void* ws,
             uint32_t* err, cudaStream_t s, const float* w_slot = nullptr, float* w_row = nullptr,
             int parts = 3, int e_lo = 0, int e_hi = -1);
size_t ffn_ws_bytes(int rows, int I, int dtype);
int grouped_ffn(const void* x_perm, const int32_t* offsets, int E, int rows, int d, int I,
                const void* w13, const void* w2, int dtype, float* y, void* h_ws, uint32_t* err,
                cudaStream_t s);
// out[t] for tokens t of the arrays passed in (slot_to_row, w, shared, out
// may point into a token range of the layer's); rows = rows of y, which
// slot_to_row indexes
int combine(const float* y, int rows, const int32_t* slot_to_row, const float* w,
            const float* shared, int T, int k, int d, float* out, const uint32_t* err,
            cudaStream_t s);
}  // namespace moe_launch
