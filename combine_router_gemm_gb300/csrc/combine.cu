// combine.cu -- gate-weighted combine of the expert outputs.
//
// The pages ("CUCo: An Agentic Framework for Compute and Communication
// Co-design", Table 4 row "MoE Dispatch/Combine") bring each token's expert
// results back to it; on one GPU that is a weighted gather:
//   out[t,:] = sum_{j<k} w[t,j] * y[slot_to_row[t*k+j], :]  (+ shared[t,:]),
// summed in slot order in fp32.  One block per token; each thread owns a few
// 16-byte column chunks and issues the k row loads of a chunk back to back.
#include "common.cuh"

namespace {

constexpr int CB_THREADS = 256;
constexpr int CB_MAXK = 32;

// KC: k known at compile time (its k row loads of a chunk are then all issued
// before the first is used), or 0 for any k.
template <int KC>
__global__ void __launch_bounds__(CB_THREADS) combine_kernel(
    const float4* __restrict__ y, const int32_t* __restrict__ slot_to_row,
    const float* __restrict__ w, const float4* __restrict__ shared, int rows, int k_rt, int d4,
    float4* __restrict__ out, const uint32_t* err) {
    const int k = KC ? KC : k_rt;
    __shared__ int s_row[CB_MAXK];
    __shared__ float s_w[CB_MAXK];
    __shared__ int s_skip, s_bad;
    const int t = blockIdx.x;  // token, relative to the arrays passed in
    if (threadIdx.x == 0) {
        s_skip = moe::read_error(err) != 0;
        s_bad = 0;
    }
    __syncthreads();
    if (threadIdx.x < k) {
        const int r = slot_to_row[(size_t)t * k + threadIdx.x];
        const bool ok = r >= 0 && r < rows;
        s_row[threadIdx.x] = ok ? r : 0;
        s_w[threadIdx.x] = w[(size_t)t * k + threadIdx.x];
        if (!ok) s_bad = 1;  // an index outside y: the output row becomes NaN
    }
    __syncthreads();
    if (s_skip) return;
    const float4 nan4 = make_float4(__int_as_float(0x7fc00000), 0.f, 0.f, 0.f);
    for (int v = threadIdx.x; v < d4; v += CB_THREADS) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (KC) {
            // all k row loads of this chunk in flight before the first is used
            float4 yv[KC ? KC : 1];
#pragma unroll
            for (int j = 0; j < KC; ++j) yv[j] = __ldcs(y + (size_t)s_row[j] * d4 + v);
#pragma unroll
            for (int j = 0; j < KC; ++j) {
                const float wj = s_w[j];
                acc.x = fmaf(wj, yv[j].x, acc.x);
                acc.y = fmaf(wj, yv[j].y, acc.y);
                acc.z = fmaf(wj, yv[j].z, acc.z);
                acc.w = fmaf(wj, yv[j].w, acc.w);
            }
        } else {
            for (int j = 0; j < k; ++j) {
                const float wj = s_w[j];
                const float4 yv = __ldcs(y + (size_t)s_row[j] * d4 + v);
                acc.x = fmaf(wj, yv.x, acc.x);
                acc.y = fmaf(wj, yv.y, acc.y);
                acc.z = fmaf(wj, yv.z, acc.z);
                acc.w = fmaf(wj, yv.w, acc.w);
            }
        }
        if (shared) {
            const float4 sv = __ldcs(shared + (size_t)t * d4 + v);
            acc.x += sv.x;
            acc.y += sv.y;
            acc.z += sv.z;
            acc.w += sv.w;
        }
        out[(size_t)t * d4 + v] = s_bad ? nan4 : acc;
    }
}

}  // namespace

namespace moe_launch {

int combine(const float* y, int rows, const int32_t* slot_to_row, const float* w,
            const float* shared, int T, int k, int d, float* out, const uint32_t* err,
            cudaStream_t s) {
    if (k > CB_MAXK) return MOE_ERR_UNSUPPORTED;
    const float4* y4 = reinterpret_cast<const float4*>(y);
    const float4* sh4 = reinterpret_cast<const float4*>(shared);
    float4* o4 = reinterpret_cast<float4*>(out);
    if (k == 8)
        combine_kernel<8><<<T, CB_THREADS, 0, s>>>(y4, slot_to_row, w, sh4, rows, k, d / 4, o4, err);
    else if (k == 2)
        combine_kernel<2><<<T, CB_THREADS, 0, s>>>(y4, slot_to_row, w, sh4, rows, k, d / 4, o4, err);
    else
        combine_kernel<0><<<T, CB_THREADS, 0, s>>>(y4, slot_to_row, w, sh4, rows, k, d / 4, o4, err);
    return moe_host::launch_status();
}

}  // namespace moe_launch
