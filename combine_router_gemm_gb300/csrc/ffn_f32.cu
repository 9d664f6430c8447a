// ffn_f32.cu -- per-expert SwiGLU FFN in fp32 on the CUDA cores.
//
// The fp32 workload (64 tokens, d=128) needs true fp32 arithmetic, which the
// bf16 tensor-core path does not give; this is the same grouped computation
//   H[r, n] = silu(<x_r, W1_e[n]>) * <x_r, W3_e[n]>,   Y[r, n] = <H_r, W2_e[n]>
// over segments [offsets[e], offsets[e+1]) with fp32 accumulation.
// Block tile: 32 rows x 32 outputs, K chunk 32, 256 threads x 4 outputs.
// Grid x covers an upper bound on the number of row tiles (rows/32 + E);
// each block maps its index to (expert, row tile) from the offsets.
#include "common.cuh"

namespace {

constexpr int FT = 32;

template <bool SWIGLU>
__global__ void __launch_bounds__(256) ffn_f32_kernel(const float* __restrict__ A,
                                                      const int32_t* __restrict__ offsets, int E,
                                                      int rows, int K,
                                                      const float* __restrict__ B,
                                                      size_t b_expert_stride, int N_out,
                                                      int up_off, float* __restrict__ Cout,
                                                      uint32_t* err) {
    __shared__ float As[FT][FT + 1];
    __shared__ float Bg[FT][FT + 1];
    __shared__ float Bu[FT][FT + 1];
    __shared__ int s_e, s_m0, s_m1;
    const int tid = threadIdx.x;
    if (tid == 0) {
        // walk experts to find which (expert, row tile) this block owns
        int tile = blockIdx.x, e = -1, m0 = 0, m1 = 0;
        if (!moe::read_error(err)) {
            for (int i = 0; i < E; ++i) {
                const int a = offsets ? offsets[i] : 0;
                const int b = offsets ? offsets[i + 1] : rows;
                if (a < 0 || b < a || b > rows) {
                    // inconsistent offsets: report them; this block computes nothing
                    moe::raise_error(err, moe::ERR_BAD_OFFSETS);
                    break;
                }
                const int nt = (b - a + FT - 1) / FT;
                if (tile < nt) {
                    e = i;
                    m0 = a + tile * FT;
                    m1 = min(b, m0 + FT);
                    break;
                }
                tile -= nt;
            }
        }
        s_e = e;
        s_m0 = m0;
        s_m1 = m1;
    }
    __syncthreads();
    const int e = s_e;
    if (e < 0) return;
    const int m0 = s_m0, m1 = s_m1;
    const int n0 = blockIdx.y * FT;
    const float* Be = B + (size_t)e * b_expert_stride;
    const int lr = tid >> 3, lk = (tid & 7) * 4;  // loader: row, 4 consecutive k
    const int orow = tid >> 3, ocol = (tid & 7) * 4;  // outputs: 1 row x 4 columns
    float ag[4] = {}, au[4] = {};
    for (int k0 = 0; k0 < K; k0 += FT) {
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int kk = k0 + lk + i;
            const int r = m0 + lr;
            As[lr][lk + i] = (r < m1 && kk < K) ? A[(size_t)r * K + kk] : 0.f;
            const int n = n0 + lr;
            Bg[lr][lk + i] = (n < N_out && kk < K) ? Be[(size_t)n * K + kk] : 0.f;
            if (SWIGLU) Bu[lr][lk + i] = (n < N_out && kk < K) ? Be[(size_t)(up_off + n) * K + kk] : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int kq = 0; kq < FT; ++kq) {
            const float a = As[orow][kq];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                ag[j] = fmaf(a, Bg[ocol + j][kq], ag[j]);
                if (SWIGLU) au[j] = fmaf(a, Bu[ocol + j][kq], au[j]);
            }
        }
    }
    const int r = m0 + orow;
    if (r >= m1) return;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int n = n0 + ocol + j;
        if (n >= N_out) continue;
        float v = ag[j];
        if (SWIGLU) v = v / (1.0f + expf(-v)) * au[j];
        Cout[(size_t)r * N_out + n] = v;
    }
}

}  // namespace

namespace moe_f32 {

int grouped_ffn_f32(const float* x_perm, const int32_t* offsets, int E, int rows, int d, int I,
                    const float* w13, const float* w2, float* y, float* h, uint32_t* err,
                    cudaStream_t s) {
    const int mtiles = moe::ceil_div(rows, FT) + E;
    dim3 g1(mtiles, moe::ceil_div(I, FT));
    ffn_f32_kernel<true><<<g1, 256, 0, s>>>(x_perm, offsets, E, rows, d, w13,
                                             (size_t)2 * I * d, I, I, h, err);
    int rc = moe_host::launch_status();
    if (rc != MOE_OK) return rc;
    dim3 g2(mtiles, moe::ceil_div(d, FT));
    ffn_f32_kernel<false><<<g2, 256, 0, s>>>(h, offsets, E, rows, I, w2, (size_t)d * I, d, 0, y,
                                              err);
    return moe_host::launch_status();
}

}  // namespace moe_f32
