// route.cu -- router scoring (GEMM) and top-k selection with gate weights.
//
// The pages ("CUCo: An Agentic Framework for Compute and Communication
// Co-design", abstract and Table 4) name a DeepSeek-V3 MoE layer; its router is
// read here as: logits = x W_r^T in fp32; Mixtral-style softmax gates over the
// top-k logits, or DeepSeek-V3 sigmoid scores with a per-expert selection bias,
// group-limited choice (best topk_group of n_group groups by the sum of each
// group's two largest biased scores) and gates normalised over the k chosen
// scores then scaled.
#include <float.h>

#include "common.cuh"

namespace {

// ---------------------------------------------------------------- router GEMM
//
// logits[t,e] = sum_i x[t,i] * W[e,i] on the CUDA cores in fp32, for fp32
// activations (bf16 activations use the tensor-core router in
// grouped_gemm_tc.cu).  Block tile 64 tokens x 64 experts, K chunk 32; 256
// threads, each owning a 4x4 block of outputs.

constexpr int RT_T = 64, RT_E = 64, RT_K = 32;

template <typename XT>
__device__ __forceinline__ void load_x8(const XT* p, float (&v)[8]);
template <>
__device__ __forceinline__ void load_x8<float>(const float* p, float (&v)[8]) {
    float4 a = *reinterpret_cast<const float4*>(p);
    float4 b = *reinterpret_cast<const float4*>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

template <typename XT>
__global__ void __launch_bounds__(256) router_gemm_kernel(const XT* __restrict__ x,
                                                          const float* __restrict__ W, int T, int d,
                                                          int E, int sigmoid,
                                                          float* __restrict__ scores) {
    __shared__ float xs[RT_K][RT_T + 4];
    __shared__ float ws[RT_K][RT_E + 4];
    const int tid = threadIdx.x;
    const int t0 = blockIdx.y * RT_T, e0 = blockIdx.x * RT_E;
    // loader mapping: row r = tid / 4 (0..63), 8 consecutive k at (tid % 4) * 8
    const int lr = tid >> 2, lk = (tid & 3) * 8;
    const int tx = tid & 15, ty = tid >> 4;  // outputs: experts tx*4.., tokens ty*4..
    float acc[4][4] = {};
    for (int k0 = 0; k0 < d; k0 += RT_K) {
        float xv[8], wv[8];
        const int kk = k0 + lk;
        if (t0 + lr < T && kk < d) {
            load_x8<XT>(x + (size_t)(t0 + lr) * d + kk, xv);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) xv[i] = 0.f;
        }
        if (e0 + lr < E && kk < d) {
            load_x8<float>(W + (size_t)(e0 + lr) * d + kk, wv);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) wv[i] = 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            xs[lk + i][lr] = xv[i];
            ws[lk + i][lr] = wv[i];
        }
        __syncthreads();
#pragma unroll
        for (int kq = 0; kq < RT_K; ++kq) {
            float4 a = *reinterpret_cast<const float4*>(&xs[kq][ty * 4]);
            float4 b = *reinterpret_cast<const float4*>(&ws[kq][tx * 4]);
            const float av[4] = {a.x, a.y, a.z, a.w};
            const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = t0 + ty * 4 + i;
        if (t >= T) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = e0 + tx * 4 + j;
            if (e >= E) continue;
            float v = acc[i][j];
            if (sigmoid) v = 1.0f / (1.0f + expf(-v));
            scores[(size_t)t * E + e] = v;
        }
    }
}

// ---------------------------------------------------------------- top-k
//
// One warp per token.  Lane l holds experts e = i*32 + l (i < EPL), so loads
// are coalesced.  Every choice is a warp-wide argmax over (key, index) that
// prefers the larger key and, on equal keys, the lower index.

struct Cand {
    float v;
    int e;  // -1: none
};

constexpr int FAST_GROUPS = 8;  // group counts up to this take the all-at-once path

__device__ __forceinline__ Cand better(Cand a, Cand b) {
    if (b.e < 0) return a;
    if (a.e < 0) return b;
    if (b.v > a.v || (b.v == a.v && b.e < a.e)) return b;
    return a;
}

__device__ __forceinline__ Cand warp_best(Cand c) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        Cand o;
        o.v = __shfl_xor_sync(0xffffffffu, c.v, off);
        o.e = __shfl_xor_sync(0xffffffffu, c.e, off);
        c = better(c, o);
    }
    return c;
}

template <int EPL>
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ scores,
                                                   const float* __restrict__ bias, int T, int E,
                                                   int k, int n_group, int topk_group, int sigmoid,
                                                   float scale, int32_t* __restrict__ idx_out,
                                                   float* __restrict__ w_out,
                                                   const float* __restrict__ partial, int ksplit,
                                                   float* __restrict__ scores_out) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    float sc[EPL], key[EPL];
    bool ok[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const int e = i * 32 + lane;
        ok[i] = e < E;
        if (partial) {
            // scores from the router's K-part partial logits, summed in order
            float v = 0.f;
            if (ok[i]) {
                v = partial[(size_t)t * E + e];
                for (int ks = 1; ks < ksplit; ++ks) v += partial[((size_t)ks * T + t) * E + e];
                if (sigmoid) v = 1.0f / (1.0f + expf(-v));
                scores_out[(size_t)t * E + e] = v;
            }
            sc[i] = v;
        } else {
            sc[i] = ok[i] ? scores[(size_t)t * E + e] : 0.f;
        }
        key[i] = ok[i] ? (bias ? sc[i] + bias[e] : sc[i]) : 0.f;
    }

    if (n_group > 1) {
        const int gs = E / n_group;
        int gid[EPL];  // group of each held expert
#pragma unroll
        for (int i = 0; i < EPL; ++i) gid[i] = (i * 32 + lane) / gs;
        unsigned keep = 0;
        if (n_group <= FAST_GROUPS) {
            // All groups at once: each lane keeps the two largest of its own
            // keys per group (-inf = none), then a butterfly merges the pairs
            // across the warp.  Top-2 of a multiset by values only: the merge
            // (max(a1,b1), max(min(a1,b1), max(a2,b2))) is exact, and every
            // group has at least two members, so no -inf survives.
            float g1[FAST_GROUPS], g2[FAST_GROUPS];
#pragma unroll
            for (int g = 0; g < FAST_GROUPS; ++g) g1[g] = g2[g] = -INFINITY;
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
#pragma unroll
                for (int g = 0; g < FAST_GROUPS; ++g) {
                    if (ok[i] && gid[i] == g) {
                        const float v = key[i];
                        g2[g] = fmaxf(g2[g], fminf(g1[g], v));
                        g1[g] = fmaxf(g1[g], v);
                    }
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
                for (int g = 0; g < FAST_GROUPS; ++g) {
                    const float o1 = __shfl_xor_sync(0xffffffffu, g1[g], off);
                    const float o2 = __shfl_xor_sync(0xffffffffu, g2[g], off);
                    g2[g] = fmaxf(fminf(g1[g], o1), fmaxf(g2[g], o2));
                    g1[g] = fmaxf(g1[g], o1);
                }
            }
            // every lane now holds every group score: pick the best groups,
            // ties to the lower group, without further communication
            float gsc[FAST_GROUPS];
#pragma unroll
            for (int g = 0; g < FAST_GROUPS; ++g) gsc[g] = g1[g] + g2[g];
            for (int r = 0; r < topk_group; ++r) {
                int best = -1;
                float bv = 0.f;
#pragma unroll
                for (int g = 0; g < FAST_GROUPS; ++g) {
                    if (g < n_group && !((keep >> g) & 1u) && (best < 0 || gsc[g] > bv)) {
                        best = g;
                        bv = gsc[g];
                    }
                }
                keep |= 1u << best;
            }
        } else {
            float my_gscore = 0.f;
            for (int g = 0; g < n_group; ++g) {
                // two largest keys of group g (values only; their sum is symmetric)
                float v1 = -INFINITY, v2 = -INFINITY;
#pragma unroll
                for (int i = 0; i < EPL; ++i) {
                    if (ok[i] && gid[i] == g) {
                        v2 = fmaxf(v2, fminf(v1, key[i]));
                        v1 = fmaxf(v1, key[i]);
                    }
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    const float o1 = __shfl_xor_sync(0xffffffffu, v1, off);
                    const float o2 = __shfl_xor_sync(0xffffffffu, v2, off);
                    v2 = fmaxf(fminf(v1, o1), fmaxf(v2, o2));
                    v1 = fmaxf(v1, o1);
                }
                if (lane == g) my_gscore = v1 + v2;
            }
            bool gtaken = false;
            for (int r = 0; r < topk_group; ++r) {
                Cand c;
                c.v = my_gscore;
                c.e = (lane < n_group && !gtaken) ? lane : -1;
                c = warp_best(c);
                if (lane == c.e) gtaken = true;
                keep |= 1u << c.e;
            }
        }
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if (ok[i] && !((keep >> gid[i]) & 1u)) ok[i] = false;
    }

    // softmax normaliser over all E logits
    float m = -FLT_MAX, z = 0.f;
    if (!sigmoid) {
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if (i * 32 + lane < E) m = fmaxf(m, sc[i]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if (i * 32 + lane < E) z += expf(sc[i] - m);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
    }

    int my_e = 0;
    float my_p = 0.f, psum = 0.f;
    for (int j = 0; j < k; ++j) {
        Cand c;
        c.e = -1;
        c.v = 0.f;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {  // ascending e: strict > keeps the lowest index
            if (ok[i] && (c.e < 0 || key[i] > c.v)) {
                c.v = key[i];
                c.e = i * 32 + lane;
            }
        }
        c = warp_best(c);
        float s_sel = 0.f;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            if (i * 32 + lane == c.e) {
                ok[i] = false;
                s_sel = sc[i];
            }
        }
        s_sel = __shfl_sync(0xffffffffu, s_sel, c.e & 31);
        const float p = sigmoid ? s_sel : expf(s_sel - m) / z;
        psum += p;  // slot order
        if (lane == j) {
            my_e = c.e;
            my_p = p;
        }
    }
    if (lane < k) {
        idx_out[(size_t)t * k + lane] = my_e;
        w_out[(size_t)t * k + lane] = my_p / psum * scale;
    }
}

}  // namespace

namespace moe_launch {

int router_gemm(const void* x, int dtype, const float* w_router, int T, int d, int E, int score_fn,
                float* scores, cudaStream_t s) {
    // fp32 activations only; bf16 activations take the tensor-core router
    if (dtype != MOE_F32) return MOE_ERR_UNSUPPORTED;
    dim3 grid(moe::ceil_div(E, RT_E), moe::ceil_div(T, RT_T));
    const int sig = score_fn == MOE_SCORE_SIGMOID;
    router_gemm_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float*>(x), w_router, T, d, E,
                                                   sig, scores);
    return moe_host::launch_status();
}

int topk(const float* scores, const float* bias, int T, const moe_route_cfg* c, int32_t* idx,
         float* w, cudaStream_t s, const float* partial, int ksplit, float* scores_out) {
    const int E = c->num_experts;
    const int blocks = moe::ceil_div(T, 8);
    const int sig = c->score_fn == MOE_SCORE_SIGMOID;
#define MOE_TOPK(EPL)                                                                          \
    topk_kernel<EPL><<<blocks, 256, 0, s>>>(scores, bias, T, E, c->top_k, c->n_group,          \
                                            c->topk_group, sig, c->routed_scale, idx, w, partial, \
                                            ksplit, scores_out)
    const int epl = moe::ceil_div(E, 32);
    if (epl <= 1) MOE_TOPK(1);
    else if (epl <= 2) MOE_TOPK(2);
    else if (epl <= 4) MOE_TOPK(4);
    else if (epl <= 8) MOE_TOPK(8);
    else if (epl <= 16) MOE_TOPK(16);
    else MOE_TOPK(32);
#undef MOE_TOPK
    return moe_host::launch_status();
}

}  // namespace moe_launch
