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
// are coalesced.  Every choice prefers the larger key and, on equal keys, the
// lower index.  Keys are compared as order-preserving unsigned integers, so
// that a warp-wide maximum is one redux.sync instead of a shuffle butterfly:
// the largest key first, then the lowest index holding it.

constexpr int FAST_GROUPS = 8;  // group counts up to this take the all-at-once path
constexpr int TOPK_THREADS = 128;
constexpr unsigned FULL = 0xffffffffu;

// a < b  <=>  ord_key(a) < ord_key(b) for non-NaN floats, with -0 mapped as
// +0 (the two compare equal as floats); every result is > 0
__device__ __forceinline__ uint32_t ord_key(float f) {
    uint32_t b = __float_as_uint(f);
    if (b == 0x80000000u) b = 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t u) {
    return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}

// the two largest of the warp's (v1 >= v2) pairs, as ordered keys: exact
// top-2 of the multiset of all pairs' values
__device__ __forceinline__ void warp_top2(uint32_t v1, uint32_t v2, uint32_t& m1, uint32_t& m2) {
    m1 = __reduce_max_sync(FULL, v1);
    const unsigned at = __ballot_sync(FULL, v1 == m1);
    m2 = __popc(at) >= 2 ? m1 : __reduce_max_sync(FULL, v1 == m1 ? v2 : v1);
}

// G32: groups of exactly 32 experts, one per lane and register slot (the
// group of held expert i is i), e.g. DeepSeek-V3's 8 groups of 32.
template <int EPL, bool G32>
__global__ void __launch_bounds__(TOPK_THREADS) topk_kernel(
    const float* __restrict__ scores, const float* __restrict__ bias, int T, int E, int k,
    int n_group, int topk_group, int sigmoid, float scale, int32_t* __restrict__ idx_out,
    float* __restrict__ w_out, const float* __restrict__ partial, int ksplit,
    float* __restrict__ scores_out) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    float sc[EPL];
    uint32_t ko[EPL];  // ordered selection keys
    uint32_t ok = 0;   // bit i: expert i*32 + lane is still a candidate
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const int e = i * 32 + lane;
        const bool in = e < E;
        if (in) ok |= 1u << i;
        if (partial) {
            // scores from the router's K-part partial logits, summed in order
            float v = 0.f;
            if (in) {
                v = partial[(size_t)t * E + e];
                for (int ks = 1; ks < ksplit; ++ks) v += partial[((size_t)ks * T + t) * E + e];
                if (sigmoid) v = 1.0f / (1.0f + expf(-v));
                scores_out[(size_t)t * E + e] = v;
            }
            sc[i] = v;
        } else {
            sc[i] = in ? scores[(size_t)t * E + e] : 0.f;
        }
        ko[i] = ord_key(in ? (bias ? sc[i] + bias[e] : sc[i]) : 0.f);
    }

    if (n_group > 1) {
        const int gs = E / n_group;
        int gid[EPL];  // group of each held expert
#pragma unroll
        for (int i = 0; i < EPL; ++i) gid[i] = G32 ? i : (i * 32 + lane) / gs;
        unsigned keep = 0;
        const uint32_t NONE = ord_key(-INFINITY);
        if (G32 || n_group <= FAST_GROUPS) {
            // every lane's two largest keys per group (-inf = none), then
            // each group's top-2 over the warp; every group has at least two
            // members, so no -inf survives
            uint32_t g1[FAST_GROUPS], g2[FAST_GROUPS];
#pragma unroll
            for (int g = 0; g < FAST_GROUPS; ++g) g1[g] = g2[g] = NONE;
            if (G32) {
#pragma unroll
                for (int i = 0; i < EPL && i < FAST_GROUPS; ++i)
                    if ((ok >> i) & 1u) g1[i] = ko[i];
            } else {
#pragma unroll
                for (int i = 0; i < EPL; ++i) {
#pragma unroll
                    for (int g = 0; g < FAST_GROUPS; ++g) {
                        if (((ok >> i) & 1u) && gid[i] == g) {
                            g2[g] = max(g2[g], min(g1[g], ko[i]));
                            g1[g] = max(g1[g], ko[i]);
                        }
                    }
                }
            }
            // every lane holds every group score: pick the best groups, ties
            // to the lower group, without further communication
            float gsc[FAST_GROUPS];
#pragma unroll
            for (int g = 0; g < FAST_GROUPS; ++g) {
                uint32_t m1 = NONE, m2 = NONE;
                if (g < n_group) warp_top2(g1[g], g2[g], m1, m2);
                gsc[g] = key_value(m1) + key_value(m2);
            }
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
            // group g's score lands in lane g
            float my_gscore = 0.f;
            for (int g = 0; g < n_group; ++g) {
                uint32_t v1 = NONE, v2 = NONE;
#pragma unroll
                for (int i = 0; i < EPL; ++i) {
                    if (((ok >> i) & 1u) && gid[i] == g) {
                        v2 = max(v2, min(v1, ko[i]));
                        v1 = max(v1, ko[i]);
                    }
                }
                uint32_t m1, m2;
                warp_top2(v1, v2, m1, m2);
                if (lane == g) my_gscore = key_value(m1) + key_value(m2);
            }
            // best groups: largest score, ties to the lower group
            uint32_t gk = lane < n_group ? ord_key(my_gscore) : 0u;
            for (int r = 0; r < topk_group; ++r) {
                const uint32_t m = __reduce_max_sync(FULL, gk);
                const int g = (int)__reduce_min_sync(FULL, gk == m ? (uint32_t)lane : FULL);
                keep |= 1u << g;
                if (lane == g) gk = 0u;
            }
        }
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if (!((keep >> gid[i]) & 1u)) ok &= ~(1u << i);
    }

    // softmax normaliser over all E logits
    float m = -FLT_MAX, z = 0.f;
    if (!sigmoid) {
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if (i * 32 + lane < E) m = fmaxf(m, sc[i]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, off));
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if (i * 32 + lane < E) z += expf(sc[i] - m);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(FULL, z, off);
    }

    int my_e = 0;
    float my_p = 0.f, psum = 0.f;
    for (int j = 0; j < k; ++j) {
        // this lane's best candidate: ascending i with strict > keeps the
        // lowest index among equal keys
        uint32_t best = 0u;
        int bi = -1;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            if (((ok >> i) & 1u) && (bi < 0 || ko[i] > best)) {
                best = ko[i];
                bi = i;
            }
        }
        const uint32_t mk = __reduce_max_sync(FULL, best);
        const int e = (int)__reduce_min_sync(
            FULL, (bi >= 0 && best == mk) ? (uint32_t)(bi * 32 + lane) : FULL);
        float s_sel = 0.f;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            if (i * 32 + lane == e) {
                ok &= ~(1u << i);
                s_sel = sc[i];
            }
        }
        s_sel = __shfl_sync(FULL, s_sel, e & 31);
        const float p = sigmoid ? s_sel : expf(s_sel - m) / z;
        psum += p;  // slot order
        if (lane == j) {
            my_e = e;
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
    const int blocks = moe::ceil_div(T, TOPK_THREADS / 32);
    const int sig = c->score_fn == MOE_SCORE_SIGMOID;
#define MOE_TOPK(EPL, G32)                                                                     \
    topk_kernel<EPL, G32><<<blocks, TOPK_THREADS, 0, s>>>(scores, bias, T, E, c->top_k, c->n_group, \
                                            c->topk_group, sig, c->routed_scale, idx, w, partial, \
                                            ksplit, scores_out)
    const int epl = moe::ceil_div(E, 32);
    const bool g32 = c->n_group > 1 && E == 32 * c->n_group;
    if (g32 && epl == 2) MOE_TOPK(2, true);
    else if (g32 && epl == 4) MOE_TOPK(4, true);
    else if (g32 && epl == 8) MOE_TOPK(8, true);
    else if (epl <= 1) MOE_TOPK(1, false);
    else if (epl <= 2) MOE_TOPK(2, false);
    else if (epl <= 4) MOE_TOPK(4, false);
    else if (epl <= 8) MOE_TOPK(8, false);
    else if (epl <= 16) MOE_TOPK(16, false);
    else MOE_TOPK(32, false);
#undef MOE_TOPK
    return moe_host::launch_status();
}

}  // namespace moe_launch
