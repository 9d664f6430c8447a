// dispatch.cu -- per-expert histogram, scan and permute of the T*k slots.
//
// The pages ("CUCo: An Agentic Framework for Compute and Communication
// Co-design", Table 4 row "MoE Dispatch/Combine") move each token to the
// experts it chose; on one GPU that is a stable counting sort of the slots
// s = t*k + j by expert followed by a row gather:
//   counts[e], offsets[e] = sum_{e'<e} counts[e'],
//   row(s) = offsets[e] + #{s' < s : idx(s') = e},  x_perm[row(s)] = x[s/k].
//
// Kernel 1 (count + scan, one pass): each block takes CH consecutive slots.
// Warps rank their slots without atomics (__match_any_sync + popc against a
// warp-private shared histogram), the block sums its per-expert counts, and a
// decoupled look-back over blocks (each block publishes its per-expert count
// vector, then its inclusive prefix vector) gives every slot its position
// inside its expert's segment.  The last block also writes counts/offsets.
// Block order comes from a ticket, so a block only ever waits for blocks that
// are already running; every wait is bounded.
// Kernel 2 (permute): one warp per slot writes the index maps and copies the
// token's row with 16-byte vectors.
#include "common.cuh"

namespace {

constexpr int DISP_WARPS = 16;
constexpr int DISP_THREADS = DISP_WARPS * 32;
constexpr int DISP_PER_WARP = 256;  // slots per warp
constexpr int DISP_CH = DISP_WARPS * DISP_PER_WARP;
constexpr int DISP_ITERS = DISP_PER_WARP / 32;

// workspace header (ints): [0] ticket; flags follow at +16 bytes
struct DispatchWs {
    int* ticket;
    int* flags;     // [nb]   0 = nothing, 1 = aggregate, 2 = inclusive prefix
    int* agg;       // [nb][E]
    int* incl;      // [nb][E]
    int* pos;       // [S]    position of each slot inside its expert's segment
};

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

__host__ __device__ inline DispatchWs carve(void* ws, int S, int E) {
    const int nb = (S + DISP_CH - 1) / DISP_CH;
    char* p = static_cast<char*>(ws);
    DispatchWs w;
    w.ticket = reinterpret_cast<int*>(p);
    w.flags = reinterpret_cast<int*>(p + 16);
    size_t off = align_up(16 + sizeof(int) * (size_t)nb, 256);
    w.agg = reinterpret_cast<int*>(p + off);
    off = align_up(off + sizeof(int) * (size_t)nb * E, 256);
    w.incl = reinterpret_cast<int*>(p + off);
    off = align_up(off + sizeof(int) * (size_t)nb * E, 256);
    w.pos = reinterpret_cast<int*>(p + off);
    return w;
}

__host__ __device__ inline size_t ws_bytes(int S, int E) {
    const int nb = (S + DISP_CH - 1) / DISP_CH;
    size_t off = align_up(16 + sizeof(int) * (size_t)nb, 256);
    off = align_up(off + sizeof(int) * (size_t)nb * E, 256);
    off = align_up(off + sizeof(int) * (size_t)nb * E, 256);
    return align_up(off + sizeof(int) * (size_t)S, 256);
}

__device__ __forceinline__ int ld_acquire(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release(int* p, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Walk back from block b-1 until a block whose inclusive prefix is published
// (flag 2), passing blocks that published only their aggregate (flag 1).
// Returns that block (-1: none before b), or -2 if a predecessor published
// nothing within limit_ns.
__device__ int lookback_walk(const int* flags, int b, uint64_t limit_ns) {
    int p = b - 1;
    const uint64_t t0 = moe::globaltimer_ns();
    while (p >= 0) {
        const int f = ld_acquire(flags + p);
        if (f == 2) return p;
        if (f == 1) { --p; continue; }
        if (moe::globaltimer_ns() - t0 > limit_ns) return -2;
    }
    return -1;
}

// Self-test of the bounded look-back wait: block 1 waits on block 0's flag,
// which nothing sets; the wait must give up and report a timeout.
__global__ void lookback_probe_kernel(const int* flags, uint64_t limit_ns, uint32_t* err) {
    if (threadIdx.x == 0 && lookback_walk(flags, 1, limit_ns) == -2)
        moe::raise_error(err, moe::ERR_TIMEOUT_SCAN);
}

__global__ void __launch_bounds__(DISP_THREADS) dispatch_count_kernel(
    const int32_t* __restrict__ idx, int S, int E, DispatchWs st, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, uint32_t* err) {
    extern __shared__ int smem[];
    int* whist = smem;                      // [DISP_WARPS][E]
    int* btot = smem + DISP_WARPS * E;      // [E]
    int* excl = btot + E;                   // [E]
    __shared__ int s_b, s_stop, s_abort;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nb = gridDim.x;

    if (tid == 0) {
        s_b = atomicAdd(st.ticket, 1);
        s_abort = 0;
    }
    for (int i = tid; i < DISP_WARPS * E; i += DISP_THREADS) whist[i] = 0;
    __syncthreads();
    const int b = s_b;

    // 1) rank slots inside each warp's sub-chunk, in slot order
    int ev[DISP_ITERS], rk[DISP_ITERS];
    int* wh = whist + warp * E;
    const unsigned lt = (1u << lane) - 1u;
#pragma unroll
    for (int it = 0; it < DISP_ITERS; ++it) {
        const int s = b * DISP_CH + warp * DISP_PER_WARP + it * 32 + lane;
        int e = -1;
        if (s < S) {
            e = idx[s];
            if (e < 0 || e >= E) {
                moe::raise_error(err, moe::ERR_BAD_INDEX);
                e = -1;
            }
        }
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        int base = 0;
        if (e >= 0) base = wh[e];
        __syncwarp();
        if (e >= 0 && lane == __ffs(peers) - 1) wh[e] = base + __popc(peers);
        __syncwarp();
        ev[it] = e;
        rk[it] = base + __popc(peers & lt);
    }
    __syncthreads();

    // 2) per expert: exclusive prefix over warps, block total
    for (int e = tid; e < E; e += DISP_THREADS) {
        int run = 0;
        for (int w = 0; w < DISP_WARPS; ++w) {
            const int c = whist[w * E + e];
            whist[w * E + e] = run;
            run += c;
        }
        btot[e] = run;
    }
    __syncthreads();

    // 3) decoupled look-back over blocks, one vector of E counts per block
    if (b == 0) {
        for (int e = tid; e < E; e += DISP_THREADS) {
            excl[e] = 0;
            st.incl[e] = btot[e];
        }
        __threadfence();
        __syncthreads();
        if (tid == 0) st_release(st.flags, 2);
    } else {
        for (int e = tid; e < E; e += DISP_THREADS) st.agg[(size_t)b * E + e] = btot[e];
        __threadfence();
        __syncthreads();
        if (tid == 0) {
            st_release(st.flags + b, 1);
            // block 0 always publishes its inclusive prefix, so a walk that
            // does not time out ends at some block >= 0
            const int stop = lookback_walk(st.flags, b, moe::WAIT_LIMIT_NS);
            if (stop < 0) {
                moe::raise_error(err, moe::ERR_TIMEOUT_SCAN);
                s_abort = 1;
            }
            s_stop = stop;
        }
        __syncthreads();
        if (s_abort) return;
        const int stop = s_stop;
        for (int e = tid; e < E; e += DISP_THREADS) {
            int v = __ldcg(st.incl + (size_t)stop * E + e);
            for (int q = stop + 1; q < b; ++q) v += __ldcg(st.agg + (size_t)q * E + e);
            excl[e] = v;
            st.incl[(size_t)b * E + e] = v + btot[e];
        }
        __threadfence();
        __syncthreads();
        if (tid == 0) st_release(st.flags + b, 2);
    }
    __syncthreads();

    // 4) position of each slot inside its expert's segment
#pragma unroll
    for (int it = 0; it < DISP_ITERS; ++it) {
        const int s = b * DISP_CH + warp * DISP_PER_WARP + it * 32 + lane;
        if (s < S && ev[it] >= 0) st.pos[s] = excl[ev[it]] + wh[ev[it]] + rk[it];
    }

    // 5) the last block owns the totals: counts and their exclusive scan
    if (b == nb - 1 && warp == 0) {
        const int per = (E + 31) / 32;
        const int lo = lane * per, hi = min(E, lo + per);
        int sum = 0;
        for (int e = lo; e < hi; ++e) sum += excl[e] + btot[e];
        int inc = sum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, inc, off);
            if (lane >= off) inc += o;
        }
        int run = inc - sum;
        for (int e = lo; e < hi; ++e) {
            const int c = excl[e] + btot[e];
            counts[e] = c;
            offsets[e] = run;
            run += c;
        }
        if (lane == 31) offsets[E] = inc;
    }
}

// One warp per slot: index maps and a 16-byte-vector copy of the token row.
__global__ void __launch_bounds__(256) permute_kernel(
    const int32_t* __restrict__ idx, const int* __restrict__ pos, const int32_t* __restrict__ offsets,
    int S, int k, int E, const uint4* __restrict__ x, int row_vecs, int32_t* __restrict__ slot_to_row,
    int32_t* __restrict__ row_to_token, uint4* __restrict__ x_perm, const float* __restrict__ w_slot,
    float* __restrict__ w_row, const uint32_t* err, int e_lo, int e_hi) {
    if (moe::read_error(err)) return;
    const int lane = threadIdx.x & 31;
    const int s = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (s >= S) return;
    const int e = idx[s];
    if (e < 0 || e >= E) return;  // already flagged by the count kernel
    if (e < e_lo || e >= e_hi) return;  // another launch's expert range
    const int row = offsets[e] + pos[s];
    const int t = s / k;
    if (lane == 0) {
        slot_to_row[s] = row;
        row_to_token[row] = t;
        if (w_row) w_row[row] = w_slot[s];  // gate weight of the row (fused combine)
    }
    if (!x_perm) return;
    const uint4* src = x + (size_t)t * row_vecs;
    uint4* dst = x_perm + (size_t)row * row_vecs;
    int v = lane;
    for (; v + 96 < row_vecs; v += 128) {
        const uint4 a = __ldg(src + v), b2 = __ldg(src + v + 32), c = __ldg(src + v + 64),
                    d = __ldg(src + v + 96);
        __stcs(dst + v, a);
        __stcs(dst + v + 32, b2);
        __stcs(dst + v + 64, c);
        __stcs(dst + v + 96, d);
    }
    for (; v < row_vecs; v += 32) __stcs(dst + v, __ldg(src + v));
}

}  // namespace

namespace moe_launch {

int lookback_probe(void* flags_zeroed, uint64_t limit_ns, uint32_t* err, cudaStream_t s) {
    lookback_probe_kernel<<<1, 32, 0, s>>>(static_cast<const int*>(flags_zeroed), limit_ns, err);
    return moe_host::launch_status();
}

size_t dispatch_ws_bytes(int T, int k, int E) { return ws_bytes(T * k, E); }

int dispatch(const int32_t* idx, const void* x, int dtype, int T, int d, int k, int E,
             int32_t* counts, int32_t* offsets, int32_t* slot_to_row, int32_t* row_to_token,
             void* x_perm, void* ws, uint32_t* err, cudaStream_t s, const float* w_slot,
             float* w_row, int parts, int e_lo, int e_hi) {
    const int S = T * k;
    const int nb = moe::ceil_div(S, DISP_CH);
    DispatchWs st = carve(ws, S, E);
    if (e_hi < 0) e_hi = E;
    if (parts & 2 && (e_lo < 0 || e_lo > e_hi || e_hi > E)) return MOE_ERR_INVALID_ARG;
    if (!(parts & 1)) {
        // the permute alone, after a count launch of the same call
        if (!(parts & 2) || e_lo == e_hi) return MOE_OK;
        const size_t esize = dtype == MOE_BF16 ? 2 : 4;
        const int row_vecs = (int)((size_t)d * esize / 16);
        permute_kernel<<<moe::ceil_div(S, 8), 256, 0, s>>>(
            idx, st.pos, offsets, S, k, E, static_cast<const uint4*>(x), row_vecs, slot_to_row,
            row_to_token, static_cast<uint4*>(x_perm), w_slot, w_row, err, e_lo, e_hi);
        return moe_host::launch_status();
    }
    if (cudaMemsetAsync(ws, 0, 16 + sizeof(int) * (size_t)nb, s) != cudaSuccess) return MOE_ERR_CUDA;
    const size_t smem = sizeof(int) * (size_t)(DISP_WARPS + 2) * E;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(dispatch_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return MOE_ERR_CUDA;
    dispatch_count_kernel<<<nb, DISP_THREADS, smem, s>>>(idx, S, E, st, counts, offsets, err);
    int rc = moe_host::launch_status();
    if (rc != MOE_OK || !(parts & 2) || e_lo == e_hi) return rc;
    const size_t esize = dtype == MOE_BF16 ? 2 : 4;
    const int row_vecs = (int)((size_t)d * esize / 16);
    permute_kernel<<<moe::ceil_div(S, 8), 256, 0, s>>>(
        idx, st.pos, offsets, S, k, E, static_cast<const uint4*>(x), row_vecs, slot_to_row,
        row_to_token, static_cast<uint4*>(x_perm), w_slot, w_row, err, e_lo, e_hi);
    return moe_host::launch_status();
}

}  // namespace moe_launch
