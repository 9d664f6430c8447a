// grouped_gemm_tc.cu -- per-expert SwiGLU FFN as tcgen05 grouped GEMMs (bf16).
//
// The pages ("CUCo: An Agentic Framework for Compute and Communication
// Co-design", abstract and Table 4 row "MoE Dispatch/Combine") put local expert
// compute between dispatch and combine, and note padding overhead on
// imbalanced loads.  Here every expert's rows form one exact, unpadded segment
// [offsets[e], offsets[e+1]) of the permuted activations, and two persistent
// kernels compute
//   gate/up:  H[r, n] = bf16( silu(<x_r, W1_e[n]>) * <x_r, W3_e[n]> )
//   down:     Y[r, n] = <H_r, W2_e[n]>                         (fp32)
// with fp32 accumulation in tensor memory.
//
// Design (sm_103a):
//  * Swap-AB: the MMA's M side (128) walks output features (weight rows), its
//    N side walks tokens (16..BN, rounded up to 16 per tile).  Small and
//    ragged segments then cost N granularity 16 rather than a 128-row tile,
//    and every weight tile of an expert is read once per BN tokens.
//  * One CTA per SM (persistent), 10 warps: warp 0 issues TMA loads, warp 1
//    allocates tensor memory and issues tcgen05.mma from one thread, warps 2-9
//    drain the accumulators (tcgen05.ld; two warps per 32-lane quarter) and
//    store.  Shared-memory stages are handed over with mbarriers; the
//    accumulator is handed over with a full/empty mbarrier pair
//    (double-buffered when tensor memory holds two).
//  * Operands are K-major bf16 tiles of 64 elements (128 B) per row, loaded by
//    TMA with the 128-byte swizzle that the tcgen05 shared-memory descriptor
//    expects; the token tile is loaded in at most four boxes of 256/128/64/32
//    rows, only as many rows (in whole 32-row boxes) as the segment needs.
//    Rows past a segment belong to the next expert (or are zero-filled past
//    the matrix); their results are computed and dropped.
//  * Tiles are enumerated expert-major, feature-tile next, token-tile last
//    (experts of many token tiles: feature tiles in blocks of four, token
//    tiles inside a block), so CTAs that run at the same time share weight
//    tiles and token tiles in L2.
//  * Every mbarrier wait is bounded (about 1 s); on expiry the kernel sets the
//    error word, waits briefly for its own copies and MMAs in flight, frees
//    tensor memory and returns.
//  * Routed launches with 256-token tiles, and routed gate/up launches with
//    160-token tiles, run the same design on CTA pairs
//    (grouped_gemm_2sm_kernel below, tcgen05.mma.cta_group::2): two weight
//    tiles and half the token tile per SM and stage, a quarter fewer bytes
//    per multiply-add than the one-SM tile.  The compute-bound down
//    projection runs two such pairs per cluster on neighbouring feature
//    tiles: each half of the token tile is loaded by one pair and multicast
//    to both, so an SM loads a quarter of the token tile per stage.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"

namespace {

constexpr int BM = 128;         // features per tile (MMA M)
// K per stage: one swizzle-atom row of bf16 (64 elements = 128 B with the
// 128-byte swizzle, 32 elements = 64 B with the 64-byte swizzle)
#ifndef MOE_BK
#define MOE_BK 64
#endif
constexpr int BK = MOE_BK;
static_assert(BK == 64 || BK == 32, "K slab of 64 or 32 bf16");
constexpr int SWZ_BYTES = BK * 2;  // swizzle span = row bytes
constexpr int B_BOX = 32;       // token rows per TMA box
constexpr int A_TILE_BYTES = BM * BK * 2;      // 16 KB
constexpr int B_BOX_BYTES = B_BOX * BK * 2;    // 4 KB
constexpr int NUM_EPI_WARPS = 8;  // two per 32-lane quarter of tensor memory
constexpr int RING = 4;           // unit indices in flight from producer to consumers
constexpr int NUM_THREADS = 32 * (2 + NUM_EPI_WARPS);
// epilogue warps of the one-SM kernel per mode (gate/up, down, router): a
// multiple of 4, each warp reaching one 32-lane quarter of tensor memory.
// Its gate/up runs the shared expert beside the router and top-k, whose
// blocks must fit beside it: with 16 warps the route stage of the
// DeepSeek-V3 Zipf layer grew from 0.29 to 0.76 ms and the prefill layer
// from 3.94 to 4.00 ms, so 8.
#ifndef MOE_EPI1_GU
#define MOE_EPI1_GU 8
#endif
__host__ __device__ constexpr int epi1_warps(int mode) { return mode == 0 ? MOE_EPI1_GU : NUM_EPI_WARPS; }
__host__ __device__ constexpr int threads1(int mode) { return 32 * (2 + epi1_warps(mode)); }
static_assert(MOE_EPI1_GU % 4 == 0 && MOE_EPI1_GU >= 4, "whole quarters of tensor memory");
constexpr int TMEM_COLS = 512;
constexpr int MAX_E = 1024;

// MODE 0: gate/up + SwiGLU (W1 and W3 tiles into two accumulators)
// MODE 1: down projection (one A tile)
// MODE 2: router, fp32 weight split into three bf16 terms (hi, mid, lo), one
//         accumulator per term (tensor-core accumulation truncates at every
//         MMA, so the small terms must not share the large term's
//         accumulator), summed in the epilogue
// BN is the token tile (MMA N upper bound).  Stages fill up to 216 KB of
// shared memory; accumulators are double-buffered when tensor memory allows.
constexpr int SMEM_BUDGET = 216 * 1024;
constexpr int SMEM_LIMIT = 227 * 1024;  // opt-in maximum per CTA

template <int MODE>
struct ModeCfg;
// rows per expert from which the gate/up and down launches use 256-row token
// tiles (below: 128)
#ifndef MOE_GU_WIDE_ROWS
#define MOE_GU_WIDE_ROWS 384
#endif
#ifndef MOE_DN_WIDE_ROWS
#define MOE_DN_WIDE_ROWS 32
#endif
// token tile of the gate/up launch below MOE_GU_WIDE_ROWS rows per expert,
// and of the down launch from MOE_DN_WIDE_ROWS rows per expert
#ifndef MOE_GU_BN
#define MOE_GU_BN 160
#endif
// below this many rows per expert on average, both launches use 32-token
// tiles (0: never)
#ifndef MOE_NARROW_ROWS
#define MOE_NARROW_ROWS 8
#endif
#ifndef MOE_DN_BN
#define MOE_DN_BN 256
#endif
template <>
struct ModeCfg<0> {
    static constexpr int NUM_A = 2;
    static constexpr bool SPLIT_ACC = true;  // one accumulator per A tile
};
template <>
struct ModeCfg<1> {
    // two 128-feature tiles (a_step = 128 rows apart) share each token tile
    static constexpr int NUM_A = 2;
    static constexpr bool SPLIT_ACC = true;
};
template <>
struct ModeCfg<2> {
    static constexpr int NUM_A = 3;
    static constexpr bool SPLIT_ACC = true;
};

template <int MODE, int BN_>
struct Cfg {
    static constexpr int NUM_A = ModeCfg<MODE>::NUM_A, BN = BN_;
    static constexpr bool SPLIT_ACC = ModeCfg<MODE>::SPLIT_ACC;
    static constexpr int STAGE_BYTES = NUM_A * A_TILE_BYTES + BN * BK * 2;
    static constexpr int STAGES = SMEM_BUDGET / STAGE_BYTES;
    // TMEM columns between the split accumulators: BN rounded up to 128, so
    // every accumulator starts on a 128-column boundary
    static constexpr int ASTRIDE = (BN + 127) / 128 * 128;
    static constexpr int ACC_COLS = SPLIT_ACC ? NUM_A * ASTRIDE : BN;  // TMEM columns per accumulator
    // output features per unit: the down projection's A tiles are distinct
    // features; gate/up (W1, W3) and the router's weight terms share features
    static constexpr int FEAT = MODE == 1 ? NUM_A * BM : BM;
    static constexpr int ACC_STAGES = TMEM_COLS / ACC_COLS >= 2 ? 2 : 1;
    // + barriers/tmem slot + schedule table
    static constexpr size_t SMEM = 1024 + (size_t)STAGES * STAGE_BYTES + 256 + sizeof(int) * 2 * (MAX_E + 1);
    static_assert(STAGES >= 2 && ACC_COLS <= TMEM_COLS, "tile does not fit");
    // token rows are loaded in whole 32-row boxes: a tile that is not a
    // multiple of 32 rows would let the last box run past its stage
    static_assert(BN % B_BOX == 0 && BN <= 256, "token tile must be whole boxes");
    static_assert(SMEM + 64 <= (size_t)SMEM_LIMIT, "shared memory over the per-CTA limit");
};

// Weight layouts.  Row-major: [rows, K] as given.  Tile-major (written by
// moe_pack_expert_weights, rows a multiple of 128, K of 64): tile (r, kb) --
// rows 128r..128r+127, columns 64kb..64kb+63 -- is one contiguous 16 KB
// block, so each TMA load of a weight tile reads 16 KB in a row of HBM
// instead of 128 pieces of 128 B one matrix row apart.  WEIGHTS_TILES orders
// the tiles (r, kb) row-tile-major; WEIGHTS_TILE_PAIRS keeps row tiles 2m and
// 2m+1 of each k-block next to each other, the two feature tiles that one
// down-projection unit loads per stage.
constexpr int WEIGHTS_ROWS = 0, WEIGHTS_TILES = 1, WEIGHTS_TILE_PAIRS = 2;

__host__ __device__ __forceinline__ int packed_tile(int rt, int kb, int num_kb, int layout) {
    return layout == WEIGHTS_TILE_PAIRS ? ((rt >> 1) * num_kb + kb) * 2 + (rt & 1)
                                        : rt * num_kb + kb;
}

// Tensor maps of one activation matrix with token boxes of 32, 64, 128 and
// 256 rows (index = log2(rows / 32)).
// token-tile maps: boxes of 32, 64, 128 and 256 rows, then one of 16 rows
// (for CTA pairs, whose half tiles are multiples of 16 rows)
struct BMaps {
    CUtensorMap m[5];
};

struct Params {
    const int32_t* offsets;  // [E+1], or NULL: one segment [0, rows)
    int E;
    int rows;                // rows of the activation matrix
    int K;                   // reduction length
    int N_out;               // output features per expert
    int a_rows;              // weight rows per expert in the 2D weight view
    int a_step;              // row distance between the A tiles of one stage
    void* out;               // H bf16 / Y fp32 / scores fp32, [rows, N_out]
    uint32_t* err;
    int flags;               // router: bit 0 = apply sigmoid
    // optional second problem run in the same launch (the shared expert): one
    // dense segment of `rows2` rows through tm_a2/tm_b2 into out2
    int rows2;
    void* out2;
    // zero before the launch: units past the first gridDim.x are claimed from it
    unsigned* work;
    // router: the K range is split into ksplit parts, each a unit of its own;
    // part ks writes its partial sums to out + ks * rows * N_out
    int ksplit;
    // down projection with fused combine (comb_out != NULL): instead of
    // writing y, add w_row[r] * y[r] into comb_out[row_token[r]] (routed
    // rows) or y[r] into comb_out[r] (second problem)
    float* comb_out;
    const int32_t* row_token;
    const float* w_row;
    // layout of the weight (A) matrix: WEIGHTS_ROWS (row-major), or one of
    // the tile-major layouts written by moe_pack_expert_weights
    int a_layout;
};

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity.  Returns false if the
// kernel is aborting (flag set by any role) or if this wait ran out.
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                       uint32_t* err, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = moe::globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (moe::globaltimer_ns() - t0 > limit_ns) {
            *abort_flag = 1;
            moe::raise_error(err, moe::ERR_TIMEOUT_PIPE);
            return false;
        }
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// tcgen05 shared-memory matrix descriptor: K-major, swizzle span SWZ_BYTES
// (128 or 64 B), 8-row core-matrix groups 8 * SWZ_BYTES apart (stride byte
// offset), version 1.
__device__ __forceinline__ uint64_t smem_desc_sw(uint32_t addr) {
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFFu) >> 4);  // start address
    d |= (uint64_t)1 << 16;                   // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)((8 * SWZ_BYTES) >> 4) << 32;  // stride byte offset
    d |= (uint64_t)1 << 46;                   // descriptor version
    d |= (uint64_t)(SWZ_BYTES == 128 ? 2 : 4) << 61;  // swizzle: 128 B or 64 B
    return d;
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major, M=128.
__device__ __forceinline__ uint32_t idesc_bf16(int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(BM >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bar)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// element i (0..3, run-time) of four values, by selects (no local memory)
__device__ __forceinline__ float pick4(const float (&a)[4], int i) {
    const float lo = (i & 1) ? a[1] : a[0];
    const float hi = (i & 1) ? a[3] : a[2];
    return (i & 2) ? hi : lo;
}
// accumulator value j0 + i (i run-time, 0..3) of a tcgen05.ld result, as float
__device__ __forceinline__ float sel4(const uint32_t (&g)[32], int j0, int i) {
    const float a[4] = {__uint_as_float(g[j0]), __uint_as_float(g[j0 + 1]),
                        __uint_as_float(g[j0 + 2]), __uint_as_float(g[j0 + 3])};
    return pick4(a, i);
}

// ---------------------------------------------------------------- schedule

struct Unit {
    int e;        // expert (E for the second, dense problem)
    int m_start;  // first activation row of the token tile
    int n_tok;    // tokens in the tile (1..BN)
    int n0;       // first output feature
    bool second;  // unit of the second problem (shared expert)
};

// The work units form two streams.  Compute stream: experts with at least
// MOE_COMPUTE_ROWS rows (their weight tiles feed many token tiles from L2),
// then the second problem's tiles.  Streaming stream: the other experts,
// whose units are bound by reading their weights from HBM.  The shorter
// stream is spread evenly through the longer one (period P = U / U_short:
// position j*P holds short-stream unit j), so that compute-bound and
// weight-streaming tiles run side by side instead of in separate phases.
// Inside a stream, units are expert-major (units of expert e occupy
// [pre[e]*nt, pre[e+1]*nt)), then feature tile, then token tile, so CTAs that
// run together share an expert's token tiles and weight tiles in L2.
// Measured: with a 128-row class threshold DeepSeek-V3 prefill (4096
// tokens) takes 4.106 ms per layer against 4.137 ms with 256 (the down
// GEMM 1.302 vs 1.325 ms), the Zipf workload (16384 tokens) 10.69 vs
// 10.71-10.75 ms; 512 and 1024 rows are slower on Zipf (10.85, 10.94 ms),
// and one stream was slower still when first measured.
#ifndef MOE_COMPUTE_ROWS
#define MOE_COMPUTE_ROWS 128
#endif

struct Sched {
    const int* pre_c;  // [E+1] token tiles of compute-class experts, prefix
    const int* pre_s;  // [E+1] token tiles of streaming-class experts, prefix
    const int* offs;
    int E, n_tiles, U, U_c, U_s, U2, rows2;
};

// Order of an expert's units.  Feature tile outermost and token tile
// innermost: an expert's few token tiles then stream each weight tile at the
// same time (one DRAM read).  An expert of many token tiles (at least
// MOE_FEAT_BLOCK_MT) would then have its whole token range in flight for
// each feature tile (a 15 K-row expert: 60 token tiles of 3.7 MB, more than
// L2, read again for every feature tile); its units go in blocks of
// MOE_FEAT_BLOCK feature tiles instead, the token tiles inside a block and
// the block's feature tiles innermost.  Measured (same box, three
// repetitions): DeepSeek-V3 Zipf(1.2) T=16384 layer 9.63-9.72 vs 9.89-9.97
// ms (routed gate/up 4.86-4.91 vs 4.98-5.02, down 3.18-3.22 vs 3.27-3.31);
// blocks of 8 feature tiles, or blocking every expert, were slower (prefill
// 2.5% with blocks of 8 for all); Mixtral and prefill, whose experts have
// fewer token tiles, are unaffected.
#ifndef MOE_FEAT_BLOCK
#define MOE_FEAT_BLOCK 4
#endif
#ifndef MOE_FEAT_BLOCK_MT
#define MOE_FEAT_BLOCK_MT 8
#endif

template <int BN, int FEAT>
__device__ __forceinline__ Unit routed_unit(int i, const int* pre, const Sched& q) {
    int lo = 0, hi = q.E;  // largest e with pre[e]*nt <= i (empty experts have no width)
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pre[mid] * q.n_tiles <= i) lo = mid; else hi = mid;
    }
    const int e = lo;
    const int mt = pre[e + 1] - pre[e];
    const int local = i - pre[e] * q.n_tiles;
    int nt, mtile;
    if (MOE_FEAT_BLOCK > 0 && mt >= MOE_FEAT_BLOCK_MT) {
        // every block but the last holds MOE_FEAT_BLOCK feature tiles
        const int b = local / (MOE_FEAT_BLOCK * mt);
        const int r = local - b * MOE_FEAT_BLOCK * mt;
        const int fb = min(MOE_FEAT_BLOCK, q.n_tiles - b * MOE_FEAT_BLOCK);
        mtile = r / fb;
        nt = b * MOE_FEAT_BLOCK + (r - mtile * fb);
    } else {
        nt = local / mt;
        mtile = local - nt * mt;
    }
    Unit r;
    r.e = e;
    r.second = false;
    r.m_start = q.offs[e] + mtile * BN;
    r.n_tok = min(BN, q.offs[e + 1] - r.m_start);
    r.n0 = nt * FEAT;
    return r;
}

template <int BN, int FEAT>
__device__ __forceinline__ Unit decode_unit(int u, const Sched& q) {
    // which stream, and which unit of it
    const bool c_short = q.U_c <= q.U_s;
    const int U_short = c_short ? q.U_c : q.U_s;
    bool in_c;
    int i;
    if (U_short > 0) {
        const int P = q.U / U_short;
        const int j = u / P;
        if (u - j * P == 0 && j < U_short) {
            in_c = c_short;
            i = j;
        } else {
            in_c = !c_short;
            i = u - min(U_short, j + 1);
        }
    } else {
        in_c = q.U_c > 0;
        i = u;
    }
    if (!in_c) return routed_unit<BN, FEAT>(i, q.pre_s, q);
    const int routed_c = (q.U_c - q.U2);
    if (i < routed_c) return routed_unit<BN, FEAT>(i, q.pre_c, q);
    // second problem: one dense segment of rows2 rows
    i -= routed_c;
    const int mt2 = (q.rows2 + BN - 1) / BN;
    const int nt = i / mt2, mtile = i - nt * mt2;
    Unit r;
    r.e = q.E;
    r.second = true;
    r.m_start = mtile * BN;
    r.n_tok = min(BN, q.rows2 - r.m_start);
    r.n0 = nt * FEAT;
    return r;
}

// The launch's schedule, by one warp: per expert the token tiles of the
// compute class (at least MOE_COMPUTE_ROWS rows) and of the streaming class,
// their prefix sums pre_c / pre_s [E+1], and total_units = {all units (-1:
// inconsistent offsets or an earlier stage failed: no work), compute-stream
// units, streaming-stream units}.  Inconsistent offsets are reported when
// `report` is set.
template <int BN>
__device__ __forceinline__ void build_schedule(const Params& p, int n_tiles, int U2, int* pre_c,
                                               int* pre_s, int* total_units, bool report) {
    const int lane = threadIdx.x & 31, E = p.E;
    // per-lane chunk of experts, then warp scans of the chunk sums
    const int per = (E + 31) / 32;
    const int lo = min(E, lane * per), hi = min(E, lo + per);
    int sum_c = 0, sum_s = 0;
    bool bad = false;
    for (int e = lo; e < hi; ++e) {
        const int a = p.offsets ? p.offsets[e] : 0;
        const int b = p.offsets ? p.offsets[e + 1] : p.rows;
        if (a < 0 || b < a || b > p.rows) bad = true;
        const int mt = (b - a + BN - 1) / BN;
        if (b - a >= MOE_COMPUTE_ROWS) sum_c += mt; else sum_s += mt;
    }
    int inc_c = sum_c, inc_s = sum_s;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int oc = __shfl_up_sync(0xffffffffu, inc_c, off);
        const int os = __shfl_up_sync(0xffffffffu, inc_s, off);
        if (lane >= off) {
            inc_c += oc;
            inc_s += os;
        }
    }
    int run_c = inc_c - sum_c, run_s = inc_s - sum_s;
    for (int e = lo; e < hi; ++e) {
        pre_c[e] = run_c;
        pre_s[e] = run_s;
        const int a = p.offsets ? p.offsets[e] : 0;
        const int b = p.offsets ? p.offsets[e + 1] : p.rows;
        const int mt = (b - a + BN - 1) / BN;
        if (b - a >= MOE_COMPUTE_ROWS) run_c += mt; else run_s += mt;
    }
    const bool any_bad = __any_sync(0xffffffffu, bad);
    if (lane == 31) {
        pre_c[E] = inc_c;
        pre_s[E] = inc_s;
        // an earlier stage that failed, or inconsistent offsets: no work
        const bool fail = any_bad || moe::read_error(p.err);
        total_units[0] = fail ? -1 : (inc_c + inc_s) * n_tiles + U2;
        total_units[1] = inc_c * n_tiles + U2;  // compute stream
        total_units[2] = inc_s * n_tiles;       // streaming stream
        if (any_bad && report) moe::raise_error(p.err, moe::ERR_BAD_OFFSETS);
    }
}

// ---------------------------------------------------------------- the kernel

template <int MODE, int BN_>
__global__ void __launch_bounds__(threads1(MODE), 1)
    grouped_gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_a,
                           const __grid_constant__ BMaps tm_b,
                           const __grid_constant__ CUtensorMap tm_a2,
                           const __grid_constant__ BMaps tm_b2, const Params p) {
    using C = Cfg<MODE, BN_>;
    constexpr int EPI1 = epi1_warps(MODE);
    constexpr int STAGES = C::STAGES, NUM_A = C::NUM_A, ACC = C::ACC_STAGES, BN = C::BN;
    constexpr int ACC_COLS = C::ACC_COLS, ASTRIDE = C::ASTRIDE;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte aligned base for the swizzled tiles
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* tiles = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)STAGES * C::STAGE_BYTES);
    uint64_t* full_bar = bars;                  // [STAGES]
    uint64_t* empty_bar = bars + STAGES;        // [STAGES]
    uint64_t* tfull_bar = bars + 2 * STAGES;    // [ACC]
    uint64_t* tempty_bar = tfull_bar + ACC;     // [ACC]
    uint64_t* drain_bar = tempty_bar + ACC;     // [1]
    uint64_t* ufull_bar = drain_bar + 1;        // [RING] unit index published
    uint64_t* uempty_bar = ufull_bar + RING;    // [RING] unit index read by all consumers
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(uempty_bar + RING);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* total_units = reinterpret_cast<int*>(tmem_slot + 2);
    volatile int* ring = reinterpret_cast<volatile int*>(tmem_slot + 5);  // [RING]
    int* mpre = reinterpret_cast<int*>(smem + (size_t)STAGES * C::STAGE_BYTES + 256);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // ---- schedule: token tiles per expert, per class, and their prefixes ---
    const int E = p.E;
    const int n_tiles = (p.N_out + C::FEAT - 1) / C::FEAT;
    const int U2 = p.rows2 > 0 ? ((p.rows2 + BN - 1) / BN) * n_tiles : 0;
    int* pre_c = mpre;             // [E+1]
    int* pre_s = mpre + (E + 1);   // [E+1]
    if (warp == 0) build_schedule<BN>(p, n_tiles, U2, pre_c, pre_s, total_units, true);
    if (tid == 0) {
        *abort_flag = 0;
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        for (int a = 0; a < ACC; ++a) {
            mbar_init(smem_u32(&tfull_bar[a]), 1);
            mbar_init(smem_u32(&tempty_bar[a]), EPI1);
        }
        mbar_init(smem_u32(drain_bar), 1);
        for (int r = 0; r < RING; ++r) {
            mbar_init(smem_u32(&ufull_bar[r]), 1);
            mbar_init(smem_u32(&uempty_bar[r]), 1 + EPI1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        tma_prefetch_desc(&tm_a);
        for (int i = 0; i < 4; ++i) tma_prefetch_desc(&tm_b.m[i]);
        if (p.rows2 > 0) {
            tma_prefetch_desc(&tm_a2);
            for (int i = 0; i < 4; ++i) tma_prefetch_desc(&tm_b2.m[i]);
        }
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // units handed out: work units x K parts (router only)
    const int KS = MODE == 2 ? max(1, p.ksplit) : 1;
    const int U = total_units[0] < 0 ? -1 : total_units[0] * KS;

    // offsets for decode: dense mode synthesises {0, rows}
    __shared__ int s_dense_offs[2];
    if (tid == 0) {
        s_dense_offs[0] = 0;
        s_dense_offs[1] = p.rows;
    }
    __syncthreads();
    const int* offs = p.offsets ? p.offsets : s_dense_offs;
    const int num_kb = (p.K + BK - 1) / BK;
    const int kb_per = (num_kb + KS - 1) / KS;  // k-blocks per K part
    const Sched sched{pre_c, pre_s,         offs, E, n_tiles, total_units[0], total_units[1],
                      total_units[2], U2,  p.rows2};

    if (U > 0 && warp == 0) {
        // ================= TMA producer (one thread) =================
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            long issued = 0;
            int slot = 0;
            uint32_t uphase = 0;
            // first unit: blockIdx.x; later ones: claimed from the launch's
            // counter, so CTAs that finish early take more of the work
            for (int u = blockIdx.x;;) {
                // publish u (or the end, -1) to the MMA and epilogue warps
                if (!mbar_wait(smem_u32(&uempty_bar[slot]), uphase ^ 1, abort_flag, p.err,
                               moe::WAIT_LIMIT_NS))
                    break;
                const bool last = u >= U || *abort_flag;
                ring[slot] = last ? -1 : u;
                mbar_arrive(smem_u32(&ufull_bar[slot]));
                if (++slot == RING) { slot = 0; uphase ^= 1; }
                if (last) break;
                const int next = (int)gridDim.x + (int)atomicAdd(p.work, 1u);
                const Unit t = decode_unit<BN, C::FEAT>(u / KS, sched);
                const int kb0 = (u % KS) * kb_per, kb1 = min(num_kb, kb0 + kb_per);
                const CUtensorMap* ma = t.second ? &tm_a2 : &tm_a;
                const CUtensorMap* mb = t.second ? tm_b2.m : tm_b.m;
                const int nbox = (t.n_tok + B_BOX - 1) / B_BOX;
                const uint32_t bytes = NUM_A * A_TILE_BYTES + nbox * B_BOX_BYTES;
                const int a_row = (t.second ? 0 : t.e * p.a_rows) + t.n0;
                bool ok = true;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1, abort_flag, p.err,
                                   moe::WAIT_LIMIT_NS)) {
                        ok = false;
                        break;
                    }
                    uint8_t* st = tiles + (size_t)stage * C::STAGE_BYTES;
                    const uint32_t fb = smem_u32(&full_bar[stage]);
                    mbar_arrive_expect_tx(fb, bytes);
                    const int kx = kb * BK;
                    if (MODE != 2 && p.a_layout != WEIGHTS_ROWS) {
                        // tile-major weights: one 128 x 64 tile is 16 KB in a row,
                        // seen through the map as 128 rows of 64 elements
#pragma unroll
                        for (int a = 0; a < NUM_A; ++a) {
                            const int rt = (a_row + a * p.a_step) / BM;  // 128-row tile
                            tma_load_2d(smem_u32(st + a * A_TILE_BYTES), ma, fb, 0,
                                        packed_tile(rt, kb, num_kb, p.a_layout) * BM);
                        }
                    } else {
#pragma unroll
                        for (int a = 0; a < NUM_A; ++a)
                            tma_load_2d(smem_u32(st + a * A_TILE_BYTES), ma, fb, kx,
                                        a_row + a * p.a_step);
                    }
                    // the token rows in at most four boxes of 256/128/64/32 rows
                    uint8_t* bdst = st + NUM_A * A_TILE_BYTES;
                    int row = 0;
#pragma unroll
                    for (int lv = 3; lv >= 0; --lv) {
                        const int h = B_BOX << lv;
                        if (h <= BN && (nbox * B_BOX - row) >= h) {
                            tma_load_2d(smem_u32(bdst + row * BK * 2), mb + lv, fb, kx,
                                        t.m_start + row);
                            row += h;
                        }
                    }
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                u = next;
            }
            if (*abort_flag) {
                // let the copies this thread started land before the CTA exits
                for (int i = 0; i < STAGES && issued > 0; ++i, --issued) {
                    if (stage == 0) { stage = STAGES; phase ^= 1; }
                    --stage;
                    const uint64_t t0 = moe::globaltimer_ns();
                    while (!mbar_try_wait(smem_u32(&full_bar[stage]), phase) &&
                           moe::globaltimer_ns() - t0 < 10000000ull) {
                    }
                }
            }
        }
    } else if (U > 0 && warp == 1) {
        // ================= MMA issuer (one thread) =================
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool issued_any = false;
            int slot = 0;
            uint32_t uphase = 0;
            while (!*abort_flag) {
                if (!mbar_wait(smem_u32(&ufull_bar[slot]), uphase, abort_flag, p.err,
                               moe::WAIT_LIMIT_NS))
                    break;
                const int u = ring[slot];
                mbar_arrive(smem_u32(&uempty_bar[slot]));
                if (++slot == RING) { slot = 0; uphase ^= 1; }
                if (u < 0) break;
                const Unit t = decode_unit<BN, C::FEAT>(u / KS, sched);
                const int kb0 = (u % KS) * kb_per, kb1 = min(num_kb, kb0 + kb_per);
                const int bn = (t.n_tok + 15) & ~15;
                const uint32_t idesc = idesc_bf16(bn);
                if (!mbar_wait(smem_u32(&tempty_bar[acc]), acc_phase ^ 1, abort_flag, p.err,
                               moe::WAIT_LIMIT_NS))
                    break;
                tc_fence_after();
                const uint32_t d0 = tmem_base + (uint32_t)(acc * ACC_COLS);
                bool ok = true;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(smem_u32(&full_bar[stage]), phase, abort_flag, p.err,
                                   moe::WAIT_LIMIT_NS)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t st = smem_u32(tiles + (size_t)stage * C::STAGE_BYTES);
                    const uint32_t bsm = st + NUM_A * A_TILE_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint64_t bdesc = smem_desc_sw(bsm + kk * 32);
#pragma unroll
                        for (int a = 0; a < NUM_A; ++a) {
                            const uint32_t dst = C::SPLIT_ACC ? d0 + (uint32_t)(a * ASTRIDE) : d0;
                            // the first product into an accumulator overwrites it
                            const bool first = kb == kb0 && kk == 0 && (C::SPLIT_ACC || a == 0);
                            mma_bf16(dst, smem_desc_sw(st + a * A_TILE_BYTES + kk * 32), bdesc,
                                     idesc, first ? 0u : 1u);
                        }
                    }
                    issued_any = true;
                    mma_commit(smem_u32(&empty_bar[stage]));  // frees the stage when done
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                mma_commit(smem_u32(&tfull_bar[acc]));  // accumulator ready
                if (++acc == ACC) { acc = 0; acc_phase ^= 1; }
            }
            if (issued_any) {
                // wait until every MMA of this thread has completed
                mma_commit(smem_u32(drain_bar));
                const uint64_t t0 = moe::globaltimer_ns();
                while (!mbar_try_wait(smem_u32(drain_bar), 0) &&
                       moe::globaltimer_ns() - t0 < moe::WAIT_LIMIT_NS) {
                }
            }
        }
    } else if (U > 0 && warp >= 2) {
        // ================= epilogue: tensor memory -> global =================
        // warps 2..: quarter q = warp % 4 of the 128 TMEM lanes (hardware
        // rule), the warps of a quarter take its 32-token chunks in turn
        const int q = warp & 3;
        const int sub = (warp - 2) >> 2;
        int acc = 0;
        uint32_t acc_phase = 0;
        int slot = 0;
        uint32_t uphase = 0;
        while (true) {
            int u = -1;
            if (lane == 0 && mbar_wait(smem_u32(&ufull_bar[slot]), uphase, abort_flag, p.err,
                                       moe::WAIT_LIMIT_NS)) {
                u = ring[slot];
                mbar_arrive(smem_u32(&uempty_bar[slot]));
            }
            u = __shfl_sync(0xffffffffu, u, 0);
            if (++slot == RING) { slot = 0; uphase ^= 1; }
            if (u < 0) break;
            const Unit t = decode_unit<BN, C::FEAT>(u / KS, sched);
            if (!mbar_wait(smem_u32(&tfull_bar[acc]), acc_phase, abort_flag, p.err,
                           moe::WAIT_LIMIT_NS))
                break;
            tc_fence_after();
            const int n = t.n0 + q * 32 + lane;
            const bool n_ok = n < p.N_out;
            // router K parts write separate partial sums (KS is 1 elsewhere)
            void* out = t.second ? p.out2
                                 : static_cast<char*>(p.out) +
                                       (size_t)(u % KS) * p.rows * p.N_out * sizeof(float);
            const uint32_t tbase =
                tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * ACC_COLS);
            for (int c0 = 32 * sub; c0 < t.n_tok; c0 += 32 * (EPI1 / 4)) {
                uint32_t g[32];
                tmem_ld32(tbase + c0, g);
                if (MODE == 0) {
                    uint32_t up[32];
                    tmem_ld32(tbase + ASTRIDE + c0, up);
                    tmem_wait_ld();
                    __nv_bfloat16* H = static_cast<__nv_bfloat16*>(out);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int tok = c0 + j;
                        if (n_ok && tok < t.n_tok) {
                            const float gv = __uint_as_float(g[j]);
                            const float uv = __uint_as_float(up[j]);
                            // silu(g) * u; the fast divide's few-ulp error
                            // vanishes in the bf16 rounding of h
                            const float h = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
                            H[(size_t)(t.m_start + tok) * p.N_out + n] = __float2bfloat16_rn(h);
                        }
                    }
                } else if (MODE == 2) {
                    uint32_t mid[32], lo[32];
                    tmem_ld32(tbase + ASTRIDE + c0, mid);
                    tmem_ld32(tbase + 2 * ASTRIDE + c0, lo);
                    tmem_wait_ld();
                    float* Y = static_cast<float*>(out);  // this K part's partial logits
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int tok = c0 + j;
                        if (n_ok && tok < t.n_tok)
                            Y[(size_t)(t.m_start + tok) * p.N_out + n] =
                                __uint_as_float(g[j]) +
                                (__uint_as_float(mid[j]) + __uint_as_float(lo[j]));
                    }
                } else {
                    uint32_t g2[32];
                    tmem_ld32(tbase + ASTRIDE + c0, g2);
                    tmem_wait_ld();
                    const int n2 = n + BM;  // the second feature tile
                    const bool n2_ok = n2 < p.N_out;
                    if (p.comb_out) {
                        // fused combine: weighted adds into the token's output
                        // row.  A 4x4 transpose inside each group of four lanes
                        // gives every lane four consecutive features of one
                        // token, added with one 16-byte vector reduction.
                        const int b = lane & 3;
                        const int nq = n - b;  // the quad's first feature
                        const bool q_ok = nq < p.N_out, q2_ok = nq + BM < p.N_out;
#pragma unroll
                        for (int j0 = 0; j0 < 32; j0 += 4) {
                            float r1[4], r2[4];  // r1[k]: feature nq + ((b + k) & 3)
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                // lane b sends its token j0 + ((b - k) & 3) and
                                // receives feature (b + k) & 3 of token j0 + b
                                const int snd = (b - k) & 3;
                                const int src = (lane & ~3) | ((b + k) & 3);
                                const float v1 = sel4(g, j0, snd), v2 = sel4(g2, j0, snd);
                                r1[k] = k == 0 ? v1 : __shfl_sync(0xffffffffu, v1, src);
                                r2[k] = k == 0 ? v2 : __shfl_sync(0xffffffffu, v2, src);
                            }
                            const int tok = c0 + j0 + b;
                            if (tok < t.n_tok) {
                                const int r = t.m_start + tok;
                                const int tk = t.second ? r : p.row_token[r];
                                const float wgt = t.second ? 1.0f : p.w_row[r];
                                float* row = p.comb_out + (size_t)tk * p.N_out + nq;
                                if (q_ok)
                                    atomicAdd(reinterpret_cast<float4*>(row),
                                              make_float4(wgt * pick4(r1, (0 - b) & 3),
                                                          wgt * pick4(r1, (1 - b) & 3),
                                                          wgt * pick4(r1, (2 - b) & 3),
                                                          wgt * pick4(r1, (3 - b) & 3)));
                                if (q2_ok)
                                    atomicAdd(reinterpret_cast<float4*>(row + BM),
                                              make_float4(wgt * pick4(r2, (0 - b) & 3),
                                                          wgt * pick4(r2, (1 - b) & 3),
                                                          wgt * pick4(r2, (2 - b) & 3),
                                                          wgt * pick4(r2, (3 - b) & 3)));
                            }
                        }
                    } else {
                        float* Y = static_cast<float*>(out);
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const int tok = c0 + j;
                            if (tok < t.n_tok) {
                                float* row = Y + (size_t)(t.m_start + tok) * p.N_out;
                                if (n_ok) row[n] = __uint_as_float(g[j]);
                                if (n2_ok) row[n2] = __uint_as_float(g2[j]);
                            }
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[acc]));
            if (++acc == ACC) { acc = 0; acc_phase ^= 1; }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(TMEM_COLS)
                     : "memory");
    }
}

// ---------------------------------------------------------------- two-SM variant
//
// The same grouped GEMM on CTA pairs (clusters of two CTAs, one per SM of a
// TPC) with tcgen05.mma.cta_group::2: one MMA computes 256 output features x
// N tokens, the leader CTA (rank 0) holding 128 of the features and token
// rows [0, N/2) of the tile, the follower (rank 1) the other 128 features
// and token rows [N/2, N).  Each CTA loads two weight tiles per stage (gate/up:
// its W1 and W3 tiles; down: two 128-feature tiles) and its half of the token
// tile: 48 KB per SM and stage for 256 x 256 x 64 multiply-adds per SM, where
// the one-SM tile loads 64 KB for the same work.  The grouped GEMMs are fed
// at a rate bounded by the bytes each SM keeps in flight (measured: the MMA
// thread of the one-SM kernel waits 20-27% of the time for its stages), so a
// quarter fewer bytes per MMA is what the pair buys.
//
// Roles per CTA as in the one-SM kernel.  The leader's producer claims units
// and publishes each unit index into both CTAs' rings (the follower's
// through distributed shared memory); both producers load into their own
// shared memory, completing on the LEADER's full barrier (the follower's
// copies use the cta_group::2 form that may signal the peer's barrier).  The
// leader's single MMA thread issues the pair's MMAs; its commits arrive on
// both CTAs' stage-empty and accumulator-full barriers (multicast).  Both
// CTAs' epilogue warps drain their own tensor memory and release the
// accumulator on the leader's barrier.  Tensor memory is allocated and freed
// collectively by one warp of each CTA.  Every wait is bounded; both CTAs
// meet at a cluster barrier before tensor memory is freed and they exit.

constexpr int BN2 = 256;  // token tile of a CTA pair (each CTA: 128 rows)
// epilogue warps of a CTA in a pair, per mode: a multiple of 4 (each warp
// reaches one 32-lane quarter of tensor memory; the warps of a quarter take
// its 32-token column chunks in turn).  The accumulator pair fills tensor
// memory, so the MMAs of the next unit wait for the drain: the SwiGLU drain
// (two accumulators, two MUFU operations per output) is latency-bound with
// two warps per scheduler.  Measured (same box, two repetitions, 8 / 12 / 16
// warps): Mixtral routed gate/up 1.171-1.181 / 1.136 / 1.107-1.114 ms, Zipf
// (DeepSeek-V3, T=16384) 5.13 / 5.00 / 4.96-4.97 ms; the down projection's
// fp32 drain gained nothing (Zipf 3.26 / 3.24 / 3.28-3.29 ms).
#ifndef MOE_EPI2_GU
#define MOE_EPI2_GU 16
#endif
#ifndef MOE_EPI2_DN
#define MOE_EPI2_DN 8
#endif
__host__ __device__ constexpr int epi2_warps(int mode) { return mode == 0 ? MOE_EPI2_GU : MOE_EPI2_DN; }
__host__ __device__ constexpr int threads2(int mode) { return 32 * (2 + epi2_warps(mode)); }
static_assert(MOE_EPI2_GU % 4 == 0 && MOE_EPI2_DN % 4 == 0 && MOE_EPI2_GU >= 4 && MOE_EPI2_DN >= 4,
              "whole quarters of tensor memory");

// routed launches with 256-token tiles on CTA pairs (two-SM MMAs)
#ifndef MOE_PAIR_GU
#define MOE_PAIR_GU 1
#endif
#ifndef MOE_PAIR_DN
#define MOE_PAIR_DN 1
#endif
// the shared expert's own dense launches on pairs as well
#ifndef MOE_PAIR_DENSE
#define MOE_PAIR_DENSE 0
#endif
// routed gate/up with fewer rows per expert (weight streaming) on pairs with
// 128-token tiles
#ifndef MOE_PAIR_GU128
#define MOE_PAIR_GU128 0
#endif
// the same with 160-token tiles (80 rows per CTA, exact 64 + 16-row boxes;
// 5 stages of 42 KB per SM, 160 KB of weight tiles in flight instead of the
// one-SM tile's 128 KB).  DeepSeek-V3 prefill, same box, three repetitions:
// routed gate/up 2.267-2.271 ms vs 2.282-2.284 ms on one SM.
#ifndef MOE_PAIR_GU160
#define MOE_PAIR_GU160 1
#endif
// clusters of two CTA pairs sharing the token tile by multicast, for the
// compute-bound routed launches (0: one pair per cluster).  The GPU holds 36
// clusters of four (144 SMs) against 76 pairs (152), so the quarter fewer
// token-tile bytes per SM must pay for 5% fewer SMs.  Measured on one box,
// one pair per cluster vs two: Mixtral down 0.566 -> 0.556 ms, gate/up
// 1.17 -> 1.22 ms (slower); on the power-capped DeepSeek-V3 Zipf(1.2)
// T=16384 layer (~512 rows per expert) the layer took 10.03 ms with one
// pair and 10.07-10.14 ms with two on the down projection.  So the down
// projection only, from 768 rows per expert.
#ifndef MOE_QUAD_GU
#define MOE_QUAD_GU 0
#endif
#ifndef MOE_QUAD_DN
#define MOE_QUAD_DN 1
#endif
// rows per expert from which the down projection takes two pairs per cluster
#ifndef MOE_QUAD_DN_ROWS
#define MOE_QUAD_DN_ROWS 768
#endif
// token tile of the wide (compute-bound) routed gate/up on pairs: 256, or 128
// (double-buffered accumulators, more bytes per MMA)
#ifndef MOE_PAIR_GU_BN
#define MOE_PAIR_GU_BN 256
#endif

template <int MODE, int BN_ = BN2>
struct Cfg2 {
    static constexpr int BN = BN_;
    static constexpr int NUM_A = 2;       // weight tiles per CTA and stage
    static constexpr int HB = BN / 2;     // token rows per CTA
    static constexpr int STAGE_BYTES = NUM_A * A_TILE_BYTES + HB * BK * 2;
    static constexpr int STAGES = SMEM_BUDGET / STAGE_BYTES;
    // TMEM columns between the two accumulators (each starts on a 128-column
    // boundary)
    static constexpr int ASTRIDE = (BN + 127) / 128 * 128;
    static constexpr int ACC_COLS = NUM_A * ASTRIDE;
    static constexpr int ACC_STAGES = TMEM_COLS / ACC_COLS;
    // output features per unit: gate/up, 256 features of W1 and the same of
    // W3; down, 512 features (MMA a: features [n0 + 256a, n0 + 256a + 256),
    // rank r holding the 128 from n0 + 256a + 128r)
    static constexpr int FEAT = MODE == 1 ? 4 * BM : 2 * BM;
    // row distance between a CTA's two weight tiles (gate/up: p.a_step = I)
    static constexpr int A_STEP_DN = 2 * BM;
    static constexpr size_t SMEM = 1024 + (size_t)STAGES * STAGE_BYTES + 256 + sizeof(int) * 2 * (MAX_E + 1);
    static_assert(STAGES >= 2 && ACC_COLS <= TMEM_COLS && ACC_STAGES >= 1, "tile does not fit");
    static_assert(HB % (B_BOX / 2) == 0, "half tile must be whole 16-row boxes");
    static_assert(SMEM + 64 <= (size_t)SMEM_LIMIT, "shared memory over the per-CTA limit");
    // barriers + tensor-memory slot + flags + ring must fit the 256-byte area
    static_assert((2 * STAGES + 2 * ACC_STAGES + 1 + 2 * RING) * 8 + 4 * (5 + RING) <= 256,
                  "barrier area");
};

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// address of the same shared-memory location in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t peer_addr(uint32_t local, uint32_t rank) {
    uint32_t d;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(local), "r"(rank));
    return d;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

// arrive on an mbarrier of another CTA of the cluster (cluster-scope release)
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}

__device__ __forceinline__ void st_remote_u32(uint32_t cluster_addr, int v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// bounded wait with cluster-scope acquire (for barriers that the other CTA
// arrives on, with data it wrote before arriving)
__device__ __noinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity,
                                               volatile int* abort_flag, uint32_t* err,
                                               uint64_t limit_ns) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = moe::globaltimer_ns();
    while (true) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if (*abort_flag) return false;
        if (moe::globaltimer_ns() - t0 > limit_ns) {
            *abort_flag = 1;
            moe::raise_error(err, moe::ERR_TIMEOUT_PIPE);
            return false;
        }
    }
}

// TMA load into this CTA's shared memory completing on a barrier of the
// CTA pair (the leader's), cta_group::2 form
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes."
        "cta_group::2 [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster)
        : "memory");
}

// The same, multicast: the tile lands at this shared-memory offset in every
// CTA of `mask`, and each destination's bytes complete on the barrier at the
// given offset in that destination's pair leader
__device__ __forceinline__ void tma_load_2d_pair_mc(uint32_t dst, const CUtensorMap* map,
                                                    uint32_t bar_cluster, int x, int y,
                                                    uint16_t mask) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes."
        "multicast::cluster.cta_group::2 [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster), "h"(mask)
        : "memory");
}

__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t a, uint64_t b,
                                              uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// commit the leader's MMAs so far to the barrier at this offset in the CTAs
// of `mask` (cluster ranks)
__device__ __forceinline__ void mma_commit_pair(uint32_t bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
        "[%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
}

__device__ __forceinline__ void mma_commit_pair_local(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bar)
                 : "memory");
}

// CL: CTAs per cluster.  2: one pair.  4: two pairs that work on neighbouring
// feature tiles of the same token tile; each half of the token tile is loaded
// once, by the two pairs in turn (alternate k-blocks), and multicast to the
// CTA of the same rank in both pairs, so that each SM loads a quarter of the
// tile per stage instead of half; a stage is released only when both pairs
// have consumed it.
template <int MODE, int BN_ = BN2, int CL = 2>
__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(threads2(MODE), 1)
    grouped_gemm_2sm_kernel(const __grid_constant__ CUtensorMap tm_a,
                            const __grid_constant__ BMaps tm_b,
                            const __grid_constant__ CUtensorMap tm_a2,
                            const __grid_constant__ BMaps tm_b2, const Params p) {
    using C = Cfg2<MODE, BN_>;
    constexpr int EPI2 = epi2_warps(MODE);
    constexpr int STAGES = C::STAGES, NUM_A = C::NUM_A, ACC = C::ACC_STAGES, BN = C::BN;
    constexpr int ACC_COLS = C::ACC_COLS, ASTRIDE = C::ASTRIDE, HB = C::HB;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* tiles = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)STAGES * C::STAGE_BYTES);
    uint64_t* full_bar = bars;                // [STAGES] leader: both CTAs' copies
    uint64_t* empty_bar = bars + STAGES;      // [STAGES] each CTA: its stage is free
    uint64_t* tfull_bar = bars + 2 * STAGES;  // [ACC] each CTA: accumulator ready
    uint64_t* tempty_bar = tfull_bar + ACC;   // [ACC] leader: both CTAs drained it
    uint64_t* drain_bar = tempty_bar + ACC;   // [1]
    uint64_t* ufull_bar = drain_bar + 1;      // [RING] each CTA: unit index published
    uint64_t* uempty_bar = ufull_bar + RING;  // [RING] leader: read by all consumers
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(uempty_bar + RING);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* total_units = reinterpret_cast<int*>(tmem_slot + 2);
    volatile int* ring = reinterpret_cast<volatile int*>(tmem_slot + 5);  // [RING]
    int* mpre = reinterpret_cast<int*>(smem + (size_t)STAGES * C::STAGE_BYTES + 256);
    static_assert(CL == 2 || CL == 4, "one or two CTA pairs per cluster");
    constexpr int FEATC = (CL / 2) * C::FEAT;  // output features per cluster unit
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t crank = cluster_rank();      // rank in the cluster
    const uint32_t rank = crank & 1u;           // rank in the CTA pair
    const uint32_t pl = crank & ~1u;            // the pair leader's cluster rank
    const int cpair = (int)(crank >> 1);        // which pair of the cluster
    const bool leader = rank == 0;              // pair leader (issues the MMAs)
    const bool cleader = crank == 0;            // cluster leader (claims units)
    const int cluster = blockIdx.x / CL, nclusters = gridDim.x / CL;

    // ---- schedule (every CTA computes the same tables) ----
    const int E = p.E;
    const int n_tiles = (p.N_out + FEATC - 1) / FEATC;
    const int U2 = p.rows2 > 0 ? ((p.rows2 + BN - 1) / BN) * n_tiles : 0;
    int* pre_c = mpre;
    int* pre_s = mpre + (E + 1);
    if (warp == 0) build_schedule<BN>(p, n_tiles, U2, pre_c, pre_s, total_units, cleader);
    if (tid == 0) {
        *abort_flag = 0;
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            // released by the commits of every pair leader of the cluster
            mbar_init(smem_u32(&empty_bar[s]), CL / 2);
        }
        for (int a = 0; a < ACC; ++a) {
            mbar_init(smem_u32(&tfull_bar[a]), 1);
            mbar_init(smem_u32(&tempty_bar[a]), 2 * EPI2);
        }
        mbar_init(smem_u32(drain_bar), 1);
        for (int r = 0; r < RING; ++r) {
            mbar_init(smem_u32(&ufull_bar[r]), 1);
            // cluster leader: every pair leader's MMA thread, every CTA's
            // epilogue warps, the other CTAs' producers
            mbar_init(smem_u32(&uempty_bar[r]), CL / 2 + CL * EPI2 + (CL - 1));
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        tma_prefetch_desc(&tm_a);
        for (int i = 0; i < 5; ++i) tma_prefetch_desc(&tm_b.m[i]);
        if (p.rows2 > 0) {
            tma_prefetch_desc(&tm_a2);
            for (int i = 0; i < 5; ++i) tma_prefetch_desc(&tm_b2.m[i]);
        }
    }
    if (warp == 1) {
        // collective: one warp of each CTA of the pair
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // every CTA's barriers initialised before any remote arrive
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int U = total_units[0];

    __shared__ int s_dense_offs[2];
    if (tid == 0) {
        s_dense_offs[0] = 0;
        s_dense_offs[1] = p.rows;
    }
    __syncthreads();
    const int* offs = p.offsets ? p.offsets : s_dense_offs;
    const int num_kb = (p.K + BK - 1) / BK;
    const Sched sched{pre_c, pre_s, offs, E, n_tiles, total_units[0], total_units[1],
                      total_units[2], U2, p.rows2};
    // the pair leader's and the cluster leader's barriers as cluster addresses
    const uint32_t leader_full0 = peer_addr(smem_u32(&full_bar[0]), pl);
    const uint32_t leader_tempty0 = peer_addr(smem_u32(&tempty_bar[0]), pl);
    const uint32_t cl_uempty0 = peer_addr(smem_u32(&uempty_bar[0]), 0);

    if (U > 0 && warp == 0) {
        // ================= TMA producer (one thread per CTA) =================
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int slot = 0;
            uint32_t uphase = 0;
            long issued = 0;
            int u = cluster;
            while (true) {
                if (cleader) {
                    // publish u (or the end, -1) to every CTA of the cluster
                    if (!mbar_wait_cluster(smem_u32(&uempty_bar[slot]), uphase ^ 1, abort_flag,
                                           p.err, moe::WAIT_LIMIT_NS))
                        break;
                    const int v = (u >= U || *abort_flag) ? -1 : u;
                    ring[slot] = v;
#pragma unroll
                    for (int r = 1; r < CL; ++r)
                        st_remote_u32(peer_addr(smem_u32((const void*)&ring[slot]), r), v);
                    mbar_arrive(smem_u32(&ufull_bar[slot]));
#pragma unroll
                    for (int r = 1; r < CL; ++r)
                        mbar_arrive_remote(peer_addr(smem_u32(&ufull_bar[slot]), r));
                    u = v;
                } else {
                    if (!mbar_wait_cluster(smem_u32(&ufull_bar[slot]), uphase, abort_flag, p.err,
                                           moe::WAIT_LIMIT_NS))
                        break;
                    u = ring[slot];
                    mbar_arrive_remote(cl_uempty0 + 8 * slot);
                }
                if (++slot == RING) { slot = 0; uphase ^= 1; }
                if (u < 0) break;
                const int next = cleader ? nclusters + (int)atomicAdd(p.work, 1u) : 0;
                const Unit t = decode_unit<BN, FEATC>(u, sched);
                const CUtensorMap* ma = t.second ? &tm_a2 : &tm_a;
                const CUtensorMap* mb = t.second ? tm_b2.m : tm_b.m;
                const int bn = (t.n_tok + 31) & ~31;  // MMA N: a multiple of 32
                const int hb = bn / 2;                // token rows per CTA, a multiple of 16
                const uint32_t cta_bytes = NUM_A * A_TILE_BYTES + hb * BK * 2;
                const int a_row =
                    (t.second ? 0 : t.e * p.a_rows) + t.n0 + cpair * C::FEAT + (int)rank * BM;
                const int a_step = MODE == 1 ? C::A_STEP_DN : p.a_step;
                const int m0 = t.m_start + (int)rank * hb;
                bool ok = true;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1, abort_flag, p.err,
                                   moe::WAIT_LIMIT_NS)) {
                        ok = false;
                        break;
                    }
                    uint8_t* st = tiles + (size_t)stage * C::STAGE_BYTES;
                    const uint32_t fb = smem_u32(&full_bar[stage]);
                    const uint32_t fb_pair = leader_full0 + 8 * stage;
                    if (leader) mbar_arrive_expect_tx(fb, 2 * cta_bytes);
                    const int kx = kb * BK;
#pragma unroll
                    for (int a = 0; a < NUM_A; ++a) {
                        const int row = a_row + a * a_step;
                        const int x = p.a_layout != WEIGHTS_ROWS ? 0 : kx;
                        const int y = p.a_layout != WEIGHTS_ROWS
                                          ? packed_tile(row / BM, kb, num_kb, p.a_layout) * BM
                                          : row;
                        if (leader)
                            tma_load_2d(smem_u32(st + a * A_TILE_BYTES), ma, fb, x, y);
                        else
                            tma_load_2d_pair(smem_u32(st + a * A_TILE_BYTES), ma, fb_pair, x, y);
                    }
                    uint8_t* bdst = st + NUM_A * A_TILE_BYTES;
                    // two pairs: this CTA's half of the token tile comes from
                    // the pairs in turn, multicast to the same rank of both
                    const bool load_b = CL == 2 || (kb & 1) == cpair;
                    const uint16_t bmask = (uint16_t)((1u << rank) | (1u << (rank + 2)));
                    // exactly hb rows, in boxes of 128/64/32/16 rows (hb / 16
                    // <= 8, so each box size is needed at most once)
                    int row = 0;
#pragma unroll
                    for (int lv = 3; lv >= 0; --lv) {
                        const int h = (B_BOX / 2) << lv;
                        if (load_b && h <= HB && hb - row >= h) {
                            const CUtensorMap* mbox = lv == 0 ? mb + 4 : mb + (lv - 1);
                            if (CL == 4)
                                tma_load_2d_pair_mc(smem_u32(bdst + row * BK * 2), mbox, fb_pair,
                                                    kx, m0 + row, bmask);
                            else if (leader)
                                tma_load_2d(smem_u32(bdst + row * BK * 2), mbox, fb, kx,
                                            m0 + row);
                            else
                                tma_load_2d_pair(smem_u32(bdst + row * BK * 2), mbox, fb_pair,
                                                 kx, m0 + row);
                            row += h;
                        }
                    }
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                if (cleader) u = next;
            }
            if (*abort_flag && leader && CL == 2) {
                // let the copies of this stage ring land before the CTA exits
                for (int i = 0; i < STAGES && issued > 0; ++i, --issued) {
                    if (stage == 0) { stage = STAGES; phase ^= 1; }
                    --stage;
                    const uint64_t t0 = moe::globaltimer_ns();
                    while (!mbar_try_wait(smem_u32(&full_bar[stage]), phase) &&
                           moe::globaltimer_ns() - t0 < 10000000ull) {
                    }
                }
            } else if (*abort_flag && issued > 0) {
                // copies that complete on another CTA's barriers (the follower's,
                // and every multicast one) cannot be waited on here: give any
                // still in flight into shared memory a fixed, bounded time
                // (10 ms) to land
                const uint64_t t0 = moe::globaltimer_ns();
                while (moe::globaltimer_ns() - t0 < 10000000ull) {
                }
            }
        }
    } else if (U > 0 && warp == 1) {
        // ================= MMA issuer (one thread of each pair leader) =================
        if (lane == 0 && leader) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool issued_any = false;
            int slot = 0;
            uint32_t uphase = 0;
            // stage releases go to every CTA of the cluster (each may hold
            // token rows this pair reads); accumulators to this pair's two
            const uint16_t all_mask = (uint16_t)((1u << CL) - 1u);
            const uint16_t pair_mask = (uint16_t)(3u << (2 * cpair));
            while (!*abort_flag) {
                if (!mbar_wait_cluster(smem_u32(&ufull_bar[slot]), uphase, abort_flag, p.err,
                                       moe::WAIT_LIMIT_NS))
                    break;
                const int u = ring[slot];
                if (cleader)
                    mbar_arrive(smem_u32(&uempty_bar[slot]));
                else
                    mbar_arrive_remote(cl_uempty0 + 8 * slot);
                if (++slot == RING) { slot = 0; uphase ^= 1; }
                if (u < 0) break;
                const Unit t = decode_unit<BN, FEATC>(u, sched);
                const int bn = (t.n_tok + 31) & ~31;
                // M = 256 over the pair (bits 24-28: M / 16), N = bn
                const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) |
                                       ((uint32_t)(bn >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);
                if (!mbar_wait_cluster(smem_u32(&tempty_bar[acc]), acc_phase ^ 1, abort_flag, p.err,
                                       moe::WAIT_LIMIT_NS))
                    break;
                tc_fence_after();
                const uint32_t d0 = tmem_base + (uint32_t)(acc * ACC_COLS);
                bool ok = true;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(smem_u32(&full_bar[stage]), phase, abort_flag, p.err,
                                   moe::WAIT_LIMIT_NS)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t st = smem_u32(tiles + (size_t)stage * C::STAGE_BYTES);
                    const uint32_t bsm = st + NUM_A * A_TILE_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint64_t bdesc = smem_desc_sw(bsm + kk * 32);
#pragma unroll
                        for (int a = 0; a < NUM_A; ++a)
                            mma_bf16_pair(d0 + (uint32_t)(a * ASTRIDE),
                                          smem_desc_sw(st + a * A_TILE_BYTES + kk * 32), bdesc, idesc,
                                          (kb == 0 && kk == 0) ? 0u : 1u);
                    }
                    issued_any = true;
                    mma_commit_pair(smem_u32(&empty_bar[stage]), all_mask);  // stage consumed
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                mma_commit_pair(smem_u32(&tfull_bar[acc]), pair_mask);  // accumulator ready
                if (++acc == ACC) { acc = 0; acc_phase ^= 1; }
            }
            if (issued_any) {
                mma_commit_pair_local(smem_u32(drain_bar));
                const uint64_t t0 = moe::globaltimer_ns();
                while (!mbar_try_wait(smem_u32(drain_bar), 0) &&
                       moe::globaltimer_ns() - t0 < moe::WAIT_LIMIT_NS) {
                }
            }
        }
    } else if (U > 0 && warp >= 2) {
        // ================= epilogue: this CTA's tensor memory -> global =================
        const int q = warp & 3;
        const int sub = (warp - 2) >> 2;
        int acc = 0;
        uint32_t acc_phase = 0;
        int slot = 0;
        uint32_t uphase = 0;
        while (true) {
            int u = -1;
            if (lane == 0 && mbar_wait_cluster(smem_u32(&ufull_bar[slot]), uphase, abort_flag, p.err,
                                               moe::WAIT_LIMIT_NS)) {
                u = ring[slot];
                if (cleader)
                    mbar_arrive(smem_u32(&uempty_bar[slot]));
                else
                    mbar_arrive_remote(cl_uempty0 + 8 * slot);
            }
            u = __shfl_sync(0xffffffffu, u, 0);
            if (++slot == RING) { slot = 0; uphase ^= 1; }
            if (u < 0) break;
            const Unit t = decode_unit<BN, FEATC>(u, sched);
            if (!mbar_wait(smem_u32(&tfull_bar[acc]), acc_phase, abort_flag, p.err,
                           moe::WAIT_LIMIT_NS))
                break;
            tc_fence_after();
            const int n = t.n0 + cpair * C::FEAT + (int)rank * BM + q * 32 + lane;
            const bool n_ok = n < p.N_out;
            void* out = t.second ? p.out2 : p.out;
            const uint32_t tbase =
                tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * ACC_COLS);
            for (int c0 = 32 * sub; c0 < t.n_tok; c0 += 32 * (EPI2 / 4)) {
                uint32_t g[32];
                tmem_ld32(tbase + c0, g);
                if (MODE == 0) {
                    uint32_t up[32];
                    tmem_ld32(tbase + ASTRIDE + c0, up);
                    tmem_wait_ld();
                    __nv_bfloat16* H = static_cast<__nv_bfloat16*>(out);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int tok = c0 + j;
                        if (n_ok && tok < t.n_tok) {
                            const float gv = __uint_as_float(g[j]);
                            const float uv = __uint_as_float(up[j]);
                            const float h = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
                            H[(size_t)(t.m_start + tok) * p.N_out + n] = __float2bfloat16_rn(h);
                        }
                    }
                } else {
                    uint32_t g2[32];
                    tmem_ld32(tbase + ASTRIDE + c0, g2);
                    tmem_wait_ld();
                    const int n2 = n + 2 * BM;  // the second MMA's features
                    const bool n2_ok = n2 < p.N_out;
                    float* Y = static_cast<float*>(out);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int tok = c0 + j;
                        if (tok < t.n_tok) {
                            float* row = Y + (size_t)(t.m_start + tok) * p.N_out;
                            if (n_ok) row[n] = __uint_as_float(g[j]);
                            if (n2_ok) row[n2] = __uint_as_float(g2[j]);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (leader)
                    mbar_arrive(smem_u32(&tempty_bar[acc]));
                else
                    mbar_arrive_remote(leader_tempty0 + 8 * acc);
            }
            if (++acc == ACC) { acc = 0; acc_phase ^= 1; }
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // the pair's MMAs and remote arrivals are done
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(TMEM_COLS)
                     : "memory");
    }
}

// Self-test of the bounded pipeline wait: an mbarrier that nothing arrives
// on; the wait must give up and report a timeout.
__global__ void mbar_probe_kernel(uint64_t limit_ns, uint32_t* err) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(smem_u32(&bar), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, &abort_flag, err, limit_ns);
}

// Self-test of the CTA pair's bounded cluster-scope wait: in a cluster of
// two, each CTA waits (acquire.cluster, as the pair kernel's ring and
// accumulator waits do) on a barrier that the peer would arrive on but never
// does; the waits must give up and report a timeout, then both CTAs meet at
// the cluster barrier and exit.
__global__ void __cluster_dims__(2, 1, 1) cluster_probe_kernel(uint64_t limit_ns, uint32_t* err) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(smem_u32(&bar), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    cluster_sync_all();
    if (threadIdx.x == 0) mbar_wait_cluster(smem_u32(&bar), 0, &abort_flag, err, limit_ns);
    __syncthreads();
    cluster_sync_all();
}

// Router weight split: w = hi + mid + lo with each term the bf16 rounding of
// what the previous terms leave (every subtraction is exact in fp32; the sum
// is exact for |w| >= 2^-110, below which bf16's spacing drops the last bits).
__global__ void split_weight_kernel(const float* __restrict__ w, long n,
                                    __nv_bfloat16* __restrict__ out) {
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n;
         i += (long)gridDim.x * blockDim.x) {
        const float v = w[i];
        const __nv_bfloat16 hi = __float2bfloat16_rn(v);
        const float r1 = v - __bfloat162float(hi);
        const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
        const float r2 = r1 - __bfloat162float(mid);
        out[i] = hi;
        out[n + i] = mid;
        out[2 * n + i] = __float2bfloat16_rn(r2);
    }
}

// Expert weights [E, rows, K] into the tile-major layouts (see WEIGHTS_*):
// one thread per 16-byte vector of the output, read from its source row.
__global__ void pack_weights_kernel(const uint4* __restrict__ w, long n_vec, int rows, int K,
                                    int pairs, uint4* __restrict__ out) {
    const int kv = K / 8, KB = K / BK;
    const long tiles_per_expert = (long)(rows / BM) * KB;
    for (long v = blockIdx.x * (long)blockDim.x + threadIdx.x; v < n_vec;
         v += (long)gridDim.x * blockDim.x) {
        const long tile = v / (BM * BK / 8);
        const int in = (int)(v % (BM * BK / 8));  // 128 rows of 8 vectors
        const long e = tile / tiles_per_expert;
        const int t = (int)(tile % tiles_per_expert);
        int rt, kb;
        if (pairs) {
            const int pr = t / (2 * KB), rem = t % (2 * KB);
            kb = rem >> 1;
            rt = 2 * pr + (rem & 1);
        } else {
            rt = t / KB;
            kb = t % KB;
        }
        const long src_row = e * rows + (long)rt * BM + in / 8;
        out[v] = w[src_row * kv + (long)kb * 8 + in % 8];
    }
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
    return fn;
}

// 2D bf16 tensor map over a row-major [rows, cols] matrix, box {64, box_rows},
// 128-byte swizzle, zero fill outside.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     SWZ_BYTES == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_bmaps(BMaps* m, const void* base, uint64_t rows, uint64_t cols) {
    for (int i = 0; i < 4; ++i)
        if (!make_map(&m->m[i], base, rows, cols, (uint32_t)(B_BOX << i))) return false;
    return make_map(&m->m[4], base, rows, cols, (uint32_t)(B_BOX / 2));
}

#ifndef MOE_BALANCED_GRID
#define MOE_BALANCED_GRID 1
#endif

// units: the launch's work units when the host knows them (dense problems,
// the router), else 0.  With a known count the grid is the smallest one that
// still needs the same number of waves (256 equal units: 128 CTAs in two
// waves rather than 152 CTAs in 1.7), which leaves the other SMs to kernels
// on other streams at no cost to this launch.
template <int MODE, int BN>
int launch(const CUtensorMap& a, const BMaps& b, const CUtensorMap& a2, const BMaps& b2,
           const Params& p, cudaStream_t s, long long units = 0) {
    // the shared-memory limit is a per-device attribute of the kernel: set it
    // once per device (setting it twice is harmless, so no lock is needed)
    static bool attr_done[64] = {};
    const size_t smem = Cfg<MODE, BN>::SMEM;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= 64 || !attr_done[dev]) {
        if (cudaFuncSetAttribute(grouped_gemm_tc_kernel<MODE, BN>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess)
            return MOE_ERR_CUDA;
        if (dev >= 0 && dev < 64) attr_done[dev] = true;
    }
    const int sms = moe_host::num_sms();
    int grid = sms;
    if (MOE_BALANCED_GRID && units > 0) {
        const long long waves = (units + sms - 1) / sms;
        grid = (int)((units + waves - 1) / waves);
    }
    grouped_gemm_tc_kernel<MODE, BN><<<grid, threads1(MODE), smem, s>>>(a, b, a2, b2, p);
    return moe_host::launch_status();
}

// Two-CTA clusters of the pair kernel that the current device can hold at
// once (queried once per device; 0 if none or the query fails, in which case
// the one-SM kernel runs instead).  The kernel's shared-memory limit is set
// on the same first use.
template <int MODE, int BN = BN2, int CL = 2>
int pair_capacity() {
    static int cap[64];
    static bool done[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (!done[dev]) {
        const size_t smem = Cfg2<MODE, BN>::SMEM;
        int n = 0;
        if (cudaFuncSetAttribute(grouped_gemm_2sm_kernel<MODE, BN, CL>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) == cudaSuccess) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(CL * std::max(1, moe_host::num_sms() / CL));
            cfg.blockDim = dim3(threads2(MODE));
            cfg.dynamicSmemBytes = smem;
            // the cluster size (CL) is the kernel's own (__cluster_dims__)
            if (cudaOccupancyMaxActiveClusters(&n, grouped_gemm_2sm_kernel<MODE, BN, CL>, &cfg) !=
                cudaSuccess)
                n = 0;
        }
        cudaGetLastError();  // a refused query leaves no error behind
        cap[dev] = n;
        done[dev] = true;
    }
    return cap[dev];
}

// The two-SM kernel over CTA pairs: as many pairs as the device holds at once
// (one per TPC: half the SMs), or the smallest pair count with the same
// number of waves when the host knows the units.
template <int MODE, int BN = BN2, int CL = 2>
int launch_pair(const CUtensorMap& a, const BMaps& b, const CUtensorMap& a2, const BMaps& b2,
                const Params& p, cudaStream_t s, long long units = 0) {
    const size_t smem = Cfg2<MODE, BN>::SMEM;
    int clusters = std::min(std::max(1, moe_host::num_sms() / CL), pair_capacity<MODE, BN, CL>());
    if (clusters < 1) return MOE_ERR_UNSUPPORTED;
    if (MOE_BALANCED_GRID && units > 0) {
        const long long waves = (units + clusters - 1) / clusters;
        clusters = (int)((units + waves - 1) / waves);
    }
    grouped_gemm_2sm_kernel<MODE, BN, CL><<<CL * clusters, threads2(MODE), smem, s>>>(a, b, a2, b2,
                                                                                      p);
    return moe_host::launch_status();
}

}  // namespace

namespace moe_tc {

// A weight matrix of `rows` rows and K columns (bf16) in the given layout.
bool make_weight_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t K, bool packed) {
    if (!packed) return make_map(m, base, rows, K, BM);
    // tile-major: every 64 columns of every row become one 128-byte row
    return make_map(m, base, rows * ((K + BK - 1) / BK), BK, BM);
}

// Both GEMMs of the SwiGLU FFN over bf16 rows; offsets == NULL means one
// segment [0, rows) with expert 0 (dense).  When sh is given, the shared
// expert (dense over sh->x, I_sh == I) runs inside the same launches (those
// its in_gate_up / in_down flags name).  When fc is given, the down launch
// adds its results into fc->out instead of writing y.  packed: the weights
// (and the shared expert's) are in the tile-major layouts of
// moe_pack_expert_weights.
int grouped_ffn_bf16(const void* x_perm, const int32_t* offsets, int E, int rows, int d, int I,
                     const void* w13, const void* w2, float* y, void* h, uint32_t* err,
                     unsigned* work, cudaStream_t s, cudaEvent_t between,
                     const SharedExpert* sh, const FusedCombine* fc, int parts,
                     cudaEvent_t before_down, bool packed, int heur_E) {
    if (E > MAX_E) return MOE_ERR_UNSUPPORTED;
    const int HE = heur_E > 0 ? heur_E : E;  // experts the rows are averaged over
    CUtensorMap a1, a2, a1s, a2s;
    BMaps b1, b2, b1s, b2s;
    if (!make_weight_map(&a1, w13, (uint64_t)E * 2 * I, d, packed) ||
        !make_bmaps(&b1, x_perm, rows, d) ||
        !make_weight_map(&a2, w2, (uint64_t)E * d, I, packed) || !make_bmaps(&b2, h, rows, I))
        return MOE_ERR_CUDA;
    const bool two = sh != nullptr && sh->T > 0;
    if (two) {
        if (!make_weight_map(&a1s, sh->w13, 2ull * I, d, packed) ||
            !make_bmaps(&b1s, sh->x, sh->T, d) ||
            !make_weight_map(&a2s, sh->w2, (uint64_t)d, I, packed) ||
            !make_bmaps(&b2s, sh->h, sh->T, I))
            return MOE_ERR_CUDA;
    } else {
        a1s = a1; b1s = b1; a2s = a2; b2s = b2;
    }
    const bool two_gu = two && sh->in_gate_up, two_dn = two && sh->in_down;
    Params p1{offsets, E,   rows, d, I, 2 * I, I, h, err, 0, two_gu ? sh->T : 0,
              two_gu ? sh->h : nullptr, work, 1, nullptr, nullptr, nullptr,
              packed ? WEIGHTS_TILES : WEIGHTS_ROWS};
    Params p2{offsets, E, rows, I, d, d, BM, y, err, 0, two_dn ? sh->T : 0,
              two_dn ? sh->y : nullptr, work + 1, 1, fc ? fc->out : nullptr,
              fc ? fc->row_token : nullptr, fc ? fc->w_row : nullptr,
              packed ? WEIGHTS_TILE_PAIRS : WEIGHTS_ROWS};
    // Token tile per launch, from the average rows per expert (the host does
    // not see the device-side offsets).  A weight-streaming GEMM runs at the
    // rate (k-blocks in flight per SM) / (load latency), so the tile trades
    // stages against passes over the weights: every token tile of an expert
    // is one more pass over its weight tiles (from L2 after the first).
    //   gate/up: 160 rows below 384 rows per expert (one-SM tile: 4 stages
    //            of 52 KB; on CTA pairs 5 of 42 KB per SM; one pass for
    //            experts of up to 160 rows; single-buffered accumulator
    //            pair), else 256.  Measured on DeepSeek-V3 prefill (one SM,
    //            row-major weights): 2.38 ms with 160, 2.45 ms with 128 (4
    //            stages, double-buffered), 2.85 ms with 256 (3 stages);
    //   down:    128 only below 32 rows per expert (decode), else 256
    //            (prefill: 1.57 ms vs 2.01 ms with 128).
    const bool gu_wide = (long long)rows >= (long long)MOE_GU_WIDE_ROWS * HE;
    const bool dn_wide = (long long)rows >= (long long)MOE_DN_WIDE_ROWS * HE;
    // a few rows per expert (decode): 32-token tiles, whose 36 KB stages let
    // each SM keep 6 weight-tile pairs in flight instead of 4
    const bool narrow = MOE_NARROW_ROWS > 0 && (long long)rows < (long long)MOE_NARROW_ROWS * HE;
    // a dense problem alone (offsets == NULL, no second problem): the unit
    // counts are known here
    const bool dense = offsets == nullptr;
    const int gu_bn = gu_wide ? 256 : narrow ? 32 : MOE_GU_BN;
    const int dn_bn = dn_wide ? MOE_DN_BN : narrow ? 32 : 128;
    const long long gu_units =
        dense && !two_gu ? (long long)((rows + gu_bn - 1) / gu_bn) * ((I + BM - 1) / BM) : 0;
    const long long dn_units =
        dense && !two_dn ? (long long)((rows + dn_bn - 1) / dn_bn) * ((d + 2 * BM - 1) / (2 * BM)) : 0;
    // routed launches with 256-token tiles may run on CTA pairs (two-SM
    // MMAs); not the fused combine's down projection, whose vector-reduction
    // epilogue is written for the one-SM tile
    const bool gu_pair = MOE_PAIR_GU && gu_wide && (!dense || MOE_PAIR_DENSE) &&
                         (MOE_PAIR_GU_BN == 128 ? pair_capacity<0, 128>() : pair_capacity<0>()) > 0;
    const bool dn_pair = MOE_PAIR_DN && dn_wide && MOE_DN_BN == 256 && !fc &&
                         (!dense || MOE_PAIR_DENSE) && pair_capacity<1>() > 0;
    // two pairs per cluster sharing the token tile (down projection from
    // MOE_QUAD_DN_ROWS rows per expert)
    const bool gu_quad = MOE_QUAD_GU && gu_pair && MOE_PAIR_GU_BN == 256 &&
                         pair_capacity<0, BN2, 4>() > 0;
    const bool dn_quad = MOE_QUAD_DN && dn_pair && (long long)rows >= (long long)MOE_QUAD_DN_ROWS * HE &&
                         pair_capacity<1, BN2, 4>() > 0;
    // a dense problem alone: its units on pairs (256 features x 256 tokens for
    // gate/up, 512 x 256 for down), for the balanced grid
    const long long gu_pair_units =
        dense && !two_gu ? (long long)((rows + 255) / 256) * ((I + 255) / 256) : 0;
    const long long dn_pair_units =
        dense && !two_dn ? (long long)((rows + 255) / 256) * ((d + 511) / 512) : 0;
    // routed gate/up below the wide threshold (and above the narrow one):
    // 160-token tiles on CTA pairs (or, off by default, 128-token ones)
    // instead of 160-token one-SM tiles
    const bool gu_pair128 =
        MOE_PAIR_GU128 && !gu_wide && !narrow && !dense && pair_capacity<0, 128>() > 0;
    const bool gu_pair160 = MOE_PAIR_GU160 && !gu_wide && !narrow && !dense && MOE_GU_BN == 160 &&
                            pair_capacity<0, 160>() > 0;
    int rc = MOE_OK;
    if (parts & 1)
        rc = gu_pair128 ? launch_pair<0, 128>(a1, b1, a1s, b1s, p1, s)
             : gu_pair160 ? launch_pair<0, 160>(a1, b1, a1s, b1s, p1, s)
             : gu_quad ? launch_pair<0, BN2, 4>(a1, b1, a1s, b1s, p1, s)
             : gu_pair ? (MOE_PAIR_GU_BN == 128 ? launch_pair<0, 128>(a1, b1, a1s, b1s, p1, s)
                                                : launch_pair<0>(a1, b1, a1s, b1s, p1, s,
                                                                 gu_pair_units))
             : gu_wide ? launch<0, 256>(a1, b1, a1s, b1s, p1, s, gu_units)
             : narrow  ? launch<0, 32>(a1, b1, a1s, b1s, p1, s, gu_units)
                       : launch<0, MOE_GU_BN>(a1, b1, a1s, b1s, p1, s, gu_units);
    if (rc != MOE_OK) return rc;
    if (between && cudaEventRecord(between, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (!(parts & 2)) return MOE_OK;
    if (before_down && cudaStreamWaitEvent(s, before_down, 0) != cudaSuccess) return MOE_ERR_CUDA;
    if (dn_quad) return launch_pair<1, BN2, 4>(a2, b2, a2s, b2s, p2, s);
    if (dn_pair) return launch_pair<1>(a2, b2, a2s, b2s, p2, s, dn_pair_units);
    if (narrow && !dn_wide) return launch<1, 32>(a2, b2, a2s, b2s, p2, s, dn_units);
    return dn_wide ? launch<1, MOE_DN_BN>(a2, b2, a2s, b2s, p2, s, dn_units)
                   : launch<1, 128>(a2, b2, a2s, b2s, p2, s, dn_units);
}

int pack_weights(const void* w, int E, int rows, int K, bool pairs, void* out, cudaStream_t s) {
    const long n_vec = (long)E * rows * (K / 8);
    if (n_vec == 0) return MOE_OK;
    const int blocks = (int)std::min<long>((n_vec + 255) / 256, 8L * moe_host::num_sms());
    pack_weights_kernel<<<blocks, 256, 0, s>>>(static_cast<const uint4*>(w), n_vec, rows, K,
                                               pairs ? 1 : 0, static_cast<uint4*>(out));
    return moe_host::launch_status();
}

int mbar_probe(uint64_t limit_ns, uint32_t* err, cudaStream_t s) {
    mbar_probe_kernel<<<1, 32, 0, s>>>(limit_ns, err);
    return moe_host::launch_status();
}

int cluster_probe(uint64_t limit_ns, uint32_t* err, cudaStream_t s) {
    cluster_probe_kernel<<<2, 32, 0, s>>>(limit_ns, err);
    return moe_host::launch_status();
}

// Router: weight split (3 bf16 terms) + partial logits of up to MAX_KSPLIT
// K parts, each [T,E] fp32.
constexpr int MAX_KSPLIT = 8;
size_t router_ws_bytes(int T, int E, int d) {
    const size_t split = ((size_t)3 * E * d * 2 + 255) / 256 * 256;
    return split + (size_t)MAX_KSPLIT * T * E * 4;
}

// Partial logits of x W^T (fp32 accumulate) with W split into three bf16
// terms: K is cut into *ksplit parts (chosen so that the units fill the SMs),
// part ks written to partial + ks * T * E.  ws: router_ws_bytes(T, E, d).
int split_router_weight(const float* w_router, int E, int d, void* out, cudaStream_t s) {
    const long n = (long)E * d;
    const int blocks = (int)std::min<long>((n + 255) / 256, 4L * moe_host::num_sms());
    split_weight_kernel<<<blocks, 256, 0, s>>>(w_router, n, static_cast<__nv_bfloat16*>(out));
    return moe_host::launch_status();
}

int router_bf16(const void* x, const float* w_router, int T, int d, int E, void* ws,
                uint32_t* err, unsigned* work, float** partial, int* ksplit, cudaStream_t s,
                cudaEvent_t after_split, const void* presplit) {
    const size_t split = ((size_t)3 * E * d * 2 + 255) / 256 * 256;
    float* part = reinterpret_cast<float*>(static_cast<char*>(ws) + split);
    const void* wsplit = presplit;
    if (!wsplit) {
        wsplit = ws;
        const int rc = split_router_weight(w_router, E, d, ws, s);
        if (rc != MOE_OK) return rc;
    }
    if (after_split && cudaEventRecord(after_split, s) != cudaSuccess) return MOE_ERR_CUDA;
    CUtensorMap a;
    BMaps b;
    if (!make_map(&a, wsplit, 3ull * E, d, BM) || !make_bmaps(&b, x, T, d)) return MOE_ERR_CUDA;
    constexpr int RBN = 128;
    const int units = ((T + RBN - 1) / RBN) * ((E + BM - 1) / BM);
    const int num_kb = (d + BK - 1) / BK;
    int ks = std::max(1, std::min(MAX_KSPLIT, moe_host::num_sms() / std::max(1, units)));
    while (ks > 1 && num_kb / ks < 8) --ks;  // keep each part at least 8 k-blocks long
    Params p{nullptr, 1, T, d, E, 0, E, part, err, 0, 0, nullptr, work, ks};
    *partial = part;
    *ksplit = ks;
    return launch<2, RBN>(a, b, a, b, p, s, (long long)units * ks);
}

}  // namespace moe_tc
