// dispatch_noalloc.cu -- moe_dispatch for callers that cannot allocate.
//
// Some callers may not allocate device memory at all while they run: a
// serving runtime that fixed its memory pool at start-up and forbids
// allocation on the request path, a plug-in hosted by another framework that
// owns the allocator, or code certified to allocate only at initialisation.
// They cannot provide the scratch workspace that moe_dispatch asks for, so
// this variant keeps that scratch in a fixed array in the library's own
// device memory instead.  The array is a file-scope __device__ variable: every
// GPU that loads the library holds it until the process exits.
//
// Host code must not use the array's name as a device address (on the host it
// names a host-side stand-in).  The device address is looked up with
// cudaGetSymbolAddress, with the device current, on the first call made on
// that device, and cached together with the identity of the CUDA context it
// was looked up in.  If that context is later replaced (cudaDeviceReset, or
// the primary context released and created again), the module is loaded
// anew and the array may move: the next call sees a different context and
// looks the address up again instead of using a stale one.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace {

// Scratch capacity: MOE_DISPATCH_NOALLOC_MAX_SLOTS slots (16384 tokens x 8,
// the largest workload measured here) over up to 1024 experts need 0.77 MiB.
constexpr size_t NOALLOC_SCRATCH_BYTES = 1u << 20;  // 1 MiB
constexpr size_t NOALLOC_ERR_BYTES = 256;           // error word, then dispatch scratch
constexpr int MAX_DEVICES = 64;

static __device__ __align__(256) unsigned char g_dispatch_scratch[NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
struct CachedAddr {
    unsigned long long ctx_id;  // context the address belongs to (0 = none yet)
    void* addr;
};
CachedAddr g_scratch_addr[MAX_DEVICES] = {};

// Unique id of the calling thread's current CUDA context (driver API through
// the runtime's entry-point query; context ids are never reused, unlike
// context handles).  Returns false if there is no current context.
bool current_context_id(unsigned long long* id) {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static bool resolved = false;
    if (!resolved) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
        resolved = true;
    }
    if (!get_current || !get_id) return false;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch array in the current device's current
// context: looked up on the first call per device, and again whenever the
// context has changed since.  Returns nullptr if the lookup fails.
void* scratch_address() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    unsigned long long id = 0;
    const bool have_id = current_context_id(&id);
    CachedAddr& c = g_scratch_addr[dev];
    if (have_id && c.addr && c.ctx_id == id) return c.addr;
    void* p = nullptr;
    // (creates the device's primary context first if the thread has none)
    if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess) return nullptr;
    if (!have_id && !current_context_id(&id)) id = 0;  // no id: not cached
    c.ctx_id = id;
    c.addr = id ? p : nullptr;
    return p;
}

}  // namespace

extern "C" {

int moe_dispatch_noalloc(const int32_t* topk_idx, const void* x, int dtype, int T, int d, int k,
                         int E, int32_t* counts, int32_t* offsets, int32_t* slot_to_row,
                         int32_t* row_to_token, void* x_perm, uint32_t* device_error,
                         void* stream) {
    if (k < 1 || k > 32 || E < 1) return MOE_ERR_INVALID_ARG;
    if (T < 0 || d < 8 || d % 8 != 0 || (dtype != MOE_F32 && dtype != MOE_BF16))
        return MOE_ERR_INVALID_ARG;
    // sizes beyond the fixed scratch array are refused, not truncated
    if (E > 1024 || (long long)T * k > MOE_DISPATCH_NOALLOC_MAX_SLOTS) return MOE_ERR_UNSUPPORTED;
    if (moe_launch::dispatch_ws_bytes(T, k, E) > NOALLOC_SCRATCH_BYTES - NOALLOC_ERR_BYTES)
        return MOE_ERR_UNSUPPORTED;
    if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!topk_idx || !slot_to_row || !row_to_token)) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (x_perm != nullptr) != (x != nullptr)) return MOE_ERR_INVALID_ARG;
    if (x && (!moe_host::aligned16(x) || !moe_host::aligned16(x_perm))) return MOE_ERR_INVALID_ARG;
    char* scratch = static_cast<char*>(scratch_address());
    if (!scratch) return MOE_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t* err = reinterpret_cast<uint32_t*>(scratch);
    // the array keeps the previous call's contents: the error word starts at
    // zero here; the dispatch launcher clears its own ticket and flags
    if (cudaMemsetAsync(err, 0, sizeof(uint32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
    int rc = MOE_OK;
    if (T == 0) {
        if (cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s) != cudaSuccess ||
            cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s) != cudaSuccess)
            rc = MOE_ERR_CUDA;
    } else {
        rc = moe_launch::dispatch(topk_idx, x, dtype, T, d, k, E, counts, offsets, slot_to_row,
                                  row_to_token, x_perm, scratch + NOALLOC_ERR_BYTES, err, s);
    }
    if (rc == MOE_OK && device_error &&
        cudaMemcpyAsync(device_error, err, sizeof(uint32_t), cudaMemcpyDeviceToDevice, s) !=
            cudaSuccess)
        rc = MOE_ERR_CUDA;
    return rc;
}

}  // extern "C"
