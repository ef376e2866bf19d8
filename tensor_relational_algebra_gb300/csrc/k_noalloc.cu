// Squared-distance join + aggregate without a caller-provided workspace.
//
// The squared-distance EinSum sum_j (x - y)^2 runs as ||x||^2 + ||y||^2 - 2 x.y and
// keeps the per-row and per-column norms, and one guard word per 128 x 128 output tile
// (tiles where the expansion cancelled, recomputed in the direct form), in device scratch.  ein_execute takes that
// scratch from the caller; this entry point takes it instead from a fixed array that
// lives in the library's own device memory, so the caller never has to allocate.
// That is for callers that cannot call cudaMalloc or any allocating routine on the
// path: a host program whose device memory is entirely owned by another allocator
// or budgeted up front, a plugin inside a framework that forbids device allocation,
// or a latency-critical path that must not pay for an allocation (and the device
// synchronisation cudaFree implies).
//
// The array is a file-scope __device__ variable: every GPU that loads libtra.so holds
// its kTraNoallocScratchBytes until the process exits.  Host code cannot use the
// array's name as a device address, so the address is fetched with cudaGetSymbolAddress
// on the first call made while a device is current, and cached for that device and its
// current context: after cudaDeviceReset (a new context, the module loaded again) the
// next call looks the address up again.  All calls share the one array: two calls whose
// kernels overlap on the GPU (different streams, no ordering between them) race on it.
// The norm kernels write every norm, and every tile's CTA writes its guard word, before
// anything reads them, so nothing needs clearing between calls.
#include <cstring>
#include <mutex>

#include "plan.h"

namespace tra {
namespace {

constexpr size_t kTraNoallocScratchBytes = size_t(1) << 20;  // 1 MiB: row + column norms

__device__ __align__(256) unsigned char g_noalloc_scratch[kTraNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {};
void* g_noalloc_ctx[kMaxDevices] = {};  // the context the cached address belongs to

// cuCtxGetCurrent through the runtime's entry-point query (no link against libcuda)
using CtxGetCurrentFn = int (*)(void**);
CtxGetCurrentFn ctx_get_current() {
    static CtxGetCurrentFn fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<CtxGetCurrentFn>(f);
        return static_cast<CtxGetCurrentFn>(nullptr);
    }();
    return fn;
}

// Device address of the scratch array on the current device: looked up on the first call for
// a device, and again whenever that device's current context has changed since.
int scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(TRA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(TRA_ERR_UNSUPPORTED, "device ordinal %d above %d", dev, kMaxDevices);
    const CtxGetCurrentFn get = ctx_get_current();
    if (!get) return fail(TRA_ERR_CUDA, "cuCtxGetCurrent unavailable");
    // the context current on this thread (null before the runtime has set one up here)
    void* ctx = nullptr;
    if (get(&ctx) != 0) ctx = nullptr;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!ctx || !g_noalloc_ptr[dev] || g_noalloc_ctx[dev] != ctx) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // sets up the device's context if needed
        if (e != cudaSuccess || !p)
            return fail(TRA_ERR_CUDA, "cudaGetSymbolAddress of the scratch array: %s", cudaGetErrorString(e));
        if (get(&ctx) != 0 || !ctx) return fail(TRA_ERR_CUDA, "no current context after the address lookup");
        g_noalloc_ptr[dev] = p;
        g_noalloc_ctx[dev] = ctx;
    }
    *out = g_noalloc_ptr[dev];
    return TRA_OK;
}

}  // namespace
}  // namespace tra

using namespace tra;

extern "C" int ein_execute_sqdist_noalloc(tra_plan_t plan, const void* in0, const void* in1, void* out,
                                          tra_stream_t stream) {
    clear_error();
    if (!plan) return fail(TRA_ERR_ARG, "NULL plan");
    const Plan& p = *reinterpret_cast<const Plan*>(plan);
    // a squared distance with an empty range needs no scratch: ein_execute fills it (or has
    // nothing to write) with the same argument rules
    if (p.op == kSqdiff && p.agg == kSum && !p.unary && (p.kernel == TRA_KERNEL_EMPTY || p.kernel == TRA_KERNEL_FILL))
        return ein_execute(plan, in0, in1, out, nullptr, 0, stream);
    if (!in0 || !in1 || !out) return fail(TRA_ERR_ARG, "NULL input or output");
    if (p.kernel != TRA_KERNEL_SEMIRING_F32 || p.op != kSqdiff || p.agg != kSum || !p.sqdiff_expand)
        return fail(TRA_ERR_UNSUPPORTED,
                    "ein_execute_sqdist_noalloc runs only fp32 squared-distance plans in the expanded form");
    if (p.ws_bytes > kTraNoallocScratchBytes)
        return fail(TRA_ERR_WORKSPACE,
                    "squared-distance norms need %llu bytes of scratch; the built-in scratch holds %llu bytes "
                    "(use ein_execute with a caller workspace)",
                    (unsigned long long)p.ws_bytes, (unsigned long long)kTraNoallocScratchBytes);
    void* scratch = nullptr;
    const int rc = scratch_address(&scratch);
    if (rc != TRA_OK) return rc;
    return ein_execute(plan, in0, in1, out, scratch, kTraNoallocScratchBytes, stream);
}
