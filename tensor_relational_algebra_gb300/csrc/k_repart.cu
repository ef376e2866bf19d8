// Repartition by tensor-memory-access (TMA) copies: "EinDecomp ... tensor relational
// algebra", section 2.2 (repartition: the same tensor re-cut under another partition vector).
//
// Along every dimension, pieces of extent gcd(source block extent, destination block
// extent) lie inside one source block and one destination block.  A piece (or a box that
// tiles it) is therefore a plain strided box in both relations: local indices of one block
// plus that block's linear key.  Each relation is described by a tensor map of rank
// (dimensions) + 1 -- the block-local dimensions, innermost first, then the block index --
// and a box goes global -> shared memory under the source map and shared -> global memory
// under the destination map, with no register traffic.  The two boxes list their elements in
// the same order (both relations lay a block out row-major over the same index order).
//
// One issuing thread per CTA (one CTA per SM) keeps a ring of stages in flight.  Every wait
// is bounded; a wait that gives up records TRA_ERR_TIMEOUT in this file's status word.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <numeric>

#include "tra_internal.h"

namespace tra {

__device__ int g_rp_status;  // TRA_ERR_* of a bounded wait that gave up; 0 otherwise

namespace {

constexpr int kMaxDims = 4;               // block-local dimensions (the tensor map adds the block index)
constexpr uint32_t kBoxBudget = 32768;    // bytes per box
constexpr uint32_t kMinBox = 4096;        // smaller boxes: the warp-cooperative kernel is faster
constexpr uint32_t kStageBytes = 196608;  // shared memory for the ring of stages

struct RpTmaParams {
    int32_t nd;  // dimensions kept (extent > 1), outermost first
    uint32_t nbox[kMaxDims], box[kMaxDims];
    uint32_t bs[kMaxDims], bd[kMaxDims];  // block extents, source / destination
    uint32_t ds[kMaxDims], dd[kMaxDims];  // partition counts, source / destination
    uint32_t n_boxes, box_bytes, stride, stages;
    uint64_t timeout_ns;
};

__device__ __forceinline__ uint64_t now_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ bool bar_try(uint32_t bar, uint32_t parity) {
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
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
    if (bar_try(bar, parity)) return true;
    const uint64_t t0 = now_ns();
    while (!bar_try(bar, parity))
        if (now_ns() - t0 > timeout_ns) return false;
    return true;
}

// Tensor-map coordinates of box `id` in the source (cs) and destination (cd) relations.
__device__ __forceinline__ void box_coords(const RpTmaParams& p, uint32_t id, int cs[5], int cd[5]) {
#pragma unroll
    for (int j = 0; j < 5; ++j) cs[j] = cd[j] = 0;
    uint32_t ks_lin = 0, kd_lin = 0, ms = 1, md = 1;
    for (int k = p.nd - 1; k >= 0; --k) {
        const uint32_t idx = id % p.nbox[k];
        id /= p.nbox[k];
        const uint32_t x = idx * p.box[k];
        const uint32_t ks = x / p.bs[k], kd = x / p.bd[k];
        cs[p.nd - 1 - k] = (int)(x - ks * p.bs[k]);
        cd[p.nd - 1 - k] = (int)(x - kd * p.bd[k]);
        ks_lin += ks * ms;
        kd_lin += kd * md;
        ms *= p.ds[k];
        md *= p.dd[k];
    }
    cs[p.nd] = (int)ks_lin;
    cd[p.nd] = (int)kd_lin;
}

__global__ void __launch_bounds__(32, 1) repart_tma_kernel(const __grid_constant__ CUtensorMap ms,
                                                           const __grid_constant__ CUtensorMap md,
                                                           const __grid_constant__ RpTmaParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (threadIdx.x != 0) return;
    const uint32_t base = ((uint32_t)__cvta_generic_to_shared(smem_raw) + 1023u) & ~1023u;
    const uint32_t bars = base + p.stages * p.stride;
    for (uint32_t s = 0; s < p.stages; ++s)
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bars + 8 * s) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    const uint32_t n = blockIdx.x < p.n_boxes ? (p.n_boxes - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    auto load = [&](uint32_t i) {
        int cs[5], cd[5];
        box_coords(p, blockIdx.x + i * gridDim.x, cs, cd);
        const uint32_t s = i % p.stages, bar = bars + 8 * s;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(p.box_bytes) : "memory");
        asm volatile(
            "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(base + s * p.stride),
            "l"(reinterpret_cast<uint64_t>(&ms)), "r"(cs[0]), "r"(cs[1]), "r"(cs[2]), "r"(cs[3]), "r"(cs[4]), "r"(bar)
            : "memory");
    };
    uint32_t issued = 0;
    for (; issued < p.stages && issued < n; ++issued) load(issued);
    uint32_t i = 0;
    for (; i < n; ++i) {
        const uint32_t s = i % p.stages;
        if (!bar_wait(bars + 8 * s, (i / p.stages) & 1u, p.timeout_ns)) {
            atomicExch(&g_rp_status, (int)TRA_ERR_TIMEOUT);
            break;
        }
        int cs[5], cd[5];
        box_coords(p, blockIdx.x + i * gridDim.x, cs, cd);
        asm volatile(
            "cp.async.bulk.tensor.5d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3, %4, %5}], [%6];" ::"l"(
                reinterpret_cast<uint64_t>(&md)),
            "r"(cd[0]), "r"(cd[1]), "r"(cd[2]), "r"(cd[3]), "r"(cd[4]), "r"(base + s * p.stride)
            : "memory");
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        if (issued < n) {
            // the stage is reloaded once the store just issued has read it
            asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
            load(issued++);
        }
    }
    // after a wait that gave up: let the loads still in flight land before the CTA leaves
    for (uint32_t j = i; j < issued; ++j) bar_wait(bars + 8 * (j % p.stages), (j / p.stages) & 1u, p.timeout_ns);
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// Rank-5 tensor map over one relation: block-local dimensions (extents blk[], innermost first)
// then the block index (n_blocks); boxes box[] and 1.
bool encode_relation(const void* base, int nd, const uint64_t* blk, uint64_t n_blocks, const uint32_t* box,
                     int elem_bytes, CUtensorMap* map) {
    auto fn = encoder();
    if (!fn) return false;
    CUtensorMapDataType dt = elem_bytes == 1   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                             : elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16
                             : elem_bytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_UINT32
                                               : CU_TENSOR_MAP_DATA_TYPE_UINT64;
    cuuint64_t dims[5], strides[4];
    cuuint32_t bx[5], es[5] = {1, 1, 1, 1, 1};
    uint64_t span = (uint64_t)elem_bytes;  // bytes of one step along the next dimension
    for (int j = 0; j < 5; ++j) {
        if (j < nd) {
            dims[j] = blk[j];
            bx[j] = box[j];
        } else if (j == nd) {
            dims[j] = n_blocks;
            bx[j] = 1;
        } else {
            dims[j] = 1;
            bx[j] = 1;
        }
        if (j > 0) strides[j - 1] = span;
        span *= dims[j];
    }
    return fn(map, dt, 5, const_cast<void*>(base), dims, strides, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Largest divisor of v that is at most cap and, with `mult` > 1, whose byte size
// (d * elem_bytes) is a multiple of mult; 0 when there is none.
uint32_t best_divisor(uint64_t v, uint64_t cap, int elem_bytes, uint32_t mult) {
    for (uint64_t d = cap < v ? cap : v; d >= 1; --d)
        if (v % d == 0 && (d * (uint64_t)elem_bytes) % mult == 0) return (uint32_t)d;
    return 0;
}

}  // namespace

cudaError_t launch_repartition_tma(int rank, const int64_t* shape, const int32_t* src_d, const int32_t* dst_d,
                                   int elem_bytes, const void* src, void* dst, cudaStream_t s) {
    if (((uintptr_t)src | (uintptr_t)dst) % 16) return cudaErrorNotSupported;
    // the dimensions of extent > 1, outermost first
    RpTmaParams p;
    memset(&p, 0, sizeof(p));
    uint64_t g[kMaxDims];
    for (int i = 0; i < rank; ++i) {
        if (shape[i] == 1) continue;
        if (p.nd == kMaxDims) return cudaErrorNotSupported;
        const int k = p.nd++;
        p.ds[k] = (uint32_t)src_d[i];
        p.dd[k] = (uint32_t)dst_d[i];
        p.bs[k] = (uint32_t)(shape[i] / src_d[i]);
        p.bd[k] = (uint32_t)(shape[i] / dst_d[i]);
        g[k] = std::gcd((uint64_t)p.bs[k], (uint64_t)p.bd[k]);
    }
    if (p.nd == 0) return cudaErrorNotSupported;
    const int last = p.nd - 1;
    // every row of a block starts on a 16-byte boundary in both relations (tensor-map strides)
    if (((uint64_t)p.bs[last] * elem_bytes) % 16 || ((uint64_t)p.bd[last] * elem_bytes) % 16)
        return cudaErrorNotSupported;
    // boxes, innermost first: the innermost extent a whole number of 16-byte units (so every box
    // starts on a 16-byte boundary), at most 256 per dimension, at most kBoxBudget bytes
    uint64_t bytes = (uint64_t)elem_bytes;
    for (int k = last; k >= 0; --k) {
        const uint64_t cap = std::min<uint64_t>(256, kBoxBudget / bytes);
        const uint32_t b = best_divisor(g[k], cap, elem_bytes, k == last ? 16u : 1u);
        if (b == 0) return cudaErrorNotSupported;
        p.box[k] = b;
        bytes *= b;
    }
    if (bytes < kMinBox) return cudaErrorNotSupported;
    uint64_t n_boxes = 1, nbs = 1, nbd = 1;
    for (int k = 0; k < p.nd; ++k) {
        p.nbox[k] = (uint32_t)((uint64_t)p.bs[k] * p.ds[k] / p.box[k]);
        n_boxes *= p.nbox[k];
        nbs *= p.ds[k];
        nbd *= p.dd[k];
    }
    if (n_boxes > 0xffffffffull) return cudaErrorNotSupported;
    p.n_boxes = (uint32_t)n_boxes;
    p.box_bytes = (uint32_t)bytes;
    p.stride = (uint32_t)((bytes + 1023) / 1024 * 1024);
    p.stages = std::min<uint32_t>(8, std::max<uint32_t>(2, kStageBytes / p.stride));
    p.timeout_ns = 2000000000ull;
    // tensor maps: block-local dimensions innermost first, then the block index
    uint64_t blk_s[kMaxDims], blk_d[kMaxDims];
    uint32_t box[kMaxDims];
    for (int j = 0; j < p.nd; ++j) {
        blk_s[j] = p.bs[last - j];
        blk_d[j] = p.bd[last - j];
        box[j] = p.box[last - j];
    }
    CUtensorMap ms, md;
    if (!encode_relation(src, p.nd, blk_s, nbs, box, elem_bytes, &ms) ||
        !encode_relation(dst, p.nd, blk_d, nbd, box, elem_bytes, &md))
        return cudaErrorNotSupported;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const size_t smem = (size_t)p.stages * p.stride + 1024 + 8 * p.stages;
    e = cudaFuncSetAttribute(repart_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)std::min<uint64_t>(n_boxes, (uint64_t)sms);
    repart_tma_kernel<<<grid, 32, smem, s>>>(ms, md, p);
    return cudaGetLastError();
}

cudaError_t read_and_clear_rp_status(int* value, cudaStream_t s) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(value, g_rp_status, sizeof(int), 0, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    const int zero = 0;
    e = cudaMemcpyToSymbolAsync(g_rp_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(s);
}

}  // namespace tra
