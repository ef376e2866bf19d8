// FP32 issue ceilings of the CUDA-core semiring kernels' inner step (a measurement aid; the
// EinDecomp page has no counterpart).
//
// Each CTA (256 threads, two per SM as the semiring kernels run) keeps the same 8 x 8 register
// tile per thread and reads its operands from shared memory in the same [m][32 k] / [k][n]
// staging, but never touches global memory inside the timed loop, so the loop measures the
// instruction mix alone:
//   kind 0  sum of products: two FFMA per two tuples (consecutive k)
//   kind 1  max-plus: FADD, FADD and one 3-input max.f32 per two tuples
//   kind 2  max-plus with the packed add: one add.rn.f32x2 and one 3-input max per two tuples
// Thread 0 of each CTA records the SM clock (clock64) and the global timer (ns) around the
// loop, so the host obtains tuples per clock per SM and the clock the SM actually ran at.
#include <cstdint>

#include "plan.h"

namespace tra {
namespace {

constexpr int kProbeThreads = 256;

__device__ __forceinline__ float probe_max3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
__device__ __forceinline__ uint64_t probe_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ uint64_t probe_add2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t probe_globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

template <int KIND>
__global__ void __launch_bounds__(kProbeThreads, 2)
    fp32_probe_kernel(int iters, float* sink, unsigned long long* cycles, unsigned long long* nanos) {
    // two copies of the staged tiles (dynamic shared memory, 64 KB), alternated per iteration
    // so the shared-memory reads stay inside the loop
    extern __shared__ __align__(16) float probe_smem[];
    constexpr int kTile = 128 * 32;  // [x copy 0][x copy 1][y copy 0][y copy 1]
    for (int i = threadIdx.x; i < kTile; i += kProbeThreads) {
        const float x = (float)(i * 37 % 101) * 0.01f, y = (float)(i * 53 % 97) * 0.01f;
        probe_smem[i] = x;
        probe_smem[kTile + i] = x + 1.f;
        probe_smem[2 * kTile + i] = y;
        probe_smem[3 * kTile + i] = y - 1.f;
    }
    __syncthreads();
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = KIND == 0 ? 0.f : -1e30f;
    const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
    const unsigned long long c0 = clock64();
    const uint64_t t0 = probe_globaltimer();
    for (int it = 0; it < iters; ++it) {
        const float4* xs4 = reinterpret_cast<const float4*>(probe_smem + (it & 1) * kTile);
        const float4* ys4 = reinterpret_cast<const float4*>(probe_smem + (2 + (it & 1)) * kTile);
#pragma unroll 2
        for (int kq = 0; kq < 8; ++kq) {  // 32 k per iteration, 4 at a time
            float4 a[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) a[i] = xs4[((i < 4) ? ty * 4 + i : 64 + ty * 4 + (i - 4)) * 8 + kq];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int k = kq * 4 + 2 * h;
                const float4 b0 = ys4[k * 32 + tx], b1 = ys4[k * 32 + 16 + tx];
                const float4 d0 = ys4[(k + 1) * 32 + tx], d1 = ys4[(k + 1) * 32 + 16 + tx];
                const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
                const float dd[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float x0 = h == 0 ? a[i].x : a[i].z;
                    const float x1 = h == 0 ? a[i].y : a[i].w;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (KIND == 0) {
                            acc[i][j] = fmaf(x1, dd[j], fmaf(x0, bb[j], acc[i][j]));
                        } else if (KIND == 1) {
                            acc[i][j] = probe_max3(acc[i][j], x0 + bb[j], x1 + dd[j]);
                        } else {
                            const uint64_t s = probe_add2(probe_pack(x0, x1), probe_pack(bb[j], dd[j]));
                            acc[i][j] = probe_max3(acc[i][j], __uint_as_float((uint32_t)s),
                                                   __uint_as_float((uint32_t)(s >> 32)));
                        }
                    }
                }
            }
        }
    }
    const unsigned long long c1 = clock64();
    const uint64_t t1 = probe_globaltimer();
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) s += acc[i][j];
    sink[(size_t)blockIdx.x * kProbeThreads + threadIdx.x] = s;  // keeps the loop alive
    if (threadIdx.x == 0) {
        cycles[blockIdx.x] = c1 - c0;
        nanos[blockIdx.x] = t1 - t0;
    }
}

}  // namespace
}  // namespace tra

using namespace tra;

extern "C" int ein_probe_fp32(int kind, int iters, int ctas, void* sink, void* cycles, void* nanos,
                              uint64_t* tuples_per_cta, tra_stream_t stream) {
    clear_error();
    if (kind < 0 || kind > 2) return fail(TRA_ERR_ARG, "probe kind %d not in 0..2", kind);
    if (iters < 1 || ctas < 1) return fail(TRA_ERR_ARG, "iters and ctas must be positive");
    if (!sink || !cycles || !nanos || !tuples_per_cta) return fail(TRA_ERR_ARG, "NULL buffer");
    // per iteration each thread covers 32 k x 64 outputs
    *tuples_per_cta = (uint64_t)iters * 32u * 64u * kProbeThreads;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    auto* sk = reinterpret_cast<float*>(sink);
    auto* cy = reinterpret_cast<unsigned long long*>(cycles);
    auto* ns = reinterpret_cast<unsigned long long*>(nanos);
    constexpr int smem = 4 * 128 * 32 * (int)sizeof(float);
    cudaError_t e = cudaSuccess;
    switch (kind) {
        case 0:
            e = cudaFuncSetAttribute(fp32_probe_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e == cudaSuccess) fp32_probe_kernel<0><<<ctas, kProbeThreads, smem, s>>>(iters, sk, cy, ns);
            break;
        case 1:
            e = cudaFuncSetAttribute(fp32_probe_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e == cudaSuccess) fp32_probe_kernel<1><<<ctas, kProbeThreads, smem, s>>>(iters, sk, cy, ns);
            break;
        default:
            e = cudaFuncSetAttribute(fp32_probe_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e == cudaSuccess) fp32_probe_kernel<2><<<ctas, kProbeThreads, smem, s>>>(iters, sk, cy, ns);
            break;
    }
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? TRA_OK : fail(TRA_ERR_CUDA, "probe launch: %s", cudaGetErrorString(e));
}
