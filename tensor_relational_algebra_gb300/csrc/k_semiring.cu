// Join + aggregate on CUDA cores for the extended EinSum semirings
// ("EinDecomp ... tensor relational algebra", section 2.1: any commutative,
// associative aggregation -- sum, max, min, logsumexp -- over any binary scalar
// function -- multiply, add, (x-y)^2).
//
// Each CTA owns one 128 x 128 output tile of one batch index.  A tile never
// straddles two output keys in the sense that matters here: every element is
// addressed through the relation layout (RoleMap), so the tile walks the whole
// contracted range -- all contracted keys, then the local indices inside each
// -- and the aggregation across join tuples of one output key (section 2.2,
// aggregation) happens in the same registers as the aggregation inside one
// sub-tensor.
#include <cuda_bf16.h>

#include <cfloat>
#include <cstdint>

#include "tra_internal.h"

namespace tra {
namespace {

constexpr int BM = 128, BN = 128, BK = 16, NT = 256;

template <typename T>
__device__ __forceinline__ float ld_in(const void* p, int64_t off);
template <>
__device__ __forceinline__ float ld_in<float>(const void* p, int64_t off) {
    return __ldg(reinterpret_cast<const float*>(p) + off);
}
template <>
__device__ __forceinline__ float ld_in<__nv_bfloat16>(const void* p, int64_t off) {
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[off]);
}

__device__ __forceinline__ void st_out(void* p, int64_t off, float v, int bf16) {
    if (bf16)
        reinterpret_cast<__nv_bfloat16*>(p)[off] = __float2bfloat16_rn(v);
    else
        reinterpret_cast<float*>(p)[off] = v;
}

__device__ __forceinline__ float apply_op(int op, float x, float y) {
    switch (op) {
        case kMul: return x * y;
        case kAdd: return x + y;
        case kSqdiff: { float t = x - y; return t * t; }
        case kSub: return x - y;
        case kExpsub: return expf(x - y);
        default: return x;
    }
}

// ---------------------------------------------------------------- semiring functors
struct MulSum {
    static __host__ __device__ constexpr float init() { return 0.f; }
    static __device__ __forceinline__ float step(float acc, float x, float y) { return fmaf(x, y, acc); }
};
struct SqdiffSum {
    static __host__ __device__ constexpr float init() { return 0.f; }
    static __device__ __forceinline__ float step(float acc, float x, float y) {
        float t = x - y;
        return fmaf(t, t, acc);
    }
};
struct AddMax {
    static __host__ __device__ constexpr float init() { return -INFINITY; }
    static __device__ __forceinline__ float step(float acc, float x, float y) { return fmaxf(acc, x + y); }
};
struct AddMin {
    static __host__ __device__ constexpr float init() { return INFINITY; }
    static __device__ __forceinline__ float step(float acc, float x, float y) { return fminf(acc, x + y); }
};

// Online logsumexp of one output over the contracted range, read straight from the
// operands (used by the factored form when its sum underflows, and by the simple kernel).
template <typename TIn>
__device__ float direct_lse(const SemiringParams& p, const void* x, const void* y, int64_t xo, int64_t yo) {
    float m = -INFINITY, s = 0.f;
    for (uint32_t k = 0; k < p.K; ++k) {
        float v = ld_in<TIn>(x, xo + role_offset(p.xk, k)) + ld_in<TIn>(y, yo + role_offset(p.yk, k));
        if (v > m) {
            s = s * expf(m - v) + 1.f;
            m = v;
        } else {
            s += expf(v - m);
        }
    }
    return m == -INFINITY ? m : m + logf(s);
}

// ---------------------------------------------------------------- tiled kernel
template <class S, typename TIn>
__global__ void __launch_bounds__(NT, 2) semiring_tiled(const __grid_constant__ SemiringParams p) {
    __shared__ __align__(16) float Xs[2][BK][BM];
    __shared__ __align__(16) float Ys[2][BK][BN];
    __shared__ int64_t rowX[BM], colY[BN], rowZ[BM], colZ[BN];
    __shared__ int64_t kX[2][BK], kY[2][BK];

    const int tid = threadIdx.x;
    const uint32_t tiles_m = (p.M + BM - 1) / BM, tiles_n = (p.N + BN - 1) / BN;
    uint32_t t = blockIdx.x;
    const uint32_t tn = t % tiles_n;
    t /= tiles_n;
    const uint32_t tm = t % tiles_m;
    const uint32_t b = t / tiles_m;
    const uint32_t m0 = tm * BM, n0 = tn * BN;

    const int64_t xb = role_offset(p.xb, b), yb = role_offset(p.yb, b), zb = role_offset(p.zb, b);
    if (tid < BM) {
        uint32_t m = min(m0 + tid, p.M - 1);
        rowX[tid] = xb + role_offset(p.xm, m);
        rowZ[tid] = zb + role_offset(p.zm, m);
    } else {
        uint32_t n = min(n0 + (tid - BM), p.N - 1);
        colY[tid - BM] = yb + role_offset(p.yn, n);
        colZ[tid - BM] = role_offset(p.zn, n);
    }
    const uint32_t nkt = (p.K + BK - 1) / BK;
    if (tid < BK) {
        uint32_t k = min((uint32_t)tid, p.K - 1);
        kX[0][tid] = role_offset(p.xk, k);
    } else if (tid < 2 * BK) {
        uint32_t k = min((uint32_t)(tid - BK), p.K - 1);
        kY[0][tid - BK] = role_offset(p.yk, k);
    }
    __syncthreads();

    // global -> register staging of one K-tile
    float rx[8], ry[8];
    const bool xk_map = p.x_kcontig;
    const bool yk_map = p.y_kcontig && !p.y_ncontig;
    auto load_tile = [&](int buf, uint32_t k0) {
        const uint32_t kv = min((uint32_t)BK, p.K - k0);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            int m, k;
            if (xk_map) { k = tid % BK; m = tid / BK + 16 * i; }
            else { m = tid % BM; k = tid / BM + 2 * i; }
            rx[i] = (uint32_t)k < kv ? ld_in<TIn>(p.x, rowX[m] + kX[buf][k]) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            int n, k;
            if (yk_map) { k = tid % BK; n = tid / BK + 16 * i; }
            else { n = tid % BN; k = tid / BN + 2 * i; }
            ry[i] = (uint32_t)k < kv ? ld_in<TIn>(p.y, colY[n] + kY[buf][k]) : 0.f;
        }
    };
    auto store_tile = [&](int buf) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            int m, k;
            if (xk_map) { k = tid % BK; m = tid / BK + 16 * i; }
            else { m = tid % BM; k = tid / BM + 2 * i; }
            Xs[buf][k][m] = rx[i];
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            int n, k;
            if (yk_map) { k = tid % BK; n = tid / BK + 16 * i; }
            else { n = tid % BN; k = tid / BN + 2 * i; }
            Ys[buf][k][n] = ry[i];
        }
    };

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = S::init();

    const int ty = tid / 16, tx = tid % 16;
    load_tile(0, 0);
    store_tile(0);
    __syncthreads();

    for (uint32_t kt = 0; kt < nkt; ++kt) {
        const int buf = kt & 1;
        const uint32_t k0 = kt * BK;
        const bool has_next = kt + 1 < nkt;
        if (has_next) {
            // offsets of the next K-tile, then its loads (overlap with the math below)
            const uint32_t k1 = k0 + BK;
            if (tid < BK) {
                uint32_t k = min(k1 + tid, p.K - 1);
                kX[buf ^ 1][tid] = role_offset(p.xk, k);
            } else if (tid < 2 * BK) {
                uint32_t k = min(k1 + tid - BK, p.K - 1);
                kY[buf ^ 1][tid - BK] = role_offset(p.yk, k);
            }
        }
        __syncthreads();
        if (has_next) load_tile(buf ^ 1, k0 + BK);
        const uint32_t kv = min((uint32_t)BK, p.K - k0);
        if (kv == BK) {
#pragma unroll
            for (int k = 0; k < BK; ++k) {
                float4 a0 = *reinterpret_cast<const float4*>(&Xs[buf][k][ty * 4]);
                float4 a1 = *reinterpret_cast<const float4*>(&Xs[buf][k][64 + ty * 4]);
                float4 b0 = *reinterpret_cast<const float4*>(&Ys[buf][k][tx * 4]);
                float4 b1 = *reinterpret_cast<const float4*>(&Ys[buf][k][64 + tx * 4]);
                float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
                for (int i = 0; i < 8; ++i)
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[i][j] = S::step(acc[i][j], a[i], bb[j]);
            }
        } else {
            for (uint32_t k = 0; k < kv; ++k) {
                float4 a0 = *reinterpret_cast<const float4*>(&Xs[buf][k][ty * 4]);
                float4 a1 = *reinterpret_cast<const float4*>(&Xs[buf][k][64 + ty * 4]);
                float4 b0 = *reinterpret_cast<const float4*>(&Ys[buf][k][tx * 4]);
                float4 b1 = *reinterpret_cast<const float4*>(&Ys[buf][k][64 + tx * 4]);
                float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
                for (int i = 0; i < 8; ++i)
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[i][j] = S::step(acc[i][j], a[i], bb[j]);
            }
        }
        if (has_next) store_tile(buf ^ 1);
        __syncthreads();
    }

    // epilogue
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int mi = (i < 4) ? ty * 4 + i : 64 + ty * 4 + (i - 4);
        const uint32_t m = m0 + mi;
        if (m >= p.M) continue;
        const float rmax = p.rowmax ? p.rowmax[(uint64_t)b * p.M + m] : 0.f;
        const float xn = p.xnorm ? p.xnorm[(uint64_t)b * p.M + m] : 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int nj = (j < 4) ? tx * 4 + j : 64 + tx * 4 + (j - 4);
            const uint32_t n = n0 + nj;
            if (n >= p.N) continue;
            float v = acc[i][j];
            if (p.rowmax) {
                const float cmax = p.colmax[(uint64_t)b * p.N + n];
                if (v > 1e-30f) {
                    v = rmax + cmax + logf(v);
                } else {
                    // every shifted term underflowed: evaluate this output directly
                    const int64_t xo = role_offset(p.xb, b) + role_offset(p.xm, m);
                    const int64_t yo = role_offset(p.yb, b) + role_offset(p.yn, n);
                    v = p.in_bf16 ? direct_lse<__nv_bfloat16>(p, p.x_raw, p.y_raw, xo, yo)
                                  : direct_lse<float>(p, p.x_raw, p.y_raw, xo, yo);
                }
            } else if (p.xnorm) {
                v = fmaxf(xn + p.ynorm[(uint64_t)b * p.N + n] - 2.f * v, 0.f);
            }
            st_out(p.z, rowZ[mi] + colZ[nj], p.alpha * v, p.out_bf16);
        }
    }
}

// ---------------------------------------------------------------- generic fallback
// One thread per output; any op / aggregation (logsumexp evaluated online).
template <typename TIn>
__global__ void semiring_simple(const __grid_constant__ SemiringParams p) {
    const uint64_t total = (uint64_t)p.nb * p.M * p.N;
    for (uint64_t o = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; o < total;
         o += (uint64_t)gridDim.x * blockDim.x) {
        const uint32_t n = o % p.N;
        const uint32_t m = (o / p.N) % p.M;
        const uint32_t b = o / ((uint64_t)p.N * p.M);
        const int64_t xo = role_offset(p.xb, b) + role_offset(p.xm, m);
        const int64_t yo = role_offset(p.yb, b) + role_offset(p.yn, n);
        float acc;
        if (p.agg == kLse) {
            float mx = -INFINITY, s = 0.f;
            for (uint32_t k = 0; k < p.K; ++k) {
                float v = apply_op(p.op, ld_in<TIn>(p.x, xo + role_offset(p.xk, k)),
                                   ld_in<TIn>(p.y, yo + role_offset(p.yk, k)));
                if (v > mx) {
                    s = s * expf(mx - v) + 1.f;
                    mx = v;
                } else {
                    s += expf(v - mx);
                }
            }
            acc = mx == -INFINITY ? mx : mx + logf(s);
        } else {
            acc = p.agg == kMax ? -INFINITY : (p.agg == kMin ? INFINITY : 0.f);
            for (uint32_t k = 0; k < p.K; ++k) {
                float v = apply_op(p.op, ld_in<TIn>(p.x, xo + role_offset(p.xk, k)),
                                   ld_in<TIn>(p.y, yo + role_offset(p.yk, k)));
                if (p.agg == kMax) acc = fmaxf(acc, v);
                else if (p.agg == kMin) acc = fminf(acc, v);
                else acc += v;
            }
        }
        st_out(p.z, role_offset(p.zb, b) + role_offset(p.zm, m) + role_offset(p.zn, n), p.alpha * acc, p.out_bf16);
    }
}

// ---------------------------------------------------------------- factored-logsumexp / norm preparation
// mode 0: per row, max over the contracted range, then dst = exp(v - max) for every element.
// mode 1: per row, sum of squares over the contracted range (squared-distance expansion).
template <typename TIn>
__global__ void lse_prep_kernel(const __grid_constant__ LsePrepParams p, int row_per_thread) {
    if (!row_per_thread) {
        // one warp per row (contracted index contiguous in memory)
        const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) / 32, lane = threadIdx.x % 32;
        const uint64_t rows = (uint64_t)p.nb * p.R;
        if (warp >= rows) return;
        const uint32_t r = warp % p.R, b = warp / p.R;
        const int64_t base = role_offset(p.b, b) + role_offset(p.r, r);
        float m = p.mode == 0 ? -INFINITY : 0.f;
        for (uint32_t k = lane; k < p.K; k += 32) {
            float v = ld_in<TIn>(p.src, base + role_offset(p.k, k));
            m = p.mode == 0 ? fmaxf(m, v) : fmaf(v, v, m);
        }
        for (int o = 16; o; o >>= 1) {
            float w = __shfl_xor_sync(0xffffffffu, m, o);
            m = p.mode == 0 ? fmaxf(m, w) : m + w;
        }
        if (lane == 0) p.rmax[warp] = m;
        if (p.mode == 0)
            for (uint32_t k = lane; k < p.K; k += 32) {
                int64_t off = base + role_offset(p.k, k);
                p.dst[off] = expf(ld_in<TIn>(p.src, off) - m);
            }
    } else {
        // one thread per row (rows contiguous in memory): coalesced across the warp
        const uint64_t row = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x;
        if (row >= (uint64_t)p.nb * p.R) return;
        const uint32_t r = row % p.R, b = row / p.R;
        const int64_t base = role_offset(p.b, b) + role_offset(p.r, r);
        float m = p.mode == 0 ? -INFINITY : 0.f;
        for (uint32_t k = 0; k < p.K; ++k) {
            float v = ld_in<TIn>(p.src, base + role_offset(p.k, k));
            m = p.mode == 0 ? fmaxf(m, v) : fmaf(v, v, m);
        }
        p.rmax[row] = m;
        if (p.mode == 0)
            for (uint32_t k = 0; k < p.K; ++k) {
                int64_t off = base + role_offset(p.k, k);
                p.dst[off] = expf(ld_in<TIn>(p.src, off) - m);
            }
    }
}

}  // namespace

cudaError_t launch_semiring(const SemiringParams& p, cudaStream_t s) {
    if (p.nb == 0 || p.M == 0 || p.N == 0) return cudaSuccess;
    if (p.K == 0) return cudaErrorInvalidValue;
    const uint64_t grid = (uint64_t)p.nb * ((p.M + BM - 1) / BM) * ((p.N + BN - 1) / BN);
    if (grid > 0x7fffffffull) return cudaErrorInvalidValue;
    const bool bf = p.in_bf16;
    if (p.rowmax || p.xnorm) {
        // factored logsumexp / squared-distance expansion: the operands are fp32 here
        // (exp-shifted scratch, or the fp32 inputs); in_bf16 describes x_raw / y_raw
        semiring_tiled<MulSum, float><<<(unsigned)grid, NT, 0, s>>>(p);
        return cudaGetLastError();
    }
    switch (p.op * 8 + p.agg) {
        case kMul * 8 + kSum:
            if (bf) semiring_tiled<MulSum, __nv_bfloat16><<<(unsigned)grid, NT, 0, s>>>(p);
            else semiring_tiled<MulSum, float><<<(unsigned)grid, NT, 0, s>>>(p);
            break;
        case kSqdiff * 8 + kSum:
            if (bf) semiring_tiled<SqdiffSum, __nv_bfloat16><<<(unsigned)grid, NT, 0, s>>>(p);
            else semiring_tiled<SqdiffSum, float><<<(unsigned)grid, NT, 0, s>>>(p);
            break;
        case kAdd * 8 + kMax:
            if (bf) semiring_tiled<AddMax, __nv_bfloat16><<<(unsigned)grid, NT, 0, s>>>(p);
            else semiring_tiled<AddMax, float><<<(unsigned)grid, NT, 0, s>>>(p);
            break;
        case kAdd * 8 + kMin:
            if (bf) semiring_tiled<AddMin, __nv_bfloat16><<<(unsigned)grid, NT, 0, s>>>(p);
            else semiring_tiled<AddMin, float><<<(unsigned)grid, NT, 0, s>>>(p);
            break;
        default:
            return launch_semiring_simple(p, s);
    }
    return cudaGetLastError();
}

cudaError_t launch_semiring_simple(const SemiringParams& p, cudaStream_t s) {
    const uint64_t total = (uint64_t)p.nb * p.M * p.N;
    if (total == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((total + 255) / 256 < 65536 ? (total + 255) / 256 : 65536);
    if (p.in_bf16) semiring_simple<__nv_bfloat16><<<blocks, 256, 0, s>>>(p);
    else semiring_simple<float><<<blocks, 256, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_lse_prep(const LsePrepParams& p, cudaStream_t s) {
    const uint64_t rows = (uint64_t)p.nb * p.R;
    if (rows == 0) return cudaSuccess;
    // rows contiguous (the contracted index is not the fastest-moving one): thread per row
    const bool rpt = !(p.k.n > 0 && p.k.t[0].div == 1 && p.k.t[0].loc_stride == 1);
    const uint64_t threads = rpt ? rows : rows * 32;
    const unsigned blocks = (unsigned)((threads + 255) / 256);
    if (p.in_bf16) lse_prep_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(p, rpt);
    else lse_prep_kernel<float><<<blocks, 256, 0, s>>>(p, rpt);
    return cudaGetLastError();
}

}  // namespace tra
