// Join + aggregate on CUDA cores for the extended EinSum semirings
// ("EinDecomp ... tensor relational algebra", section 2.1: any commutative,
// associative aggregation -- sum, max, min, logsumexp -- over any binary scalar
// function -- multiply, add, (x-y)^2).
//
// Each CTA owns one 128 x 128 output tile of one batch index and walks the whole
// contracted range -- every contracted key, then the local indices inside it --
// so the aggregation across the join tuples of one output key (section 2.2,
// aggregation) happens in the same registers as the aggregation inside one
// sub-tensor.  Every element is addressed through the relation layout
// (RoleMap), so one kernel serves every binary EinSum and every partition vector.
//
// Per thread: an 8 x 8 register tile; K is staged through shared memory 16 at a
// time (double-buffered, prefetched into registers during the math).  Operands
// are loaded as float4 / 4 x bf16 when the layout makes 4 consecutive indices
// contiguous, else gathered element by element.  The K tail is padded with
// values whose join is the aggregation's identity, so the inner loop never
// branches.  For max-plus / min-plus the inner step works on pairs of
// consecutive k: one packed add (add.rn.f32x2) and one 3-input max/min per two
// join tuples.
#include <cuda_bf16.h>

#include <cfloat>
#include <cstdint>

#include "tra_internal.h"

namespace tra {
namespace {

constexpr int BM = 128, BN = 128, BK = 16, NT = 256;
enum { kEpiPlain = 0, kEpiLse = 1, kEpiSqExpand = 2 };
enum { kLoadGather = 0, kLoadVecK = 1, kLoadVecMN = 2 };

template <typename T>
__device__ __forceinline__ float ld1(const void* p, int64_t off);
template <>
__device__ __forceinline__ float ld1<float>(const void* p, int64_t off) {
    return __ldg(reinterpret_cast<const float*>(p) + off);
}
template <>
__device__ __forceinline__ float ld1<__nv_bfloat16>(const void* p, int64_t off) {
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[off]);
}

// four consecutive elements starting at a multiple of 4 (16-byte / 8-byte aligned)
template <typename T>
__device__ __forceinline__ float4 ld4(const void* p, int64_t off);
template <>
__device__ __forceinline__ float4 ld4<float>(const void* p, int64_t off) {
    return __ldg(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p) + off));
}
template <>
__device__ __forceinline__ float4 ld4<__nv_bfloat16>(const void* p, int64_t off) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(p) + off));
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u), __uint_as_float(u.y << 16),
                       __uint_as_float(u.y & 0xffff0000u));
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

// packed pair helpers
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ float lo_of(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi_of(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }
__device__ __forceinline__ float max3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
__device__ __forceinline__ float min3(float a, float b, float c) {
    float r;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// ---------------------------------------------------------------- semiring functors
// pad_x / pad_y: operand values for k beyond K whose join is the aggregation's identity
struct MulSum {
    static constexpr bool kPacked = false;
    static __device__ __forceinline__ float init() { return 0.f; }
    static __device__ __forceinline__ float pad_x() { return 0.f; }
    static __device__ __forceinline__ float pad_y() { return 0.f; }
    static __device__ __forceinline__ void step(float& acc, float x, float y) { acc = fmaf(x, y, acc); }
    static __device__ __forceinline__ void step2(float&, uint64_t, uint64_t) {}
};
struct SqdiffSum {
    static constexpr bool kPacked = false;
    static __device__ __forceinline__ float init() { return 0.f; }
    static __device__ __forceinline__ float pad_x() { return 0.f; }
    static __device__ __forceinline__ float pad_y() { return 0.f; }
    static __device__ __forceinline__ void step(float& acc, float x, float y) {
        const float t = x - y;
        acc = fmaf(t, t, acc);
    }
    static __device__ __forceinline__ void step2(float&, uint64_t, uint64_t) {}
};
struct AddMax {
    static constexpr bool kPacked = true;
    static __device__ __forceinline__ float init() { return -INFINITY; }
    static __device__ __forceinline__ float pad_x() { return -INFINITY; }
    static __device__ __forceinline__ float pad_y() { return 0.f; }
    static __device__ __forceinline__ void step(float& acc, float x, float y) { acc = fmaxf(acc, x + y); }
    static __device__ __forceinline__ void step2(float& acc, uint64_t x2, uint64_t y2) {
        const uint64_t t = add2(x2, y2);
        acc = max3(acc, lo_of(t), hi_of(t));
    }
};
struct AddMin {
    static constexpr bool kPacked = true;
    static __device__ __forceinline__ float init() { return INFINITY; }
    static __device__ __forceinline__ float pad_x() { return INFINITY; }
    static __device__ __forceinline__ float pad_y() { return 0.f; }
    static __device__ __forceinline__ void step(float& acc, float x, float y) { acc = fminf(acc, x + y); }
    static __device__ __forceinline__ void step2(float& acc, uint64_t x2, uint64_t y2) {
        const uint64_t t = add2(x2, y2);
        acc = min3(acc, lo_of(t), hi_of(t));
    }
};

// Online logsumexp of one output over the contracted range, read straight from the
// operands (the factored form's fallback when its sum underflows; the simple kernel).
template <typename TIn>
__device__ __noinline__ float direct_lse(const SemiringParams& p, const void* x, const void* y, int64_t xo,
                                         int64_t yo) {
    float m = -INFINITY, s = 0.f;
    for (uint32_t k = 0; k < p.K; ++k) {
        float v = ld1<TIn>(x, xo + role_offset(p.xk, k)) + ld1<TIn>(y, yo + role_offset(p.yk, k));
        if (v > m) {
            s = s * expf(m - v) + 1.f;
            m = v;
        } else {
            s += expf(v - m);
        }
    }
    return m == -INFINITY ? m : m + logf(s);
}

__device__ __noinline__ float lse_fallback(const SemiringParams& p, uint32_t b, uint32_t m, uint32_t n) {
    const int64_t xo = role_offset(p.xb, b) + role_offset(p.xm, m);
    const int64_t yo = role_offset(p.yb, b) + role_offset(p.yn, n);
    return p.in_bf16 ? direct_lse<__nv_bfloat16>(p, p.x_raw, p.y_raw, xo, yo)
                     : direct_lse<float>(p, p.x_raw, p.y_raw, xo, yo);
}

// offset of contracted index k in X / Y: one multiply-high division when the contracted
// composite is a single label, the general role map otherwise
__device__ __forceinline__ int64_t koff_x(const SemiringParams& p, uint32_t k) {
    if (p.xk_simple) {
        const uint32_t q = fdiv(k, p.xk_sub);
        return (int64_t)q * p.xk_ks + (int64_t)(k - q * p.xk_sub.d) * p.xk_ls;
    }
    return role_offset(p.xk, k);
}
__device__ __forceinline__ int64_t koff_y(const SemiringParams& p, uint32_t k) {
    if (p.yk_simple) {
        const uint32_t q = fdiv(k, p.yk_sub);
        return (int64_t)q * p.yk_ks + (int64_t)(k - q * p.yk_sub.d) * p.yk_ls;
    }
    return role_offset(p.yk, k);
}

// shared-memory index of (k, row) in the unpacked [k][row] or packed [k/2][row][k%2] layout
template <bool P>
__device__ __forceinline__ int sidx(int k, int r) {
    return P ? (((k >> 1) * BM + r) << 1) + (k & 1) : k * BM + r;
}

// ---------------------------------------------------------------- tiled kernel
template <class S, typename TIn, int EPI>
__global__ void __launch_bounds__(NT, 2) semiring_tiled(const __grid_constant__ SemiringParams p) {
    constexpr bool P = S::kPacked;
    __shared__ __align__(16) float Xs[2][BK * BM];
    __shared__ __align__(16) float Ys[2][BK * BN];
    __shared__ int64_t rowX[BM], colY[BN];

    const int tid = threadIdx.x;
    const uint32_t tiles_m = (p.M + BM - 1) / BM, tiles_n = (p.N + BN - 1) / BN;
    uint32_t t = blockIdx.x;
    const uint32_t tn = t % tiles_n;
    t /= tiles_n;
    const uint32_t tm = t % tiles_m;
    const uint32_t b = t / tiles_m;
    const uint32_t m0 = tm * BM, n0 = tn * BN;

    if (tid < BM) {
        rowX[tid] = role_offset(p.xb, b) + role_offset(p.xm, clamp_row(m0 + tid, p.M, p.x_mode == kLoadVecMN));
    } else {
        colY[tid - BM] =
            role_offset(p.yb, b) + role_offset(p.yn, clamp_row(n0 + (tid - BM), p.N, p.y_mode == kLoadVecMN));
    }
    __syncthreads();

    const int xmode = p.x_mode, ymode = p.y_mode;
    float rx[8], ry[8];

    // ---- global -> registers for the K-tile starting at k0 (each thread maps its own k)
    auto load = [&](uint32_t k0) {
        const int kv = (int)min((uint32_t)BK, p.K - k0);
        const float px = S::pad_x(), py = S::pad_y();
        if (xmode == kLoadVecK) {
            const int m = tid & (BM - 1);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int k = ((tid >> 7) + 2 * i) * 4;
                float4 v = k < kv ? ld4<TIn>(p.x, rowX[m] + koff_x(p, k0 + k)) : make_float4(px, px, px, px);
                rx[4 * i] = v.x, rx[4 * i + 1] = v.y, rx[4 * i + 2] = v.z, rx[4 * i + 3] = v.w;
            }
        } else if (xmode == kLoadVecMN) {
            const int m = (tid & 31) * 4;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int k = (tid >> 5) + 8 * i;
                float4 v = k < kv ? ld4<TIn>(p.x, rowX[m] + koff_x(p, k0 + k)) : make_float4(px, px, px, px);
                rx[4 * i] = v.x, rx[4 * i + 1] = v.y, rx[4 * i + 2] = v.z, rx[4 * i + 3] = v.w;
            }
        } else {
            const int m = tid & (BM - 1);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int k = (tid >> 7) + 2 * i;
                rx[i] = k < kv ? ld1<TIn>(p.x, rowX[m] + koff_x(p, k0 + k)) : px;
            }
        }
        if (ymode == kLoadVecMN) {
            const int n = (tid & 31) * 4;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                // packed layout: rows 2*kp and 2*kp+1; unpacked: rows kk and kk+8
                const int k = P ? 2 * (tid >> 5) + i : (tid >> 5) + 8 * i;
                float4 v = k < kv ? ld4<TIn>(p.y, colY[n] + koff_y(p, k0 + k)) : make_float4(py, py, py, py);
                ry[4 * i] = v.x, ry[4 * i + 1] = v.y, ry[4 * i + 2] = v.z, ry[4 * i + 3] = v.w;
            }
        } else if (ymode == kLoadVecK) {
            const int n = tid & (BN - 1);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int k = ((tid >> 7) + 2 * i) * 4;
                float4 v = k < kv ? ld4<TIn>(p.y, colY[n] + koff_y(p, k0 + k)) : make_float4(py, py, py, py);
                ry[4 * i] = v.x, ry[4 * i + 1] = v.y, ry[4 * i + 2] = v.z, ry[4 * i + 3] = v.w;
            }
        } else {
            const int n = tid & (BN - 1);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int k = (tid >> 7) + 2 * i;
                ry[i] = k < kv ? ld1<TIn>(p.y, colY[n] + koff_y(p, k0 + k)) : py;
            }
        }
    };

    // ---- registers -> shared memory
    auto store = [&](int buf) {
        float* xs = Xs[buf];
        float* ys = Ys[buf];
        if (xmode == kLoadVecK) {
            const int m = tid & (BM - 1);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int k = ((tid >> 7) + 2 * i) * 4;
                if (P) {
                    *reinterpret_cast<float2*>(&xs[sidx<P>(k, m)]) = make_float2(rx[4 * i], rx[4 * i + 1]);
                    *reinterpret_cast<float2*>(&xs[sidx<P>(k + 2, m)]) = make_float2(rx[4 * i + 2], rx[4 * i + 3]);
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c) xs[sidx<P>(k + c, m)] = rx[4 * i + c];
                }
            }
        } else if (xmode == kLoadVecMN) {
            const int m = (tid & 31) * 4;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int k = (tid >> 5) + 8 * i;
                if (P) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) xs[sidx<P>(k, m + c)] = rx[4 * i + c];
                } else {
                    *reinterpret_cast<float4*>(&xs[sidx<P>(k, m)]) =
                        make_float4(rx[4 * i], rx[4 * i + 1], rx[4 * i + 2], rx[4 * i + 3]);
                }
            }
        } else {
            const int m = tid & (BM - 1);
#pragma unroll
            for (int i = 0; i < 8; ++i) xs[sidx<P>((tid >> 7) + 2 * i, m)] = rx[i];
        }
        if (ymode == kLoadVecMN) {
            const int n = (tid & 31) * 4;
            if (P) {
                const int kp = tid >> 5;  // rows 2kp (ry[0..3]) and 2kp+1 (ry[4..7])
                float4* dst = reinterpret_cast<float4*>(&ys[((kp * BN + n) << 1)]);
                dst[0] = make_float4(ry[0], ry[4], ry[1], ry[5]);
                dst[1] = make_float4(ry[2], ry[6], ry[3], ry[7]);
            } else {
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int k = (tid >> 5) + 8 * i;
                    *reinterpret_cast<float4*>(&ys[sidx<P>(k, n)]) =
                        make_float4(ry[4 * i], ry[4 * i + 1], ry[4 * i + 2], ry[4 * i + 3]);
                }
            }
        } else if (ymode == kLoadVecK) {
            const int n = tid & (BN - 1);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int k = ((tid >> 7) + 2 * i) * 4;
                if (P) {
                    *reinterpret_cast<float2*>(&ys[sidx<P>(k, n)]) = make_float2(ry[4 * i], ry[4 * i + 1]);
                    *reinterpret_cast<float2*>(&ys[sidx<P>(k + 2, n)]) = make_float2(ry[4 * i + 2], ry[4 * i + 3]);
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c) ys[sidx<P>(k + c, n)] = ry[4 * i + c];
                }
            }
        } else {
            const int n = tid & (BN - 1);
#pragma unroll
            for (int i = 0; i < 8; ++i) ys[sidx<P>((tid >> 7) + 2 * i, n)] = ry[i];
        }
    };

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = S::init();

    const int ty = tid >> 4, tx = tid & 15;
    load(0);
    store(0);
    __syncthreads();

    const uint32_t nkt = (p.K + BK - 1) / BK;
    for (uint32_t kt = 0; kt < nkt; ++kt) {
        const int buf = kt & 1;
        const bool has_next = kt + 1 < nkt;
        // one barrier per K-tile: this tile computes from buf while the next one is
        // loaded into registers and then stored to buf ^ 1
        if (has_next) load((kt + 1) * BK);
        const float* xs = Xs[buf];
        const float* ys = Ys[buf];
        if constexpr (P) {
#pragma unroll 2
            for (int kp = 0; kp < BK / 2; ++kp) {
                // x pairs for rows ty*4..+3 and 64+ty*4..+3; y pairs for columns g*32 + tx*2 + {0,1}
                uint64_t xa[8];
                const ulonglong2* xr0 = reinterpret_cast<const ulonglong2*>(&xs[((kp * BM + ty * 4) << 1)]);
                const ulonglong2* xr1 = reinterpret_cast<const ulonglong2*>(&xs[((kp * BM + 64 + ty * 4) << 1)]);
                const ulonglong2 q0 = xr0[0], q1 = xr0[1], q2 = xr1[0], q3 = xr1[1];
                xa[0] = q0.x, xa[1] = q0.y, xa[2] = q1.x, xa[3] = q1.y;
                xa[4] = q2.x, xa[5] = q2.y, xa[6] = q3.x, xa[7] = q3.y;
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    // one group of two y pairs at a time keeps fewer values live
                    const ulonglong2 w = *reinterpret_cast<const ulonglong2*>(&ys[((kp * BN + g * 32 + tx * 2) << 1)]);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        S::step2(acc[i][2 * g], xa[i], w.x);
                        S::step2(acc[i][2 * g + 1], xa[i], w.y);
                    }
                }
            }
        } else {
#pragma unroll 8
            for (int k = 0; k < BK; ++k) {
                const float4 a0 = *reinterpret_cast<const float4*>(&xs[k * BM + ty * 4]);
                const float4 a1 = *reinterpret_cast<const float4*>(&xs[k * BM + 64 + ty * 4]);
                const float4 b0 = *reinterpret_cast<const float4*>(&ys[k * BN + tx * 4]);
                const float4 b1 = *reinterpret_cast<const float4*>(&ys[k * BN + 64 + tx * 4]);
                const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
                for (int i = 0; i < 8; ++i)
#pragma unroll
                    for (int j = 0; j < 8; ++j) S::step(acc[i][j], a[i], bb[j]);
            }
        }
        if (has_next) store(buf ^ 1);
        __syncthreads();
    }

    // ---- epilogue: output offsets through Z's relation layout.  The row / column offset
    // tables reuse rowX / colY (every thread is past its last load: the loop ends on a barrier).
    if (tid < BM) {
        rowX[tid] = role_offset(p.zb, b) + role_offset(p.zm, min(m0 + tid, p.M - 1));
    } else {
        colY[tid - BM] = role_offset(p.zn, min(n0 + (tid - BM), p.N - 1));
    }
    __syncthreads();
    constexpr int G = P ? 2 : 4;  // consecutive output columns a thread owns
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int mi = (i < 4) ? ty * 4 + i : 64 + ty * 4 + (i - 4);
        const uint32_t m = m0 + mi;
        if (m >= p.M) continue;
        const int64_t zrow = rowX[mi];
        float rterm = 0.f;
        if (EPI == kEpiLse) rterm = p.rowmax[(uint64_t)b * p.M + m];
        if (EPI == kEpiSqExpand) rterm = p.xnorm[(uint64_t)b * p.M + m];
#pragma unroll
        for (int g = 0; g < 8 / G; ++g) {
            const int nb = P ? g * 32 + tx * 2 : g * 64 + tx * 4;
            const uint32_t n = n0 + nb;
            float v[G];
#pragma unroll
            for (int c = 0; c < G; ++c) {
                float a = acc[i][g * G + c];
                if (EPI == kEpiLse) {
                    if (n + c < p.N) {
                        if (a > 1e-30f) a = rterm + p.colmax[(uint64_t)b * p.N + n + c] + logf(a);
                        else a = lse_fallback(p, b, m, n + c);  // every exp-shifted product underflowed
                    }
                } else if (EPI == kEpiSqExpand) {
                    if (n + c < p.N) a = fmaxf(rterm + p.ynorm[(uint64_t)b * p.N + n + c] - 2.f * a, 0.f);
                }
                v[c] = p.alpha * a;
            }
            if (p.z_vec4 && n + G - 1 < p.N) {
                const int64_t off = zrow + colY[nb];
                if (p.out_bf16) {
                    uint32_t w[G / 2];
#pragma unroll
                    for (int h = 0; h < G / 2; ++h) {
                        const __nv_bfloat162 pr = __floats2bfloat162_rn(v[2 * h], v[2 * h + 1]);
                        w[h] = *reinterpret_cast<const uint32_t*>(&pr);
                    }
                    if (G == 4)
                        *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.z) + off) = make_uint2(w[0], w[G / 2 - 1]);
                    else
                        *reinterpret_cast<uint32_t*>(reinterpret_cast<__nv_bfloat16*>(p.z) + off) = w[0];
                } else if (G == 4) {
                    *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.z) + off) = make_float4(v[0], v[1 % G], v[2 % G], v[3 % G]);
                } else {
                    *reinterpret_cast<float2*>(reinterpret_cast<float*>(p.z) + off) = make_float2(v[0], v[1 % G]);
                }
            } else {
#pragma unroll
                for (int c = 0; c < G; ++c)
                    if (n + c < p.N) st_out(p.z, zrow + colY[nb + c], v[c], p.out_bf16);
            }
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
                float v = apply_op(p.op, ld1<TIn>(p.x, xo + role_offset(p.xk, k)),
                                   ld1<TIn>(p.y, yo + role_offset(p.yk, k)));
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
                float v = apply_op(p.op, ld1<TIn>(p.x, xo + role_offset(p.xk, k)),
                                   ld1<TIn>(p.y, yo + role_offset(p.yk, k)));
                if (p.agg == kMax) acc = fmaxf(acc, v);
                else if (p.agg == kMin) acc = fminf(acc, v);
                else acc += v;
            }
        }
        st_out(p.z, role_offset(p.zb, b) + role_offset(p.zm, m) + role_offset(p.zn, n), p.alpha * acc, p.out_bf16);
    }
}

// ---------------------------------------------------------------- factored-logsumexp / norm preparation
__device__ __forceinline__ int64_t prep_koff(const LsePrepParams& p, uint32_t k) {
    if (p.k_simple) {
        const uint32_t q = fdiv(k, p.k_sub);
        return (int64_t)q * p.k_ks + (int64_t)(k - q * p.k_sub.d) * p.k_ls;
    }
    return role_offset(p.k, k);
}

// mode 0: per row, max over the contracted range, then dst = exp(v - max) for every element.
// mode 1: per row, sum of squares over the contracted range (squared-distance expansion).
template <typename TIn>
__global__ void lse_prep_kernel(const __grid_constant__ LsePrepParams p, int row_per_thread) {
    if (!row_per_thread) {
        // one warp per row (contracted index contiguous in memory)
        const uint64_t warp = (blockIdx.x * (uint64_t)blockDim.x + threadIdx.x) / 32;
        const uint32_t lane = threadIdx.x % 32;
        const uint64_t rows = (uint64_t)p.nb * p.R;
        if (warp >= rows) return;
        const uint32_t r = warp % p.R, b = warp / p.R;
        const int64_t base = role_offset(p.b, b) + role_offset(p.r, r);
        float m = p.mode == 0 ? -INFINITY : 0.f;
        for (uint32_t k = lane; k < p.K; k += 32) {
            float v = ld1<TIn>(p.src, base + prep_koff(p, k));
            m = p.mode == 0 ? fmaxf(m, v) : fmaf(v, v, m);
        }
        for (int o = 16; o; o >>= 1) {
            float w = __shfl_xor_sync(0xffffffffu, m, o);
            m = p.mode == 0 ? fmaxf(m, w) : m + w;
        }
        if (lane == 0) p.rmax[warp] = m;
        if (p.mode == 0)
            for (uint32_t k = lane; k < p.K; k += 32) {
                int64_t off = base + prep_koff(p, k);
                p.dst[off] = expf(ld1<TIn>(p.src, off) - m);
            }
    } else {
        // rows contiguous in memory: 32 consecutive rows per CTA (one per lane, coalesced
        // across the warp), the 8 warps split the contracted range, shared-memory reduction
        __shared__ float red[8][32];
        const uint32_t lane = threadIdx.x & 31, w = threadIdx.x >> 5;
        const uint64_t rows = (uint64_t)p.nb * p.R;
        const uint64_t row = blockIdx.x * 32ull + lane;
        const bool valid = row < rows;
        const uint32_t r = valid ? (uint32_t)(row % p.R) : 0u, b = valid ? (uint32_t)(row / p.R) : 0u;
        const int64_t base = role_offset(p.b, b) + role_offset(p.r, r);
        float m = p.mode == 0 ? -INFINITY : 0.f;
        if (valid)
            for (uint32_t k = w; k < p.K; k += 8) {
                const float v = ld1<TIn>(p.src, base + prep_koff(p, k));
                m = p.mode == 0 ? fmaxf(m, v) : fmaf(v, v, m);
            }
        red[w][lane] = m;
        __syncthreads();
        if (w == 0) {
            for (int q = 1; q < 8; ++q) m = p.mode == 0 ? fmaxf(m, red[q][lane]) : m + red[q][lane];
            red[0][lane] = m;
            if (valid) p.rmax[row] = m;
        }
        __syncthreads();
        m = red[0][lane];
        if (p.mode == 0 && valid)
            for (uint32_t k = w; k < p.K; k += 8) {
                const int64_t off = base + prep_koff(p, k);
                p.dst[off] = expf(ld1<TIn>(p.src, off) - m);
            }
    }
}

template <class S, typename TIn, int EPI>
cudaError_t launch_tiled(const SemiringParams& p, unsigned grid, cudaStream_t s) {
    semiring_tiled<S, TIn, EPI><<<grid, NT, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_semiring(const SemiringParams& p, cudaStream_t s) {
    if (p.nb == 0 || p.M == 0 || p.N == 0) return cudaSuccess;
    if (p.K == 0) return cudaErrorInvalidValue;
    const uint64_t grid64 = (uint64_t)p.nb * ((p.M + BM - 1) / BM) * ((p.N + BN - 1) / BN);
    if (grid64 > 0x7fffffffull) return cudaErrorInvalidValue;
    const unsigned grid = (unsigned)grid64;
    const bool bf = p.in_bf16;
    if (p.rowmax) return launch_tiled<MulSum, float, kEpiLse>(p, grid, s);       // fp32 exp-shifted scratch
    if (p.xnorm) return launch_tiled<MulSum, float, kEpiSqExpand>(p, grid, s);   // fp32 inputs
    switch (p.op * 8 + p.agg) {
        case kMul * 8 + kSum:
            return bf ? launch_tiled<MulSum, __nv_bfloat16, kEpiPlain>(p, grid, s)
                      : launch_tiled<MulSum, float, kEpiPlain>(p, grid, s);
        case kSqdiff * 8 + kSum:
            return bf ? launch_tiled<SqdiffSum, __nv_bfloat16, kEpiPlain>(p, grid, s)
                      : launch_tiled<SqdiffSum, float, kEpiPlain>(p, grid, s);
        case kAdd * 8 + kMax:
            return bf ? launch_tiled<AddMax, __nv_bfloat16, kEpiPlain>(p, grid, s)
                      : launch_tiled<AddMax, float, kEpiPlain>(p, grid, s);
        case kAdd * 8 + kMin:
            return bf ? launch_tiled<AddMin, __nv_bfloat16, kEpiPlain>(p, grid, s)
                      : launch_tiled<AddMin, float, kEpiPlain>(p, grid, s);
        default:
            return launch_semiring_simple(p, s);
    }
}

cudaError_t launch_semiring_simple(const SemiringParams& p, cudaStream_t s) {
    const uint64_t total = (uint64_t)p.nb * p.M * p.N;
    if (total == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((total + 255) / 256 < 65536 ? (total + 255) / 256 : 65536);
    if (p.in_bf16) semiring_simple<__nv_bfloat16><<<blocks, 256, 0, s>>>(p);
    else semiring_simple<float><<<blocks, 256, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_lse_prep(const LsePrepParams& pin, cudaStream_t s) {
    LsePrepParams p = pin;
    p.k_simple = p.k.n == 1 && p.k.t[0].div == 1 && p.k.t[0].ext == p.K;
    if (p.k_simple) {
        p.k_sub = FastDiv(p.k.t[0].sub);
        p.k_ks = p.k.t[0].key_stride;
        p.k_ls = p.k.t[0].loc_stride;
    }
    const uint64_t rows = (uint64_t)p.nb * p.R;
    if (rows == 0) return cudaSuccess;
    // rows contiguous (the contracted index is not the fastest-moving one): thread per row
    const bool rpt = !(p.k.n > 0 && p.k.t[0].div == 1 && p.k.t[0].loc_stride == 1);
    const unsigned blocks = (unsigned)(rpt ? (rows + 31) / 32 : (rows * 32 + 255) / 256);
    if (p.in_bf16) lse_prep_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(p, rpt);
    else lse_prep_kernel<float><<<blocks, 256, 0, s>>>(p, rpt);
    return cudaGetLastError();
}

}  // namespace tra
