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
// Per thread: an 8 x 8 register tile.  Two kernels share the tile mapping and the
// epilogue:
//  * semiring_async -- fp32 operands laid out K-contiguous (X) and N-contiguous (Y)
//    in runs of 4: a 3-stage cp.async pipeline of 32-deep K tiles, no register
//    staging, one barrier per tile;
//  * semiring_tiled -- every other layout / bf16: 16-deep K tiles staged through
//    registers (float4 / 4 x bf16 loads where the layout allows, gathers otherwise).
// The K tail is padded with values whose join is the aggregation's identity, so the
// inner loop never branches.  Tuples are taken in pairs of consecutive k: max-plus and
// min-plus become two FADD and one 3-input FMNMX per two tuples.
#include <cuda_bf16.h>

#include <cfloat>
#include <cstdint>

#include "tra_internal.h"

namespace tra {
namespace {

constexpr int BM = 128, BN = 128, BK = 16, NT = 256;
constexpr int ABK = 32, ASTAGES = 3;  // async kernel: K-tile depth and pipeline stages
constexpr size_t kAsyncSmem = (size_t)ASTAGES * (BM * ABK + ABK * BN) * sizeof(float);
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

// the loads above with the check build's bounds test (n elements; pad where it fails)
template <typename T>
__device__ __forceinline__ float ld1c(const void* p, int64_t off, uint64_t n, int site, float pad) {
    return chk(off, n, site) ? ld1<T>(p, off) : pad;
}
template <typename T>
__device__ __forceinline__ float4 ld4c(const void* p, int64_t off, uint64_t n, int site, float pad) {
    return chk(off + 3, n, site) ? ld4<T>(p, off) : make_float4(pad, pad, pad, pad);
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

__device__ __forceinline__ void cp_async16(float* dst, const float* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------- semiring functors
// step: one join tuple; step2: two tuples of the same output (consecutive k).
// pad_x / pad_y: operand values for k beyond K whose join is the aggregation's identity.
struct MulSum {
    static __device__ __forceinline__ float init() { return 0.f; }
    static __device__ __forceinline__ float pad_x() { return 0.f; }
    static __device__ __forceinline__ float pad_y() { return 0.f; }
    static __device__ __forceinline__ void step2(float& acc, float x0, float y0, float x1, float y1) {
        acc = fmaf(x1, y1, fmaf(x0, y0, acc));
    }
};
struct SqdiffSum {
    static __device__ __forceinline__ float init() { return 0.f; }
    static __device__ __forceinline__ float pad_x() { return 0.f; }
    static __device__ __forceinline__ float pad_y() { return 0.f; }
    static __device__ __forceinline__ void step2(float& acc, float x0, float y0, float x1, float y1) {
        const float t0 = x0 - y0, t1 = x1 - y1;
        acc = fmaf(t1, t1, fmaf(t0, t0, acc));
    }
};
struct AddMax {
    static __device__ __forceinline__ float init() { return -INFINITY; }
    static __device__ __forceinline__ float pad_x() { return -INFINITY; }
    static __device__ __forceinline__ float pad_y() { return 0.f; }
    static __device__ __forceinline__ void step2(float& acc, float x0, float y0, float x1, float y1) {
        acc = max3(acc, x0 + y0, x1 + y1);
    }
};
struct AddMin {
    static __device__ __forceinline__ float init() { return INFINITY; }
    static __device__ __forceinline__ float pad_x() { return INFINITY; }
    static __device__ __forceinline__ float pad_y() { return 0.f; }
    static __device__ __forceinline__ void step2(float& acc, float x0, float y0, float x1, float y1) {
        acc = min3(acc, x0 + y0, x1 + y1);
    }
};

// Online logsumexp of one output over the contracted range, read straight from the
// operands (the factored form's fallback when its sum underflows; the simple kernel).
template <typename TIn>
__device__ __noinline__ float direct_lse(const SemiringParams& p, const void* x, const void* y, int64_t xo,
                                         int64_t yo) {
    float m = -INFINITY, s = 0.f;
    for (uint32_t k = 0; k < p.K; ++k) {
        float v = ld1c<TIn>(x, xo + role_offset(p.xk, k), p.x_elems, 114, -INFINITY) +
                  ld1c<TIn>(y, yo + role_offset(p.yk, k), p.y_elems, 114, 0.f);
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

__device__ __forceinline__ uint32_t n_tiles(const SemiringParams& p) {
    return p.nb * ((p.M + BM - 1) / BM) * ((p.N + BN - 1) / BN);
}

__device__ __forceinline__ void decode_tile(const SemiringParams& p, uint32_t t, uint32_t& b, uint32_t& m0,
                                            uint32_t& n0) {
    const uint32_t tiles_m = (p.M + BM - 1) / BM, tiles_n = (p.N + BN - 1) / BN;
    const uint32_t tn = t % tiles_n;
    t /= tiles_n;
    const uint32_t tm = t % tiles_m;
    b = t / tiles_m;
    m0 = tm * BM;
    n0 = tn * BN;
}

// Thread (ty, tx) owns rows ty*4+{0..3}, 64+ty*4+{0..3} and columns tx*4+{0..3},
// 64+tx*4+{0..3} of the tile.  The caller guarantees every shared buffer passed here is
// free (all threads past their last read of it).
// stg (BULK): a free 64 KB of shared memory.  When the output is fp32 and each of the tile's
// 128-column row segments is contiguous and 16-byte aligned in Z, the tile is staged there
// and leaves as one 512-byte bulk copy per row: the CTA waits only until shared memory has
// been read, and the writes to HBM drain while the next CTA on the SM computes (the CTAs of
// a wave finish together, so direct stores would all stall on the same write burst).
template <int EPI, bool BULK = false>
__device__ __forceinline__ void tile_epilogue(const SemiringParams& p, float (&acc)[8][8], uint32_t b, uint32_t m0,
                                              uint32_t n0, int64_t* rowZ, int64_t* colZ, float* rterms,
                                              float* cterms, float* stg = nullptr) {
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    if (tid < BM) {
        const uint32_t m = min(m0 + tid, p.M - 1);
        rowZ[tid] = role_offset(p.zb, b) + role_offset(p.zm, m);
        if (EPI == kEpiLse) rterms[tid] = p.rowmax[(uint64_t)b * p.M + m];
        if (EPI == kEpiSqExpand) rterms[tid] = p.xnorm[(uint64_t)b * p.M + m];
    } else {
        const uint32_t n = min(n0 + (tid - BM), p.N - 1);
        colZ[tid - BM] = role_offset(p.zn, n);
        if (EPI == kEpiLse) cterms[tid - BM] = p.colmax[(uint64_t)b * p.N + n];
        if (EPI == kEpiSqExpand) cterms[tid - BM] = p.ynorm[(uint64_t)b * p.N + n];
    }
    __syncthreads();
    // squared-distance guard: this thread saw an output whose expansion cancelled
    bool marked = false;
    if (BULK) {
        const bool rows_contiguous = __syncthreads_and(
            !p.out_bf16 && p.z_vec4 && p.z_device && (reinterpret_cast<uintptr_t>(p.z) & 15) == 0 && n0 + BN <= p.N &&
            (tid >= BN || colZ[tid] == colZ[0] + tid));
        if (rows_contiguous) {
            // guard, bounded per thread: min over its outputs of d against tau * (largest row norm
            // + largest column norm); this marks every tile the exact test would (and rows past M,
            // computed from a clamped row, can only add a mark)
            float dmin = INFINITY, rmx = 0.f, cmx = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int mi = (i < 4) ? ty * 4 + i : 64 + ty * 4 + (i - 4);
                const float rterm = EPI == kEpiPlain ? 0.f : rterms[mi];
                if (EPI == kEpiSqExpand) rmx = fmaxf(rmx, rterm);
#pragma unroll
                for (int g = 0; g < 2; ++g) {
                    const int nb = g * 64 + tx * 4;
                    float v[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        float a = acc[i][g * 4 + c];
                        if (EPI == kEpiLse) {
                            a = a > 1e-30f ? rterm + cterms[nb + c] + logf(a) : __int_as_float(0x7fc00000);
                        } else if (EPI == kEpiSqExpand) {
                            const float d = rterm + cterms[nb + c] - 2.f * a;
                            dmin = fminf(dmin, d);
                            if (i == 0) cmx = fmaxf(cmx, cterms[nb + c]);
                            a = fmaxf(d, 0.f);
                        }
                        v[c] = p.alpha * a;
                    }
                    *reinterpret_cast<float4*>(stg + mi * BN + nb) = make_float4(v[0], v[1], v[2], v[3]);
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            if (EPI == kEpiSqExpand) {
                const int any = __syncthreads_or(dmin < p.sq_tau * (rmx + cmx));
                if (tid == 0 && p.tile_mark) {
                    p.tile_mark[blockIdx.x] = any ? 1u : 0u;
                    if (any) p.tile_mark[gridDim.x] = p.gate_tag;  // this launch marked a tile
                }
            } else {
                __syncthreads();
            }
            if (tid < BM) {
                if (m0 + tid < p.M && chk(rowZ[tid] + colZ[0] + BN - 1, p.z_elems, 103)) {
                    float* dst = reinterpret_cast<float*>(p.z) + rowZ[tid] + colZ[0];
                    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                                 "r"((uint32_t)__cvta_generic_to_shared(stg + tid * BN)), "r"(BN * 4)
                                 : "memory");
                }
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
            }
            return;
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int mi = (i < 4) ? ty * 4 + i : 64 + ty * 4 + (i - 4);
        const uint32_t m = m0 + mi;
        if (m >= p.M) continue;
        const int64_t zrow = rowZ[mi];
        const float rterm = EPI == kEpiPlain ? 0.f : rterms[mi];
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            const int nb = g * 64 + tx * 4;
            const uint32_t n = n0 + nb;
            float v[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float a = acc[i][g * 4 + c];
                if (EPI == kEpiLse) {
                    // every exp-shifted product underflowed: mark the output, lse_fixup recomputes it
                    a = a > 1e-30f ? rterm + cterms[nb + c] + logf(a) : __int_as_float(0x7fc00000);
                } else if (EPI == kEpiSqExpand) {
                    const float s = rterm + cterms[nb + c], d = s - 2.f * a;
                    marked |= d < p.sq_tau * s && n + c < p.N;
                    a = fmaxf(d, 0.f);
                }
                v[c] = p.alpha * a;
            }
            if (p.z_vec4 && n + 3 < p.N) {
                const int64_t off = zrow + colZ[nb];
                if (!chk(off + 3, p.z_elems, 104)) continue;
                if (p.out_bf16) {
                    const __nv_bfloat162 lo = __floats2bfloat162_rn(v[0], v[1]);
                    const __nv_bfloat162 hi = __floats2bfloat162_rn(v[2], v[3]);
                    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.z) + off) =
                        make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
                } else {
                    *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.z) + off) = make_float4(v[0], v[1], v[2], v[3]);
                }
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    if (n + c < p.N && chk(zrow + colZ[nb + c], p.z_elems, 105))
                        st_out(p.z, zrow + colZ[nb + c], v[c], p.out_bf16);
            }
        }
    }
    if (EPI == kEpiSqExpand) {
        const int any = __syncthreads_or(marked);
        if (tid == 0 && p.tile_mark) {
            p.tile_mark[blockIdx.x] = any ? 1u : 0u;
            if (any) p.tile_mark[gridDim.x] = p.gate_tag;
        }
    }
}

// ---------------------------------------------------------------- cp.async pipelined kernel
// X tile in shared memory as [m][k] (32 floats per row, copied straight from the
// K-contiguous operand), Y tile as [k][n].  Per thread per 4 k: 8 LDS.128 of X (one per
// owned row), 2 LDS.128 of Y per k.
template <class S, int EPI>
__device__ __forceinline__ void async_tile(const SemiringParams& p, uint32_t tile) {
    extern __shared__ __align__(16) float dsm[];
    float* Xs = dsm;                          // [ASTAGES][BM * ABK]
    float* Ys = dsm + ASTAGES * BM * ABK;     // [ASTAGES][ABK * BN]
    __shared__ int64_t rowX[BM], colY[BN];

    const int tid = threadIdx.x;
    uint32_t b, m0, n0;
    decode_tile(p, tile, b, m0, n0);
    if (tid < BM) {
        rowX[tid] = role_offset(p.xb, b) + role_offset(p.xm, clamp_row(m0 + tid, p.M, false));
    } else {
        colY[tid - BM] = role_offset(p.yb, b) + role_offset(p.yn, clamp_row(n0 + (tid - BM), p.N, true));
    }
    __syncthreads();

    const float* __restrict__ xg = reinterpret_cast<const float*>(p.x);
    const float* __restrict__ yg = reinterpret_cast<const float*>(p.y);
    // copy assignment: X chunk (row (tid>>3) + 32i, k (tid&7)*4); Y chunk (k row (tid>>5) + 8i, n (tid&31)*4)
    const int xk = (tid & 7) * 4, xr = tid >> 3;
    const int yn = (tid & 31) * 4, yr = tid >> 5;
    auto issue = [&](int stage, uint32_t k0) {
        float* xs = Xs + stage * (BM * ABK);
        float* ys = Ys + stage * (ABK * BN);
        if (k0 + xk < p.K) {
            const int64_t ko = koff_x(p, k0 + xk);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if (chk(rowX[xr + 32 * i] + ko + 3, p.x_elems, 101)) {
                    cp_async16(&xs[(xr + 32 * i) * ABK + xk], xg + rowX[xr + 32 * i] + ko);
                } else {
                    const float px = S::pad_x();
                    *reinterpret_cast<float4*>(&xs[(xr + 32 * i) * ABK + xk]) = make_float4(px, px, px, px);
                }
            }
        } else {
            const float px = S::pad_x();
#pragma unroll
            for (int i = 0; i < 4; ++i)
                *reinterpret_cast<float4*>(&xs[(xr + 32 * i) * ABK + xk]) = make_float4(px, px, px, px);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int kr = yr + 8 * i;
            if (k0 + kr < p.K && chk(colY[yn] + koff_y(p, k0 + kr) + 3, p.y_elems, 102)) {
                cp_async16(&ys[kr * BN + yn], yg + colY[yn] + koff_y(p, k0 + kr));
            } else {
                const float py = S::pad_y();
                *reinterpret_cast<float4*>(&ys[kr * BN + yn]) = make_float4(py, py, py, py);
            }
        }
        cp_async_commit();
    };

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = S::init();

    const int ty = tid >> 4, tx = tid & 15;
    const uint32_t nkt = (p.K + ABK - 1) / ABK;
    issue(0, 0);
    if (nkt > 1) issue(1, ABK);
    else cp_async_commit();
    for (uint32_t kt = 0; kt < nkt; ++kt) {
        cp_async_wait<ASTAGES - 2>();  // this thread's copies of tile kt have landed
        __syncthreads();               // everyone's have, and tile kt-1's buffer is free
        if (kt + 2 < nkt) issue((kt + 2) % ASTAGES, (kt + 2) * ABK);
        else cp_async_commit();
        const int st = kt % ASTAGES;
        const float4* xs4 = reinterpret_cast<const float4*>(Xs + st * (BM * ABK));
        const float4* ys4 = reinterpret_cast<const float4*>(Ys + st * (ABK * BN));
#pragma unroll 2
        for (int kq = 0; kq < ABK / 4; ++kq) {
            float4 a[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r = (i < 4) ? ty * 4 + i : 64 + ty * 4 + (i - 4);
                a[i] = xs4[r * (ABK / 4) + kq];
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int k = kq * 4 + 2 * h;
                const float4 b0 = ys4[k * (BN / 4) + tx], b1 = ys4[k * (BN / 4) + 16 + tx];
                const float4 d0 = ys4[(k + 1) * (BN / 4) + tx], d1 = ys4[(k + 1) * (BN / 4) + 16 + tx];
                const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
                const float dd[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float x0 = h == 0 ? a[i].x : a[i].z;
                    const float x1 = h == 0 ? a[i].y : a[i].w;
#pragma unroll
                    for (int j = 0; j < 8; ++j) S::step2(acc[i][j], x0, bb[j], x1, dd[j]);
                }
            }
        }
    }
    cp_async_wait<0>();
    __syncthreads();
    // staging: the first 64 KB of the pipeline stages; row / column terms past it (in the last
    // Y stage)
    float* terms = Ys + 2 * (ABK * BN);
    tile_epilogue<EPI, true>(p, acc, b, m0, n0, rowX, colY, terms, terms + BM, dsm);
}

// One CTA per output tile; GATED (the squared-distance guard's fix-up pass): a persistent
// sweep over the tiles, computing only those whose word in p.tile_gate is nonzero.
template <class S, int EPI, bool GATED>
__global__ void __launch_bounds__(NT, 2) semiring_async(const __grid_constant__ SemiringParams p) {
    if (!GATED) {
        async_tile<S, EPI>(p, blockIdx.x);
        return;
    }
    const uint32_t n = n_tiles(p);
    if (p.tile_gate[n] != p.gate_tag) return;  // the producing launch marked no tile
    for (uint32_t t = blockIdx.x; t < n; t += gridDim.x) {
        if (p.tile_gate[t] == 0) continue;
        async_tile<S, EPI>(p, t);
        __syncthreads();  // shared memory is free again (the epilogue's bulk reads are done)
    }
}

// ---------------------------------------------------------------- register-staged kernel
template <class S, typename TIn, int EPI>
__device__ __forceinline__ void tiled_tile(const SemiringParams& p, uint32_t tile) {
    __shared__ __align__(16) float Xs[2][BK * BM];
    __shared__ __align__(16) float Ys[2][BK * BN];
    __shared__ int64_t rowX[BM], colY[BN];

    const int tid = threadIdx.x;
    uint32_t b, m0, n0;
    decode_tile(p, tile, b, m0, n0);
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
                float4 v = k < kv ? ld4c<TIn>(p.x, rowX[m] + koff_x(p, k0 + k), p.x_elems, 106, px) : make_float4(px, px, px, px);
                rx[4 * i] = v.x, rx[4 * i + 1] = v.y, rx[4 * i + 2] = v.z, rx[4 * i + 3] = v.w;
            }
        } else if (xmode == kLoadVecMN) {
            const int m = (tid & 31) * 4;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int k = (tid >> 5) + 8 * i;
                float4 v = k < kv ? ld4c<TIn>(p.x, rowX[m] + koff_x(p, k0 + k), p.x_elems, 106, px) : make_float4(px, px, px, px);
                rx[4 * i] = v.x, rx[4 * i + 1] = v.y, rx[4 * i + 2] = v.z, rx[4 * i + 3] = v.w;
            }
        } else {
            const int m = tid & (BM - 1);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int k = (tid >> 7) + 2 * i;
                rx[i] = k < kv ? ld1c<TIn>(p.x, rowX[m] + koff_x(p, k0 + k), p.x_elems, 107, px) : px;
            }
        }
        if (ymode == kLoadVecMN) {
            const int n = (tid & 31) * 4;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int k = (tid >> 5) + 8 * i;
                float4 v = k < kv ? ld4c<TIn>(p.y, colY[n] + koff_y(p, k0 + k), p.y_elems, 108, py) : make_float4(py, py, py, py);
                ry[4 * i] = v.x, ry[4 * i + 1] = v.y, ry[4 * i + 2] = v.z, ry[4 * i + 3] = v.w;
            }
        } else if (ymode == kLoadVecK) {
            const int n = tid & (BN - 1);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int k = ((tid >> 7) + 2 * i) * 4;
                float4 v = k < kv ? ld4c<TIn>(p.y, colY[n] + koff_y(p, k0 + k), p.y_elems, 108, py) : make_float4(py, py, py, py);
                ry[4 * i] = v.x, ry[4 * i + 1] = v.y, ry[4 * i + 2] = v.z, ry[4 * i + 3] = v.w;
            }
        } else {
            const int n = tid & (BN - 1);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int k = (tid >> 7) + 2 * i;
                ry[i] = k < kv ? ld1c<TIn>(p.y, colY[n] + koff_y(p, k0 + k), p.y_elems, 109, py) : py;
            }
        }
    };

    // ---- registers -> shared memory, [k][row] layout
    auto store = [&](int buf) {
        float* xs = Xs[buf];
        float* ys = Ys[buf];
        if (xmode == kLoadVecK) {
            const int m = tid & (BM - 1);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int k = ((tid >> 7) + 2 * i) * 4;
#pragma unroll
                for (int c = 0; c < 4; ++c) xs[(k + c) * BM + m] = rx[4 * i + c];
            }
        } else if (xmode == kLoadVecMN) {
            const int m = (tid & 31) * 4;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int k = (tid >> 5) + 8 * i;
                *reinterpret_cast<float4*>(&xs[k * BM + m]) = make_float4(rx[4 * i], rx[4 * i + 1], rx[4 * i + 2], rx[4 * i + 3]);
            }
        } else {
            const int m = tid & (BM - 1);
#pragma unroll
            for (int i = 0; i < 8; ++i) xs[((tid >> 7) + 2 * i) * BM + m] = rx[i];
        }
        if (ymode == kLoadVecMN) {
            const int n = (tid & 31) * 4;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int k = (tid >> 5) + 8 * i;
                *reinterpret_cast<float4*>(&ys[k * BN + n]) = make_float4(ry[4 * i], ry[4 * i + 1], ry[4 * i + 2], ry[4 * i + 3]);
            }
        } else if (ymode == kLoadVecK) {
            const int n = tid & (BN - 1);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int k = ((tid >> 7) + 2 * i) * 4;
#pragma unroll
                for (int c = 0; c < 4; ++c) ys[(k + c) * BN + n] = ry[4 * i + c];
            }
        } else {
            const int n = tid & (BN - 1);
#pragma unroll
            for (int i = 0; i < 8; ++i) ys[((tid >> 7) + 2 * i) * BN + n] = ry[i];
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
        const float4* xs4 = reinterpret_cast<const float4*>(Xs[buf]);
        const float4* ys4 = reinterpret_cast<const float4*>(Ys[buf]);
#pragma unroll 4
        for (int k = 0; k < BK; k += 2) {
            const float4 a0 = xs4[k * (BM / 4) + ty], a1 = xs4[k * (BM / 4) + 16 + ty];
            const float4 c0 = xs4[(k + 1) * (BM / 4) + ty], c1 = xs4[(k + 1) * (BM / 4) + 16 + ty];
            const float4 b0 = ys4[k * (BN / 4) + tx], b1 = ys4[k * (BN / 4) + 16 + tx];
            const float4 d0 = ys4[(k + 1) * (BN / 4) + tx], d1 = ys4[(k + 1) * (BN / 4) + 16 + tx];
            const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
            const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
            const float dd[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) S::step2(acc[i][j], a[i], bb[j], c[i], dd[j]);
        }
        if (has_next) store(buf ^ 1);
        __syncthreads();
    }
    // every thread is past its last read of Xs / Ys / rowX / colY (the loop ends on a barrier)
    tile_epilogue<EPI>(p, acc, b, m0, n0, rowX, colY, Xs[0], Ys[0]);
}

template <class S, typename TIn, int EPI, bool GATED>
__global__ void __launch_bounds__(NT, 2) semiring_tiled(const __grid_constant__ SemiringParams p) {
    if (!GATED) {
        tiled_tile<S, TIn, EPI>(p, blockIdx.x);
        return;
    }
    const uint32_t n = n_tiles(p);
    if (p.tile_gate[n] != p.gate_tag) return;
    for (uint32_t t = blockIdx.x; t < n; t += gridDim.x) {
        if (p.tile_gate[t] == 0) continue;
        tiled_tile<S, TIn, EPI>(p, t);
        __syncthreads();
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
                float v = apply_op(p.op, ld1c<TIn>(p.x, xo + role_offset(p.xk, k), p.x_elems, 110, 0.f),
                                   ld1c<TIn>(p.y, yo + role_offset(p.yk, k), p.y_elems, 111, 0.f));
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
                float v = apply_op(p.op, ld1c<TIn>(p.x, xo + role_offset(p.xk, k), p.x_elems, 110, 0.f),
                                   ld1c<TIn>(p.y, yo + role_offset(p.yk, k), p.y_elems, 111, 0.f));
                if (p.agg == kMax) acc = fmaxf(acc, v);
                else if (p.agg == kMin) acc = fminf(acc, v);
                else acc += v;
            }
        }
        const int64_t zo = role_offset(p.zb, b) + role_offset(p.zm, m) + role_offset(p.zn, n);
        if (chk(zo, p.z_elems, 112)) st_out(p.z, zo, p.alpha * acc, p.out_bf16);
    }
}

// ---------------------------------------------------------------- factored-logsumexp underflow fix-up
// Outputs whose exp-shifted sum underflowed carry a NaN mark from the tiled kernel; this pass
// (same 128 x 128 tiling) finds them and recomputes each with an online max / sum straight
// from the operands.  With finite inputs no true result is NaN.
__global__ void __launch_bounds__(NT) lse_fixup_kernel(const __grid_constant__ SemiringParams p) {
    __shared__ int64_t rowZ[BM], colZ[BN];
    if (p.mark_count && *p.mark_count == 0) return;  // the producer counted its marks: none
    const int tid = threadIdx.x;
    const uint32_t tiles_m = (p.M + BM - 1) / BM, tiles_n = (p.N + BN - 1) / BN;
    uint32_t t = blockIdx.x;
    const uint32_t tn = t % tiles_n;
    t /= tiles_n;
    const uint32_t tm = t % tiles_m;
    const uint32_t b = t / tiles_m;
    const uint32_t m0 = tm * BM, n0 = tn * BN;
    if (tid < BM) rowZ[tid] = role_offset(p.zb, b) + role_offset(p.zm, min(m0 + tid, p.M - 1));
    else colZ[tid - BM] = role_offset(p.zn, min(n0 + (tid - BM), p.N - 1));
    __syncthreads();
    const int c = tid & (BN - 1);
    if (n0 + c >= p.N) return;
    for (int r = tid >> 7; r < BM && m0 + r < p.M; r += NT / BN) {
        const int64_t off = rowZ[r] + colZ[c];
        if (!chk(off, p.z_elems, 113)) continue;
        const float v = p.out_bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.z)[off])
                                   : reinterpret_cast<const float*>(p.z)[off];
        if (v == v) continue;
        st_out(p.z, off, p.alpha * lse_fallback(p, b, m0 + r, n0 + c), p.out_bf16);
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
#pragma unroll 8
        for (uint32_t k = lane; k < p.K; k += 32) {
            float v = ld1c<TIn>(p.src, base + prep_koff(p, k), p.src_elems, 115, p.mode == 0 ? -INFINITY : 0.f);
            m = p.mode == 0 ? fmaxf(m, v) : fmaf(v, v, m);
        }
        for (int o = 16; o; o >>= 1) {
            float w = __shfl_xor_sync(0xffffffffu, m, o);
            m = p.mode == 0 ? fmaxf(m, w) : m + w;
        }
        if (lane == 0) p.rmax[warp] = m;
        if (p.mode == 0 && p.dst)
            for (uint32_t k = lane; k < p.K; k += 32) {
                int64_t off = base + prep_koff(p, k);
                if (chk(off, p.src_elems, 116)) p.dst[off] = expf(ld1<TIn>(p.src, off) - m);
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
#pragma unroll 8
            for (uint32_t k = w; k < p.K; k += 8) {
                const float v = ld1c<TIn>(p.src, base + prep_koff(p, k), p.src_elems, 115, p.mode == 0 ? -INFINITY : 0.f);
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
        if (p.mode == 0 && p.dst && valid)
            for (uint32_t k = w; k < p.K; k += 8) {
                const int64_t off = base + prep_koff(p, k);
                if (chk(off, p.src_elems, 116)) p.dst[off] = expf(ld1<TIn>(p.src, off) - m);
            }
    }
}

template <class S, typename TIn, int EPI, bool GATED = false>
cudaError_t launch_tiled(const SemiringParams& p, unsigned grid, cudaStream_t s) {
    if (!p.in_bf16 && p.x_mode == kLoadVecK && p.y_mode == kLoadVecMN) {
        // fp32, X contiguous along K and Y along N: the cp.async pipelined kernel
        cudaError_t e = cudaFuncSetAttribute(semiring_async<S, EPI, GATED>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kAsyncSmem);
        if (e != cudaSuccess) return e;
        semiring_async<S, EPI, GATED><<<grid, NT, kAsyncSmem, s>>>(p);
        return cudaGetLastError();
    }
    semiring_tiled<S, TIn, EPI, GATED><<<grid, NT, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

TRA_CHECK_READER(read_and_clear_check_semiring)

cudaError_t launch_semiring(const SemiringParams& p, cudaStream_t s) {
    if (p.nb == 0 || p.M == 0 || p.N == 0) return cudaSuccess;
    if (p.K == 0) return cudaErrorInvalidValue;
    const uint64_t grid64 = (uint64_t)p.nb * ((p.M + BM - 1) / BM) * ((p.N + BN - 1) / BN);
    if (grid64 > 0x7fffffffull) return cudaErrorInvalidValue;
    const unsigned grid = (unsigned)grid64;
    const bool bf = p.in_bf16;
    if (p.rowmax) {  // fp32 exp-shifted scratch, then the underflow fix-up
        SemiringParams q = p;
        q.in_bf16 = 0;
        cudaError_t e = launch_tiled<MulSum, float, kEpiLse>(q, grid, s);
        if (e != cudaSuccess) return e;
        lse_fixup_kernel<<<grid, NT, 0, s>>>(p);
        return cudaGetLastError();
    }
    if (p.xnorm) {  // fp32 inputs: the expansion, then the direct form over the tiles it marked
        cudaError_t e = launch_tiled<MulSum, float, kEpiSqExpand>(p, grid, s);
        if (e != cudaSuccess || !p.tile_mark) return e;
        SemiringParams q = p;
        q.op = kSqdiff;
        q.xnorm = q.ynorm = nullptr;
        q.tile_gate = p.tile_mark;
        q.tile_mark = nullptr;
        return launch_sqdist_fixup(q, s);
    }
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

cudaError_t launch_sqdist_fixup(const SemiringParams& p, cudaStream_t s) {
    if (p.nb == 0 || p.M == 0 || p.N == 0) return cudaSuccess;
    if (!p.tile_gate || p.in_bf16) return cudaErrorInvalidValue;
    const uint64_t tiles = (uint64_t)p.nb * ((p.M + BM - 1) / BM) * ((p.N + BN - 1) / BN);
    if (tiles > 0x7fffffffull) return cudaErrorInvalidValue;
    // persistent sweep: two CTAs per SM (the kernels' occupancy) walk the tiles' words and
    // compute the marked tiles; with none marked the pass costs one read per tile
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const uint64_t grid = tiles < 2ull * (uint64_t)sms ? tiles : 2ull * (uint64_t)sms;
    return launch_tiled<SqdiffSum, float, kEpiPlain, true>(p, (unsigned)grid, s);
}

cudaError_t launch_lse_fixup(const SemiringParams& p, cudaStream_t s) {
    if (p.nb == 0 || p.M == 0 || p.N == 0) return cudaSuccess;
    const uint64_t grid64 = (uint64_t)p.nb * ((p.M + BM - 1) / BM) * ((p.N + BN - 1) / BN);
    if (grid64 > 0x7fffffffull) return cudaErrorInvalidValue;
    lse_fixup_kernel<<<(unsigned)grid64, NT, 0, s>>>(p);
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
