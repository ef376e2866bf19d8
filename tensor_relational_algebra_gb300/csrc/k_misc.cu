// HBM-bound kernels of the TRA path ("EinDecomp ... tensor relational algebra"):
//   * repartition (section 2.2: change the partitioning of a relation),
//   * unary aggregation over contracted labels (section 2.2 aggregation with no
//     join partner; the logsumexp / max rows of the attention softmax in the
//     multi-head-attention example of section 2.1),
//   * join with aggregation "none" (the element-wise example of section 2.1, with
//     broadcast operands, e.g. exp(Scores - L)),
//   * ordered combine of per-join-tuple partials (section 2.2 aggregation, GROUP BY
//     the output key).
#include <cuda_bf16.h>

#include <cstdint>

#include "tra_internal.h"

namespace tra {

namespace {

__device__ __forceinline__ float ld_f(const void* p, int64_t off, int bf16) {
    return bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[off])
                : reinterpret_cast<const float*>(p)[off];
}
__device__ __forceinline__ void st_f(void* p, int64_t off, float v, int bf16) {
    if (bf16)
        reinterpret_cast<__nv_bfloat16*>(p)[off] = __float2bfloat16_rn(v);
    else
        reinterpret_cast<float*>(p)[off] = v;
}

// ---------------------------------------------------------------- repartition
// Source offset (in elements) of the element that sits at destination position e:
// decode e into (destination key, local index) per dimension, rebuild the global index
// g, and re-encode g under the source partition.
__device__ __forceinline__ int64_t repart_src_offset(const RepartParams& p, uint32_t e) {
    uint32_t key = fdiv(e, p.dst_sub_total);
    uint32_t loc = e - key * p.dst_sub_total.d;
    int64_t so = 0;
    for (int i = p.rank - 1; i >= 0; --i) {
        const uint32_t kq = fdiv(key, p.dst_grid[i]);
        const uint32_t ki = key - kq * p.dst_grid[i].d;
        key = kq;
        const uint32_t lq = fdiv(loc, p.dst_sub[i]);
        const uint32_t li = loc - lq * p.dst_sub[i].d;
        loc = lq;
        const uint32_t g = ki * p.dst_sub[i].d + li;
        const uint32_t sq = fdiv(g, p.src_sub[i]);
        so += (int64_t)sq * p.src_key_stride[i] + (int64_t)(g - sq * p.src_sub[i].d) * p.src_loc_stride[i];
    }
    return so;
}

// Destination-ordered copy.  A warp takes chunks of 128 consecutive destination vectors
// (V = up to 16 bytes).  The source is contiguous over runs of G vectors (G = 1, 2 or 4
// divides the run length shared by both layouts), so each lane decodes the source offset
// of 4 / G segments and the lanes that copy a segment read its offset by shuffle.  Copy
// instruction j of the warp then reads segments 32j / G .. and writes 32 consecutive
// vectors, and each lane has 4 loads in flight before its stores.  Grid: persistent.
template <typename V, int G>
__global__ void __launch_bounds__(256) repartition_kernel(const __grid_constant__ RepartParams p) {
    const V* __restrict__ src = reinterpret_cast<const V*>(p.src);
    V* __restrict__ dst = reinterpret_cast<V*>(p.dst);
    const int lane = threadIdx.x & 31;
    const int vsh = __ffs(p.vec_elems) - 1;  // vec_elems is a power of two; segments start on vectors
    const uint64_t n_chunks = (p.n_vec + 127) / 128;
    const uint64_t warps = ((uint64_t)gridDim.x * blockDim.x) >> 5;
    for (uint64_t chunk = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; chunk < n_chunks; chunk += warps) {
        const uint64_t c0 = chunk * 128;
        int64_t seg[4 / G];
#pragma unroll
        for (int i = 0; i < 4 / G; ++i) {
            const uint64_t v = c0 + (uint64_t)(lane + 32 * i) * G;
            seg[i] = v < p.n_vec ? repart_src_offset(p, (uint32_t)(v << vsh)) >> vsh : 0;
        }
        V val[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int pos = 32 * j + lane;
            const int64_t so = __shfl_sync(0xffffffffu, seg[(32 * j) / (32 * G)], (pos / G) & 31) + pos % G;
            if (c0 + pos < p.n_vec) val[j] = chk(so, p.n_vec, 201) ? __ldcs(src + so) : V{};
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (c0 + 32 * j + lane < p.n_vec) dst[c0 + 32 * j + lane] = val[j];
    }
}

template <typename V>
cudaError_t launch_repartition_v(const RepartParams& p, unsigned g, cudaStream_t s) {
    switch (p.group) {
        case 4: repartition_kernel<V, 4><<<g, 256, 0, s>>>(p); break;
        case 2: repartition_kernel<V, 2><<<g, 256, 0, s>>>(p); break;
        default: repartition_kernel<V, 1><<<g, 256, 0, s>>>(p); break;
    }
    return cudaGetLastError();
}

// ---------------------------------------------------------------- unary aggregation
template <int AGG>
__device__ __forceinline__ void agg_step(float& m, float& s, float v) {
    if (AGG == kLse) {
        if (v > m) {
            s = s * __expf(m - v) + 1.f;
            m = v;
        } else {
            s += __expf(v - m);
        }
    } else if (AGG == kMax) {
        m = fmaxf(m, v);
    } else if (AGG == kMin) {
        m = fminf(m, v);
    } else {
        s += v;
    }
}

template <int AGG>
__device__ __forceinline__ void agg_merge(float& m, float& s, float m2, float s2) {
    if (AGG == kLse) {
        const float mm = fmaxf(m, m2);
        if (mm == -INFINITY) return;
        if (mm == INFINITY) {
            m = INFINITY;
            s = 1.f;
            return;
        }
        s = s * __expf(m - mm) + s2 * __expf(m2 - mm);
        m = mm;
    } else if (AGG == kMax) {
        m = fmaxf(m, m2);
    } else if (AGG == kMin) {
        m = fminf(m, m2);
    } else {
        s += s2;
    }
}

template <int AGG>
__device__ __forceinline__ void agg_group16(float& m, float& s, const float4 (&v)[4]) {
    if (AGG == kLse) {
        float cm = m;
#pragma unroll
        for (int u = 0; u < 4; ++u) cm = fmaxf(cm, fmaxf(fmaxf(v[u].x, v[u].y), fmaxf(v[u].z, v[u].w)));
        if (cm == -INFINITY) return;  // nothing but empty / -inf values so far
        if (cm == INFINITY) {         // the result is +inf from here on
            m = INFINITY;
            s = 1.f;
            return;
        }
        s *= __expf(m - cm);  // m == -inf gives 0
        m = cm;
#pragma unroll
        for (int u = 0; u < 4; ++u)
            s += (__expf(v[u].x - m) + __expf(v[u].y - m)) + (__expf(v[u].z - m) + __expf(v[u].w - m));
    } else {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            agg_step<AGG>(m, s, v[u].x);
            agg_step<AGG>(m, s, v[u].y);
            agg_step<AGG>(m, s, v[u].z);
            agg_step<AGG>(m, s, v[u].w);
        }
    }
}

// One warp per output row.
template <int AGG>
__global__ void row_reduce_kernel(const __grid_constant__ RowReduceParams p) {
    const uint64_t warp = (blockIdx.x * (uint64_t)blockDim.x + threadIdx.x) / 32;
    const int lane = threadIdx.x % 32;
    if (warp >= p.R) return;
    const uint32_t r = (uint32_t)warp;
    const int64_t xo = role_offset(p.xr, r);
    float m = AGG == kMin ? INFINITY : -INFINITY, s = 0.f;
    if (p.k_affine && !p.in_bf16 && (xo % 4) == 0 && (p.K % 4) == 0 && ((uintptr_t)p.x % 16) == 0 &&
        chk(xo + (int64_t)p.K - 1, p.x_elems, 202)) {
        // 4 float4 loads in flight per lane; each group of 16 values folds in at once (for
        // logsumexp: one rescale per group, one exp per value); padding is the identity of the
        // aggregation
        const float4* row = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p.x) + xo);
        const uint32_t K4 = p.K / 4;
        const float pad = AGG == kMin ? INFINITY : (AGG == kSum ? 0.f : -INFINITY);
        for (uint32_t k0 = lane; k0 < K4; k0 += 128) {
            float4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                v[u] = k0 + 32 * u < K4 ? __ldcs(row + k0 + 32 * u) : make_float4(pad, pad, pad, pad);
            agg_group16<AGG>(m, s, v);
        }
    } else if (p.k_affine) {
        for (uint32_t k = lane; k < p.K; k += 32)
            if (chk(xo + k, p.x_elems, 203)) agg_step<AGG>(m, s, ld_f(p.x, xo + k, p.in_bf16));
    } else {
        for (uint32_t k = lane; k < p.K; k += 32) {
            const int64_t o = xo + role_offset(p.xk, k);
            if (chk(o, p.x_elems, 203)) agg_step<AGG>(m, s, ld_f(p.x, o, p.in_bf16));
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        agg_merge<AGG>(m, s, m2, s2);
    }
    if (lane == 0) {
        float v;
        if (AGG == kLse) v = m == -INFINITY ? m : m + logf(s);
        else if (AGG == kSum) v = s;
        else v = m;
        const int64_t zo = role_offset(p.zr, r);
        if (chk(zo, p.z_elems, 204)) st_f(p.z, zo, p.alpha * v, p.out_bf16);
    }
}

// ---------------------------------------------------------------- join with aggregation "none"
__device__ __forceinline__ float ew_op(int op, float x, float y) {
    switch (op) {
        case kMul: return x * y;
        case kAdd: return x + y;
        case kSqdiff: { float t = x - y; return t * t; }
        case kSub: return x - y;
        case kExpsub: return __expf(x - y);
        default: return x;
    }
}

// One warp per run of I contiguous output elements.
__global__ void elementwise_kernel(const __grid_constant__ ElementwiseParams p) {
    const uint64_t run = (blockIdx.x * (uint64_t)blockDim.x + threadIdx.x) / 32;
    const int lane = threadIdx.x % 32;
    if (run >= p.n_runs) return;
    const uint32_t e = (uint32_t)(run * p.I);
    uint32_t key = fdiv(e, p.sub_total);
    uint32_t loc = e - key * p.sub_total.d;
    int64_t xo = 0, yo = 0;
    for (int i = p.rank - 1; i >= 0; --i) {
        const uint32_t kq = fdiv(key, p.grid[i]);
        const uint32_t ki = key - kq * p.grid[i].d;
        key = kq;
        const uint32_t lq = fdiv(loc, p.sub[i]);
        const uint32_t li = loc - lq * p.sub[i].d;
        loc = lq;
        xo += (int64_t)ki * p.x_ks[i] + (int64_t)li * p.x_ls[i];
        yo += (int64_t)ki * p.y_ks[i] + (int64_t)li * p.y_ls[i];
    }
    const int last = p.rank - 1;
    const int64_t xs = p.x_ls[last], ys = p.y_ls[last];
    // fp32 operands, X contiguous along the run, Y contiguous or broadcast, everything
    // 4-aligned: 16-byte loads, 4 outputs per lane per step
    if (!p.in_bf16 && xs == 1 && (ys == 0 || ys == 1 || !p.y) && (p.I & 3) == 0 && (e & 3) == 0 &&
        (xo & 3) == 0 && (ys != 1 || (yo & 3) == 0) && ((uintptr_t)p.x & 15) == 0 &&
        (!p.y || ys != 1 || ((uintptr_t)p.y & 15) == 0) && ((uintptr_t)p.z & (p.out_bf16 ? 7 : 15)) == 0 &&
        chk(xo + p.I - 1, p.x_elems, 205) && (!p.y || chk(yo + (ys ? p.I - 1 : 0), p.y_elems, 206)) &&
        chk((int64_t)e + p.I - 1, p.total, 207)) {
        const float* xr = reinterpret_cast<const float*>(p.x) + xo;
        const float* yr = p.y ? reinterpret_cast<const float*>(p.y) + yo : nullptr;
        const float yb = (p.y && ys == 0) ? yr[0] : 0.f;
        for (uint32_t j = lane * 4; j < p.I; j += 128) {
            const float4 xv = __ldcs(reinterpret_cast<const float4*>(xr + j));
            const float4 yv = (p.y && ys == 1) ? __ldg(reinterpret_cast<const float4*>(yr + j)) : make_float4(yb, yb, yb, yb);
            const float r0 = p.alpha * ew_op(p.op, xv.x, yv.x), r1 = p.alpha * ew_op(p.op, xv.y, yv.y);
            const float r2 = p.alpha * ew_op(p.op, xv.z, yv.z), r3 = p.alpha * ew_op(p.op, xv.w, yv.w);
            if (p.out_bf16) {
                const __nv_bfloat162 lo = __floats2bfloat162_rn(r0, r1), hi = __floats2bfloat162_rn(r2, r3);
                __stcs(reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.z) + e + j),
                       make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi)));
            } else {
                __stcs(reinterpret_cast<float4*>(reinterpret_cast<float*>(p.z) + e + j), make_float4(r0, r1, r2, r3));
            }
        }
        return;
    }
    for (uint32_t j = lane; j < p.I; j += 32) {
        const int64_t xi = xo + (int64_t)j * xs, yi = yo + (int64_t)j * ys;
        if (!chk(xi, p.x_elems, 205) || (p.y && !chk(yi, p.y_elems, 206)) || !chk((int64_t)e + j, p.total, 207))
            continue;
        const float x = ld_f(p.x, xi, p.in_bf16);
        const float y = p.y ? ld_f(p.y, yi, p.in_bf16) : 0.f;
        st_f(p.z, (int64_t)e + j, p.alpha * ew_op(p.op, x, y), p.out_bf16);
    }
}

// Flat form of the join above (see ElementwiseParams::flat): one thread per 8 consecutive
// elements of Z, two 16-byte loads of X (and of Y when laid out as Z), one store of 8 results.
template <int OP, bool OUT_BF16>
__global__ void __launch_bounds__(256) elementwise_flat_kernel(const __grid_constant__ ElementwiseParams p) {
    const uint64_t c = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x;
    if (c * 8 >= p.total) return;
    const uint64_t e = c * 8;
    if (!chk((int64_t)e + 7, p.total, 208) || !chk((int64_t)e + 7, p.x_elems, 208) ||
        (p.y && !chk(p.flat == 1 ? (int64_t)e + 7 : (int64_t)(e / p.y_div), p.y_elems, 209)))
        return;
    const float* xr = reinterpret_cast<const float*>(p.x) + e;
    const float4 x0 = *reinterpret_cast<const float4*>(xr), x1 = *reinterpret_cast<const float4*>(xr + 4);
    float4 y0 = make_float4(0.f, 0.f, 0.f, 0.f), y1 = y0;
    if (p.y) {
        if (p.flat == 1) {
            const float* yr = reinterpret_cast<const float*>(p.y) + e;
            y0 = *reinterpret_cast<const float4*>(yr);
            y1 = *reinterpret_cast<const float4*>(yr + 4);
        } else {
            const float yb = __ldg(reinterpret_cast<const float*>(p.y) + e / p.y_div);
            y0 = y1 = make_float4(yb, yb, yb, yb);
        }
    }
    const float r[8] = {p.alpha * ew_op(OP, x0.x, y0.x), p.alpha * ew_op(OP, x0.y, y0.y), p.alpha * ew_op(OP, x0.z, y0.z),
                        p.alpha * ew_op(OP, x0.w, y0.w), p.alpha * ew_op(OP, x1.x, y1.x), p.alpha * ew_op(OP, x1.y, y1.y),
                        p.alpha * ew_op(OP, x1.z, y1.z), p.alpha * ew_op(OP, x1.w, y1.w)};
    if (OUT_BF16) {
        __nv_bfloat162 h[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(r[2 * i], r[2 * i + 1]);
        *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.z) + e) = *reinterpret_cast<const uint4*>(h);
    } else {
        float* zr = reinterpret_cast<float*>(p.z) + e;
        *reinterpret_cast<float4*>(zr) = make_float4(r[0], r[1], r[2], r[3]);
        *reinterpret_cast<float4*>(zr + 4) = make_float4(r[4], r[5], r[6], r[7]);
    }
}

template <int OP>
cudaError_t launch_flat(const ElementwiseParams& p, cudaStream_t s) {
    const unsigned blocks = (unsigned)((p.total / 8 + 255) / 256);
    if (p.out_bf16) elementwise_flat_kernel<OP, true><<<blocks, 256, 0, s>>>(p);
    else elementwise_flat_kernel<OP, false><<<blocks, 256, 0, s>>>(p);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- ordered combine of partials
__global__ void combine_kernel(const __grid_constant__ CombineParams p) {
    const uint64_t total = p.n_groups * p.z_sub;
    for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < total;
         i += (uint64_t)gridDim.x * blockDim.x) {
        const uint64_t g = i / p.z_sub, l = i % p.z_sub;
        const float* part = p.partials + g * p.n_agg * p.z_sub + l;
        float acc = part[0];
        for (uint64_t c = 1; c < p.n_agg; ++c) {
            const float v = part[c * p.z_sub];
            switch (p.agg) {
                case kMax: acc = fmaxf(acc, v); break;
                case kMin: acc = fminf(acc, v); break;
                case kLse: {
                    const float m = fmaxf(acc, v);
                    if (m != -INFINITY) acc = m + logf(expf(acc - m) + expf(v - m));
                    break;
                }
                default: acc += v;
            }
        }
        st_f(p.z, (int64_t)i, p.alpha * acc, p.out_bf16);
    }
}

unsigned grid_for(uint64_t work, unsigned per_block) {
    uint64_t b = (work + per_block - 1) / per_block;
    if (b > 152ull * 64) b = 152ull * 64;
    return (unsigned)(b ? b : 1);
}

// CTAs for a grid-stride kernel: enough to fill every SM at its occupancy, no more than
// the work needs.
template <typename K>
unsigned persistent_grid(uint64_t work, unsigned per_block, K kernel, int max_per_sm = 64) {
    int dev = 0, sms = 0, per_sm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 256, 0) != cudaSuccess || per_sm < 1) {
        (void)cudaGetLastError();
        per_sm = 4;
    }
    if (per_sm > max_per_sm) per_sm = max_per_sm;
    const uint64_t need = (work + per_block - 1) / per_block;
    const uint64_t full = (uint64_t)(sms > 0 ? sms : 1) * per_sm;
    return (unsigned)(need < full ? (need ? need : 1) : full);
}

}  // namespace

TRA_CHECK_READER(read_and_clear_check_misc)

cudaError_t launch_repartition(const RepartParams& p, cudaStream_t s) {
    if (p.n_vec == 0) return cudaSuccess;
    const unsigned g = persistent_grid(p.n_vec, 256 * 4, repartition_kernel<uint4, 4>);
    switch (p.vec_bytes) {
        case 16: return launch_repartition_v<uint4>(p, g, s);
        case 8: return launch_repartition_v<uint2>(p, g, s);
        case 4: return launch_repartition_v<uint32_t>(p, g, s);
        case 2: return launch_repartition_v<uint16_t>(p, g, s);
        case 1: return launch_repartition_v<uint8_t>(p, g, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_row_reduce(const RowReduceParams& p, cudaStream_t s) {
    if (p.R == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)(((uint64_t)p.R * 32 + 255) / 256);
    switch (p.agg) {
        case kLse: row_reduce_kernel<kLse><<<blocks, 256, 0, s>>>(p); break;
        case kMax: row_reduce_kernel<kMax><<<blocks, 256, 0, s>>>(p); break;
        case kMin: row_reduce_kernel<kMin><<<blocks, 256, 0, s>>>(p); break;
        case kSum: row_reduce_kernel<kSum><<<blocks, 256, 0, s>>>(p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_elementwise(const ElementwiseParams& p, cudaStream_t s) {
    if (p.n_runs == 0) return cudaSuccess;
    if (p.flat && p.total / 8 <= 0xffffffffull * 256) {
        switch (p.op) {
            case kMul: return launch_flat<kMul>(p, s);
            case kAdd: return launch_flat<kAdd>(p, s);
            case kSqdiff: return launch_flat<kSqdiff>(p, s);
            case kSub: return launch_flat<kSub>(p, s);
            case kExpsub: return launch_flat<kExpsub>(p, s);
            case kId: return launch_flat<kId>(p, s);
            default: break;
        }
    }
    const uint64_t threads = p.n_runs * 32;
    elementwise_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(p);
    return cudaGetLastError();
}

namespace {

// One CTA per 32 rows x 128 contracted indices of one batch: the tile's row and contracted
// offsets are formed once (shared memory), the tile is read along the index that is contiguous
// in the operand (k when k_fast), staged in shared memory, and written along k as bf16 pairs,
// so both sides coalesce whatever the operand's relation layout.
constexpr uint32_t kSplitTR = 32, kSplitTK = 128;

__global__ void __launch_bounds__(256) split3_kernel(const __grid_constant__ Split3Params p) {
    constexpr uint32_t TR = kSplitTR, TK = kSplitTK;
    __shared__ float t[TR][TK + 1];
    __shared__ int64_t roff[TR], koff[TK];
    __shared__ float rsh[TR];
    const uint32_t tiles_k = (p.K + TK - 1) / TK, tiles_r = (p.R + TR - 1) / TR;
    const uint32_t kt = blockIdx.x % tiles_k, rest = blockIdx.x / tiles_k;
    const uint32_t rt = rest % tiles_r, b = rest / tiles_r;
    const uint32_t r0 = rt * TR, k0 = kt * TK;
    const uint32_t tid = threadIdx.x;
    if (tid < TR) {
        const uint32_t r = min(r0 + tid, p.R - 1);
        roff[tid] = role_offset(p.b, b) + role_offset(p.r, r);
        rsh[tid] = p.shift ? p.shift[(uint64_t)b * p.R + r] : 0.f;
    } else if (tid < TR + TK && !p.k_dense) {
        koff[tid - TR] = role_offset(p.k, min(k0 + tid - TR, p.K - 1));
    }
    __syncthreads();
    const uint32_t lane = tid & 31, w = tid >> 5;
    if (p.k_fast) {
        // warp w reads rows w, w + 8, ...; lanes along k
#pragma unroll
        for (uint32_t i = 0; i < TR / 8; ++i) {
            const uint32_t rl = w + 8 * i;
            if (r0 + rl >= p.R) continue;
            const float* row = p.src + roff[rl];
#pragma unroll
            for (uint32_t h = 0; h < TK / 32; ++h) {
                const uint32_t kl = lane + 32 * h;
                const int64_t o = p.k_dense ? (int64_t)(k0 + kl) : koff[kl];
                if (k0 + kl < p.K) t[rl][kl] = chk(roff[rl] + o, p.src_elems, 210) ? row[o] : 0.f;
            }
        }
    } else {
        // lanes along the rows
        const bool rv = r0 + lane < p.R;
        const float* row = p.src + roff[lane];
#pragma unroll 4
        for (uint32_t i = 0; i < TK / 8; ++i) {
            const uint32_t kl = w + 8 * i;
            const int64_t o = p.k_dense ? (int64_t)(k0 + kl) * p.k_ls : koff[kl];
            if (rv && k0 + kl < p.K) t[lane][kl] = chk(roff[lane] + o, p.src_elems, 210) ? row[o] : 0.f;
        }
    }
    __syncthreads();
    // write: warp w, rows w, w + 8, ...; lane holds k = 2 lane, 2 lane + 1 of each 64
    const uint64_t K = p.K;
#pragma unroll
    for (uint32_t i = 0; i < TR / 8; ++i) {
        const uint32_t rl = w + 8 * i, r = r0 + rl;
        if (r >= p.R) continue;
        __nv_bfloat16* out = p.dst + ((uint64_t)b * p.Rp + r) * p.K3p;
        if (!chk(((int64_t)b * p.Rp + r) * p.K3p + p.K3p - 1, (uint64_t)p.nb * p.Rp * p.K3p, 211)) continue;
#pragma unroll
        for (uint32_t h = 0; h < TK / 64; ++h) {
            const uint32_t kl = 2 * lane + 64 * h, k = k0 + kl;
            if (k >= p.K) continue;
            float v0 = t[rl][kl], v1 = k + 1 < p.K ? t[rl][kl + 1] : 0.f;
            if (p.shift) {
                v0 = expf(v0 - rsh[rl]);
                v1 = k + 1 < p.K ? expf(v1 - rsh[rl]) : 0.f;
            }
            const __nv_bfloat162 hi = __floats2bfloat162_rn(v0, v1);
            const float2 hf = __bfloat1622float2(hi);
            const __nv_bfloat162 lo = __floats2bfloat162_rn(v0 - hf.x, v1 - hf.y);
            if ((K & 1) == 0) {  // k even, so every pair is 4-byte aligned
                *reinterpret_cast<__nv_bfloat162*>(out + k) = hi;
                *reinterpret_cast<__nv_bfloat162*>(out + K + k) = p.is_y ? lo : hi;
                *reinterpret_cast<__nv_bfloat162*>(out + 2 * K + k) = p.is_y ? hi : lo;
            } else {
                const __nv_bfloat16 e[3][2] = {{hi.x, hi.y}, {p.is_y ? lo.x : hi.x, p.is_y ? lo.y : hi.y},
                                               {p.is_y ? hi.x : lo.x, p.is_y ? hi.y : lo.y}};
                for (int sgm = 0; sgm < 3; ++sgm) {
                    out[sgm * K + k] = e[sgm][0];
                    if (k + 1 < p.K) out[sgm * K + k + 1] = e[sgm][1];
                }
            }
        }
        if (kt == tiles_k - 1)  // the row's zero padding
            for (uint64_t j = 3 * K + lane; j < p.K3p; j += 32) out[j] = __float2bfloat16_rn(0.f);
    }
}

}  // namespace

namespace {

// Phase 1 of the row statistics: one CTA per 32 rows x one chunk of the contracted range.
// k_fast: warp w takes rows w, w + 8, w + 16, w + 24 with its lanes along k; otherwise the lanes
// take the 32 rows and the 8 warps split the chunk.  Loads are unrolled for memory parallelism.
constexpr uint32_t kStatsChunk = 2048;  // contracted indices per phase-1 CTA at most

__global__ void __launch_bounds__(256) split3_stats_kernel(const __grid_constant__ Split3StatsParams p) {
    __shared__ float red[8][32];
    __shared__ int64_t koff[kStatsChunk];
    const uint32_t tiles_r = (p.R + 31) / 32;
    const uint32_t c = blockIdx.x % p.kc, rest = blockIdx.x / p.kc;
    const uint32_t rt = rest % tiles_r, b = rest / tiles_r;
    const uint32_t r0 = rt * 32;
    const uint32_t per = (p.K + p.kc - 1) / p.kc, k_lo = c * per, k_hi = min(p.K, k_lo + per);
    const uint32_t lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const float init = p.mode == 0 ? -INFINITY : 0.f;
    const int64_t bo = role_offset(p.b, b);
    auto acc = [&](float a, float v) { return p.mode == 0 ? fmaxf(a, v) : fmaf(v, v, a); };
    const uint64_t rows = (uint64_t)p.nb * p.R;
    for (uint32_t k = k_lo + threadIdx.x; k < k_hi; k += blockDim.x) koff[k - k_lo] = role_offset(p.k, k);
    __syncthreads();
    const int64_t* ko = koff - k_lo;  // indexed by k
    // check build: the chunk's offsets against the operand (a row's offset is added below)
    int64_t kmax = 0;
    if (kCheckBuild)
        for (uint32_t k = k_lo; k < k_hi; ++k) kmax = kmax > ko[k] ? kmax : ko[k];
    if (p.k_fast) {
#pragma unroll
        for (uint32_t i = 0; i < 4; ++i) {
            const uint32_t r = r0 + w + 8 * i;
            float a0 = init, a1 = init;
            if (r < p.R && chk(bo + role_offset(p.r, r) + kmax, p.src_elems, 212)) {
                const float* row = p.src + bo + role_offset(p.r, r);
                uint32_t k = k_lo + lane;
#pragma unroll 4
                for (; k + 32 < k_hi; k += 64) {
                    a0 = acc(a0, row[ko[k]]);
                    a1 = acc(a1, row[ko[k + 32]]);
                }
                if (k < k_hi) a0 = acc(a0, row[ko[k]]);
            }
            float a = p.mode == 0 ? fmaxf(a0, a1) : a0 + a1;
            for (int o = 16; o; o >>= 1) {
                const float v = __shfl_xor_sync(0xffffffffu, a, o);
                a = p.mode == 0 ? fmaxf(a, v) : a + v;
            }
            if (lane == 0 && r < p.R) p.partials[(uint64_t)c * rows + (uint64_t)b * p.R + r] = a;
        }
    } else {
        const uint32_t r = r0 + lane;
        float a0 = init, a1 = init;
        if (r < p.R && chk(bo + role_offset(p.r, r) + kmax, p.src_elems, 212)) {
            const float* row = p.src + bo + role_offset(p.r, r);
            uint32_t k = k_lo + w;
#pragma unroll 4
            for (; k + 8 < k_hi; k += 16) {
                a0 = acc(a0, row[ko[k]]);
                a1 = acc(a1, row[ko[k + 8]]);
            }
            if (k < k_hi) a0 = acc(a0, row[ko[k]]);
        }
        red[w][lane] = p.mode == 0 ? fmaxf(a0, a1) : a0 + a1;
        __syncthreads();
        if (w == 0 && r < p.R) {
            float a = red[0][lane];
            for (int q = 1; q < 8; ++q) a = p.mode == 0 ? fmaxf(a, red[q][lane]) : a + red[q][lane];
            p.partials[(uint64_t)c * rows + (uint64_t)b * p.R + r] = a;
        }
    }
}

__global__ void split3_stats_combine(const __grid_constant__ Split3StatsParams p) {
    const uint64_t rows = (uint64_t)p.nb * p.R;
    const uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x;
    if (i >= rows) return;
    float a = p.partials[i];
    for (uint32_t c = 1; c < p.kc; ++c) {
        const float v = p.partials[(uint64_t)c * rows + i];
        a = p.mode == 0 ? fmaxf(a, v) : a + v;
    }
    p.out[i] = a;
}

}  // namespace

uint32_t split3_stats_chunks(uint64_t rows, uint64_t K) {
    // about 2048 CTAs in phase 1, and at least 256 contracted indices per chunk
    const uint64_t tiles = (rows + 31) / 32;
    uint64_t kc = (2048 + tiles - 1) / tiles;
    const uint64_t kmax = (K + 255) / 256;
    if (kc > kmax) kc = kmax;
    const uint64_t kmin = (K + kStatsChunk - 1) / kStatsChunk;  // chunks fit the offset table
    if (kc < kmin) kc = kmin;
    if (kc < 1) kc = 1;
    return (uint32_t)kc;
}

cudaError_t launch_split3_stats(const Split3StatsParams& pin, cudaStream_t s) {
    Split3StatsParams p = pin;
    p.k_fast = p.k.n > 0 && p.k.t[0].div == 1 && p.k.t[0].loc_stride == 1;
    const uint64_t rows = (uint64_t)p.nb * p.R;
    if (rows == 0) return cudaSuccess;
    if (p.kc < 1 || p.kc != split3_stats_chunks(rows, p.K)) return cudaErrorInvalidValue;
    const uint64_t ctas = (uint64_t)p.nb * ((p.R + 31) / 32) * p.kc;
    if (ctas > 0x7fffffffull) return cudaErrorInvalidValue;
    split3_stats_kernel<<<(unsigned)ctas, 256, 0, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    split3_stats_combine<<<(unsigned)((rows + 255) / 256), 256, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_split3(const Split3Params& pin, cudaStream_t s) {
    Split3Params p = pin;
    p.k_fast = p.k.n > 0 && p.k.t[0].div == 1 && p.k.t[0].loc_stride == 1;
    // one contracted label, not split into keys: offset = k * its local stride
    p.k_dense = p.k.n == 1 && p.k.t[0].div == 1 && p.k.t[0].sub == p.K && p.k.t[0].ext == p.K;
    p.k_ls = p.k_dense ? p.k.t[0].loc_stride : 0;
    const uint64_t ctas = (uint64_t)p.nb * ((p.R + kSplitTR - 1) / kSplitTR) * ((p.K + kSplitTK - 1) / kSplitTK);
    if (ctas == 0) return cudaSuccess;
    if (ctas > 0x7fffffffull) return cudaErrorInvalidValue;
    split3_kernel<<<(unsigned)ctas, 256, 0, s>>>(p);
    return cudaGetLastError();
}

// Every element of z set to v (fp32, or bf16 rounded to nearest even): the outputs of an
// EinSum whose contracted range is empty, each the identity of its aggregation times alpha.
__global__ void fill_kernel(void* z, uint64_t n, float v, int bf16) {
    for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n; i += (uint64_t)gridDim.x * blockDim.x) {
        if (bf16) reinterpret_cast<__nv_bfloat16*>(z)[i] = __float2bfloat16_rn(v);
        else reinterpret_cast<float*>(z)[i] = v;
    }
}

cudaError_t launch_fill(void* z, uint64_t n, float v, bool bf16, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    fill_kernel<<<grid_for(n, 256), 256, 0, s>>>(z, n, v, bf16 ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t s) {
    const uint64_t total = p.n_groups * p.z_sub;
    if (total == 0) return cudaSuccess;
    combine_kernel<<<grid_for(total, 256), 256, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace tra
