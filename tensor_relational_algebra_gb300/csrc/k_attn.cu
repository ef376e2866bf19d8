// The attention chain of the multi-head-attention EinGraph, fused: Scores -> logsumexp ->
// exp(S - L) -> A.V in one tcgen05 kernel that never writes the scores.
//
// "EinDecomp ... tensor relational algebra", section 2.1 (multi-head attention as EinSums):
//   S[h,s,t] = scale * sum_d Q[h,s,d] K[h,t,d],  L[h,s] = logsumexp_t S[h,s,t],
//   A[h,s,t] = exp(S[h,s,t] - L[h,s]),           O[s,h,d] = sum_t A[h,s,t] V[h,t,d].
// Here the t axis is walked in blocks of 128 keys with a running maximum m and running sum
// l per query row (the logsumexp of the blocks seen so far is m + log l); O is rescaled by
// exp(m_old - m_new) whenever m moves, so after the last block O / l is the chained result
// and m + log l is L.
//
// One CTA per (head, 128 query rows); 7 warps:
//   warp 0   TMA loads of Q (once) and of each K block,   warp 1   TMA loads of each V block,
//   warp 2   tensor memory and the MMAs: S_j = Q K_j^T into one of two TMEM buffers, then
//            O += P_j V_j with P_j (bf16) read from shared memory,
//   warps 3-6 (TMEM lane quarter warp % 4, one query row per thread): the softmax update,
//            P_j in the 128-byte-swizzled K-major layout the MMA reads, the rescale of O, and
//            the epilogue (O / l as bf16 in [s][h][d]; L as fp32 in [h][s]).
// Every mbarrier wait is bounded; a wait that gives up records TRA_ERR_TIMEOUT in this unit's
// status word (read by ein_status), raises the CTA's abort flag and the CTA leaves after its
// copies and MMAs in flight have landed.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "plan.h"
#include "tc_ptx.h"

namespace tra {

__device__ int g_attn_status;  // TRA_ERR_* set by a bounded wait that gave up; 0 otherwise

namespace {

constexpr int kHead = 128;     // head dimension d
constexpr int kRows = 128;     // query rows per CTA
constexpr int kKeys = 128;     // keys per block
constexpr int kThreadsA = 7 * 32;
constexpr uint32_t kTile = 128 * 128 * 2;   // one 128 x 128 bf16 operand tile (two 16 KB boxes)
constexpr uint32_t kHalf = kTile / 2;       // one box: 64 columns x 128 rows
// shared memory: Q | K0 V0 | K1 V1 | P0 | P1 | barriers (all tiles 1024-aligned)
constexpr uint32_t kSmemA = 7 * kTile + 1024 + 256;

struct AttnParams {
    uint32_t s, t, h, nb;   // query rows, keys, heads, key blocks
    float scale_log2;       // scale * log2(e)
    __nv_bfloat16* o;       // [s][h][d]
    float* lse;             // [h][s] or null
    uint64_t timeout_ns;
};

__device__ __forceinline__ bool wait_a(uint32_t bar, uint32_t parity, volatile int* abort, uint64_t ns) {
    return mbar_wait_status(bar, parity, abort, ns, &g_attn_status);
}

__device__ __forceinline__ void tma_load_rows(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int row) {
    const int c[5] = {x, row, 0, 0, 0};
    tma_load_5d(dst, map, bar, c);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__global__ void __launch_bounds__(kThreadsA, 1)
    attn_fwd(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
             const __grid_constant__ CUtensorMap map_v, const __grid_constant__ AttnParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t sq = base;
    auto sk = [&](uint32_t st) { return base + kTile + st * 2 * kTile; };
    auto sv = [&](uint32_t st) { return base + 2 * kTile + st * 2 * kTile; };
    auto sp = [&](uint32_t b) { return base + 5 * kTile + b * kTile; };
    const uint32_t bar = base + 7 * kTile;
    // barriers: q_full, kv_full[2], kv_empty[2], s_full[2], s_free[2], p_full[2], o_done, mma_done,
    // then the TMEM slot and the abort flag
    const uint32_t q_full = bar, kv_full = bar + 8, kv_empty = bar + 24, s_full = bar + 40, s_free = bar + 56,
                   p_full = bar + 72, o_done = bar + 88, mma_done = bar + 96;
    uint8_t* gbase = smem_raw + (base - raw);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + (bar + 104 - base));
    volatile int* abort = reinterpret_cast<volatile int*>(gbase + (bar + 108 - base));

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t hd = blockIdx.y, q0 = blockIdx.x * kRows;
    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(kv_full + 8 * i, 2);   // the K and the V producer each arrive with their bytes
            mbar_init(kv_empty + 8 * i, 1);  // MMA commit after the block's P.V
            mbar_init(s_full + 8 * i, 1);    // MMA commit after S_j
            mbar_init(s_free + 8 * i, 4);    // one lane of each softmax warp
            mbar_init(p_full + 8 * i, 4);
        }
        mbar_init(o_done, 1);
        mbar_init(mma_done, 1);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 2) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(512)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t t_s0 = tmem, t_o = tmem + 256;  // S buffers at columns 0 and 128, O at 256

    if (warp <= 1) {
        // ------------------------------------------------------------------ producers
        if (lane == 0) {
            const CUtensorMap* map = warp == 0 ? &map_k : &map_v;
            if (warp == 0) {
                mbar_expect_tx(q_full, kTile);
                tma_load_rows(sq, &map_q, q_full, 0, (int)(hd * p.s + q0));
                tma_load_rows(sq + kHalf, &map_q, q_full, 64, (int)(hd * p.s + q0));
            }
            for (uint32_t j = 0; j < p.nb; ++j) {
                const uint32_t st = j & 1, ph = (j >> 1) & 1;
                if (!wait_a(kv_empty + 8 * st, ph ^ 1, abort, p.timeout_ns)) break;
                mbar_expect_tx(kv_full + 8 * st, kTile);
                const uint32_t dst = warp == 0 ? sk(st) : sv(st);
                const int row = (int)(hd * p.t + j * kKeys);
                tma_load_rows(dst, map, kv_full + 8 * st, 0, row);
                tma_load_rows(dst + kHalf, map, kv_full + 8 * st, 64, row);
            }
            if (*abort) __nanosleep(20000);  // let copies already issued land before leaving
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            // S = Q K^T: M = 128, N = 128 keys, both K-major; O += P V: M = 128, N = 128, P K-major,
            // V M/N-major (d innermost; its two 64-column boxes are 16 KB apart)
            const uint32_t id_s = (1u << 4) | (1u << 7) | (1u << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
            const uint32_t id_o = id_s | (1u << 16);
            bool ok = wait_a(q_full, 0, abort, p.timeout_ns);
            auto issue_s = [&](uint32_t j) {
                const uint32_t st = j & 1;
                if (!wait_a(kv_full + 8 * st, (j >> 1) & 1, abort, p.timeout_ns)) return false;
                tc_fence_after();
                for (uint32_t kk = 0; kk < kHead / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
                    tc_mma(t_s0 + st * 128, smem_desc(sq + off, 16, 1024), smem_desc(sk(st) + off, 16, 1024), id_s,
                           kk != 0);
                }
                tc_commit(s_full + 8 * st);
                return true;
            };
            if (ok) ok = issue_s(0);
            if (ok && p.nb > 1) ok = issue_s(1);
            for (uint32_t j = 0; ok && j < p.nb; ++j) {
                const uint32_t b = j & 1, ph = (j >> 1) & 1;
                if (!wait_a(p_full + 8 * b, ph, abort, p.timeout_ns)) break;
                tc_fence_after();
                for (uint32_t kk = 0; kk < kKeys / 16; ++kk) {
                    const uint64_t ad = smem_desc(sp(b) + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd = smem_desc(sv(b) + kk * 2048, kHalf, 1024);
                    tc_mma(t_o, ad, bd, id_o, (j | kk) != 0);
                }
                tc_commit(o_done);
                tc_commit(kv_empty + 8 * b);
                if (j + 2 < p.nb) {
                    // S_{j+2} reuses S buffer b once the softmax warps have read S_j
                    if (!wait_a(s_free + 8 * b, ph, abort, p.timeout_ns)) break;
                    if (!issue_s(j + 2)) break;
                }
            }
            // every MMA issued so far has completed once this commit arrives
            tc_commit(mma_done);
            volatile int never = 0;
            mbar_wait_status(mma_done, 0, &never, p.timeout_ns, &g_attn_status);
        }
    } else {
        // ------------------------------------------------------------------ softmax, rescale, epilogue
        const uint32_t qr = warp & 3;                 // TMEM lane quarter
        const uint32_t row = qr * 32 + lane;          // query row inside the tile
        const uint32_t lanebase = (qr * 32u) << 16;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (uint32_t j = 0; j < p.nb; ++j) {
            const uint32_t b = j & 1, ph = (j >> 1) & 1;
            if (!wait_a(s_full + 8 * b, ph, abort, p.timeout_ns)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sr[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32_nowait(t_s0 + lanebase + b * 128 + c * 32, sr[c]);
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_free + 8 * b);  // S buffer b may be overwritten
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int i = 0; i < 32; ++i) mx = fmaxf(mx, __uint_as_float(sr[c][i]));
            const float m_new = fmaxf(m, mx * p.scale_log2);
            const float corr = fast_exp2(m - m_new);  // 0 on the first block (m = -inf)
            // P_j as bf16 pairs in registers while P V_{j-1} may still run
            uint32_t pk[64];
            float sum = 0.f;
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float p0 = fast_exp2(__uint_as_float(sr[c][2 * i]) * p.scale_log2 - m_new);
                    const float p1 = fast_exp2(__uint_as_float(sr[c][2 * i + 1]) * p.scale_log2 - m_new);
                    sum += p0 + p1;
                    const __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
                    pk[c * 16 + i] = *reinterpret_cast<const uint32_t*>(&h2);
                }
            // the P buffer b was last read by P V_{j-2}, and O is rescaled after P V_{j-1}: wait for
            // P V_{j-1} (they complete in order)
            if (j > 0 && !wait_a(o_done, (j - 1) & 1, abort, p.timeout_ns)) {
                ok = false;
                break;
            }
            const uint32_t pbase = sp(b) + row * 128;
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    // keys 32c + 8u .. +7: 64-key chunk c / 2, 16-byte unit (c % 2) * 4 + u, swizzled by row
                    const uint32_t unit = (uint32_t)((c & 1) * 4 + u);
                    const uint32_t addr = pbase + (uint32_t)(c >> 1) * kHalf + ((unit ^ (row & 7u)) << 4);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[c * 16 + 4 * u]),
                                 "r"(pk[c * 16 + 4 * u + 1]), "r"(pk[c * 16 + 4 * u + 2]), "r"(pk[c * 16 + 4 * u + 3])
                                 : "memory");
                }
            l = l * corr + sum;
            m = m_new;
            if (j > 0) {
                // O *= corr (PV_{j-1} has completed: waited above)
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t orr[32];
                    tmem_ld32_nowait(t_o + lanebase + c * 32, orr);
                    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                    for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * corr);
                    tmem_st32(t_o + lanebase + c * 32, orr);
                }
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            }
            fence_async_smem();  // P_j visible to the tensor core's (async proxy) reads
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full + 8 * b);
        }
        // epilogue: O / l and L
        if (ok && wait_a(o_done, (p.nb - 1) & 1, abort, p.timeout_ns)) {
            tc_fence_after();
            const float inv = 1.f / l;
            __nv_bfloat16* orow = p.o + ((uint64_t)(q0 + row) * p.h + hd) * kHead;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t orr[32];
                tmem_ld32_nowait(t_o + lanebase + c * 32, orr);
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(orr[8 * v + 2 * e]) * inv,
                                                                       __uint_as_float(orr[8 * v + 2 * e + 1]) * inv);
                        w[e] = *reinterpret_cast<const uint32_t*>(&h2);
                    }
                    *reinterpret_cast<uint4*>(orow + c * 32 + v * 8) = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            if (p.lse) p.lse[(uint64_t)hd * p.s + q0 + row] = m * 0.6931471805599453f + logf(l);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_a() {
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

// rows x 128 bf16 (row pitch 256 bytes), boxes of 64 columns x 128 rows, 128-byte swizzle
bool encode_rows(const void* base, uint64_t rows, CUtensorMap* map) {
    auto fn = encode_fn_a();
    if (!fn) return false;
    cuuint64_t dims[5] = {(cuuint64_t)kHead, rows, 1, 1, 1};
    cuuint64_t strides[4] = {kHead * 2, rows * kHead * 2, rows * kHead * 2, rows * kHead * 2};
    cuuint32_t box[5] = {64, 128, 1, 1, 1}, es[5] = {1, 1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t read_and_clear_attn_status(int* value, cudaStream_t s) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(value, g_attn_status, sizeof(int), 0, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    const int zero = 0;
    e = cudaMemcpyToSymbolAsync(g_attn_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(s);
}

}  // namespace tra

using namespace tra;

extern "C" int ein_attention(int s, int t, int h, int d, float scale, const void* q, const void* k, const void* v,
                             void* o, void* lse, tra_stream_t stream) {
    clear_error();
    if (!q || !k || !v || !o) return fail(TRA_ERR_ARG, "NULL argument");
    if (d != kHead) return fail(TRA_ERR_UNSUPPORTED, "head dimension %d (the fused kernel takes %d)", d, kHead);
    if (s < kRows || s % kRows || t < kKeys || t % kKeys || h < 1 || h > 65535)
        return fail(TRA_ERR_UNSUPPORTED, "s and t must be multiples of 128, 1 <= h <= 65535");
    if ((uint64_t)h * s >= (1ull << 31) || (uint64_t)h * t >= (1ull << 31))
        return fail(TRA_ERR_UNSUPPORTED, "h * s and h * t must stay below 2^31 rows");
    if (((uintptr_t)q | (uintptr_t)k | (uintptr_t)v | (uintptr_t)o) % 16 || (lse && (uintptr_t)lse % 4))
        return fail(TRA_ERR_ARG, "misaligned buffer");
    if (!(scale > 0.f) || !std::isfinite(scale)) return fail(TRA_ERR_ARG, "scale must be positive and finite");
    CUtensorMap mq, mk, mv;
    if (!encode_rows(q, (uint64_t)h * s, &mq) || !encode_rows(k, (uint64_t)h * t, &mk) ||
        !encode_rows(v, (uint64_t)h * t, &mv))
        return fail(TRA_ERR_CUDA, "tensor map encoding failed");
    AttnParams ap;
    memset(&ap, 0, sizeof(ap));
    ap.s = (uint32_t)s;
    ap.t = (uint32_t)t;
    ap.h = (uint32_t)h;
    ap.nb = (uint32_t)(t / kKeys);
    ap.scale_log2 = scale * 1.4426950408889634f;
    ap.o = reinterpret_cast<__nv_bfloat16*>(o);
    ap.lse = reinterpret_cast<float*>(lse);
    ap.timeout_ns = 2000000000ull;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaFuncSetAttribute(attn_fwd, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemA);
    if (e != cudaSuccess) return fail(TRA_ERR_CUDA, "smem attribute: %s", cudaGetErrorString(e));
    attn_fwd<<<dim3((unsigned)(s / kRows), (unsigned)h), kThreadsA, kSmemA, st>>>(mq, mk, mv, ap);
    e = cudaGetLastError();
    return e == cudaSuccess ? TRA_OK : fail(TRA_ERR_CUDA, "attention launch: %s", cudaGetErrorString(e));
}
