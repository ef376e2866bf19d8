// The attention chain of the multi-head-attention EinGraph, fused: Scores -> logsumexp ->
// exp(S - L) -> A.V in one tcgen05 kernel that never writes the scores.
//
// "EinDecomp ... tensor relational algebra", section 2.1 (multi-head attention as EinSums):
//   S[h,s,t] = scale * sum_d Q[h,s,d] K[h,t,d],  L[h,s] = logsumexp_t S[h,s,t],
//   A[h,s,t] = exp(S[h,s,t] - L[h,s]),           O[s,h,d] = sum_t A[h,s,t] V[h,t,d].
// Here the t axis is walked in blocks of 128 keys with a reference maximum m and running sum
// l per query row (the logsumexp of the blocks seen so far is m + log l).  m moves only when
// a block's maximum exceeds it by more than 2^8 (so every exponent stays below 2^8); then l
// and O are rescaled by exp(m_old - m_new).  After the last block O / l is the chained
// result and m + log l is L.
//
// Persistent CTAs, one per SM, each taking work units (128 query rows of one head)
// blockIdx.x, blockIdx.x + grid, ...; the key blocks of its units are counted in one sequence,
// so the pipelines run on across unit boundaries (the next unit's Q loads into the other of two
// Q buffers, its first S blocks compute while the current unit's last blocks finish, and its
// first P V waits only until the softmax warps have read the previous unit's O).  12 warps:
//   warp 0   TMA loads of Q (once per unit) and of each K block (three slots, each freed once
//            S_j is computed), one 32 KB copy per tile,
//   warp 1   TMA loads of each V block (two slots, freed once P_j V_j is computed),
//   warp 2   tensor memory and the S MMAs: S_j = Q K_j^T into one of two TMEM buffers,
//   warp 7   the P V MMAs: O += P_j V_j with P_j (bf16) read from tensor memory (two buffers),
//   warps 3-6 and 8-11, two sets of softmax warps taking alternate key blocks (TMEM lane
//            quarter warp % 4, one query row per thread, all 128 keys of a block in
//            registers): the softmax update, P_j stored to tensor memory, the rescale of O, and
//            the epilogue (O as bf16 in [s][h][d]; L as fp32 in [h][s]).  With whole rows per
//            thread no warp waits on another for a row maximum or sum within a block; the
//            reference maximum passes from one set to the other once per block.
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
constexpr int kThreadsA = 12 * 32;
constexpr uint32_t kTile = 128 * 128 * 2;   // one 128 x 128 bf16 operand tile (two 16 KB boxes)
constexpr uint32_t kHalf = kTile / 2;       // one box: 64 columns x 128 rows
constexpr uint32_t kKStages = 3;            // K tiles in flight; V has two
constexpr uint32_t kTiles = 2 + kKStages + 2;
// shared memory: Q0 Q1 | K0 K1 K2 | V0 V1 | barriers, TMEM slot, abort flag (256 B); tiles 1024-aligned
// after the barrier block: 4 hand-off barriers (one per TMEM lane quarter) and the hand-off
// message (per query row: reference maximum, a row sum and that sum's reference)
constexpr uint32_t kHandoff = 32 + 3 * 128 * 4;
constexpr uint32_t kSmemA = kTiles * kTile + 1024 + 256 + kHandoff;

struct AttnParams {
    uint32_t s, t, h, nb;   // query rows, keys, heads, key blocks
    uint32_t qtiles, units; // query tiles of 128 rows per head; units = qtiles * h
    float scale_log2;       // scale * log2(e)
    __nv_bfloat16* o;       // [s][h][d]
    float* lse;             // [h][s] or null
    uint64_t timeout_ns;
};

__device__ __forceinline__ bool wait_a(uint32_t bar, uint32_t parity, volatile int* abort, uint64_t ns) {
    return mbar_wait_status(bar, parity, abort, ns, &g_attn_status);
}

// one 128-row x 128-column bf16 tile: the map's box covers both 64-column halves, the
// second landing 16 KB after the first
__device__ __forceinline__ void tma_load_tile(uint32_t dst, const CUtensorMap* map, uint32_t bar, int row) {
    const int c[5] = {0, row, 0, 0, 0};
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

// Two lanes of fp32 work per instruction (sm_100 packed forms; each lane rounds as the scalar
// instruction does): d = a * b + c and d = a + b.
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b, float c) {
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %4};\n\t"
        "mov.b64 rc, {%5, %5};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b), "f"(c));
}
__device__ __forceinline__ void fadd2(float& s0, float& s1, float a0, float a1) {
    asm("{\n\t.reg .b64 rs, ra;\n\t"
        "mov.b64 rs, {%0, %1};\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "add.rn.f32x2 rs, rs, ra;\n\t"
        "mov.b64 {%0, %1}, rs;\n\t}"
        : "+f"(s0), "+f"(s1)
        : "f"(a0), "f"(a1));
}
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
__global__ void __launch_bounds__(kThreadsA, 1)
    attn_fwd(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
             const __grid_constant__ CUtensorMap map_v, const __grid_constant__ AttnParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    auto sq = [&](uint32_t qb) { return base + qb * kTile; };
    auto sk = [&](uint32_t st) { return base + (2 + st) * kTile; };
    auto sv = [&](uint32_t st) { return base + (2 + kKStages + st) * kTile; };
    const uint32_t bar = base + kTiles * kTile;
    // barriers: q_full (Q buffer 0), k_full[3], k_empty[3], v_full[2], v_empty[2], s_full[2],
    // s_free[2], p_full[2], o_done[2], mma_done[2], q_full (Q buffer 1), q_empty[2] (a unit's last
    // S has read its Q), o_free (the softmax warps have read a unit's O); then the TMEM slot and
    // the abort flag
    const uint32_t q_full = bar, k_full = bar + 8, k_empty = bar + 32, v_full = bar + 56, v_empty = bar + 72,
                   s_full = bar + 88, s_free = bar + 104, o_done = bar + 136, mma_done = bar + 152,
                   q_full2 = bar + 168, q_empty = bar + 176, o_free = bar + 192;
    auto qf = [&](uint32_t qb) { return qb ? q_full2 : q_full; };
    // one "P_j published" barrier per P buffer: softmax can finish block j + 1 before the MMA warp
    // waits for block j (P_{j+1} does not wait for P V_j), so a single barrier could run two
    // phases ahead of its waiter; per buffer, block j + 2's phase needs P V_j, issued after the wait
    auto p_full = [&](uint32_t b_) { return bar + 120 + 8 * b_; };
    uint8_t* gbase = smem_raw + (base - raw);
    const uint32_t hand0 = bar + 256;
    float* msg_m = reinterpret_cast<float*>(gbase + (bar + 288 - base));
    float* msg_l = msg_m + 128;
    float* msg_r = msg_m + 256;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + (bar + 216 - base));
    volatile int* abort = reinterpret_cast<volatile int*>(gbase + (bar + 220 - base));

    // warp index and tensor-memory base made provably warp-uniform (shuffled from lane 0), so the
    // tcgen05 operands derived from them live in uniform registers
    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x / 32), 0), lane = threadIdx.x % 32;
    const uint32_t nu = (p.units - blockIdx.x + gridDim.x - 1) / gridDim.x;
    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_full2, 1);
        mbar_init(q_empty, 1);
        mbar_init(q_empty + 8, 1);
        mbar_init(o_free, 4);  // one lane of each softmax warp of the set writing the unit's O
        for (int i = 0; i < kKStages; ++i) {
            mbar_init(k_full + 8 * i, 1);   // the K producer's arrive with its bytes
            mbar_init(k_empty + 8 * i, 1);  // MMA commit after S_j (K_j read)
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(v_full + 8 * i, 1);
            mbar_init(v_empty + 8 * i, 1);  // MMA commit after P_j V_j
            mbar_init(s_full + 8 * i, 1);   // MMA commit after S_j
            mbar_init(s_free + 8 * i, 4);   // one lane of each softmax warp of the block's set: S_j read
            mbar_init(o_done + 8 * i, 1);   // MMA commit after P_j V_j
        }
        mbar_init(p_full(0), 4);            // one lane of each softmax warp of the set: P_j stored, O rescaled
        mbar_init(p_full(1), 4);
        for (int i = 0; i < 4; ++i) mbar_init(hand0 + 8 * i, 1);  // one lane of the quarter's softmax warp
        mbar_init(mma_done, 1);      // the S issuer's last commit
        mbar_init(mma_done + 8, 1);  // the P V issuer's last commit
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
    const uint32_t tmem = __shfl_sync(0xffffffffu, *tmem_slot, 0);
    // columns: S buffers 0-127 and 128-255 (fp32), O 256-383 (fp32), P buffers 384-447 and
    // 448-511 (bf16 pairs: column c holds keys 2c and 2c + 1); P_j goes to buffer j % 2
    const uint32_t t_s0 = tmem, t_o = tmem + 256, t_p = tmem + 384;

    // producer and MMA warps run their loops with the whole warp (waits taken by every lane, the
    // result shuffled from lane 0 so that control flow stays uniform); one elected lane issues
    auto wait_u = [&](uint32_t b_, uint32_t parity) {
        return __shfl_sync(0xffffffffu, (int)wait_a(b_, parity, abort, p.timeout_ns), 0) != 0;
    };
    if (warp <= 1) {
        // ------------------------------------------------------------------ producers (K: warp 0, V: warp 1)
        // one 32 KB copy per tile (both 64-column halves)
        bool ok = true;
        uint32_t g = 0;
        for (uint32_t i = 0; ok && i < nu; ++i) {
            const uint32_t u = blockIdx.x + i * gridDim.x, hd = u / p.qtiles, q0 = (u % p.qtiles) * kRows;
            if (warp == 0) {
                const uint32_t qb = i & 1;
                if (i >= 2 && !wait_u(q_empty + 8 * qb, ((i - 2) >> 1) & 1)) break;
                if (elect_one()) {
                    mbar_expect_tx(qf(qb), kTile);
                    tma_load_tile(sq(qb), &map_q, qf(qb), (int)(hd * p.s + q0));
                }
                __syncwarp();
            }
            for (uint32_t j = 0; j < p.nb; ++j, ++g) {
                if (warp == 0) {
                    const uint32_t st = g % kKStages, ph = (g / kKStages) & 1;
                    if (!wait_u(k_empty + 8 * st, ph ^ 1)) { ok = false; break; }
                    if (elect_one()) {
                        mbar_expect_tx(k_full + 8 * st, kTile);
                        tma_load_tile(sk(st), &map_k, k_full + 8 * st, (int)(hd * p.t + j * kKeys));
                    }
                } else {
                    const uint32_t st = g & 1, ph = (g >> 1) & 1;
                    if (!wait_u(v_empty + 8 * st, ph ^ 1)) { ok = false; break; }
                    if (elect_one()) {
                        mbar_expect_tx(v_full + 8 * st, kTile);
                        tma_load_tile(sv(st), &map_v, v_full + 8 * st, (int)(hd * p.t + j * kKeys));
                    }
                }
                __syncwarp();
            }
        }
        if (*abort) __nanosleep(20000);  // let copies already issued land before leaving
    } else if (warp == 2 || warp == 7) {
        // ------------------------------------------------------------------ MMA issuers
        // S = Q K^T: M = 128, N = 128 keys, Q and K K-major in shared memory (warp 2).
        // O += P V: M = 128, N = 128, P (A) in tensor memory, V M/N-major in shared memory
        // (d innermost; its two 64-column boxes are 16 KB apart) (warp 7).
        // Two issuing warps: a thread's mbarrier wait that follows its own tcgen05.commit stalls
        // until the committed MMAs have drained, so one issuer would leave the tensor core idle
        // between the S and P V streams (a clock64 trace showed ~500 cycles per block).  Apart,
        // each stream's waits stall only on its own MMAs, and the tensor core interleaves the two.
        // The streams touch separate tensor memory (S buffers / O and the P buffers they read),
        // ordered through the softmax warps' barriers.  Descriptors are formed once; a tile or
        // K-step offset is added to the start-address field (addresses stay below 2^18, so the
        // field does not carry).
        const uint32_t id_s = (1u << 4) | (1u << 7) | (1u << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
        const uint32_t id_o = id_s | (1u << 16);
        const uint64_t dq = smem_desc(sq(0), 16, 1024), dk = smem_desc(sk(0), 16, 1024), dv = smem_desc(sv(0), kHalf, 1024);
        bool ok = true;
        if (warp == 2) {
            // S_j = Q K_j^T into S buffer j % 2, as soon as the softmax warps have read S_{j-2}
            // from that buffer and K_j has landed
            uint32_t g = 0;
            for (uint32_t i = 0; ok && i < nu; ++i) {
                const uint32_t qb = i & 1;
                ok = wait_u(qf(qb), (i >> 1) & 1);
                for (uint32_t j = 0; ok && j < p.nb; ++j, ++g) {
                    const uint32_t st = g % kKStages, b = g & 1;
                    if (g >= 2 && !wait_u(s_free + 8 * b, ((g - 2) >> 1) & 1)) { ok = false; break; }
                    if (!wait_u(k_full + 8 * st, (g / kKStages) & 1)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t dqs = dq + ((qb * kTile) >> 4), dks = dk + ((st * kTile) >> 4);
#pragma unroll
                    for (uint32_t kk = 0; kk < kHead / 16; ++kk) {
                        const uint32_t off = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
                        tc_mma_elect(t_s0 + b * 128, dqs + off, dks + off, id_s, kk != 0);
                    }
                    tc_commit_elect(s_full + 8 * b);
                    tc_commit_elect(k_empty + 8 * st);
                }
                if (ok) tc_commit_elect(q_empty + 8 * qb);  // this unit's Q has been read
            }
        } else {
            // P V_j once P_j is published and V_j has landed
            uint32_t g = 0;
            for (uint32_t i = 0; ok && i < nu; ++i) {
                for (uint32_t j = 0; j < p.nb; ++j, ++g) {
                    const uint32_t b = g & 1, ph = (g >> 1) & 1;
                    if (!wait_u(p_full(b), ph) || !wait_u(v_full + 8 * b, ph)) { ok = false; break; }
                    if (j == 0 && i >= 1 && !wait_u(o_free, (i - 1) & 1)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t dvb = dv + ((b * kTile) >> 4);
#pragma unroll
                    for (uint32_t kk = 0; kk < kKeys / 16; ++kk)  // keys 16kk..16kk+15: P columns 8kk..8kk+7
                        tc_mma_ts_elect(t_o, t_p + b * 64 + kk * 8, dvb + ((kk * 2048) >> 4), id_o, (j | kk) != 0);
                    tc_commit_elect(o_done + 8 * b);
                    tc_commit_elect(v_empty + 8 * b);
                }
            }
        }
        // every MMA this warp issued has completed once this commit arrives
        const uint32_t done = warp == 2 ? mma_done : mma_done + 8;
        tc_commit_elect(done);
        volatile int never = 0;
        mbar_wait_status(done, 0, &never, p.timeout_ns, &g_attn_status);
        __syncwarp();
    } else {
        // ------------------------------------------------------------------ softmax, rescale, epilogue
        // Warps 3-6: TMEM lane quarter warp % 4, one query row per thread, all 128 keys of a
        // block in registers (so the row maximum and sum need no exchange between warps).  m
        // moves only when a block's maximum exceeds it by more than 8 (log2 units): P stays below
        // 2^8, and O is rescaled through tensor memory only on such blocks, once P V_{j-1} has
        // completed.  P_j goes to P buffer j % 2 once P V_{j-2}, the last reader of that buffer,
        // has completed -- long before, so softmax(j) does not wait for P V_{j-1}.  The parity
        // waits on o_done stay unambiguous: P V_j cannot complete before P_j is published.
        // Two sets of four softmax warps (warps 3-6 and 8-11) take alternate key blocks: set k
        // handles the blocks g with g % 2 = k, always in S and P buffer k, so two softmax warps
        // share each scheduler and one block's exponentials overlap the next one's.  The
        // reference maximum passes from block g to block g + 1 through a message per lane quarter
        // (hand-off barrier, phase g), published right after block g's maximum: the maximum
        // after block g, and the sender's row sum just before block g with that sum's reference.
        // A set rescales its own sum whenever the maximum it receives has moved.  The set that
        // handles a unit's last block writes O / l: the other set's sum reaches it in the next
        // message (the first block of the next unit, or a closing message after the last unit).
        const uint32_t set = warp >= 8 ? 1u : 0u;
        const uint32_t qr = warp & 3;         // TMEM lane quarter
        const uint32_t row = qr * 32 + lane;  // query row inside the tile
        const uint32_t lanebase = (qr * 32u) << 16;
        const uint32_t hb = hand0 + 8 * qr;
        bool ok = true;
        uint32_t g = 0;
        float m_used = -INFINITY, l = 0.f;  // this set's reference maximum and row sum (current unit)
        uint32_t my_unit = 0xffffffffu;     // the unit m_used and l belong to
        for (uint32_t i = 0; ok && i < nu; ++i) {
        const uint32_t u = blockIdx.x + i * gridDim.x, hd = u / p.qtiles, q0 = (u % p.qtiles) * kRows;
        for (uint32_t j = 0; j < p.nb; ++j, ++g) {
            if ((g & 1) != set) continue;
            const uint32_t b = g & 1, ph = (g >> 1) & 1;
            float m_in = -INFINITY;
            if (g >= 1) {
                if (!wait_a(hb, (g - 1) & 1, abort, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                m_in = msg_m[row];
            }
            const float l_before = l, r_before = m_used;
            if (my_unit != i) {  // this set's first block of the unit (j = 0 or 1)
                my_unit = i;
                m_used = -INFINITY;
                l = 0.f;
            }
            if (j > 0 && m_in > m_used) {  // block g - 1 (the other set's) moved the reference
                l *= fast_exp2(m_used - m_in);
                m_used = m_in;
            }
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
            float mc[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint32_t* v = &sr[c >> 1][(c & 1) * 16];
                float x = max3f(__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]));
#pragma unroll
                for (int i = 3; i < 15; i += 2) x = max3f(x, __uint_as_float(v[i]), __uint_as_float(v[i + 1]));
                mc[c] = fmaxf(x, __uint_as_float(v[15]));
            }
            const float m_blk = max3f(max3f(mc[0], mc[1], mc[2]), max3f(mc[3], mc[4], mc[5]), fmaxf(mc[6], mc[7])) *
                                p.scale_log2;
            const bool need = m_blk > m_used + 8.f;
            const float m_use = need ? m_blk : m_used;
            const float corr = fast_exp2(m_used - m_use);  // 1 when m_used stays; 0 on the first block
            // message g: the maximum after this block, and this set's sum before it
            msg_m[row] = m_use;
            msg_l[row] = l_before;
            msg_r[row] = r_before;
            __syncwarp();
            if (lane == 0) mbar_arrive(hb);
            uint32_t pk[2][32];
            float sc[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float s0 = 0.f, s1 = 0.f;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float x0, x1;
                    ffma2(x0, x1, __uint_as_float(sr[c][2 * i]), __uint_as_float(sr[c][2 * i + 1]), p.scale_log2, -m_use);
                    const float p0 = fast_exp2(x0);
                    const float p1 = fast_exp2(x1);
                    fadd2(s0, s1, p0, p1);
                    const __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
                    pk[c >> 1][(c & 1) * 16 + i] = *reinterpret_cast<const uint32_t*>(&h2);
                }
                sc[c] = s0 + s1;
            }
            if (g >= 2 && !wait_a(o_done + 8 * b, ((g - 2) >> 1) & 1, abort, p.timeout_ns)) {
                ok = false;  // P buffer b is free once P V_{g-2} has completed
                break;
            }
            tc_fence_after();
            tmem_st32(t_p + b * 64 + lanebase, pk[0]);  // keys 0-63
            tmem_st32(t_p + b * 64 + lanebase + 32, pk[1]);  // keys 64-127
            l = fmaf(l, corr, (sc[0] + sc[1]) + (sc[2] + sc[3]));
            m_used = m_use;
            if (j > 0 && __any_sync(0xffffffffu, need)) {
                // O *= corr, once P V_{g-1} has completed (rows whose m_used stayed multiply by 1)
                if (!wait_a(o_done + 8 * ((g - 1) & 1), ((g - 1) >> 1) & 1, abort, p.timeout_ns)) {
                    ok = false;
                    break;
                }
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
            }
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full(b));
        }
        if (!ok) break;
        // epilogue by the set that handled the unit's last block, once the last P V has completed
        // (they complete in order): O / l as bf16, and L = (m ln 2) + log(l)
        const uint32_t gl = g - 1;
        if ((gl & 1) != set) continue;
        float l_tot = l;
        if (p.nb >= 2) {  // the other set's sum over its blocks of this unit, from message g
            ok = wait_a(hb, g & 1, abort, p.timeout_ns);
            if (!ok) break;
            l_tot += msg_l[row] * fast_exp2(msg_r[row] - m_used);
        }
        ok = wait_a(o_done + 8 * (gl & 1), (gl >> 1) & 1, abort, p.timeout_ns);
        if (ok) {
            const float inv = 1.f / l_tot;
            tc_fence_after();
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
            if (p.lse) p.lse[(uint64_t)hd * p.s + q0 + row] = m_used * 0.6931471805599453f + logf(l_tot);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(o_free);
        }
        }
        // closing message (index g = all blocks): the sum of this set's last unit, for the set
        // that handled that unit's last block
        if (ok && (g & 1) == set && g >= 1) {
            if (wait_a(hb, (g - 1) & 1, abort, p.timeout_ns)) {
                msg_l[row] = l;
                msg_r[row] = m_used;
                __syncwarp();
                if (lane == 0) mbar_arrive(hb);
            }
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

// rows x 128 bf16 (row pitch 256 bytes) seen as [2 column halves][rows][64 columns]: the box
// {64 columns, 128 rows, 2 halves} is one 32 KB copy, 128-byte swizzle
bool encode_rows(const void* base, uint64_t rows, CUtensorMap* map) {
    auto fn = encode_fn_a();
    if (!fn) return false;
    cuuint64_t dims[5] = {64, rows, 2, 1, 1};
    cuuint64_t strides[4] = {kHead * 2, 128, rows * kHead * 2, rows * kHead * 2};
    cuuint32_t box[5] = {64, 128, 2, 1, 1}, es[5] = {1, 1, 1, 1, 1};
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
    ap.qtiles = (uint32_t)(s / kRows);
    ap.units = ap.qtiles * (uint32_t)h;
    ap.scale_log2 = scale * 1.4426950408889634f;
    ap.o = reinterpret_cast<__nv_bfloat16*>(o);
    ap.lse = reinterpret_cast<float*>(lse);
    ap.timeout_ns = 2000000000ull;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaFuncSetAttribute(attn_fwd, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemA);
    if (e != cudaSuccess) return fail(TRA_ERR_CUDA, "smem attribute: %s", cudaGetErrorString(e));
    // persistent: one CTA per SM (its shared and tensor memory allow no second one)
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess || sms < 1) return fail(TRA_ERR_CUDA, "SM count: %s", cudaGetErrorString(e));
    const unsigned grid = ap.units < (uint32_t)sms ? ap.units : (unsigned)sms;
    attn_fwd<<<grid, kThreadsA, kSmemA, st>>>(mq, mk, mv, ap);
    e = cudaGetLastError();
    return e == cudaSuccess ? TRA_OK : fail(TRA_ERR_CUDA, "attention launch: %s", cudaGetErrorString(e));
}
