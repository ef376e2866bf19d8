// BF16 sum-of-products join + aggregate on the 5th-generation tensor cores
// (tcgen05.mma with the accumulator in tensor memory, operands staged by TMA).
//
// "EinDecomp ... tensor relational algebra", section 2.2: under a partition
// vector every join tuple multiplies one X sub-tensor with one key-matched Y
// sub-tensor, and the aggregation sums the tuples that share an output key.
// Here each CTA tile of the output lies inside one output key; its K loop walks
// every contracted key (one more run of K-steps at another block coordinate),
// so the aggregation across join tuples is the TMEM accumulation itself.
//
// Relations are addressed through rank-5 TMA tensor maps over the blocked
// layout: the dimensions are the block-local and the key parts of each label
// (unit dimensions dropped), and a tile coordinate along a dimension is
// (composite index / div) % mod.  The planner accepts a shape only when every
// tile is one TMA box, which keeps every load inside one sub-tensor.
//
// Kernels: persistent, one CTA per SM, 13 warps: warps 0-3 issue TMA loads,
// warp 4 owns tensor memory and issues tcgen05.mma (fp32 accumulate, K = 16 per
// instruction), warps 5-12 drain the double-buffered accumulator (tcgen05.ld)
// into global memory while the next tile is computed.  tc_gemm: one CTA per
// 128 x BLOCK_N tile.  tc_gemm_2sm: a cluster of two CTAs per 256 x BLOCK_N tile
// (cta_group::2 instructions issued by the even CTA).
// Every mbarrier wait is bounded; a wait that gives up sets the device status
// word (TRA_ERR_TIMEOUT) and makes the whole CTA leave after its copies and
// MMAs in flight have landed.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <chrono>
#include <cstring>
#include <mutex>

#include "plan.h"
#include "tc_ptx.h"

namespace tra {

__device__ int g_status;  // TRA_ERR_* set by a bounded wait that gave up; 0 otherwise

namespace {

constexpr int kBlockM = 128;
constexpr int kBlockK = 64;  // one 128-byte swizzle row of bf16
// Warp roles: 0-3 TMA producers (global K step g goes to producer g % kProducers: the
// copy engine completes the copies of one issuing thread in order, so a single issuing
// thread caps a CTA at one box per L2 round trip), 4 MMA issuer, 5-12 epilogue (two warps
// per TMEM lane quarter, each taking half of the tile's columns).
constexpr int kProducers = 4;
constexpr int kMmaWarp = kProducers;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 32 * (kProducers + 1 + kEpiWarps);
constexpr uint32_t kMaxSmem = 227 * 1024;
// Epilogue staging per epilogue warp: a 32 x 32 fp32 tile (16-byte groups swizzled by row).
constexpr uint32_t kEpiTile = 32 * 32 * 4;
constexpr uint32_t kEpiBytes = kEpiWarps * kEpiTile;

struct TcOpDev {
    int32_t mn_major;  // 1: innermost dimension is M (X) / N (Y); 0: innermost is K
    int32_t n_loads;   // TMA loads per stage (MN-major: one per 64 rows of M/N)
    int32_t role[5];
    FastDiv div[5], mod[5];  // coordinate along dimension j = (composite / div) % mod
};

struct TcParams {
    TcOpDev zt;     // output tensor-map dimensions (TMA-store epilogue)
    uint32_t z_tma;  // 1: the epilogue stores through the output tensor map
    TcOpDev a, b;
    uint32_t nb, M, N, K;
    uint32_t tiles_m, tiles_n, n_tiles, group_m;
    uint32_t block_n, stages, num_kb, tmem_cols;
    uint32_t idesc;
    uint32_t a_bytes, b_bytes;
    RoleMap zb, zm, zn;
    void* z;
    float alpha;
    int32_t out_bf16;
    uint64_t timeout_ns;
    // epilogue terms (TcExtra): 0 plain; 1 max(r[m] + c[n] - 2 acc, 0); 2 r[m] + c[n] + log(acc),
    // NaN where acc <= 1e-30 (the caller's fix-up recomputes those); r, c indexed b * M + m, b * N + n
    uint32_t epi;
    const float* row_term;
    const float* col_term;
    uint32_t zM, zN;  // output rows / columns stored (M, N unless the operands are padded)
    int* mark_count;  // epilogue 2: incremented once per output marked NaN (may be null)
    // epilogue 1: guard of the expansion (r + c - 2 acc < sq_tau (r + c) sets the word of the
    // output's 128 x 128 tile in fix_flags; may be null)
    float sq_tau;
    uint32_t* fix_flags;
    uint32_t fix_tiles_m, fix_tiles_n;
    uint64_t fix_tag_index;  // fix_flags[fix_tag_index] = 1 once anything is marked
    uint64_t z_elems;        // elements of z: the check build's bound on the warp stores
    // Work units (see unit_of): tiles [0, n_full) whole; tiles [n_full, n_tiles) of the last,
    // partly filled wave split into `split` runs of K steps on as many idle workers.  Parts
    // 0 .. split-2 each leave fp32 partial sums in a slot of `part` and release them through one
    // flag per (tile, part, epilogue warp); the last part adds them in part order.
    uint32_t n_full, split, n_units;
    // split == 2 with an fp32 output tensor map: instead of passing partial sums, both parts add
    // their sums into the output with TMA reduce-add, after the worker of part 0 has zeroed the
    // tile at the start of the launch (flag per tile and epilogue warp, as for the partial sums)
    uint32_t split_reduce;
    float* part;                 // [tile - n_full][part][lane quarter][column block][register][lane]
    unsigned long long* flags;   // [tile - n_full][part][epilogue warp]: tag | 1 once released
    unsigned long long tag;      // this launch's flag tag (the low 8 bits are zero)
};

constexpr uint32_t kWhole = 0xffffffffu;  // unit_of: the unit is a whole tile

// Unit u -> its tile, its run of K steps [kb0, kb1) and its part (kWhole for a whole tile).
// Worker w (CTA or CTA pair) takes units w, w + workers, ...; n_full is a multiple of the
// worker count (or 0), so each worker owns at most one split unit, and it is its last.
__device__ __forceinline__ void unit_of(const TcParams& p, uint32_t u, uint32_t& tile, uint32_t& kb0, uint32_t& kb1,
                                        uint32_t& part) {
    if (u < p.n_full) {
        tile = u;
        kb0 = 0;
        kb1 = p.num_kb;
        part = kWhole;
        return;
    }
    const uint32_t v = u - p.n_full, j = v % p.split;
    tile = p.n_full + v / p.split;
    part = j;
    kb0 = j * p.num_kb / p.split;
    kb1 = (j + 1) * p.num_kb / p.split;
}

// ------------------------------------------------------------------ PTX wrappers (tc_ptx.h)
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort, uint64_t timeout_ns) {
    return mbar_wait_status(bar, parity, abort, timeout_ns, &g_status);
}

__device__ __forceinline__ int dim_coord(const TcOpDev& o, int j, uint32_t v) {
    const uint32_t q = fdiv(v, o.div[j]);
    return (int)(q - fdiv(q, o.mod[j]) * o.mod[j].d);
}

// Coordinates of the dimensions that do not move along K (batch and M or N): once per tile.
__device__ __forceinline__ void fixed_coords(const TcOpDev& o, uint32_t cb, uint32_t cmn, int c[5]) {
#pragma unroll
    for (int j = 0; j < 5; ++j) c[j] = o.role[j] == kK ? 0 : dim_coord(o, j, o.role[j] == kBatch ? cb : cmn);
}

// Coordinates of the contracted dimensions at composite K index ck: once per K step.
__device__ __forceinline__ void k_coords(const TcOpDev& o, uint32_t ck, int c[5]) {
#pragma unroll
    for (int j = 0; j < 5; ++j) c[j] = o.role[j] == kK ? dim_coord(o, j, ck) : 0;
}

__device__ __forceinline__ void tile_of(const TcParams& p, uint32_t t, uint32_t& b, uint32_t& mt, uint32_t& nt) {
    const uint32_t per = p.tiles_m * p.tiles_n;
    b = t / per;
    const uint32_t r = t % per;
    const uint32_t gsize = p.group_m * p.tiles_n;
    const uint32_t g = r / gsize;
    const uint32_t first = g * p.group_m;
    const uint32_t gm = min(p.group_m, p.tiles_m - first);
    const uint32_t w = r % gsize;
    mt = first + w % gm;
    nt = w / gm;
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cl(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// bounded wait on a barrier that other CTAs of the cluster signal (cluster-scope acquire)
__device__ __forceinline__ bool mbar_wait_cl(uint32_t bar, uint32_t parity, volatile int* abort, uint64_t timeout_ns) {
    if (mbar_try_wait_cl(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait_cl(bar, parity)) return true;
        if ((n & 63) == 0) {
            if (*abort) return false;
            if (globaltimer() - t0 > timeout_ns) {
                *abort = 1;
                atomicExch(&g_status, (int)TRA_ERR_TIMEOUT);
                return false;
            }
        }
    }
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster_addr) : "memory");
}
// TMA load into this CTA's shared memory whose completion is counted on a barrier that may
// live in the peer CTA of the pair
__device__ __forceinline__ void tma_load_5d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                 const int c[5]) {
    asm volatile(
        "cp.async.bulk.tensor.5d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]), "r"(c[4]), "r"(bar_cluster)
        : "memory");
}
// tcgen05.mma / commit with cta_group::2 (M = 256 across the pair), issued by the elected lane
// of a converged warp (see tc_mma_elect); the commit arrives once on the barrier at this shared
// offset in every CTA of ctamask when the MMAs issued so far have completed
__device__ __forceinline__ void tc_mma_pair_elect(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                  uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void tc_commit_pair_elect(uint32_t bar, uint16_t ctamask) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}" ::"r"(bar),
        "h"(ctamask)
        : "memory");
}

// One producer warp's share of the K steps of every tile this CTA (or CTA pair) owns:
// steps g = pw, pw + kProducers, ...  Stage g % stages, phase (g / stages) & 1.  A parity
// wait cannot alias an older phase because stages >= kProducers: when this warp reaches
// step g it has seen step g - kProducers - stages released, and releases are in order.
// Lane 0 waits for the stage and arms its full barrier; then lane L issues box L of the step
// (the A boxes, then the B boxes).  The copies of one issuing thread complete one after
// another (a fixed ~560 cycles per box, whatever its size), so one box per lane lets the
// step's boxes travel together.
// PAIR: the copy of this CTA's half counts on the even CTA's full barrier (cta_group::2).
template <bool PAIR>
__device__ __forceinline__ void producer_steps(const CUtensorMap* map_a, const CUtensorMap* map_b, const TcParams& p,
                                               uint32_t pw, int lane, uint32_t first_tile, uint32_t tile_step,
                                               uint32_t rank, uint32_t base, uint32_t full0, uint32_t empty0,
                                               volatile int* abort) {
    const uint32_t stage_bytes = p.a_bytes + p.b_bytes;
    // this lane's box: operand, map, index within the operand and offset within the stage
    const uint32_t na = (uint32_t)p.a.n_loads, nbox = na + (uint32_t)p.b.n_loads;
    const bool mine = (uint32_t)lane < nbox, is_a = (uint32_t)lane < na;
    const TcOpDev& op = is_a ? p.a : p.b;
    const CUtensorMap* map = is_a ? map_a : map_b;
    const uint32_t l = is_a ? (uint32_t)lane : (uint32_t)lane - na;
    const uint32_t box_off = (is_a ? 0u : p.a_bytes) + 8192u * l;
    // this worker's units: n_whole whole tiles, then at most one split unit (K steps skb0 .. skb1)
    const uint32_t n_whole = first_tile < p.n_full ? (p.n_full - first_tile + tile_step - 1) / tile_step : 0u;
    const uint32_t split_u = p.n_full + first_tile;
    uint32_t stile = 0, skb0 = 0, skb1 = 0, spart = 0;
    if (p.split > 1 && split_u < p.n_units) unit_of(p, split_u, stile, skb0, skb1, spart);
    const uint32_t whole_steps = n_whole * p.num_kb;
    const uint32_t total = whole_steps + (skb1 - skb0);
    uint32_t cur = 0xffffffffu;
    int fc[5];
    uint32_t pend_stage[2] = {0, 0}, pend_phase[2] = {0, 0}, n_pend = 0;
    bool ok = true;
    for (uint32_t g = pw; g < total; g += kProducers) {
        uint32_t i, kb, tile;
        if (g < whole_steps) {
            i = g / p.num_kb;
            kb = g - i * p.num_kb;
            tile = first_tile + i * tile_step;
        } else {
            i = n_whole;
            kb = skb0 + (g - whole_steps);
            tile = stile;
        }
        if (i != cur) {
            cur = i;
            uint32_t b, mt, nt;
            tile_of(p, tile, b, mt, nt);
            const uint32_t m0 = PAIR ? mt * 2 * kBlockM + rank * kBlockM : mt * kBlockM;
            const uint32_t n0 = PAIR ? nt * p.block_n + rank * (p.block_n / 2) : nt * p.block_n;
            if (mine) fixed_coords(op, b, (is_a ? m0 : n0) + 64u * l, fc);
        }
        const uint32_t stage = g % p.stages, phase = (g / p.stages) & 1u;
        const uint32_t fb = full0 + 8 * stage;
        int got = 1;
        if (lane == 0) {
            got = PAIR ? mbar_wait_cl(empty0 + 8 * stage, phase ^ 1, abort, p.timeout_ns)
                       : mbar_wait(empty0 + 8 * stage, phase ^ 1, abort, p.timeout_ns);
            if (got) {
                if (!PAIR) mbar_expect_tx(fb, stage_bytes);
                else if (rank == 0) mbar_expect_tx(fb, 2 * stage_bytes);  // both CTAs' bytes land on the even CTA's barrier
            }
        }
        if (!__shfl_sync(0xffffffffu, got, 0)) {
            ok = false;
            break;
        }
        if (mine) {
            int kc[5], c[5];
            k_coords(op, kb * kBlockK, kc);
#pragma unroll
            for (int j = 0; j < 5; ++j) c[j] = fc[j] + kc[j];
            const uint32_t dst = base + stage * stage_bytes + box_off;
            if (PAIR) tma_load_5d_pair(dst, map, mapa_shared(fb, 0), c);
            else tma_load_5d(dst, map, fb, c);
        }
        pend_stage[n_pend & 1] = stage;
        pend_phase[n_pend & 1] = phase;
        ++n_pend;
    }
    if (!ok && lane == 0) {
        // let the copies this warp issued land before the CTA leaves (at most
        // ceil(stages / kProducers) <= 2 steps are outstanding)
        if (PAIR) {
            __nanosleep(20000);  // the pair's copies count on the even CTA's barriers
        } else {
            volatile int never = 0;
            for (uint32_t j = 0; j < 2 && j < n_pend; ++j) mbar_wait(full0 + 8 * pend_stage[j], pend_phase[j], &never, p.timeout_ns);
        }
    }
    __syncwarp();
}

// Output tensor-map coordinates of the box starting at (b, m, n).
__device__ __forceinline__ void z_coords(const TcOpDev& o, uint32_t b, uint32_t m, uint32_t n, int c[5]) {
#pragma unroll
    for (int j = 0; j < 5; ++j)
        c[j] = o.role[j] == kK ? 0 : dim_coord(o, j, o.role[j] == kBatch ? b : (o.role[j] == kM ? m : n));
}

// Store one 32 x 32 accumulator block (thread = row, r = its 32 columns starting at n; zr =
// this lane's row offset in Z, -1 for a row past the end; zc = the block's column offset).
// The block goes through shared memory as 16-byte groups, group g of row w at slot
// g ^ (w & 7): the row-wise writes (8 rows per phase) and the column-wise reads (one row
// per 8 lanes) are both conflict-free, and each global store instruction of the warp writes
// whole row segments (4 rows x 128 bytes fp32, or 8 rows x 64 bytes bf16).
__device__ __forceinline__ void store_block(const TcParams& p, float4* stg, int64_t zr, int64_t zc, int lane,
                                            const uint32_t (&r)[32], uint32_t n) {
    if (n >= p.zN) return;  // uniform over the warp
#pragma unroll
    for (int g = 0; g < 8; ++g)
        stg[lane * 8 + (g ^ (lane & 7))] =
            make_float4(p.alpha * __uint_as_float(r[4 * g]), p.alpha * __uint_as_float(r[4 * g + 1]),
                        p.alpha * __uint_as_float(r[4 * g + 2]), p.alpha * __uint_as_float(r[4 * g + 3]));
    __syncwarp();
    if (p.out_bf16) {
        __nv_bfloat16* z = reinterpret_cast<__nv_bfloat16*>(p.z);
        const int sub = lane & 3;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int row = 8 * i + (lane >> 2);
            const float4 v0 = stg[row * 8 + ((2 * sub) ^ (row & 7))];
            const float4 v1 = stg[row * 8 + ((2 * sub + 1) ^ (row & 7))];
            const int64_t o = __shfl_sync(0xffffffffu, zr, row);
            __nv_bfloat162 h[4] = {__floats2bfloat162_rn(v0.x, v0.y), __floats2bfloat162_rn(v0.z, v0.w),
                                   __floats2bfloat162_rn(v1.x, v1.y), __floats2bfloat162_rn(v1.z, v1.w)};
            if (o >= 0 && chk(o + zc + 8 * sub + 7, p.z_elems, 301))
                *reinterpret_cast<uint4*>(z + o + zc + 8 * sub) = *reinterpret_cast<const uint4*>(h);
        }
    } else {
        float* z = reinterpret_cast<float*>(p.z);
        const int g = lane & 7;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int row = 4 * i + (lane >> 3);
            const float4 v = stg[row * 8 + (g ^ (row & 7))];
            const int64_t o = __shfl_sync(0xffffffffu, zr, row);
            if (o >= 0 && chk(o + zc + 4 * g + 3, p.z_elems, 302)) *reinterpret_cast<float4*>(z + o + zc + 4 * g) = v;
        }
    }
    __syncwarp();
}

// Epilogue of one tile for one epilogue warp: TMEM lane quarter q holds 32 rows of the
// accumulator (thread = row m).  The tile's columns go out in pairs of 32-column blocks (both
// TMEM loads in flight before the wait); the two warps of a quarter (half 0 / 1) take
// alternate pairs.  With an output tensor map the blocks leave by TMA stores; otherwise by
// warp stores, with row and column offsets computed once per tile, one per lane, and passed
// by shuffle.
// Rank-one epilogue terms of the rewritten non-sum semirings, applied to one 32-column block
// (this lane's row m, columns n .. n + 31) before the stores scale by alpha.
template <int EPI>
__device__ __forceinline__ void apply_terms(const TcParams& p, uint32_t (&r)[32], float rt, uint32_t b, uint32_t m,
                                            uint32_t n) {
    if (EPI == 0) return;
    const float* ct = p.col_term + (uint64_t)b * p.zN;
    bool marked = false;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const float c = __ldg(ct + min(n + (uint32_t)i, p.zN - 1));
        const float a = __uint_as_float(r[i]);
        float v;
        if (EPI == 1) {
            const float s = rt + c, d = s - 2.f * a;
            marked |= d < p.sq_tau * s && n + (uint32_t)i < p.zN;
            v = fmaxf(d, 0.f);
        } else if (a > 1e-30f) {
            v = rt + c + logf(a);
        } else {
            v = __int_as_float(0x7fc00000);
            if (p.mark_count) atomicAdd(p.mark_count, 1);
        }
        r[i] = __float_as_uint(v);
    }
    // the 32 columns n .. n + 31 lie in one 128-column tile (n is a multiple of 32)
    if (EPI == 1 && marked && m < p.zM && p.fix_flags) {
        p.fix_flags[((uint64_t)b * p.fix_tiles_m + m / 128u) * p.fix_tiles_n + n / 128u] = 1u;
        p.fix_flags[p.fix_tag_index] = 1u;
    }
}

// out[box] += smem box (fp32 add in L2), through the output tensor map
__device__ __forceinline__ void tma_reduce_add_5d(const CUtensorMap* map, const int c[5], uint32_t src) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.5d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2, %3, %4, %5}], [%6];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]), "r"(c[4]), "r"(src)
        : "memory");
}

// Partial sums of a split tile, for one epilogue warp: column block c (32 columns) holds
// register i of every lane at c * 1024 + i * 32 + lane, so each access of the warp is one
// contiguous 128-byte line.  L2 only (the other parts run on other SMs).
__device__ __forceinline__ void add_partial(uint32_t (&r)[32], const float* pw, uint32_t c, int lane) {
    const float* s = pw + (size_t)c * 1024u + (uint32_t)lane;
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) + __ldcg(s + 32 * i));
}
__device__ __forceinline__ void put_partial(const uint32_t (&r)[32], float* pw, uint32_t c, int lane) {
    float* s = pw + (size_t)c * 1024u + (uint32_t)lane;
#pragma unroll
    for (int i = 0; i < 32; ++i) __stcg(s + 32 * i, __uint_as_float(r[i]));
}

// Bounded wait, by every lane, until the flag holds `want` (acquire at GPU scope: the partial
// sums written before the flag's release are visible afterwards).
__device__ __forceinline__ bool wait_flag(const unsigned long long* f, unsigned long long want, volatile int* abort,
                                          uint64_t timeout_ns) {
    const uint64_t t0 = globaltimer();
    bool ok = true;
    for (uint32_t n = 0;; ++n) {
        unsigned long long v;
        asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(f) : "memory");
        if (v == want) break;
        if ((n & 15) == 15) {
            if (*abort || globaltimer() - t0 > timeout_ns) {
                if (!*abort) {
                    *abort = 1;
                    atomicExch(&g_status, (int)TRA_ERR_TIMEOUT);
                }
                ok = false;
                break;
            }
        }
        __nanosleep(100);
    }
    return __all_sync(0xffffffffu, ok);
}
__device__ __forceinline__ void set_flag(unsigned long long* f, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(f), "l"(v) : "memory");
}

// The worker of part 0 of a tile split in two (split_reduce): this epilogue warp zeroes its
// share of the tile's output (the 32-column blocks it also stores: c = 2 half + 4 i, + 1) from
// its zeroed staging tile by TMA stores, waits for them to complete and releases the flag.
__device__ __forceinline__ void zero_split_share(const TcParams& p, const CUtensorMap* map_z, uint8_t* epi,
                                                 uint32_t q, uint32_t half, int lane, uint32_t b, uint32_t m,
                                                 uint32_t n0, unsigned long long* flag) {
    float4* stg = reinterpret_cast<float4*>(epi + (q + 4 * half) * kEpiTile);
#pragma unroll
    for (int g = 0; g < 8; ++g) stg[lane * 8 + g] = make_float4(0.f, 0.f, 0.f, 0.f);
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
        const uint32_t row0 = m - (uint32_t)lane;
        for (uint32_t c = 2 * half; c < p.block_n / 32; c += 4)
            for (uint32_t k = 0; k < 2; ++k) {
                int cc[5];
                z_coords(p.zt, b, row0, n0 + (c + k) * 32u, cc);
                tma_store_5d(map_z, cc, smem_u32(stg));
            }
        bulk_commit();
        bulk_wait_all();  // the zeros are written
        asm volatile("fence.proxy.async.global;" ::: "memory");
        set_flag(flag, p.tag | 1u);
    }
    __syncwarp();
}

// A part of a split tile other than the last: leave this warp's sums in the part's own slot of
// the partial buffer and release them (no wait: every such part runs at once).
__device__ __forceinline__ void split_partial(const TcParams& p, uint32_t tmem_acc, uint32_t q, uint32_t half,
                                              int lane, float* pw, unsigned long long* flag) {
    const uint32_t nblk = p.block_n / 32;
    const uint32_t taddr = tmem_acc + ((q * 32u) << 16);
    for (uint32_t c = 2 * half; c < nblk; c += 4) {
        uint32_t ra[32], rb[32];
        tmem_ld32_nowait(taddr + c * 32u, ra);
        tmem_ld32_nowait(taddr + c * 32u + 32u, rb);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        put_partial(ra, pw, c, lane);
        put_partial(rb, pw, c + 1, lane);
    }
    __threadfence();
    __syncwarp();
    if (lane == 0) set_flag(flag, p.tag | 1u);
}

template <int EPI>
__device__ __forceinline__ void epilogue_tile(const TcParams& p, const CUtensorMap* map_z, uint8_t* epi,
                                              uint32_t tmem_acc, uint32_t q, uint32_t half, int lane, uint32_t b,
                                              uint32_t m, uint32_t n0, const float* addp = nullptr, uint32_t nadd = 0,
                                              size_t add_stride = 0, bool reduce = false) {
    float4* stg = reinterpret_cast<float4*>(epi + (q + 4 * half) * kEpiTile);
    const uint32_t nblk = p.block_n / 32;  // block_n is a multiple of 64
    const uint32_t taddr = tmem_acc + ((q * 32u) << 16);
    const float rt = EPI ? __ldg(p.row_term + (uint64_t)b * p.zM + min(m, p.zM - 1)) : 0.f;
    if (p.z_tma) {
        // TMA stores: the warp writes its 32 rows into its (1024-aligned) staging tile in the
        // 128-byte swizzle the output map uses, then one lane stores the box.  fp32: one box
        // per 32 columns; bf16: one box per 64 columns.  The tile is rewritten once the previous
        // box has left shared memory.  (A second staging tile per warp measured no faster and
        // costs the pair kernel a pipeline stage.)
        const uint32_t row0 = m - (uint32_t)lane;
        auto next_tile = [&]() -> float4* {
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
            return stg;
        };
        auto store_tile = [&](float4* t, uint32_t n) {
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
                int cc[5];
                z_coords(p.zt, b, row0, n, cc);
                if (reduce) tma_reduce_add_5d(map_z, cc, smem_u32(t));
                else tma_store_5d(map_z, cc, smem_u32(t));
                bulk_commit();
            }
        };
        for (uint32_t c = 2 * half; c < nblk; c += 4) {
            uint32_t ra[32], rb[32];
            tmem_ld32_nowait(taddr + c * 32u, ra);
            tmem_ld32_nowait(taddr + c * 32u + 32u, rb);
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            for (uint32_t j = 0; j < nadd; ++j) {  // the other parts' sums, in part order
                add_partial(ra, addp + j * add_stride, c, lane);
                add_partial(rb, addp + j * add_stride, c + 1, lane);
            }
            apply_terms<EPI>(p, ra, rt, b, m, n0 + c * 32u);
            apply_terms<EPI>(p, rb, rt, b, m, n0 + c * 32u + 32u);
            if (!p.out_bf16) {
#pragma unroll
                for (int blk = 0; blk < 2; ++blk) {
                    float4* t = next_tile();
#pragma unroll
                    for (int g = 0; g < 8; ++g) {
                        const uint32_t* r = blk ? rb : ra;
                        t[lane * 8 + (g ^ (lane & 7))] = make_float4(
                            p.alpha * __uint_as_float(r[4 * g]), p.alpha * __uint_as_float(r[4 * g + 1]),
                            p.alpha * __uint_as_float(r[4 * g + 2]), p.alpha * __uint_as_float(r[4 * g + 3]));
                    }
                    store_tile(t, n0 + (c + blk) * 32u);
                }
            } else {
                float4* t = next_tile();
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                    const uint32_t* r = g < 4 ? ra : rb;
                    const int o = 8 * (g & 3);
                    __nv_bfloat162 h[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        h[i] = __floats2bfloat162_rn(p.alpha * __uint_as_float(r[o + 2 * i]),
                                                     p.alpha * __uint_as_float(r[o + 2 * i + 1]));
                    t[lane * 8 + (g ^ (lane & 7))] = *reinterpret_cast<const float4*>(h);
                }
                store_tile(t, n0 + c * 32u);
            }
        }
        return;
    }
    const int64_t zr = m < p.zM ? role_offset(p.zb, b) + role_offset(p.zm, m) : (int64_t)-1;
    const int64_t zc_lane = (uint32_t)lane < nblk && n0 + 32u * lane < p.zN ? role_offset(p.zn, n0 + 32u * lane) : 0;
    for (uint32_t c = 2 * half; c < nblk; c += 4) {
        uint32_t ra[32], rb[32];
        tmem_ld32_nowait(taddr + c * 32u, ra);
        tmem_ld32_nowait(taddr + c * 32u + 32u, rb);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        for (uint32_t j = 0; j < nadd; ++j) {
            add_partial(ra, addp + j * add_stride, c, lane);
            add_partial(rb, addp + j * add_stride, c + 1, lane);
        }
        apply_terms<EPI>(p, ra, rt, b, m, n0 + c * 32u);
        apply_terms<EPI>(p, rb, rt, b, m, n0 + c * 32u + 32u);
        store_block(p, stg, zr, __shfl_sync(0xffffffffu, zc_lane, c), lane, ra, n0 + c * 32u);
        store_block(p, stg, zr, __shfl_sync(0xffffffffu, zc_lane, c + 1), lane, rb, n0 + c * 32u + 32u);
    }
}

// One unit's epilogue for one epilogue warp.  A whole tile goes out as before.  Of a split tile
// (plain epilogue only), the parts before the last each leave their sums in a slot of their
// own; the last part waits for all of them, adds them to its accumulator in part order (a fixed
// order: results are deterministic), stores the tile and clears the flags.  rank: the CTA's rank
// in its pair (0 for one CTA per tile); regions: TMEM lane quarters per tile (4 per CTA).  False
// when a wait gave up.
__device__ __forceinline__ bool epilogue_unit(const TcParams& p, const CUtensorMap* map_z, uint8_t* epi,
                                              uint32_t tmem_acc, uint32_t q, uint32_t half, int lane, uint32_t b,
                                              uint32_t mrow, uint32_t n0, uint32_t tile, uint32_t part, uint32_t rank,
                                              uint32_t regions, volatile int* abort) {
    if (part == kWhole) {
        if (p.epi == 0) epilogue_tile<0>(p, map_z, epi, tmem_acc, q, half, lane, b, mrow, n0);
        else if (p.epi == 1) epilogue_tile<1>(p, map_z, epi, tmem_acc, q, half, lane, b, mrow, n0);
        else epilogue_tile<2>(p, map_z, epi, tmem_acc, q, half, lane, b, mrow, n0);
        return true;
    }
    // slot (tile, part j) of this warp's lane quarter: partial sums and one flag per epilogue warp
    const uint32_t others = p.split - 1;
    const size_t region = (size_t)p.block_n * 32u;
    float* slot0 = p.part + ((size_t)(tile - p.n_full) * others * regions + rank * 4u + q) * region;
    unsigned long long* flag0 = p.flags + (size_t)(tile - p.n_full) * others * (2u * regions) + rank * 8u + half * 4u + q;
    if (p.split_reduce) {
        // both parts add into the output zeroed by part 0's worker at the start of the launch
        if (part == 1) {
            if (!wait_flag(flag0, p.tag | 1u, abort, p.timeout_ns)) return false;
            asm volatile("fence.proxy.async.global;" ::: "memory");
        }
    } else if (part < others) {
        split_partial(p, tmem_acc, q, half, lane, slot0 + part * regions * region, flag0 + part * 2u * regions);
        return true;
    } else {
        for (uint32_t j = 0; j < others; ++j)
            if (!wait_flag(flag0 + j * 2u * regions, p.tag | 1u, abort, p.timeout_ns)) return false;
    }
    const bool red = p.split_reduce != 0;
    epilogue_tile<0>(p, map_z, epi, tmem_acc, q, half, lane, b, mrow, n0, red ? nullptr : slot0, red ? 0u : others,
                     regions * region, red);
    if (lane == 0 && (!red || part == 1))  // ready for the next call
        for (uint32_t j = 0; j < (red ? 1u : others); ++j)
            *reinterpret_cast<volatile unsigned long long*>(flag0 + j * 2u * regions) = 0ull;
    return true;
}

// ------------------------------------------------------------------ the kernel
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
            const __grid_constant__ CUtensorMap map_z, const __grid_constant__ TcParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t stage_bytes = p.a_bytes + p.b_bytes;
    const uint32_t epi_s = base + p.stages * stage_bytes;  // epilogue staging, 1024-aligned (TMA swizzle)
    const uint32_t bar0 = epi_s + kEpiBytes;
    // barrier block: full[S], empty[S], tfull[2], tempty[2], done, then tmem slot and abort flag
    const uint32_t full0 = bar0, empty0 = bar0 + 8 * p.stages, tfull0 = bar0 + 16 * p.stages;
    const uint32_t tempty0 = tfull0 + 16, done_bar = tempty0 + 16;
    uint8_t* gbase = smem_raw + (base - raw);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + (done_bar + 8 - base));
    volatile int* abort = reinterpret_cast<volatile int*>(gbase + (done_bar + 12 - base));
    uint8_t* epi = gbase + (epi_s - base);

    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x / 32), 0), lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < p.stages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull0 + 8 * a, 1);
            mbar_init(tempty0 + 8 * a, 32 * kEpiWarps);
        }
        mbar_init(done_bar, 1);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(p.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = __shfl_sync(0xffffffffu, *tmem_slot, 0);  // warp-uniform

    if (warp < kProducers) {
        // ---------------------------------------------------------------- TMA producers
        producer_steps<false>(&map_a, &map_b, p, (uint32_t)warp, lane, blockIdx.x, gridDim.x, 0u, base, full0, empty0, abort);
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------------- MMA issuer
        // The whole warp runs the loop (waits by every lane, results shuffled from lane 0 so
        // that control flow and operands stay warp-uniform); the elected lane issues.
        // Descriptors are formed once; stage and K-step offsets go into the start-address
        // field (shared addresses stay below 2^18, so the field does not carry).
        auto wait_u = [&](uint32_t b_, uint32_t parity) {
            return __shfl_sync(0xffffffffu, (int)mbar_wait(b_, parity, abort, p.timeout_ns), 0) != 0;
        };
        uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
        bool ok = true;
        const uint32_t a_lbo = p.a.mn_major ? 8192u : 16u, b_lbo = p.b.mn_major ? 8192u : 16u;
        const uint32_t a_kstep = (p.a.mn_major ? 2048u : 32u) >> 4, b_kstep = (p.b.mn_major ? 2048u : 32u) >> 4;
        const uint64_t da0 = smem_desc(base, a_lbo, 1024), db0 = smem_desc(base + p.a_bytes, b_lbo, 1024);
        for (uint32_t u = blockIdx.x; u < p.n_units && ok; u += gridDim.x) {
            uint32_t tile, kb0, kb1, part;
            unit_of(p, u, tile, kb0, kb1, part);
            if (!wait_u(tempty0 + 8 * acc, acc_phase ^ 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + acc * p.block_n;
            for (uint32_t kb = kb0; kb < kb1; ++kb) {
                if (!wait_u(full0 + 8 * stage, phase)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t so = (stage * stage_bytes) >> 4;
#pragma unroll
                for (uint32_t k = 0; k < kBlockK / 16; ++k)
                    tc_mma_elect(d_tmem, da0 + so + k * a_kstep, db0 + so + k * b_kstep, p.idesc,
                                 (kb != kb0 || k != 0));
                tc_commit_elect(empty0 + 8 * stage);  // frees the stage once these MMAs have read it
                if (++stage == p.stages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (!ok) break;
            tc_commit_elect(tfull0 + 8 * acc);  // accumulator ready for the epilogue
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1;
            }
        }
        // every MMA issued so far has completed once this commit arrives
        tc_commit_elect(done_bar);
        volatile int never = 0;
        mbar_wait(done_bar, 0, &never, p.timeout_ns);
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- epilogue (warps 5-12)
        const uint32_t q = warp & 3;  // TMEM lane quarter this warp may access
        const uint32_t half = (uint32_t)(warp - kMmaWarp - 1) >> 2;
        uint32_t acc = 0, acc_phase = 0;
        if (p.split_reduce && p.n_full + blockIdx.x < p.n_units) {  // this worker's split unit
            uint32_t tile, kb0, kb1, part, b, mt, nt;
            unit_of(p, p.n_full + blockIdx.x, tile, kb0, kb1, part);
            if (part == 0) {
                tile_of(p, tile, b, mt, nt);
                zero_split_share(p, &map_z, epi, q, half, lane, b, mt * kBlockM + q * 32 + lane, nt * p.block_n,
                                 p.flags + (size_t)(tile - p.n_full) * 8u + half * 4u + q);
            }
        }
        for (uint32_t u = blockIdx.x; u < p.n_units; u += gridDim.x) {
            uint32_t tile, kb0, kb1, part, b, mt, nt;
            unit_of(p, u, tile, kb0, kb1, part);
            tile_of(p, tile, b, mt, nt);
            if (!mbar_wait(tfull0 + 8 * acc, acc_phase, abort, p.timeout_ns)) break;
            tc_fence_after();
            const uint32_t mrow = mt * kBlockM + q * 32 + lane;
            if (!epilogue_unit(p, &map_z, epi, tmem_base + acc * p.block_n, q, half, lane, b, mrow, nt * p.block_n, tile,
                               part, 0u, 4u, abort))
                break;
            tc_fence_before();
            mbar_arrive(tempty0 + 8 * acc);
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1;
            }
        }
        if (lane == 0) bulk_wait_all();  // this warp's TMA stores have completed
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(p.tmem_cols)
                     : "memory");
    }
}

// ------------------------------------------------------------------ CTA-pair kernel
// Two CTAs of a cluster share one 256 x 256 output tile: tcgen05.mma.cta_group::2
// (M = 256, N = 256) issued by the even CTA reads A rows 0-127 and B rows 0-127 from its
// own shared memory and A rows 128-255 / B rows 128-255 from the odd CTA's, and writes
// accumulator rows 0-127 to the even CTA's tensor memory, rows 128-255 to the odd CTA's.
// Each SM therefore loads half of B per K step (32 KB instead of 48 KB for the same MMA
// work).
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    tc_gemm_2sm(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                const __grid_constant__ CUtensorMap map_z, const __grid_constant__ TcParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t stage_bytes = p.a_bytes + p.b_bytes;  // this CTA's half of one K step
    const uint32_t epi_s = base + p.stages * stage_bytes;  // epilogue staging, 1024-aligned (TMA swizzle)
    const uint32_t bar0 = epi_s + kEpiBytes;
    const uint32_t full0 = bar0, empty0 = bar0 + 8 * p.stages, tfull0 = bar0 + 16 * p.stages;
    const uint32_t tempty0 = tfull0 + 16, done_bar = tempty0 + 16;
    uint8_t* gbase = smem_raw + (base - raw);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + (done_bar + 8 - base));
    volatile int* abort = reinterpret_cast<volatile int*>(gbase + (done_bar + 12 - base));
    uint8_t* epi = gbase + (epi_s - base);

    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x / 32), 0), lane = threadIdx.x % 32;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    const uint32_t pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < p.stages; ++s) {
            mbar_init(full0 + 8 * s, 1);   // the even CTA's producer arrives; both CTAs' bytes count
            mbar_init(empty0 + 8 * s, 1);  // one multicast commit
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull0 + 8 * a, 1);
            mbar_init(tempty0 + 8 * a, 2 * kEpiWarps);  // one lane of each epilogue warp of both CTAs
        }
        mbar_init(done_bar, 1);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(p.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers exist before anyone signals across the pair
    tc_fence_after();
    const uint32_t tmem_base = __shfl_sync(0xffffffffu, *tmem_slot, 0);  // warp-uniform

    if (warp < kProducers) {
        // ---------------------------------------------------------------- TMA producers (both CTAs)
        producer_steps<true>(&map_a, &map_b, p, (uint32_t)warp, lane, pair, n_pairs, rank, base, full0, empty0, abort);
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------------- MMA issuer (even CTA)
        // whole warp, uniform waits, elected issue, descriptors formed once (as in tc_gemm)
        if (leader) {
            auto wait_u = [&](uint32_t b_, uint32_t parity) {
                return __shfl_sync(0xffffffffu, (int)mbar_wait_cl(b_, parity, abort, p.timeout_ns), 0) != 0;
            };
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            const uint32_t a_lbo = p.a.mn_major ? 8192u : 16u, b_lbo = p.b.mn_major ? 8192u : 16u;
            const uint32_t a_kstep = (p.a.mn_major ? 2048u : 32u) >> 4, b_kstep = (p.b.mn_major ? 2048u : 32u) >> 4;
            const uint64_t da0 = smem_desc(base, a_lbo, 1024), db0 = smem_desc(base + p.a_bytes, b_lbo, 1024);
            for (uint32_t u = pair; u < p.n_units && ok; u += n_pairs) {
                uint32_t tile, kb0, kb1, part;
                unit_of(p, u, tile, kb0, kb1, part);
                if (!wait_u(tempty0 + 8 * acc, acc_phase ^ 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * p.block_n;
                for (uint32_t kb = kb0; kb < kb1; ++kb) {
                    if (!wait_u(full0 + 8 * stage, phase)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t so = (stage * stage_bytes) >> 4;
#pragma unroll
                    for (uint32_t k = 0; k < kBlockK / 16; ++k)
                        tc_mma_pair_elect(d_tmem, da0 + so + k * a_kstep, db0 + so + k * b_kstep, p.idesc,
                                          (kb != kb0 || k != 0));
                    tc_commit_pair_elect(empty0 + 8 * stage, 3);  // frees this stage in both CTAs
                    if (++stage == p.stages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                tc_commit_pair_elect(tfull0 + 8 * acc, 3);  // accumulator ready in both CTAs
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1;
                }
            }
            tc_commit_pair_elect(done_bar, 1);  // all MMAs issued so far have completed
            volatile int never = 0;
            mbar_wait_cl(done_bar, 0, &never, p.timeout_ns);
            __syncwarp();
        }
    } else {
        // ---------------------------------------------------------------- epilogue (warps 5-12, both CTAs)
        const uint32_t q = warp & 3;
        const uint32_t half = (uint32_t)(warp - kMmaWarp - 1) >> 2;
        uint32_t acc = 0, acc_phase = 0;
        if (p.split_reduce && p.n_full + pair < p.n_units) {  // this worker's split unit
            uint32_t tile, kb0, kb1, part, b, mt, nt;
            unit_of(p, p.n_full + pair, tile, kb0, kb1, part);
            if (part == 0) {
                tile_of(p, tile, b, mt, nt);
                zero_split_share(p, &map_z, epi, q, half, lane, b, mt * 2 * kBlockM + rank * kBlockM + q * 32 + lane,
                                 nt * p.block_n, p.flags + (size_t)(tile - p.n_full) * 16u + rank * 8u + half * 4u + q);
            }
        }
        for (uint32_t u = pair; u < p.n_units; u += n_pairs) {
            uint32_t tile, kb0, kb1, part, b, mt, nt;
            unit_of(p, u, tile, kb0, kb1, part);
            tile_of(p, tile, b, mt, nt);
            if (!mbar_wait_cl(tfull0 + 8 * acc, acc_phase, abort, p.timeout_ns)) break;
            tc_fence_after();
            const uint32_t mrow = mt * 2 * kBlockM + rank * kBlockM + q * 32 + lane;
            if (!epilogue_unit(p, &map_z, epi, tmem_base + acc * p.block_n, q, half, lane, b, mrow, nt * p.block_n, tile,
                               part, rank, 8u, abort))
                break;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(tempty0 + 8 * acc, 0));
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1;
            }
        }
        if (lane == 0) bulk_wait_all();  // this warp's TMA stores have completed
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the even CTA's MMAs have finished with the odd CTA's memory
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(p.tmem_cols)
                     : "memory");
    }
}

// Test hook: one thread waits on an mbarrier that nothing arrives on; the bounded
// wait must give up after timeout_ns and record TRA_ERR_TIMEOUT.
__global__ void wait_timeout_probe(uint64_t timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        mbar_wait(smem_u32(&bar), 0, &abort, timeout_ns);
    }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

}  // namespace

struct TcDim {
    int role;
    uint32_t div, mod, box;
    uint64_t extent, stride;  // stride in elements
};

struct TcOperandPlan {
    int ndims = 0;
    TcDim dims[5];
    TcOpDev dev;
};

struct TcPlan {
    TcOperandPlan a, b;
    TcOperandPlan z;     // output tensor map (TMA-store epilogue), valid when z_tma
    bool z_tma = false;
    bool pair = false;  // 256 x block_n tile on a cluster of two CTAs
    uint32_t b_rows = 0;  // rows of Y one CTA loads per K step
    uint32_t block_n = 0, stages = 0, tiles_m = 0, tiles_n = 0, n_tiles = 0, num_kb = 0, tmem_cols = 0;
    uint32_t idesc = 0, smem = 0;
    // K split of the last wave's tiles, chosen for `workers` co-resident CTAs (one CTA per
    // tile) or CTA pairs; split = 1 when it does not apply
    uint32_t workers = 0, split = 1, n_full = 0;
    uint64_t ws_part = 0, ws_flags = 0;  // workspace bytes of the partial sums and of the flags
};

void tc_free(TcPlan* t) { delete t; }
bool tc_tma_store(const TcPlan* t) { return t && t->z_tma; }

namespace {

// Physical dimensions of a relation's blocked layout, innermost first: the local part of every
// label (last index first), then the key part; unit dimensions dropped.  Boxes: tiles[role]
// consecutive composite indices of each role, one TMA box that stays inside one block.
bool box_dims(const Plan& p, const Operand& t, const uint32_t (&tiles)[4], int elem_bytes, TcOperandPlan& out) {
    struct Phys {
        int label, key;
        uint64_t extent, stride;
    };
    Phys ph[2 * TRA_MAX_RANK];
    int n = 0;
    for (int i = t.rank - 1; i >= 0; --i) {
        const int l = t.label[i];
        if (p.B[l] / p.D[l] > 1) ph[n++] = {l, 0, (uint64_t)(p.B[l] / p.D[l]), (uint64_t)t.loc_stride[i]};
    }
    for (int i = t.rank - 1; i >= 0; --i) {
        const int l = t.label[i];
        if (p.D[l] > 1) ph[n++] = {l, 1, (uint64_t)p.D[l], (uint64_t)t.key_stride[i]};
    }
    if (n == 0) return false;
    if (ph[0].stride != 1 || ph[0].key) return false;
    // composite stride of every label in its role
    uint64_t div[TRA_MAX_LABELS] = {};
    for (int r = 0; r < 4; ++r) {
        uint64_t d = 1;
        for (int l : p.comp[r]) {
            div[l] = d;
            d *= (uint64_t)p.B[l];
        }
    }
    TcDim dims[2 * TRA_MAX_RANK];
    for (int j = 0; j < n; ++j) {
        const int l = ph[j].label;
        TcDim& dm = dims[j];
        dm.role = p.role[l];
        dm.extent = ph[j].extent;
        dm.stride = ph[j].stride;
        const uint64_t b = (uint64_t)(p.B[l] / p.D[l]);
        dm.div = (uint32_t)(ph[j].key ? div[l] * b : div[l]);
        dm.mod = (uint32_t)ph[j].extent;
        dm.box = 1;
    }
    // boxes: walk each role's labels innermost first with the tile extent (1: box 1 everywhere)
    for (int r = 0; r < 4; ++r) {
        uint64_t rem = tiles[r];
        int last_dim = -1;
        for (int l : p.comp[r]) {
            if (t.pos_of(l) < 0) {
                if (rem != 1) return false;  // the tile would span a label this operand lacks
                continue;
            }
            for (int key = 0; key < 2; ++key) {
                int j = -1;
                for (int q = 0; q < n; ++q)
                    if (ph[q].label == l && ph[q].key == key) j = q;
                if (j < 0) continue;  // unit dimension
                const uint64_t ext = ph[j].extent;
                uint64_t box;
                if (rem >= ext) {
                    if (rem % ext) return false;
                    box = ext;
                } else {
                    if (ext % rem) return false;
                    box = rem;
                }
                rem /= box;
                dims[j].box = (uint32_t)box;
                if (box > 1) {
                    if (j <= last_dim) return false;  // box order must follow the composite order
                    last_dim = j;
                }
            }
        }
        if (rem != 1) return false;
    }
    // Merge neighbours that are one dimension in memory and in their role's composite index
    // (the outer's stride and composite divisor continue the inner's): the box stays one
    // contiguous range of the merged coordinate when the inner box is whole or the outer box is
    // 1, and its bytes land in shared memory in the same order.  A relation with more than five
    // physical dimensions (a blocked output, say) then fits a rank-5 tensor map.
    int m = 0;
    for (int j = 0; j < n; ++j) {
        if (m > 0) {
            TcDim& a = dims[m - 1];
            const TcDim& b = dims[j];
            const uint64_t box = b.box == 1 ? a.box : (uint64_t)a.box * b.box;
            if (a.role == b.role && b.stride == a.stride * a.extent && (uint64_t)b.div == (uint64_t)a.div * a.mod &&
                (a.box == a.extent || b.box == 1) && box <= 256 && a.extent * b.extent <= 0xffffffffull) {
                a.box = (uint32_t)box;
                a.extent *= b.extent;
                a.mod = (uint32_t)a.extent;
                continue;
            }
        }
        dims[m++] = dims[j];
    }
    if (m > 5) return false;
    for (int j = 1; j < m; ++j)
        if ((dims[j].stride * (uint64_t)elem_bytes) % 16) return false;
    out.ndims = m;
    for (int j = 0; j < m; ++j) out.dims[j] = dims[j];
    return true;
}

// Physical dimensions and TMA boxes of an operand: a tile of mn_tile rows along M (X) or N (Y)
// and kBlockK along K, loaded in mn_loads boxes.
bool operand_dims(const Plan& p, const Operand& t, int mn_role, uint32_t mn_tile, int mn_loads, TcOperandPlan& out) {
    const uint32_t tiles[4] = {1u, mn_role == kM ? mn_tile : 1u, mn_role == kN ? mn_tile : 1u, (uint32_t)kBlockK};
    if (!box_dims(p, t, tiles, 2, out)) return false;
    const int n = out.ndims;
    // shared-memory layout: K-major (innermost K, 64 wide; the other boxes are the M/N rows)
    // or MN-major (innermost M/N, 64 wide per load; the other boxes are K rows)
    const int r0 = out.dims[0].role;
    if (out.dims[0].box != 64 || out.dims[0].extent % 64) return false;
    if (r0 == kK) {
        if (mn_loads != 1) return false;
        for (int j = 1; j < n; ++j)
            if (out.dims[j].box > 1 && out.dims[j].role != mn_role) return false;
        out.dev.mn_major = 0;
        out.dev.n_loads = 1;
    } else if (r0 == mn_role) {
        for (int j = 1; j < n; ++j)
            if (out.dims[j].box > 1 && out.dims[j].role != kK) return false;
        out.dev.mn_major = 1;
        out.dev.n_loads = mn_loads;
    } else {
        return false;
    }
    for (int j = 0; j < 5; ++j) {
        out.dev.role[j] = j < n ? out.dims[j].role : kK;
        out.dev.div[j] = FastDiv(j < n ? out.dims[j].div : 1u);
        out.dev.mod[j] = FastDiv(j < n ? out.dims[j].mod : 1u);
    }
    return true;
}

}  // namespace

namespace {

// The output's tensor map for TMA stores from the epilogue: boxes of 32 rows (M) by n_tile
// columns (N), the innermost dimension being the innermost N label (n_tile wide, 128 bytes).
bool z_dims(const Plan& p, uint32_t n_tile, TcOperandPlan& out) {
    const uint32_t tiles[4] = {1u, 32u, n_tile, 1u};
    const int eb = p.out_bf16 ? 2 : 4;
    if (!box_dims(p, p.Z, tiles, eb, out)) return false;
    if (out.dims[0].role != kN || out.dims[0].box != n_tile || n_tile * (uint32_t)eb != 128) return false;
    for (int j = 0; j < 5; ++j) {
        out.dev.role[j] = j < out.ndims ? out.dims[j].role : kK;
        out.dev.div[j] = FastDiv(j < out.ndims ? out.dims[j].div : 1u);
        out.dev.mod[j] = FastDiv(j < out.ndims ? out.dims[j].mod : 1u);
    }
    return true;
}

// Operand tilings for one CTA: A holds a_rows output rows x 64 K, B holds b_rows output
// columns x 64 K.  Either may be K-major (one box) or M/N-major (boxes of 64 rows).
bool plan_operands(const Plan& p, uint32_t a_rows, uint32_t b_rows, TcPlan* t) {
    bool ok = operand_dims(p, p.X, kM, a_rows, 1, t->a);
    if (!ok || t->a.dev.mn_major) {
        t->a = TcOperandPlan();
        ok = operand_dims(p, p.X, kM, 64, a_rows / 64, t->a) && t->a.dev.mn_major;
    }
    if (!ok) return false;
    bool okb = operand_dims(p, p.Y, kN, b_rows, 1, t->b);
    if (!okb || t->b.dev.mn_major) {
        t->b = TcOperandPlan();
        okb = operand_dims(p, p.Y, kN, 64, b_rows / 64, t->b) && t->b.dev.mn_major;
    }
    return okb;
}

}  // namespace

namespace {

// Fill t for one tiling: a CTA pair (256 x bn tile, each CTA loading 128 rows of X and bn / 2
// rows of Y) or a single CTA (128 x bn).  False when the operands cannot be boxed that way.
bool build_tc(const Plan& p, bool pair, uint32_t bn, TcPlan* t) {
    *t = TcPlan();
    if (!plan_operands(p, kBlockM, pair ? bn / 2 : bn, t)) return false;
    t->pair = pair;
    t->block_n = bn;
    t->b_rows = pair ? bn / 2 : bn;
    const uint32_t stage = (uint32_t)(kBlockM * kBlockK * 2 + t->b_rows * kBlockK * 2);
    t->stages = (kMaxSmem - 1024 - 256 - kEpiBytes) / stage;
    if (t->stages > 8) t->stages = 8;
    if (t->stages < (uint32_t)kProducers) return false;  // the producers' parity waits need stages >= kProducers
    t->smem = t->stages * stage + 1024 + 256 + kEpiBytes;
    const uint32_t tile_m = pair ? 2 * kBlockM : kBlockM;
    t->tiles_m = (uint32_t)(p.ext[kM] / tile_m);
    t->tiles_n = (uint32_t)(p.ext[kN] / bn);
    t->n_tiles = (uint32_t)(p.ext[kBatch] * t->tiles_m * t->tiles_n);
    t->num_kb = (uint32_t)(p.ext[kK] / kBlockK);
    if ((uint64_t)t->n_tiles * t->num_kb >= (1ull << 31)) return false;  // K steps are counted in 32 bits
    // TMA-store epilogue: boxes of 32 rows x 128 bytes of the output
    t->z_tma = p.tc_store != 0 && z_dims(p, p.out_bf16 ? 64u : 32u, t->z);
    if (p.tc_store == 1 && !t->z_tma) return false;  // TMA stores asked for and no output map fits
    t->tmem_cols = 2 * bn <= 128 ? 128 : (2 * bn <= 256 ? 256 : 512);
    t->idesc = (1u << 4)                                   // D: fp32 (M = 256 for a pair: two CTAs' rows)
               | (1u << 7) | (1u << 10)                    // A, B: bf16
               | ((uint32_t)t->a.dev.mn_major << 15)       // A major-ness
               | ((uint32_t)t->b.dev.mn_major << 16)       // B major-ness
               | ((bn >> 3) << 17)                         // N / 8
               | ((tile_m >> 4) << 24);                    // M / 16
    return true;
}

}  // namespace

namespace {
int sm_count();
uint32_t pair_clusters(int sms, uint32_t smem);

// K split of the tiles of the last, partly filled wave: T tiles on C workers leave R = T mod C
// tiles for the last wave; each is split into s = min(C / R, 4) runs of K steps (each run at
// least 8 steps), so that the last wave keeps R * s workers busy for 1 / s of a tile's time.
// Tiles [0, n_full) stay whole; n_full = T - R is a multiple of C.
void split_config(uint32_t T, uint32_t C, uint32_t num_kb, uint32_t& n_full, uint32_t& s) {
    n_full = T;
    s = 1;
    if (C == 0 || T == 0) return;
    const uint32_t R = T % C;
    if (R == 0) return;
    uint32_t c = C / R;
    if (c > 4) c = 4;
    while (c > 1 && num_kb / c < 8) --c;
    if (c < 2) return;
    n_full = T - R;
    s = c;
}

// Workers a launch of this tiling gets on the current device: co-resident CTA pairs, or SMs.
uint32_t tc_workers(const TcPlan& t) {
    const int sms = sm_count();
    if (sms <= 0) return 0;
    return t.pair ? pair_clusters(sms, t.smem) : (uint32_t)sms;
}
}  // namespace

bool tc_plan(Plan* p) {
    if (p->unary || p->op != kMul || p->agg != kSum || !p->in_bf16 || p->literal) return false;
    const uint64_t M = p->ext[kM], N = p->ext[kN], K = p->ext[kK];
    if (M % kBlockM || K % kBlockK || N % 64) return false;
    // output: 32 consecutive columns contiguous (innermost label of Z is the innermost N label)
    if (p->comp[kN].empty()) return false;
    const int zl = p->Z.label[p->Z.rank - 1];
    if (zl != p->comp[kN][0] || (p->B[zl] / p->D[zl]) % 32) return false;
    TcPlan* t = new TcPlan();
    bool ok = false;
    if (p->tc_pair != 0 && M % 256 == 0 && N % 128 == 0) {
        // 256-wide tiles where the columns allow: a 256 x 128 tile moves 3/4 of the bytes of a
        // 256 x 256 one per K step for half the MMA work, and measured ~1.7x slower per flop
        if (N % 256 == 0 && p->tc_n != 128) ok = build_tc(*p, true, 256, t);
        if (!ok && p->tc_n != 256) ok = build_tc(*p, true, 128, t);
    }
    if (!ok && p->tc_pair != 1) ok = build_tc(*p, false, N % 256 == 0 ? 256 : (N % 128 == 0 ? 128 : 64), t);
    if (!ok) {
        delete t;
        return false;
    }
    p->tc = t;
    p->kernel = t->pair ? TRA_KERNEL_TC_BF16_PAIR : TRA_KERNEL_TC_BF16;
    if (p->ksplit) {
        t->workers = tc_workers(*t);
        (void)cudaGetLastError();  // no device here: plan without the split
        uint32_t n_full = 0, s = 1;
        split_config(t->n_tiles, t->workers, t->num_kb, n_full, s);
        if (s > 1) {
            t->split = s;
            t->n_full = n_full;
            const uint64_t R = t->n_tiles - n_full, tile = (uint64_t)(t->pair ? 2 * kBlockM : kBlockM) * t->block_n;
            t->ws_part = align256(R * (s - 1) * tile * 4);
            t->ws_flags = align256(R * (s - 1) * (t->pair ? 16 : 8) * 8);
            p->ws_bytes = t->ws_part + t->ws_flags;
        }
    }
    return true;
}

namespace {

bool encode(const TcOperandPlan& o, const void* base, CUtensorMap* map,
            CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, int elem = 2) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[5], strides[4];
    cuuint32_t box[5], estr[5] = {1, 1, 1, 1, 1};
    uint64_t last = 1;
    for (int j = 0; j < 5; ++j) {
        if (j < o.ndims) {
            dims[j] = o.dims[j].extent;
            box[j] = o.dims[j].box;
            if (j > 0) strides[j - 1] = o.dims[j].stride * (uint64_t)elem;
            last = o.dims[j].stride * o.dims[j].extent;
        } else {
            dims[j] = 1;
            box[j] = 1;
            if (j > 0) strides[j - 1] = ((last * (uint64_t)elem + 15) / 16) * 16;
        }
    }
    const CUresult r = fn(map, dtype, 5, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

// Co-resident clusters of tc_gemm_2sm at this dynamic shared memory size on the current device
// (cached: the occupancy query costs more than a launch).
uint32_t pair_clusters(int sms, uint32_t smem) {
    static std::mutex mu;
    static int cache_dev[64];
    static uint32_t cache_smem[64], cache_val[64];
    static int n = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return (uint32_t)sms / 2;
    {
        std::lock_guard<std::mutex> lk(mu);
        for (int i = 0; i < n; ++i)
            if (cache_dev[i] == dev && cache_smem[i] == smem) return cache_val[i];
    }
    uint32_t clusters = (uint32_t)sms / 2;
    if (cudaFuncSetAttribute(tc_gemm_2sm, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * clusters);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
        int active = 0;
        if (cudaOccupancyMaxActiveClusters(&active, tc_gemm_2sm, &cfg) == cudaSuccess && active > 0)
            clusters = (uint32_t)active < clusters ? (uint32_t)active : clusters;
    }
    (void)cudaGetLastError();
    std::lock_guard<std::mutex> lk(mu);
    if (n < 64) {
        cache_dev[n] = dev;
        cache_smem[n] = smem;
        cache_val[n] = clusters;
        ++n;
    }
    return clusters;
}

}  // namespace

namespace {
// Flag tag of one launch: a fixed high byte and a per-process launch counter (started from the
// clock), so that flags left by an earlier launch, or bytes the workspace held before, never
// read as this launch's.  Bits 0-7 stay free for the count of parts done.
unsigned long long next_split_tag() {
    static std::atomic<unsigned long long> n{(unsigned long long)std::chrono::steady_clock::now().time_since_epoch().count()};
    const unsigned long long e = n.fetch_add(1) & 0xffffffffffull;
    return (0xa5ull << 56) | (e << 8);
}
}  // namespace

int tc_execute(const Plan& p, const void* x, const void* y, void* z, cudaStream_t s, const TcExtra* ex, void* ws) {
    if (((uintptr_t)x | (uintptr_t)y | (uintptr_t)z) % 16) return fail(TRA_ERR_ARG, "tensor-core path needs 16-byte aligned buffers");
    const int sms = sm_count();
    if (sms <= 0) return fail(TRA_ERR_CUDA, "no device");
    const TcPlan& t = *p.tc;
    uint32_t clusters = 0;
    if (t.pair) {
        clusters = pair_clusters(sms, t.smem);
        if (clusters == 0) return fail(TRA_ERR_CUDA, "no co-resident pair of SMs for the pair kernel");
    }
    CUtensorMap ma, mb, mz;
    if (!encode(t.a, x, &ma) || !encode(t.b, y, &mb)) return fail(TRA_ERR_CUDA, "tensor map encoding failed");
    memset(&mz, 0, sizeof(mz));
    // an output in pinned host memory (device-addressable under unified addressing) takes the
    // warp-store epilogue: the tiles then cross the host link while later tiles compute
    cudaPointerAttributes pa;
    const bool z_device = cudaPointerGetAttributes(&pa, z) == cudaSuccess && pa.type == cudaMemoryTypeDevice;
    (void)cudaGetLastError();
    const bool z_tma = t.z_tma && z_device;
    if (z_tma && !encode(t.z, z, &mz, p.out_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                         p.out_bf16 ? 2 : 4))
        return fail(TRA_ERR_CUDA, "output tensor map encoding failed");
    TcParams tp;
    memset(&tp, 0, sizeof(tp));
    tp.a = t.a.dev;
    tp.b = t.b.dev;
    tp.zt = t.z.dev;
    tp.z_tma = z_tma ? 1u : 0u;
    tp.nb = (uint32_t)p.ext[kBatch];
    tp.M = (uint32_t)p.ext[kM];
    tp.N = (uint32_t)p.ext[kN];
    tp.K = (uint32_t)p.ext[kK];
    tp.tiles_m = t.tiles_m;
    tp.tiles_n = t.tiles_n;
    tp.n_tiles = t.n_tiles;
    // tile raster: groups of 16 M-tiles keep the operand panels of concurrent tiles in L2 for a
    // long K loop; with a short one (write-bound: the output dominates the bytes) N runs
    // fastest, so concurrent tiles write neighbouring output rows' segments
    tp.group_m = t.num_kb <= 8 ? 1u : 16u;
    tp.block_n = t.block_n;
    tp.stages = t.stages;
    tp.num_kb = t.num_kb;
    tp.tmem_cols = t.tmem_cols;
    tp.idesc = t.idesc;
    tp.a_bytes = kBlockM * kBlockK * 2;
    tp.b_bytes = t.b_rows * kBlockK * 2;
    tp.zb = role_map(p, p.Z, kBatch);
    tp.zm = role_map(p, p.Z, kM);
    tp.zn = role_map(p, p.Z, kN);
    tp.z = z;
    tp.alpha = (float)p.alpha;
    tp.out_bf16 = p.out_bf16;
    tp.timeout_ns = 2000000000ull;  // 2 s per wait
    tp.zM = tp.M;
    tp.zN = tp.N;
    tp.z_elems = (uint64_t)p.Z.total;
    if (ex) {
        if (ex->z_override) {
            if (z_tma) return fail(TRA_ERR_UNSUPPORTED, "output addressing override needs warp stores");
            if (ex->M > tp.M || ex->N > tp.N) return fail(TRA_ERR_ARG, "output bounds exceed the product");
            // the warp stores write runs of 32 columns: the map must keep each run contiguous
            if (ex->zn.n < 1 || ex->zn.t[0].div != 1 || ex->zn.t[0].loc_stride != 1 || ex->zn.t[0].sub % 32 ||
                ex->N % 32)
                return fail(TRA_ERR_UNSUPPORTED, "output map is not contiguous along N in runs of 32");
            tp.zb = ex->zb;
            tp.zm = ex->zm;
            tp.zn = ex->zn;
            tp.zM = ex->M;
            tp.zN = ex->N;
            tp.z_elems = ex->z_elems;
        }
        tp.epi = (uint32_t)ex->epi;
        tp.row_term = ex->row_term;
        tp.col_term = ex->col_term;
        tp.mark_count = ex->mark_count;
        tp.sq_tau = ex->sq_tau;
        tp.fix_flags = ex->fix_flags;
        tp.fix_tiles_m = ex->fix_tiles_m;
        tp.fix_tiles_n = ex->fix_tiles_n;
        tp.fix_tag_index = ex->fix_tag_index;
        tp.alpha = ex->alpha;
        if (tp.epi && (!tp.row_term || !tp.col_term)) return fail(TRA_ERR_ARG, "epilogue terms missing");
    }
    // work units: the plan's K split of the last wave when the workspace is there, no epilogue
    // terms are asked for, and this device gives the split no more workspace than planned
    const uint32_t workers = t.pair ? clusters : (uint32_t)sms;
    uint32_t n_full = t.n_tiles, split = 1;
    if (t.split > 1 && !ex && ws) {
        split_config(t.n_tiles, workers, t.num_kb, n_full, split);
        const uint64_t R = t.n_tiles - n_full, tile = (uint64_t)(t.pair ? 2 * kBlockM : kBlockM) * t.block_n;
        if (split > 1 && (align256(R * (split - 1) * tile * 4) > t.ws_part ||
                          align256(R * (split - 1) * (t.pair ? 16 : 8) * 8) > t.ws_flags)) {
            split = 1;
            n_full = t.n_tiles;
        }
    }
    tp.n_full = n_full;
    tp.split = split;
    tp.n_units = n_full + (t.n_tiles - n_full) * split;
    if (split > 1) {
        tp.part = reinterpret_cast<float*>(ws);
        tp.flags = reinterpret_cast<unsigned long long*>(reinterpret_cast<char*>(ws) + t.ws_part);
        tp.tag = next_split_tag();
        // two parts into an fp32 output through its tensor map: both add into the output (fp32
        // addition of two values into zero gives the same bits in either order)
        tp.split_reduce = split == 2 && z_tma && !p.out_bf16 ? 1u : 0u;
    }
    cudaError_t e;
    if (t.pair) {
        e = cudaFuncSetAttribute(tc_gemm_2sm, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)t.smem);
        if (e != cudaSuccess) return fail(TRA_ERR_CUDA, "smem attribute: %s", cudaGetErrorString(e));
        // persistent: one cluster per co-resident SM pair, at most one per work unit (so that
        // the whole tiles fill whole waves and every worker owns at most one split unit)
        const uint32_t c = clusters < tp.n_units ? clusters : tp.n_units;
        tc_gemm_2sm<<<2 * c, kThreads, t.smem, s>>>(ma, mb, mz, tp);
    } else {
        e = cudaFuncSetAttribute(tc_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)t.smem);
        if (e != cudaSuccess) return fail(TRA_ERR_CUDA, "smem attribute: %s", cudaGetErrorString(e));
        const unsigned grid = (unsigned)(tp.n_units < (uint32_t)sms ? tp.n_units : (uint32_t)sms);
        tc_gemm<<<grid, kThreads, t.smem, s>>>(ma, mb, mz, tp);
    }
    e = cudaGetLastError();
    return e == cudaSuccess ? TRA_OK : fail(TRA_ERR_CUDA, "tensor-core launch: %s", cudaGetErrorString(e));
}

TRA_CHECK_READER(read_and_clear_check_tc)

cudaError_t read_and_clear_status(int* value, cudaStream_t s) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(value, g_status, sizeof(int), 0, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    const int zero = 0;
    e = cudaMemcpyToSymbolAsync(g_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(s);
}

cudaError_t launch_wait_timeout_probe(uint64_t timeout_ns, cudaStream_t s) {
    wait_timeout_probe<<<1, 32, 0, s>>>(timeout_ns);
    return cudaGetLastError();
}

}  // namespace tra
