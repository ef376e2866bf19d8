// Internal structures shared by the host planner and the CUDA kernels of libtra.so.
//
// Addressing model.  Every label l of a plan has a global extent B_l, a
// partition count D_l and a block-local extent b_l = B_l / D_l.  In the
// relation ("blocked") layout of an operand with labels l_0..l_{r-1}, the
// element with global indices g_l sits at
//     sum_i (g_i / b_i) * key_stride_i + (g_i % b_i) * loc_stride_i
// with loc_stride_i = prod_{j>i} b_j and key_stride_i = (prod_{j>i} D_j) * |sub|
// (key k -> index range [k*b, (k+1)*b) of the key definition in section 2.2 of
// the EinDecomp page).  Labels are grouped into roles -- batch (X, Y and Z), M
// (X and Z), N (Y and Z), K (contracted) -- and each role's labels are folded
// into one composite index; a RoleMap turns a composite index into that role's
// part of an operand offset.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/tra.h"
#include "fastdiv.h"

#ifdef __CUDACC__
#define TRA_HD __host__ __device__ __forceinline__
#else
#define TRA_HD inline
#endif

namespace tra {

constexpr int kMaxTerms = 8;

enum Role { kBatch = 0, kM = 1, kN = 2, kK = 3 };
enum Op { kMul = 0, kAdd = 1, kSqdiff = 2, kSub = 3, kExpsub = 4, kId = 5 };
enum Agg { kSum = 0, kMax = 1, kMin = 2, kLse = 3, kNone = 4 };

struct Term {
    uint32_t div;        // composite stride of the label inside its role
    uint32_t ext;        // extent of the label inside the composite
    uint32_t sub;        // block-local extent (ext when the label is not split)
    uint32_t pad_;
    int64_t key_stride;  // elements per key step
    int64_t loc_stride;  // elements per local step
};

struct RoleMap {
    int32_t n;
    int32_t pad_;
    Term t[kMaxTerms];
};

TRA_HD int64_t role_offset(const RoleMap& r, uint32_t idx) {
    int64_t off = 0;
    for (int i = 0; i < r.n; ++i) {
        uint32_t g = (idx / r.t[i].div) % r.t[i].ext;
        uint32_t k = g / r.t[i].sub;
        uint32_t l = g - k * r.t[i].sub;
        off += (int64_t)k * r.t[i].key_stride + (int64_t)l * r.t[i].loc_stride;
    }
    return off;
}

// Row index a tile uses for loads: itself when in range; past the end, the last row
// (scalar loader) or the start of the last 4-aligned group (vector loader), so a
// clamped row keeps the vector loader's alignment.
TRA_HD uint32_t clamp_row(uint32_t idx, uint32_t ext, bool vec) {
    if (idx < ext) return idx;
    return vec ? ((ext - 1u) & ~3u) : ext - 1u;
}

// Stride of consecutive composite indices when the whole run [idx, idx+len) stays
// affine in this operand: returns the element stride, or 0 when not affine.
inline int64_t affine_stride(const RoleMap& r) {
    if (r.n == 0) return 0;
    const Term& t = r.t[0];
    if (t.div != 1) return 0;
    return t.loc_stride;
}

// ---------------------------------------------------------------- check builds
// Built with -DTRA_CHECK (libtra_check.so), the plain global loads and stores of the CUDA-core
// semiring, reduction, element-wise, split and repartition kernels and the warp stores of the
// tensor-core epilogue test their index against the extent of the buffer first (chk).  An
// access outside is skipped -- a load reads the aggregation's padding or 0, a store is dropped --
// and the translation unit's check word keeps the first site number that failed; ein_status()
// then returns TRA_ERR_BOUNDS.  Nothing traps.  In the normal build chk is constant true and
// the tests compile away.  Site numbers: 1xx semiring kernels, 2xx k_misc.cu, 3xx tensor-core
// epilogue.
#ifdef TRA_CHECK
namespace {
__device__ int g_check_site;  // one per translation unit (internal linkage)
}
__device__ __forceinline__ bool chk(int64_t off, uint64_t n, int site) {
    if (off >= 0 && (uint64_t)off < n) return true;
    atomicCAS(&g_check_site, 0, site);
    return false;
}
#define TRA_CHECK_READER(fn)                                                                       \
    cudaError_t fn(int* v, cudaStream_t s) {                                                       \
        cudaError_t e = cudaMemcpyFromSymbolAsync(v, g_check_site, sizeof(int), 0,                 \
                                                  cudaMemcpyDeviceToHost, s);                      \
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);                                        \
        const int zero = 0;                                                                        \
        if (e == cudaSuccess && *v)                                                                \
            e = cudaMemcpyToSymbolAsync(g_check_site, &zero, sizeof(int), 0,                       \
                                        cudaMemcpyHostToDevice, s);                                \
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);                                        \
        return e;                                                                                  \
    }
#else
#ifdef __CUDACC__
__device__ __forceinline__ constexpr bool chk(int64_t, uint64_t, int) { return true; }
#endif
#define TRA_CHECK_READER(fn)                      \
    cudaError_t fn(int* v, cudaStream_t) {        \
        *v = 0;                                   \
        return cudaSuccess;                       \
    }
#endif
// check words of the kernels' translation units (always 0 outside check builds)
cudaError_t read_and_clear_check_semiring(int* v, cudaStream_t s);
cudaError_t read_and_clear_check_misc(int* v, cudaStream_t s);
cudaError_t read_and_clear_check_tc(int* v, cudaStream_t s);
constexpr bool kCheckBuild =
#ifdef TRA_CHECK
    true;
#else
    false;
#endif

// Join + aggregate on CUDA cores (register-tiled).  Operands may be fp32 or bf16.
struct SemiringParams {
    const void* x;
    const void* y;
    void* z;
    RoleMap xb, xm, xk;
    RoleMap yb, yn, yk;
    RoleMap zb, zm, zn;
    uint32_t nb, M, N, K;
    int32_t op, agg;
    float alpha;
    int32_t in_bf16, out_bf16;
    int32_t x_kcontig, x_mcontig, y_ncontig, y_kcontig;
    // loader of each operand: 0 generic gather, 1 float4 along K, 2 float4 along M (X) / N (Y)
    int32_t x_mode, y_mode;
    // output: every 4-aligned group of 4 consecutive N indices is contiguous and 4-aligned
    int32_t z_vec4;
    // contracted composite made of one label (div 1): offset = (k / sub) * ks + (k % sub) * ls
    int32_t xk_simple, yk_simple;
    FastDiv xk_sub, yk_sub;
    int64_t xk_ks, xk_ls, yk_ks, yk_ls;
    // logsumexp factored form: the operands are exp(x - rowmax) and exp(y - colmax)
    // (fp32 scratch), and the epilogue adds rowmax + colmax + log(sum).
    const float* rowmax;  // [nb * M] or null
    const float* colmax;  // [nb * N] or null
    const void* x_raw;    // original operands for the underflow fallback
    const void* y_raw;
    // squared distance by expansion: the epilogue forms xn + yn - 2*sum
    const float* xnorm;   // [nb * M] or null
    const float* ynorm;   // [nb * N] or null
    // Guard of the expansion: where xn + yn - 2*sum < sq_tau * (xn + yn) the subtraction has
    // cancelled too far for the fp32 bar, and the CTA records its tile in tile_mark (one word
    // per 128 x 128 output tile, in launch order: 1 marked, 0 not; every CTA writes its own
    // word), and a CTA that marked writes gate_tag to the word after the last tile's.  A launch
    // with tile_gate set returns at once unless that word holds gate_tag, and otherwise
    // computes only the tiles whose word is nonzero (the direct-form fix-up pass).
    float sq_tau;
    uint32_t* tile_mark;
    const uint32_t* tile_gate;
    uint32_t gate_tag;
    // the underflow fix-up returns at once when this count (written by the producer of the
    // marks) is zero; null: scan every output
    const int* mark_count;
    // 1 when z is device memory (the bulk-copy epilogue writes only there; pinned host memory
    // the device can address gets plain stores)
    int32_t z_device;
    // elements of x (and x_raw), y (and y_raw) and z: the check build's bounds
    uint64_t x_elems, y_elems, z_elems;
};

// Per-operand row-max / exp-shift preparation of the factored logsumexp.
struct LsePrepParams {
    const void* src;      // operand (fp32 or bf16)
    float* dst;           // exp(v - max) in the same layout as src (fp32)
    float* rmax;          // [nb * R]
    RoleMap b, r, k;      // batch, row (M or N) and contracted maps of this operand
    uint32_t nb, R, K;
    int32_t in_bf16;
    int32_t mode;         // 0: row max, and dst = exp(v - max) unless dst is null;
                          // 1: sum of squares (for sqdiff expansion)
    // contracted composite made of one label (set by the launcher)
    int32_t k_simple;
    FastDiv k_sub;
    int64_t k_ks, k_ls;
    uint64_t src_elems;   // elements of src (and dst): the check build's bound
};

// One fp32 operand of a sum-of-products split for three BF16 products (split=bf16x3):
// v = src (or exp(src - shift[row]) when shift is set) becomes hi = bf16(v), lo = bf16(v - hi),
// written dense, one row of pitch K3p >= 3K per row index r (M for X, N for Y) of batch b:
// dst[(b Rp + r) K3p + s K + k] = hi, hi, lo for X (is_y = 0) and hi, lo, hi for Y, s = 0, 1, 2,
// and zeros in [3K, K3p); rows R .. Rp - 1 are left as they are (they feed only outputs that
// are not stored).  hi.hi + hi.lo + lo.hi then runs as one GEMM over the tripled index.
// Row statistics of one fp32 operand for split=bf16x3: per row r of batch b the maximum
// (mode 0) or the sum of squares (mode 1) over the contracted index.  Phase 1: CTAs over 32 rows
// x one of kc chunks of the contracted range write partials[c][b R + r]; phase 2 combines the kc
// partials of each row in chunk order into out (deterministic).
struct Split3StatsParams {
    const float* src;
    float* partials;      // [kc][nb * R]
    float* out;           // [nb * R]
    RoleMap b, r, k;
    uint32_t nb, R, K, kc;
    int32_t mode;
    int32_t k_fast;       // set by the launcher
    uint64_t src_elems;   // the check build's bound
};
uint32_t split3_stats_chunks(uint64_t rows, uint64_t K);  // kc for nb * R rows

struct Split3Params {
    const float* src;
    __nv_bfloat16* dst;
    const float* shift;   // [nb * R] or null
    RoleMap b, r, k;      // batch, row (M or N) and contracted maps of the operand
    uint32_t nb, R, K;
    uint32_t Rp, K3p;     // padded row count and row pitch of dst
    int32_t is_y;
    int32_t k_fast;       // set by the launcher: the innermost contracted label is contiguous
    int32_t k_dense;      // set by the launcher: one unsplit contracted label (offset k * k_ls)
    int64_t k_ls;
    uint64_t src_elems;   // the check build's bound on src (dst: nb * Rp * K3p)
};

// Unary aggregation over the contracted labels (row reduction).
struct RowReduceParams {
    const void* x;
    void* z;
    RoleMap xr, xk;       // X: output-row composite (all Z labels), contracted composite
    RoleMap zr;           // Z: output-row composite
    uint32_t R, K;
    int32_t agg;
    float alpha;
    int32_t in_bf16, out_bf16;
    int32_t k_affine;     // the contracted composite is contiguous (stride 1) over all of [0, K)
    uint64_t x_elems, z_elems;  // the check build's bounds
};

// Join with aggregation "none": every output element is op(x, y); operands may broadcast.
// The kernel walks Z in its physical (blocked) order, one run of I contiguous
// elements (the innermost label's block-local extent) at a time.  Every label
// of X and Y is a label of Z with the same partition count, so an operand's
// offset is sum_i key_i * ks[i] + loc_i * ls[i] over Z's index positions i
// (ks = ls = 0 where the operand lacks that label).
struct ElementwiseParams {
    const void* x;
    const void* y;      // null for a unary (identity) join
    void* z;
    int32_t rank;       // rank of Z
    int32_t op;
    float alpha;
    int32_t in_bf16, out_bf16;
    uint32_t I;         // run length (elements)
    uint64_t n_runs;
    FastDiv sub_total;  // elements per Z block
    FastDiv grid[TRA_MAX_RANK], sub[TRA_MAX_RANK];
    int64_t x_ks[TRA_MAX_RANK], x_ls[TRA_MAX_RANK];
    int64_t y_ks[TRA_MAX_RANK], y_ls[TRA_MAX_RANK];
    // flat fast path (fp32 X laid out exactly as Z): 0 off; 1 Y absent or laid out as Z;
    // 2 Y laid out as Z without its innermost label (unsplit, extent y_div)
    int32_t flat;
    uint32_t y_div;
    uint64_t total;
    uint64_t x_elems, y_elems;  // the check build's bounds (z: total)
};

// Repartition (permute copy) between two relation layouts of one tensor: walks the
// destination in physical order, vec_elems elements per thread; a vector never
// leaves a run that is contiguous in both layouts.
struct RepartParams {
    const void* src;
    void* dst;
    int32_t rank;
    int32_t elem_bytes;
    int32_t vec_elems;
    int32_t vec_bytes;
    int32_t group;  // vectors per decoded segment (1, 2 or 4): a power of two dividing the common run
    uint64_t n_vec;
    FastDiv dst_sub_total;
    FastDiv dst_grid[TRA_MAX_RANK], dst_sub[TRA_MAX_RANK], src_sub[TRA_MAX_RANK];
    int64_t src_key_stride[TRA_MAX_RANK], src_loc_stride[TRA_MAX_RANK];
};

// Ordered combine of per-join-tuple partials (literal mode).
struct CombineParams {
    const float* partials;  // [n_groups][n_agg][z_sub]
    void* z;                // Z relation layout: group g's block at g * z_sub
    uint64_t n_groups, n_agg, z_sub;
    int32_t agg;
    float alpha;
    int32_t out_bf16;
};

cudaError_t launch_semiring(const SemiringParams& p, cudaStream_t s);
cudaError_t launch_semiring_simple(const SemiringParams& p, cudaStream_t s);
cudaError_t launch_lse_prep(const LsePrepParams& p, cudaStream_t s);
// Outputs of the factored logsumexp marked NaN (their exp-shifted sum underflowed) are
// recomputed straight from p.x_raw / p.y_raw through p's role maps.
cudaError_t launch_lse_fixup(const SemiringParams& p, cudaStream_t s);
// Squared distance in the direct form sum_k (x - y)^2 (fp32 operands) over the 128 x 128 output
// tiles whose word in p.tile_gate is nonzero, when the word after them holds p.gate_tag; the
// other tiles are left as they are.
cudaError_t launch_sqdist_fixup(const SemiringParams& p, cudaStream_t s);
// Guard threshold of the squared-distance expansion for a contracted extent K (see plan.cpp).
float sqdist_guard_tau(uint64_t K, double c);
// 128 x 128 output tiles of the CUDA-core kernels (the fix-up pass's grid)
inline uint64_t semiring_tiles(uint64_t nb, uint64_t M, uint64_t N) {
    return nb * ((M + 127) / 128) * ((N + 127) / 128);
}
// Guard words of the squared-distance expansion: one per tile, then the launch's tag word.
inline uint64_t sqdist_guard_bytes(uint64_t nb, uint64_t M, uint64_t N) {
    return (semiring_tiles(nb, M, N) + 1) * 4;
}
// A fresh nonzero tag per launch of the expanded squared distance (the tag word then tells
// the fix-up pass whether this launch marked anything).
uint32_t next_gate_tag();
cudaError_t launch_split3(const Split3Params& p, cudaStream_t s);
cudaError_t launch_split3_stats(const Split3StatsParams& p, cudaStream_t s);
cudaError_t launch_row_reduce(const RowReduceParams& p, cudaStream_t s);
cudaError_t launch_elementwise(const ElementwiseParams& p, cudaStream_t s);
cudaError_t launch_repartition(const RepartParams& p, cudaStream_t s);
// TMA path of the repartition (k_repart.cu): cudaErrorNotSupported when the layouts do not fit
// it (more than 4 dimensions of extent > 1, rows not on 16-byte boundaries, boxes under 4 KB);
// the caller then runs launch_repartition.
cudaError_t launch_repartition_tma(int rank, const int64_t* shape, const int32_t* src_d, const int32_t* dst_d,
                                   int elem_bytes, const void* src, void* dst, cudaStream_t s);
cudaError_t read_and_clear_rp_status(int* value, cudaStream_t s);
cudaError_t launch_combine(const CombineParams& p, cudaStream_t s);
cudaError_t launch_fill(void* z, uint64_t n, float v, bool bf16, cudaStream_t s);

// Device status word written by bounded waits that give up (TRA_ERR_TIMEOUT).
cudaError_t read_and_clear_status(int* value, cudaStream_t s);
cudaError_t read_and_clear_attn_status(int* value, cudaStream_t s);
cudaError_t launch_wait_timeout_probe(uint64_t timeout_ns, cudaStream_t s);

}  // namespace tra
