// Host planner of libtra.so: turns (spec, bounds, d) into a TRA plan.
// "EinDecomp ... tensor relational algebra": section 2.2 (partition vector,
// key -> index range, EinSum -> TRA lowering) and sections 3.1 / 3.2 (task
// triple, cost model, task count).
#pragma once

#include <string>
#include <vector>

#include "tra_internal.h"

namespace tra {

struct Operand {
    int rank = 0;
    int label[TRA_MAX_RANK] = {};
    int32_t d[TRA_MAX_RANK] = {};
    int64_t shape[TRA_MAX_RANK] = {};
    int64_t sub = 1;    // elements per sub-tensor
    int64_t nkeys = 1;  // number of sub-tensors
    int64_t total = 1;  // elements
    int64_t key_stride[TRA_MAX_RANK] = {};
    int64_t loc_stride[TRA_MAX_RANK] = {};
    int pos_of(int l) const {
        for (int i = 0; i < rank; ++i)
            if (label[i] == l) return i;
        return -1;
    }
};

struct TcPlan;  // tensor-core launch description (k_tc.cu)

struct Plan {
    std::string spec;
    int op = kMul, agg = kSum;
    double alpha = 1.0;
    int in_bf16 = 0, out_bf16 = 0;
    int literal = 0;
    int sqdiff_expand = 0;
    int tc_pair = -1;  // tensor-core tile: 1 CTA pair (256 x 256), 0 single CTA, -1 pair when shapes allow
    int tc_n = 0;      // width of a pair tile: 256, 128, or 0 (256 where the columns allow)
    int tc_store = -1; // tensor-core epilogue: 1 TMA stores, 0 warp stores, -1 TMA where the output map fits
    int ksplit = 1;    // tensor-core path: 1 split the K loop of the last wave's tiles over idle workers, 0 never
    int split3 = 0;    // split=bf16x3: squared distance / logsumexp rewritten onto BF16 tensor cores
    Plan* inner = nullptr;  // split3: the GEMM plan over the split operands (owned)
    int split3_direct = 0;  // split3: inner's output layout is this plan's (no override, TMA stores)
    // vector-load eligibility of the semiring kernel's operands (host scan, see scan_vec_flags)
    int vec_flags[5] = {0, 0, 0, 0, 0};  // X along K, X along M, Y along N, Y along K, Z along N
    bool unary = false;

    int n_labels = 0;
    char name[TRA_MAX_LABELS] = {};
    int64_t B[TRA_MAX_LABELS] = {};
    int32_t D[TRA_MAX_LABELS] = {};
    int role[TRA_MAX_LABELS] = {};
    std::vector<int> contracted;  // first-appearance order

    Operand X, Y, Z;
    std::vector<int> comp[4];  // labels per role, composite order (innermost first)
    uint64_t ext[4] = {1, 1, 1, 1};

    uint64_t n_tasks = 0, n_groups = 0, n_agg = 0;
    uint64_t cost_join = 0, cost_agg = 0;
    uint64_t msg_join = 0, msg_agg = 0, mem_elems = 0;
    int kernel = 0;
    uint64_t ws_bytes = 0;

    TcPlan* tc = nullptr;
    ~Plan();
};

// Error reporting (thread-local message, returned code).
int fail(int code, const char* fmt, ...);
void clear_error();
const char* last_error();

int build_plan(const char* spec, const int64_t* bounds, int n_bounds, const int32_t* d, int n_d, Plan* p);
void layout_operand(Operand& t, const Plan& p);
RoleMap role_map(const Plan& p, const Operand& t, int role);
void fill_keys(const Plan& p, int32_t* out);

// Tensor-core planning (k_tc.cu): returns true and sets p->tc when the BF16
// sum-of-products can run on tcgen05 with TMA tiles that stay inside blocks.
bool tc_plan(Plan* p);
void tc_free(TcPlan* t);
bool tc_tma_store(const TcPlan* t);  // the plan's epilogue stores through an output tensor map
// Optional epilogue of tc_execute for the rewritten non-sum semirings (split=bf16x3): rank-one
// terms per output row / column, and the output addressed through another plan's Z role maps
// (the caller's relation layout) instead of the GEMM plan's own.
struct TcExtra {
    int epi = 0;  // 0 plain, 1 squared-distance expansion, 2 factored logsumexp
    const float* row_term = nullptr;
    const float* col_term = nullptr;
    float alpha = 1.f;
    bool z_override = false;
    RoleMap zb, zm, zn;
    uint32_t M = 0, N = 0;  // with z_override: the rows / columns stored (the product may be padded)
    int* mark_count = nullptr;  // epi 2: count of outputs marked for the underflow fix-up
    // epi 1: guard of the expansion -- where r + c - 2 acc < sq_tau (r + c), the word of the
    // output's 128 x 128 tile (b, m / 128, n / 128) in fix_flags (zeroed by the caller) is set
    float sq_tau = 0.f;
    uint32_t* fix_flags = nullptr;
    uint32_t fix_tiles_m = 0, fix_tiles_n = 0;
    uint64_t fix_tag_index = 0;  // fix_flags[fix_tag_index] is set to 1 when any tile is marked
    uint64_t z_elems = 0;        // with z_override: elements of the output buffer
};
// ws: the plan's workspace (tc->ws_part + tc->ws_flags bytes) for the K split of the last
// wave's tiles; without it, or with ex, every tile runs on one worker.
int tc_execute(const Plan& p, const void* x, const void* y, void* z, cudaStream_t s, const TcExtra* ex = nullptr,
               void* ws = nullptr);

uint64_t align256(uint64_t v);
// constants c of the squared-distance guard (sqdist_guard_tau): fp32 expansion, split=bf16x3
constexpr double kSqGuardFp32 = 3.0, kSqGuardSplit3 = 4.5;
inline uint64_t split3_pad(uint64_t v, uint64_t q) { return (v + q - 1) / q * q; }
uint64_t repartition_cost_elems(int rank, const int64_t* shape, const int32_t* src_d, const int32_t* dst_d);
uint64_t repartition_messages(int rank, const int64_t* shape, const int32_t* src_d, const int32_t* dst_d);

// Exhaustive host check of the semiring kernel's 4-wide loads: an operand may load
// 4 consecutive indices of a role at once only if every 4-aligned group of that role
// maps to 4 contiguous elements at a multiple of 4, and every other offset that is
// added to it (the other role, the batch) is a multiple of 4.  flags: X along K,
// X along M, Y along N, Y along K, Z along N (vector stores of the output).
void scan_vec_flags(const RoleMap& xb, const RoleMap& xm, const RoleMap& xk, const RoleMap& yb, const RoleMap& yn,
                    const RoleMap& yk, const RoleMap& zb, const RoleMap& zm, const RoleMap& zn, uint32_t nb,
                    uint32_t M, uint32_t N, uint32_t K, int flags[5]);

}  // namespace tra
