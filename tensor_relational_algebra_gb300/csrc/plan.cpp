// Host planner: spec parsing, validation, key space, join enumeration, cost
// terms and kernel choice.  Touches no device.
//
// "EinDecomp ... tensor relational algebra":
//  * section 2.1 -- extended EinSum: labels on the right-hand side that are not in
//    the output are contracted; aggregation sum/max/min/logsumexp; any binary op.
//  * section 2.2 -- tensor [B1..] under d=[D1..] (D_i | B_i) is a relation of
//    prod D_i sub-tensors of shape [B_i/D_i]; matmul's d is [d_i, d_jX, d_jY, d_k]
//    with d_jX = d_jY; join pairs key-matched sub-tensors; aggregation groups
//    by the output key.
//  * section 3.1 -- cost model: join P*(|X_sub|+|Y_sub|), aggregation
//    (P/n_agg)*(n_agg-1)*|Z_sub|, P read here as the number of join tuples.
//  * section 3.2 -- the number of tasks is the number of tuples the join produces.
#include "plan.h"

#include <cctype>
#include <cerrno>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <algorithm>
#include <atomic>
#include <cstring>

namespace tra {

namespace {
thread_local std::string g_err;
}

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}
void clear_error() { g_err.clear(); }
const char* last_error() { return g_err.c_str(); }

uint64_t align256(uint64_t v) { return (v + 255) & ~uint64_t(255); }

// Guard of the squared-distance expansion |x|^2 + |y|^2 - 2 x.y (section 2.1's squared
// distance, D = sum_k (x - y)^2 >= 0, zero for coincident points).  With S = |x|^2 + |y|^2 the
// rounding error of the expansion in fp32 grows like c * sqrt(K) * u * S (u = 2^-24), whatever
// D is, so its relative error is unbounded as D -> 0.  An output whose computed value falls
// below tau * S, tau = c * sqrt(K) * u / 1e-5, is recomputed in the direct form; above it the
// expansion's error stays under 1e-5 * D.  c: 3 for the fp32 expansion (largest error seen in
// an fp32 simulation at K = 256 was 1.4 sqrt(K) u S, so a factor 2 of margin), 4.5 for
// split=bf16x3, whose dropped lo.lo products add about three times that (margin 1: that path's
// own bar is looser, see include/tra.h).  Capped at 2 (D <= 2 S: every output then qualifies).
uint32_t next_gate_tag() {
    static std::atomic<uint32_t> n{0x5eed0000u};
    uint32_t t = n.fetch_add(1);
    return t ? t : n.fetch_add(1);
}

float sqdist_guard_tau(uint64_t K, double c) {
    const double t = c * std::sqrt((double)K) * 0x1p-24 / 1e-5;
    return (float)(t < 2.0 ? t : 2.0);
}

// Elements whose owning block changes between two partitions of one tensor, blocks being
// owned by their row-major linear key id L: |T| - sum_L |block_L(src) n block_L(dst)|.
// Arguments already validated (every d divides its extent).
uint64_t repartition_cost_elems(int rank, const int64_t* shape, const int32_t* src_d, const int32_t* dst_d) {
    uint64_t total = 1, ns = 1, nd = 1;
    for (int i = 0; i < rank; ++i) {
        total *= (uint64_t)shape[i];
        ns *= (uint64_t)src_d[i];
        nd *= (uint64_t)dst_d[i];
    }
    uint64_t stay = 0;
    const uint64_t n = ns < nd ? ns : nd;
    for (uint64_t L = 0; L < n; ++L) {
        uint64_t ls = L, ld = L, inter = 1;
        for (int i = rank - 1; i >= 0 && inter; --i) {
            const uint64_t ks = ls % (uint64_t)src_d[i], kd = ld % (uint64_t)dst_d[i];
            ls /= (uint64_t)src_d[i];
            ld /= (uint64_t)dst_d[i];
            const uint64_t bs = (uint64_t)shape[i] / src_d[i], bd = (uint64_t)shape[i] / dst_d[i];
            const uint64_t lo = ks * bs > kd * bd ? ks * bs : kd * bd;
            const uint64_t hi = (ks + 1) * bs < (kd + 1) * bd ? (ks + 1) * bs : (kd + 1) * bd;
            inter *= hi > lo ? hi - lo : 0;
        }
        stay += inter;
    }
    return total - stay;
}

uint64_t repartition_messages(int rank, const int64_t* shape, const int32_t* src_d, const int32_t* dst_d) {
    // overlapping (source block, destination block) pairs: per dimension the union of the two
    // sets of block boundaries cuts [0, B) into Ds + Dd - gcd(Ds, Dd) segments, one per pair;
    // minus the pairs whose two blocks have the same linear id (nothing moves between them)
    uint64_t pairs = 1, ns = 1, nd = 1;
    for (int i = 0; i < rank; ++i) {
        uint64_t a = (uint64_t)src_d[i], b = (uint64_t)dst_d[i];
        while (b) {
            const uint64_t t = a % b;
            a = b;
            b = t;
        }
        pairs *= (uint64_t)src_d[i] + (uint64_t)dst_d[i] - a;
        ns *= (uint64_t)src_d[i];
        nd *= (uint64_t)dst_d[i];
    }
    uint64_t same = 0;
    const uint64_t n = ns < nd ? ns : nd;
    for (uint64_t L = 0; L < n; ++L) {
        uint64_t ls = L, ld = L;
        bool meet = true;
        for (int i = rank - 1; i >= 0 && meet; --i) {
            const uint64_t ks = ls % (uint64_t)src_d[i], kd = ld % (uint64_t)dst_d[i];
            ls /= (uint64_t)src_d[i];
            ld /= (uint64_t)dst_d[i];
            const uint64_t bs = (uint64_t)shape[i] / src_d[i], bd = (uint64_t)shape[i] / dst_d[i];
            meet = ks * bs < (kd + 1) * bd && kd * bd < (ks + 1) * bs;
        }
        same += meet;
    }
    return pairs - same;
}

Plan::~Plan() {
    if (tc) tc_free(tc);
    delete inner;
}

namespace {

std::vector<std::string> split(const std::string& s, char c) {
    std::vector<std::string> out;
    size_t start = 0;
    for (;;) {
        size_t pos = s.find(c, start);
        out.push_back(s.substr(start, pos == std::string::npos ? std::string::npos : pos - start));
        if (pos == std::string::npos) break;
        start = pos + 1;
    }
    return out;
}

int parse_op(const std::string& s) {
    if (s == "mul") return kMul;
    if (s == "add") return kAdd;
    if (s == "sqdiff") return kSqdiff;
    if (s == "sub") return kSub;
    if (s == "expsub") return kExpsub;
    return -1;
}

int parse_agg(const std::string& s) {
    if (s == "sum") return kSum;
    if (s == "max") return kMax;
    if (s == "min") return kMin;
    if (s == "lse") return kLse;
    if (s == "none") return kNone;
    return -1;
}

}  // namespace

void layout_operand(Operand& t, const Plan& p) {
    t.sub = 1;
    t.nkeys = 1;
    for (int i = 0; i < t.rank; ++i) {
        const int l = t.label[i];
        t.d[i] = p.D[l];
        t.shape[i] = p.B[l];
        t.sub *= p.B[l] / p.D[l];
        t.nkeys *= p.D[l];
    }
    t.total = t.sub * t.nkeys;
    int64_t ls = 1, ks = t.sub;
    for (int i = t.rank - 1; i >= 0; --i) {
        const int l = t.label[i];
        t.loc_stride[i] = ls;
        t.key_stride[i] = ks;
        ls *= p.B[l] / p.D[l];
        ks *= p.D[l];
    }
}

RoleMap role_map(const Plan& p, const Operand& t, int role) {
    RoleMap m;
    memset(&m, 0, sizeof(m));
    uint64_t div = 1;
    for (int l : p.comp[role]) {
        const int i = t.pos_of(l);
        if (i >= 0) {
            Term& tm = m.t[m.n++];
            tm.div = (uint32_t)div;
            tm.ext = (uint32_t)p.B[l];
            tm.sub = (uint32_t)(p.B[l] / p.D[l]);
            tm.key_stride = t.key_stride[i];
            tm.loc_stride = t.loc_stride[i];
        }
        div *= (uint64_t)p.B[l];
    }
    return m;
}

int build_plan(const char* spec, const int64_t* bounds, int n_bounds, const int32_t* d, int n_d, Plan* p) {
    if (!spec || !p) return fail(TRA_ERR_ARG, "null spec or plan");
    p->spec = spec;
    p->sqdiff_expand = -1;  // not given: expansion for fp32 inputs, direct for bf16
    std::vector<std::string> parts = split(spec, ':');
    const std::string eq = parts[0];
    const size_t arrow = eq.find("->");
    if (arrow == std::string::npos) return fail(TRA_ERR_PARSE, "spec '%s': missing '->'", spec);
    const std::string lhs = eq.substr(0, arrow), rhs = eq.substr(arrow + 2);
    std::vector<std::string> ins = split(lhs, ',');
    if (ins.size() < 1 || ins.size() > 2) return fail(TRA_ERR_PARSE, "spec '%s': one or two operands expected", spec);
    p->unary = ins.size() == 1;
    if (parts.size() < 3) return fail(TRA_ERR_PARSE, "spec '%s': expected '<eq>:<op>:<agg>'", spec);
    if (p->unary) {
        if (!parts[1].empty()) return fail(TRA_ERR_PARSE, "spec '%s': a unary EinSum takes no op", spec);
        p->op = kId;
    } else {
        p->op = parse_op(parts[1]);
        if (p->op < 0) return fail(TRA_ERR_PARSE, "spec '%s': unknown op '%s'", spec, parts[1].c_str());
    }
    p->agg = parse_agg(parts[2]);
    if (p->agg < 0) return fail(TRA_ERR_PARSE, "spec '%s': unknown aggregation '%s'", spec, parts[2].c_str());
    for (size_t i = 3; i < parts.size(); ++i) {
        const std::string& o = parts[i];
        const size_t eqp = o.find('=');
        if (eqp == std::string::npos) return fail(TRA_ERR_PARSE, "spec '%s': option '%s' needs '='", spec, o.c_str());
        const std::string k = o.substr(0, eqp), v = o.substr(eqp + 1);
        if (k == "in" && (v == "f32" || v == "bf16")) p->in_bf16 = v == "bf16";
        else if (k == "out" && (v == "f32" || v == "bf16")) p->out_bf16 = v == "bf16";
        else if (k == "mode" && (v == "fused" || v == "literal")) p->literal = v == "literal";
        else if (k == "sqdiff" && (v == "direct" || v == "expand")) p->sqdiff_expand = v == "expand" ? 1 : 0;
        else if (k == "tc" && (v == "pair" || v == "single")) p->tc_pair = v == "pair" ? 1 : 0;
        else if (k == "tc_n" && (v == "256" || v == "128")) p->tc_n = v == "256" ? 256 : 128;
        else if (k == "tc_store" && (v == "tma" || v == "lsu")) p->tc_store = v == "tma" ? 1 : 0;
        else if (k == "ksplit" && (v == "auto" || v == "off")) p->ksplit = v == "auto" ? 1 : 0;
        else if (k == "split" && (v == "bf16x3" || v == "none")) p->split3 = v == "bf16x3";
        else if (k == "alpha") {
            char* end = nullptr;
            errno = 0;
            p->alpha = strtod(v.c_str(), &end);
            if (errno || !end || *end || v.empty() || !std::isfinite(p->alpha))
                return fail(TRA_ERR_PARSE, "spec '%s': bad alpha '%s'", spec, v.c_str());
        } else {
            return fail(TRA_ERR_PARSE, "spec '%s': unknown option '%s'", spec, o.c_str());
        }
    }

    // labels, first appearance X then Y
    std::string order;
    Operand* ops[2] = {&p->X, &p->Y};
    for (size_t a = 0; a < ins.size(); ++a) {
        const std::string& s = ins[a];
        if (s.empty() || (int)s.size() > TRA_MAX_RANK)
            return fail(TRA_ERR_RANK, "operand '%s': rank must be 1..%d", s.c_str(), TRA_MAX_RANK);
        ops[a]->rank = (int)s.size();
        for (size_t i = 0; i < s.size(); ++i) {
            const char c = s[i];
            if (!std::isalpha((unsigned char)c)) return fail(TRA_ERR_PARSE, "label '%c' is not a letter", c);
            if (s.find(c) != i) return fail(TRA_ERR_PARSE, "label '%c' repeats inside operand '%s'", c, s.c_str());
            size_t pos = order.find(c);
            if (pos == std::string::npos) {
                if ((int)order.size() >= TRA_MAX_LABELS) return fail(TRA_ERR_RANK, "more than %d labels", TRA_MAX_LABELS);
                order.push_back(c);
                pos = order.size() - 1;
            }
            ops[a]->label[i] = (int)pos;
        }
    }
    if ((int)rhs.size() > TRA_MAX_RANK) return fail(TRA_ERR_RANK, "output rank above %d", TRA_MAX_RANK);
    p->Z.rank = (int)rhs.size();
    for (size_t i = 0; i < rhs.size(); ++i) {
        const char c = rhs[i];
        const size_t pos = order.find(c);
        if (pos == std::string::npos) return fail(TRA_ERR_PARSE, "output label '%c' is in no operand", c);
        if (rhs.find(c) != i) return fail(TRA_ERR_PARSE, "output label '%c' repeats", c);
        p->Z.label[i] = (int)pos;
    }
    p->n_labels = (int)order.size();
    for (int l = 0; l < p->n_labels; ++l) p->name[l] = order[l];

    if (!bounds || n_bounds != p->n_labels)
        return fail(TRA_ERR_RANK, "%d bounds given, %d labels in '%s'", n_bounds, p->n_labels, spec);
    const int nd_want = p->X.rank + (p->unary ? 0 : p->Y.rank);
    if (!d || n_d != nd_want) return fail(TRA_ERR_RANK, "%d partition counts given, %d index positions", n_d, nd_want);
    for (int l = 0; l < p->n_labels; ++l) {
        if (bounds[l] < 0 || bounds[l] > 0x7fffffffLL)
            return fail(TRA_ERR_ARG, "bound of '%c' out of range", p->name[l]);
        p->B[l] = bounds[l];
        p->D[l] = 0;
    }
    int di = 0;
    for (size_t a = 0; a < ins.size(); ++a) {
        for (int i = 0; i < ops[a]->rank; ++i, ++di) {
            const int l = ops[a]->label[i];
            if (d[di] < 1) return fail(TRA_ERR_ARG, "partition count %d < 1", d[di]);
            if (p->B[l] % d[di])
                return fail(TRA_ERR_DIVISIBILITY, "D=%d does not divide B=%lld for label '%c'", d[di],
                            (long long)p->B[l], p->name[l]);
            if (p->D[l] && p->D[l] != d[di])
                return fail(TRA_ERR_SHARED_LABEL_D, "label '%c' partitioned %d ways in X and %d in Y", p->name[l],
                            p->D[l], d[di]);
            p->D[l] = d[di];
        }
    }


    // roles
    bool inx[TRA_MAX_LABELS] = {}, iny[TRA_MAX_LABELS] = {}, inz[TRA_MAX_LABELS] = {};
    for (int i = 0; i < p->X.rank; ++i) inx[p->X.label[i]] = true;
    if (!p->unary)
        for (int i = 0; i < p->Y.rank; ++i) iny[p->Y.label[i]] = true;
    for (int i = 0; i < p->Z.rank; ++i) inz[p->Z.label[i]] = true;
    for (int l = 0; l < p->n_labels; ++l) {
        if (!inz[l]) p->role[l] = kK;
        else if (inx[l] && iny[l]) p->role[l] = kBatch;
        else if (inx[l]) p->role[l] = kM;
        else p->role[l] = kN;
        if (!inz[l]) p->contracted.push_back(l);
    }
    if (p->agg == kNone && !p->contracted.empty())
        return fail(TRA_ERR_PARSE, "aggregation 'none' with contracted label '%c'", p->name[p->contracted[0]]);
    if (p->agg != kNone && p->contracted.empty())
        return fail(TRA_ERR_PARSE, "no contracted label: use aggregation 'none'");

    layout_operand(p->X, *p);
    if (!p->unary) layout_operand(p->Y, *p);
    layout_operand(p->Z, *p);
    const int64_t lim = 0x7fffffffLL;
    if (p->X.total > lim || p->Y.total > lim || p->Z.total > lim)
        return fail(TRA_ERR_UNSUPPORTED, "tensors above 2^31-1 elements are not supported");

    // composite order (innermost first): M by X's memory order, N by Y's, K by X's
    // then Y-only contracted labels by Y's, batch by Z's
    for (int r = 0; r < 4; ++r) p->comp[r].clear();
    for (int i = p->Z.rank - 1; i >= 0; --i)
        if (p->role[p->Z.label[i]] == kBatch) p->comp[kBatch].push_back(p->Z.label[i]);
    for (int i = p->X.rank - 1; i >= 0; --i) {
        const int l = p->X.label[i];
        if (p->role[l] == kM) p->comp[kM].push_back(l);
        if (p->role[l] == kK) p->comp[kK].push_back(l);
    }
    if (!p->unary)
        for (int i = p->Y.rank - 1; i >= 0; --i) {
            const int l = p->Y.label[i];
            if (p->role[l] == kN) p->comp[kN].push_back(l);
            if (p->role[l] == kK && !inx[l]) p->comp[kK].push_back(l);
        }
    for (int r = 0; r < 4; ++r) {
        uint64_t e = 1;
        for (int l : p->comp[r]) e *= (uint64_t)p->B[l];
        if (e > 0x7fffffffull) return fail(TRA_ERR_UNSUPPORTED, "a composite extent exceeds 2^31-1");
        p->ext[r] = e;
    }

    // task count and cost terms
    p->n_tasks = 1;
    p->n_groups = 1;
    for (int l = 0; l < p->n_labels; ++l) {
        p->n_tasks *= (uint64_t)p->D[l];
        if (inz[l]) p->n_groups *= (uint64_t)p->D[l];
    }
    p->n_agg = p->n_tasks / p->n_groups;
    const uint64_t xs = (uint64_t)p->X.sub, ys = p->unary ? 0 : (uint64_t)p->Y.sub, zs = (uint64_t)p->Z.sub;
    p->cost_join = p->n_tasks * (xs + ys);
    p->cost_agg = (p->n_tasks / p->n_agg) * (p->n_agg - 1) * zs;
    // cost-model variants: one message per sub-tensor moved, and the node's memory (its output
    // plus the join's partial results when they are aggregated)
    p->msg_join = p->n_tasks * (p->unary ? 1u : 2u);
    p->msg_agg = (p->n_tasks / p->n_agg) * (p->n_agg - 1);
    p->mem_elems = (uint64_t)p->Z.total + (p->n_agg > 1 ? p->n_tasks * zs : 0);

    // kernel choice and workspace
    p->ws_bytes = 0;
    // squared distance: the expansion by default for fp32 inputs while its guard can pass
    // typical outputs (threshold below 1), the direct form otherwise
    if (p->sqdiff_expand < 0) p->sqdiff_expand = !p->in_bf16 && sqdist_guard_tau(p->ext[kK], kSqGuardFp32) < 1.f;
    for (int l = 0; l < p->n_labels; ++l)
        if (p->B[l] == 0) {
            // an empty EinSum: no output element, or only empty aggregations (agg's identity)
            p->kernel = p->Z.total == 0 ? TRA_KERNEL_EMPTY : TRA_KERNEL_FILL;
            return TRA_OK;
        }
    if (p->literal && p->agg != kNone) {
        p->kernel = TRA_KERNEL_LITERAL;
        p->ws_bytes = align256(p->n_tasks * zs * sizeof(float));
    } else if (p->agg == kNone) {
        p->kernel = TRA_KERNEL_ELEMENTWISE;
    } else if (p->unary) {
        p->kernel = TRA_KERNEL_ROW_REDUCE;
    } else if (p->split3) {
        // Squared distance sum_k (x - y)^2 = |x|^2 + |y|^2 - 2 x.y, and the factored logsumexp
        // lse_k (x + y) = mx + my + log sum_k e^(x - mx) e^(y - my): the sum of products runs as
        // one BF16 GEMM over K' = 3K with each fp32 operand split into hi + lo bf16 terms
        // (hi.hi + hi.lo + lo.hi); the rank-one terms go into its epilogue.
        if (p->in_bf16) return fail(TRA_ERR_UNSUPPORTED, "split=bf16x3 takes fp32 inputs");
        if (!((p->op == kSqdiff && p->agg == kSum) || (p->op == kAdd && p->agg == kLse)))
            return fail(TRA_ERR_UNSUPPORTED, "split=bf16x3 applies to sqdiff:sum and add:lse");
        const uint64_t nb = p->ext[kBatch], M = p->ext[kM], N = p->ext[kN], K = p->ext[kK];
        if (3 * K + 64 > 0x7fffffffull) return fail(TRA_ERR_UNSUPPORTED, "split=bf16x3: 3K exceeds 2^31-1");
        // the GEMM's warp-store epilogue writes runs of 32 output columns: Z must be contiguous
        // along N in such runs (its last label is N's innermost, with a block extent that is a
        // multiple of 32)
        const int zl = p->Z.rank ? p->Z.label[p->Z.rank - 1] : -1;
        if (p->comp[kN].empty() || zl != p->comp[kN][0] || (p->B[zl] / p->D[zl]) % 32)
            return fail(TRA_ERR_UNSUPPORTED,
                        "split=bf16x3: the output's last label must be an N label with a block extent that is a multiple of 32");
        // the GEMM's tiles take M, K' and N in multiples of 128, 64 and 64: the split operands
        // are padded (rows past M / N are never stored; the K' padding is zero)
        const uint64_t Mp = split3_pad(M, 128), Np = split3_pad(N, 64), K3p = split3_pad(3 * K, 64);
        const std::string out_opt = p->out_bf16 ? ":out=bf16" : "";
        auto is_tc = [](const Plan* q) { return q->kernel == TRA_KERNEL_TC_BF16 || q->kernel == TRA_KERNEL_TC_BF16_PAIR; };
        // Direct form: one M and one N label, no padding.  The GEMM "mk,nk->mn" takes this plan's
        // partition of m and n; with k' unsplit, the split operands' row-major layout is their
        // relation layout, and the GEMM's output relation is this plan's Z, so its TMA-store
        // epilogue writes Z directly.
        if (nb == 1 && p->comp[kM].size() == 1 && p->comp[kN].size() == 1 && p->Z.rank == 2 && Mp == M && Np == N) {
            const std::string dspec = "mk,nk->mn:mul:sum:in=bf16:ksplit=off" + out_opt;
            const int64_t db[3] = {(int64_t)M, (int64_t)K3p, (int64_t)N};
            const int32_t dd[4] = {p->D[p->comp[kM][0]], 1, p->D[p->comp[kN][0]], 1};
            Plan* in = new Plan();
            if (build_plan(dspec.c_str(), db, 3, dd, 4, in) == TRA_OK && is_tc(in) && tc_tma_store(in->tc)) {
                p->inner = in;
                p->split3_direct = 1;
            } else {
                delete in;
                clear_error();
            }
        }
        // General form: dense operands, the output addressed through this plan's Z role maps.
        if (!p->inner) {
            std::string ispec = nb > 1 ? "bmk,bnk->bmn" : "mk,nk->mn";
            ispec += ":mul:sum:in=bf16:tc_store=lsu:ksplit=off" + out_opt;
            const int64_t ib[4] = {(int64_t)nb, (int64_t)Mp, (int64_t)K3p, (int64_t)Np};  // labels b, m, k, n
            const int32_t ones[6] = {1, 1, 1, 1, 1, 1};
            Plan* in = new Plan();
            const int rc = nb > 1 ? build_plan(ispec.c_str(), ib, 4, ones, 6, in) : build_plan(ispec.c_str(), ib + 1, 3, ones, 4, in);
            if (rc != TRA_OK || !is_tc(in)) {
                delete in;
                return fail(TRA_ERR_UNSUPPORTED, "split=bf16x3: no tensor-core tiling for the %llu x %llu x %llu product",
                            (unsigned long long)M, (unsigned long long)(3 * K), (unsigned long long)N);
            }
            p->inner = in;
        }
        p->kernel = TRA_KERNEL_TC_SPLIT3;
        const uint64_t parts = std::max<uint64_t>(split3_stats_chunks(nb * M, K) * nb * M, split3_stats_chunks(nb * N, K) * nb * N);
        // operands, row / column terms, the fix-up's mark count (256 bytes), the statistics' partials
        p->ws_bytes = align256(nb * Mp * K3p * 2) + align256(nb * Np * K3p * 2) + align256(nb * M * 4) +
                      align256(nb * N * 4) + 256 + align256(parts * 4);
        // squared distance: one word per 128 x 128 output tile marked by the expansion's guard
        if (p->op == kSqdiff) p->ws_bytes += align256(sqdist_guard_bytes(nb, M, N));
    } else if (p->op == kAdd && p->agg == kLse) {
        p->kernel = TRA_KERNEL_LSE_FACTORED;
        const uint64_t nb = p->ext[kBatch];
        p->ws_bytes = align256((uint64_t)p->X.total * 4) + align256((uint64_t)p->Y.total * 4) +
                      align256(nb * p->ext[kM] * 4) + align256(nb * p->ext[kN] * 4);
    } else if (p->op == kMul && p->agg == kSum && p->in_bf16 && tc_plan(p)) {
        // tc_plan chose TRA_KERNEL_TC_BF16 or TRA_KERNEL_TC_BF16_PAIR
    } else {
        if (p->tc_pair == 1 && p->op == kMul && p->agg == kSum && p->in_bf16)
            return fail(TRA_ERR_UNSUPPORTED, "tc=pair: no 256 x 256 tensor-core tiling for this plan");
        if (p->tc_store == 1 && p->op == kMul && p->agg == kSum && p->in_bf16)
            return fail(TRA_ERR_UNSUPPORTED, "tc_store=tma: no tensor-core tiling with an output tensor map");
        p->kernel = TRA_KERNEL_SEMIRING_F32;
        if (p->op == kSqdiff && p->agg == kSum && p->sqdiff_expand) {
            if (p->in_bf16) return fail(TRA_ERR_UNSUPPORTED, "sqdiff=expand needs fp32 inputs");
            const uint64_t nb = p->ext[kBatch];
            // row norms, column norms, one guard word per 128 x 128 output tile
            p->ws_bytes = align256(nb * p->ext[kM] * 4) + align256(nb * p->ext[kN] * 4) +
                          align256(sqdist_guard_bytes(nb, p->ext[kM], p->ext[kN]));
        }
    }
    // (split=bf16x3 squared distance: the guard's direct-form pass runs the CUDA-core kernel)
    if (!p->unary && p->kernel != TRA_KERNEL_TC_BF16 && p->kernel != TRA_KERNEL_TC_BF16_PAIR &&
        p->kernel != TRA_KERNEL_ELEMENTWISE && !(p->kernel == TRA_KERNEL_TC_SPLIT3 && p->op != kSqdiff))
        scan_vec_flags(role_map(*p, p->X, kBatch), role_map(*p, p->X, kM), role_map(*p, p->X, kK),
                       role_map(*p, p->Y, kBatch), role_map(*p, p->Y, kN), role_map(*p, p->Y, kK),
                       role_map(*p, p->Z, kBatch), role_map(*p, p->Z, kM), role_map(*p, p->Z, kN),
                       (uint32_t)p->ext[kBatch], (uint32_t)p->ext[kM], (uint32_t)p->ext[kN], (uint32_t)p->ext[kK],
                       p->vec_flags);
    return TRA_OK;
}

namespace {

bool groups_of_four(const RoleMap& m, uint32_t ext) {
    if (ext % 4) return false;
    for (uint32_t i = 0; i < ext; i += 4) {
        const int64_t o = role_offset(m, i);
        if (o % 4) return false;
        for (uint32_t c = 1; c < 4; ++c)
            if (role_offset(m, i + c) != o + c) return false;
    }
    return true;
}

bool all_multiples_of_four(const RoleMap& m, uint32_t ext) {
    for (uint32_t i = 0; i < ext; ++i)
        if (role_offset(m, i) % 4) return false;
    return true;
}

}  // namespace

void scan_vec_flags(const RoleMap& xb, const RoleMap& xm, const RoleMap& xk, const RoleMap& yb, const RoleMap& yn,
                    const RoleMap& yk, const RoleMap& zb, const RoleMap& zm, const RoleMap& zn, uint32_t nb,
                    uint32_t M, uint32_t N, uint32_t K, int flags[5]) {
    const bool xb4 = all_multiples_of_four(xb, nb), yb4 = all_multiples_of_four(yb, nb);
    const bool xk_in = xk.n > 0 && xk.t[0].div == 1 && xk.t[0].loc_stride == 1;
    const bool xm_in = xm.n > 0 && xm.t[0].div == 1 && xm.t[0].loc_stride == 1;
    const bool yn_in = yn.n > 0 && yn.t[0].div == 1 && yn.t[0].loc_stride == 1;
    const bool yk_in = yk.n > 0 && yk.t[0].div == 1 && yk.t[0].loc_stride == 1;
    flags[0] = xb4 && xk_in && groups_of_four(xk, K) && all_multiples_of_four(xm, M);
    flags[1] = xb4 && xm_in && groups_of_four(xm, M) && all_multiples_of_four(xk, K);
    flags[2] = yb4 && yn_in && groups_of_four(yn, N) && all_multiples_of_four(yk, K);
    flags[3] = yb4 && yk_in && groups_of_four(yk, K) && all_multiples_of_four(yn, N);
    const bool zn_in = zn.n > 0 && zn.t[0].div == 1 && zn.t[0].loc_stride == 1;
    flags[4] = zn_in && groups_of_four(zn, N) && all_multiples_of_four(zm, M) && all_multiples_of_four(zb, nb);
}

// Join tuples in canonical order: Z key row-major, then the contracted labels' key
// components (first-appearance order) row-major.  Row = X key, Y key, Z key.
void fill_keys(const Plan& p, int32_t* out) {
    const int w = p.X.rank + (p.unary ? 0 : p.Y.rank) + p.Z.rank;
    int32_t comp[TRA_MAX_LABELS];
    uint64_t row = 0;
    for (uint64_t g = 0; g < p.n_groups; ++g) {
        uint64_t t = g;
        for (int i = p.Z.rank - 1; i >= 0; --i) {
            comp[p.Z.label[i]] = (int32_t)(t % (uint64_t)p.D[p.Z.label[i]]);
            t /= (uint64_t)p.D[p.Z.label[i]];
        }
        for (uint64_t c = 0; c < p.n_agg; ++c, ++row) {
            uint64_t u = c;
            for (int i = (int)p.contracted.size() - 1; i >= 0; --i) {
                const int l = p.contracted[i];
                comp[l] = (int32_t)(u % (uint64_t)p.D[l]);
                u /= (uint64_t)p.D[l];
            }
            int32_t* r = out + row * w;
            int o = 0;
            for (int i = 0; i < p.X.rank; ++i) r[o++] = comp[p.X.label[i]];
            if (!p.unary)
                for (int i = 0; i < p.Y.rank; ++i) r[o++] = comp[p.Y.label[i]];
            for (int i = 0; i < p.Z.rank; ++i) r[o++] = comp[p.Z.label[i]];
        }
    }
}

}  // namespace tra
