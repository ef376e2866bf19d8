// EinDecomp's optimiser over an EinGraph: one partition vector per node.
//
// "EinDecomp ... tensor relational algebra":
//  * section 3.1 -- the cost of a node under d is its join cost P*(|X_sub|+|Y_sub|) plus
//    its aggregation cost (P/n_agg)*(n_agg-1)*|Z_sub| (P read as the number of join
//    tuples, as everywhere in this library); an edge whose producer output and consumer
//    input are partitioned differently adds the repartition term.
//  * section 3.2 -- states are (node, d); d is pruned to vectors whose task count meets
//    the parallelism constraint and whose entries divide the bounds (often powers of two);
//    DP[v][d_v] = min over d_u of (DP[u][d_u] + repartition(d_u, d_v)) + cost(v, d_v),
//    read back from the output node.  A node with two inputs adds one such minimum per
//    input.
//  * section 4.3 (troubleshooting) -- the cost-model variants of tra_cost_model: a latency
//    charge per message (node: msg_join + msg_agg; edge: repartition messages), a minimum
//    block extent per label, a memory limit and weight on the node's output plus partials,
//    and task counts restricted to multiples of a given number.
// Host only; no device is touched.
#include <cstring>
#include <limits>
#include <vector>

#include "plan.h"

namespace tra {
namespace {

constexpr size_t kMaxCandidates = 1u << 16;

struct Candidate {
    int32_t D[TRA_MAX_LABELS];
    uint64_t cost;  // join + aggregation
};

struct Node {
    Plan plan;
    std::vector<Candidate> cand;
    std::vector<uint64_t> dp;
    std::vector<int> arg[2];  // per input: best producer candidate for each of this node's candidates
};

// Operand ranks of a spec "<X>,<Y>-><Z>:..." or "<X>-><Z>::..." (0 when malformed).
void spec_ranks(const char* spec, int& rx, int& ry) {
    rx = ry = 0;
    int* cur = &rx;
    for (const char* c = spec; *c && *c != '-' && *c != ':'; ++c) {
        if (*c == ',') cur = &ry;
        else ++*cur;
    }
}

struct Model {
    uint64_t latency = 0, mem_limit = 0, mem_weight = 0;
    int64_t min_block = 0, task_multiple = 0;
};

// the node's memory under D: its output plus the join's partials when they are aggregated
uint64_t node_memory(const Plan& p, const int32_t* D) {
    uint64_t tasks = 1, n_agg = 1, z_sub = 1;
    for (int l = 0; l < p.n_labels; ++l) {
        tasks *= (uint64_t)D[l];
        if (p.role[l] == kK) n_agg *= (uint64_t)D[l];
    }
    for (int i = 0; i < p.Z.rank; ++i) z_sub *= (uint64_t)(p.B[p.Z.label[i]] / D[p.Z.label[i]]);
    return (uint64_t)p.Z.total + (n_agg > 1 ? tasks * z_sub : 0);
}

void enumerate(const Plan& p, int l, Candidate& c, uint64_t prod, int64_t p_min, int64_t p_max, bool pow2,
               const Model& m, std::vector<Candidate>& out, bool& overflow) {
    if (overflow) return;
    if (l == p.n_labels) {
        if (prod < (uint64_t)p_min) return;
        if (m.task_multiple > 1 && prod % (uint64_t)m.task_multiple) return;
        if (m.mem_limit && node_memory(p, c.D) > m.mem_limit) return;
        if (out.size() >= kMaxCandidates) {
            overflow = true;
            return;
        }
        out.push_back(c);
        return;
    }
    const int64_t B = p.B[l];
    const int64_t gmin = m.min_block > 1 ? (m.min_block < B ? m.min_block : B) : 1;
    for (int64_t D = 1; D <= B; ++D) {
        if (B % D) continue;
        if (pow2 && (D & (D - 1))) continue;
        if (prod * (uint64_t)D > (uint64_t)p_max) break;
        if (B / D < gmin) break;  // block extents only shrink as D grows
        c.D[l] = (int32_t)D;
        enumerate(p, l + 1, c, prod * (uint64_t)D, p_min, p_max, pow2, m, out, overflow);
    }
}

uint64_t node_cost(const Plan& p, const int32_t* D, const Model& m) {
    uint64_t tasks = 1, x_sub = 1, y_sub = 0, z_sub = 1, n_agg = 1;
    for (int l = 0; l < p.n_labels; ++l) {
        tasks *= (uint64_t)D[l];
        if (p.role[l] == kK) n_agg *= (uint64_t)D[l];
    }
    for (int i = 0; i < p.X.rank; ++i) x_sub *= (uint64_t)(p.B[p.X.label[i]] / D[p.X.label[i]]);
    if (!p.unary) {
        y_sub = 1;
        for (int i = 0; i < p.Y.rank; ++i) y_sub *= (uint64_t)(p.B[p.Y.label[i]] / D[p.Y.label[i]]);
    }
    for (int i = 0; i < p.Z.rank; ++i) z_sub *= (uint64_t)(p.B[p.Z.label[i]] / D[p.Z.label[i]]);
    uint64_t c = tasks * (x_sub + y_sub) + (tasks / n_agg) * (n_agg - 1) * z_sub;
    if (m.latency) c += m.latency * (tasks * (p.unary ? 1u : 2u) + (tasks / n_agg) * (n_agg - 1));
    if (m.mem_weight) c += m.mem_weight * node_memory(p, D);
    return c;
}

const Operand& input_operand(const Plan& p, int k) { return k == 0 ? p.X : p.Y; }

// Repartition cost of producer u's output (candidate cu) into consumer v's input k (candidate cv).
uint64_t edge_cost(const Plan& u, const Candidate& cu, const Plan& v, int k, const Candidate& cv, const Model& m) {
    const Operand& in = input_operand(v, k);
    int64_t shape[TRA_MAX_RANK];
    int32_t src[TRA_MAX_RANK], dst[TRA_MAX_RANK];
    for (int i = 0; i < in.rank; ++i) {
        shape[i] = v.B[in.label[i]];
        dst[i] = cv.D[in.label[i]];
        src[i] = cu.D[u.Z.label[i]];
    }
    uint64_t c = repartition_cost_elems(in.rank, shape, src, dst);
    if (m.latency && c) c += m.latency * repartition_messages(in.rank, shape, src, dst);
    return c;
}

}  // namespace
}  // namespace tra

using namespace tra;

extern "C" int ein_graph_decompose(const tra_graph_node* nodes, int n_nodes, int64_t p_min, int64_t p_max, int flags,
                                   const tra_cost_model* model, int32_t* d_out, int n_d_out, uint64_t* node_cost_out,
                                   tra_graph_result* result) {
    clear_error();
    if (!nodes || n_nodes < 1 || !d_out || !result) return fail(TRA_ERR_ARG, "NULL argument or empty graph");
    if (p_min < 1 || p_max < p_min) return fail(TRA_ERR_ARG, "task bounds must satisfy 1 <= p_min <= p_max");
    const bool pow2 = (flags & TRA_DP_POW2) != 0;
    Model m;
    if (model) {
        if (model->min_block < 0 || model->task_multiple < 0) return fail(TRA_ERR_ARG, "negative cost-model parameter");
        m.latency = model->latency;
        m.min_block = model->min_block;
        m.mem_limit = model->mem_limit;
        m.mem_weight = model->mem_weight;
        m.task_multiple = model->task_multiple;
    }
    std::vector<Node> g(n_nodes);
    int d_total = 0;
    for (int v = 0; v < n_nodes; ++v) {
        const tra_graph_node& nd = nodes[v];
        if (!nd.spec || !nd.bounds) return fail(TRA_ERR_ARG, "node %d: NULL spec or bounds", v);
        int rx, ry;
        spec_ranks(nd.spec, rx, ry);
        if (rx < 1 || rx > TRA_MAX_RANK || ry > TRA_MAX_RANK)
            return fail(TRA_ERR_RANK, "node %d: operand ranks must be 1..%d", v, TRA_MAX_RANK);
        std::vector<int32_t> ones(rx + ry, 1);
        const int rc = build_plan(nd.spec, nd.bounds, nd.n_bounds, ones.data(), rx + ry, &g[v].plan);
        if (rc != TRA_OK) return rc;
        const Plan& p = g[v].plan;
        d_total += p.X.rank + (p.unary ? 0 : p.Y.rank);
        for (int k = 0; k < 2; ++k) {
            const int u = nd.input[k];
            if (u == -1) continue;
            if (k == 1 && p.unary) return fail(TRA_ERR_ARG, "node %d: a unary EinSum has no second input", v);
            if (u < 0 || u >= v) return fail(TRA_ERR_ARG, "node %d: input %d must name an earlier node", v, u);
            const Plan& pu = g[u].plan;
            const Operand& in = input_operand(p, k);
            if (pu.Z.rank != in.rank) return fail(TRA_ERR_ARG, "node %d input %d: rank differs from node %d's output", v, k, u);
            for (int i = 0; i < in.rank; ++i)
                if (pu.B[pu.Z.label[i]] != p.B[in.label[i]])
                    return fail(TRA_ERR_ARG, "node %d input %d: shape differs from node %d's output", v, k, u);
        }
        Candidate c;
        memset(&c, 0, sizeof(c));
        bool overflow = false;
        enumerate(p, 0, c, 1, p_min, p_max, pow2, m, g[v].cand, overflow);
        if (overflow) return fail(TRA_ERR_UNSUPPORTED, "node %d: more than %zu candidate partition vectors", v, kMaxCandidates);
        if (g[v].cand.empty())
            return fail(TRA_ERR_UNSUPPORTED, "node %d: no partition vector gives %lld..%lld tasks under the cost model",
                        v, (long long)p_min, (long long)p_max);
        for (Candidate& cc : g[v].cand) cc.cost = node_cost(p, cc.D, m);
    }
    if (n_d_out != d_total) return fail(TRA_ERR_ARG, "d_out holds %d entries, the graph needs %d", n_d_out, d_total);

    // the programme, in node order
    uint64_t n_cand = 0;
    for (int v = 0; v < n_nodes; ++v) {
        Node& nv = g[v];
        const size_t cv_n = nv.cand.size();
        n_cand += cv_n;
        nv.dp.assign(cv_n, 0);
        for (size_t c = 0; c < cv_n; ++c) nv.dp[c] = nv.cand[c].cost;
        for (int k = 0; k < 2; ++k) {
            const int u = nodes[v].input[k];
            if (u < 0) continue;
            const Node& nu = g[u];
            nv.arg[k].assign(cv_n, 0);
            for (size_t c = 0; c < cv_n; ++c) {
                uint64_t best = std::numeric_limits<uint64_t>::max();
                int best_i = 0;
                for (size_t cu = 0; cu < nu.cand.size(); ++cu) {
                    const uint64_t t = nu.dp[cu] + edge_cost(nu.plan, nu.cand[cu], nv.plan, k, nv.cand[c], m);
                    if (t < best) {
                        best = t;
                        best_i = (int)cu;
                    }
                }
                nv.dp[c] += best;
                nv.arg[k][c] = best_i;
            }
        }
    }

    // read the choice back from the output (the last node); a node reached from two
    // consumers keeps the choice of the later one; nodes not reaching the output decide alone
    std::vector<int> choice(n_nodes, -1);
    auto argmin = [&](int v) {
        int b = 0;
        for (size_t c = 1; c < g[v].dp.size(); ++c)
            if (g[v].dp[c] < g[v].dp[b]) b = (int)c;
        return b;
    };
    for (int v = n_nodes - 1; v >= 0; --v) {
        if (choice[v] < 0) choice[v] = argmin(v);
        for (int k = 0; k < 2; ++k) {
            const int u = nodes[v].input[k];
            if (u >= 0 && choice[u] < 0) choice[u] = g[v].arg[k][choice[v]];
        }
    }

    uint64_t total = 0;
    int pos = 0;
    for (int v = 0; v < n_nodes; ++v) {
        const Plan& p = g[v].plan;
        const Candidate& cv = g[v].cand[choice[v]];
        uint64_t own = cv.cost;
        for (int k = 0; k < 2; ++k) {
            const int u = nodes[v].input[k];
            if (u >= 0) own += edge_cost(g[u].plan, g[u].cand[choice[u]], p, k, cv, m);
        }
        total += own;
        if (node_cost_out) node_cost_out[v] = own;
        for (int i = 0; i < p.X.rank; ++i) d_out[pos++] = cv.D[p.X.label[i]];
        if (!p.unary)
            for (int i = 0; i < p.Y.rank; ++i) d_out[pos++] = cv.D[p.Y.label[i]];
    }
    result->total_cost = total;
    result->dp_cost = g[n_nodes - 1].dp[choice[n_nodes - 1]];
    result->n_candidates = n_cand;
    return TRA_OK;
}
