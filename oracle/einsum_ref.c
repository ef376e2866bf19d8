/*
 * CPU ORACLE -- test infrastructure, not product code.
 * Only the tests, the package's smoke check and the benchmark's CPU-baseline /
 * reference arm may load this library.  It shares no code with the CUDA path.
 *
 * What it computes: the extended EinSum of "EinDecomp: automatic tensor-parallel
 * decomposition via Einstein summation + tensor relational algebra", section 2.1
 * (extended Einstein notation): for every output index tuple,
 *
 *     Z[out] = alpha * AGG_{contracted index tuples c} OP( X[x-indices], Y[y-indices] )
 *
 * where the contracted labels are those that appear on the right-hand side but
 * not in the output (section 2.1, matrix-multiply example), AGG is a
 * commutative, associative aggregation (sum, max, min, logsumexp) and OP is a
 * binary scalar function (multiply, add, (x-y)^2, x-y, exp(x-y)) (section 2.1,
 * "extended" operators and the squared-distance example).  AGG "none" means no
 * label is contracted (the element-wise example of section 2.1).  A unary
 * EinSum (no Y) uses OP = identity.
 *
 * The evaluation is the definition written out: an outer loop over the output
 * tuples in row-major order, an inner loop over the contracted tuples in
 * row-major order (contracted labels in first-appearance order, X then Y),
 * accumulation in double.  logsumexp is evaluated in two passes (maximum, then
 * m + log(sum exp(v - m))), the usual overflow-free form of log(sum(exp(v))).
 * alpha multiplies the aggregated value.
 *
 * Tensors are dense, row-major over their own label order, in double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OR_OP_MUL = 0, OR_OP_ADD = 1, OR_OP_SQDIFF = 2, OR_OP_SUB = 3, OR_OP_EXPSUB = 4, OR_OP_ID = 5 };
enum { OR_AGG_SUM = 0, OR_AGG_MAX = 1, OR_AGG_MIN = 2, OR_AGG_LSE = 3, OR_AGG_NONE = 4 };

#define OR_MAX_LABELS 16

typedef struct {
    int n_labels;
    int64_t bounds[OR_MAX_LABELS];
    int rx, ry, rz;                    /* ry < 0: unary */
    int64_t sx[OR_MAX_LABELS];         /* stride of X per label (0 if absent) */
    int64_t sy[OR_MAX_LABELS];
    int lz[OR_MAX_LABELS];             /* output labels in order */
    int n_c;                           /* contracted labels */
    int lc[OR_MAX_LABELS];
} or_shape;

static double apply_op(int op, double x, double y) {
    switch (op) {
        case OR_OP_MUL: return x * y;
        case OR_OP_ADD: return x + y;
        case OR_OP_SQDIFF: { double t = x - y; return t * t; }
        case OR_OP_SUB: return x - y;
        case OR_OP_EXPSUB: return exp(x - y);
        default: return x;
    }
}

static int build_shape(or_shape* s, int n_labels, const int64_t* bounds, int rx, const int* lx, int ry,
                       const int* ly, int rz, const int* lz) {
    if (n_labels <= 0 || n_labels > OR_MAX_LABELS || rx < 0 || rx > OR_MAX_LABELS || ry > OR_MAX_LABELS ||
        rz < 0 || rz > OR_MAX_LABELS)
        return -1;
    memset(s, 0, sizeof(*s));
    s->n_labels = n_labels;
    s->rx = rx; s->ry = ry; s->rz = rz;
    for (int l = 0; l < n_labels; ++l) s->bounds[l] = bounds[l];
    int64_t st = 1;
    for (int i = rx - 1; i >= 0; --i) { s->sx[lx[i]] += st; st *= bounds[lx[i]]; }
    st = 1;
    for (int i = ry - 1; i >= 0; --i) { s->sy[ly[i]] += st; st *= bounds[ly[i]]; }
    int in_z[OR_MAX_LABELS] = {0};
    for (int i = 0; i < rz; ++i) { s->lz[i] = lz[i]; in_z[lz[i]] = 1; }
    /* contracted labels, first-appearance order over X then Y */
    int seen[OR_MAX_LABELS] = {0};
    s->n_c = 0;
    for (int i = 0; i < rx; ++i)
        if (!in_z[lx[i]] && !seen[lx[i]]) { seen[lx[i]] = 1; s->lc[s->n_c++] = lx[i]; }
    for (int i = 0; i < ry; ++i)
        if (!in_z[ly[i]] && !seen[ly[i]]) { seen[ly[i]] = 1; s->lc[s->n_c++] = ly[i]; }
    return 0;
}

/* One output element: idx[] holds the value of every output label.  The contracted
 * tuples are visited in row-major order (an odometer over the contracted labels, the
 * last one fastest); the operand offsets follow the odometer incrementally. */
static double eval_one(const or_shape* s, int64_t* idx, const double* X, const double* Y, int op, int agg,
                       double alpha) {
    int unary = s->ry < 0 || Y == NULL;
    int64_t ox0 = 0, oy0 = 0;
    for (int i = 0; i < s->rz; ++i) {
        int l = s->lz[i];
        ox0 += idx[l] * s->sx[l];
        oy0 += idx[l] * s->sy[l];
    }
    int64_t n_outer = 1, n_inner = 1, sxi = 0, syi = 0;
    if (s->n_c > 0) {
        int li = s->lc[s->n_c - 1];
        n_inner = s->bounds[li];
        sxi = s->sx[li];
        syi = s->sy[li];
        for (int c = 0; c < s->n_c - 1; ++c) n_outer *= s->bounds[s->lc[c]];
    }
    double acc = 0.0, m = -INFINITY;
    int pass_count = (agg == OR_AGG_LSE) ? 2 : 1;
    for (int pass = 0; pass < pass_count; ++pass) {
        if (agg == OR_AGG_SUM || agg == OR_AGG_NONE) acc = 0.0;
        else if (agg == OR_AGG_MAX) acc = -INFINITY;
        else if (agg == OR_AGG_MIN) acc = INFINITY;
        else acc = (pass == 0) ? -INFINITY : 0.0;
        for (int c = 0; c < s->n_c; ++c) idx[s->lc[c]] = 0;
        int64_t ox = ox0, oy = oy0;
        for (int64_t t = 0; t < n_outer; ++t) {
            for (int64_t u = 0; u < n_inner; ++u) {
                double v = unary ? X[ox + u * sxi] : apply_op(op, X[ox + u * sxi], Y[oy + u * syi]);
                switch (agg) {
                    case OR_AGG_SUM: case OR_AGG_NONE: acc += v; break;
                    case OR_AGG_MAX: if (v > acc) acc = v; break;
                    case OR_AGG_MIN: if (v < acc) acc = v; break;
                    default:
                        if (pass == 0) { if (v > acc) acc = v; }
                        else acc += exp(v - m);
                }
            }
            /* row-major odometer over the outer contracted labels */
            for (int c = s->n_c - 2; c >= 0; --c) {
                int l = s->lc[c];
                ox += s->sx[l];
                oy += s->sy[l];
                if (++idx[l] < s->bounds[l]) break;
                ox -= s->sx[l] * s->bounds[l];
                oy -= s->sy[l] * s->bounds[l];
                idx[l] = 0;
            }
        }
        if (agg == OR_AGG_LSE && pass == 0) m = acc;
    }
    if (agg == OR_AGG_LSE) acc = (m == -INFINITY) ? -INFINITY : m + log(acc);
    return alpha * acc;
}

static void decode_out(const or_shape* s, int64_t o, int64_t* idx) {
    for (int i = s->rz - 1; i >= 0; --i) {
        int l = s->lz[i];
        idx[l] = o % s->bounds[l];
        o /= s->bounds[l];
    }
}

/* Full output, dense row-major over lz.  Returns 0 or -1 on bad arguments. */
int oracle_einsum(int n_labels, const int64_t* bounds, int rx, const int* lx, const double* X, int ry,
                  const int* ly, const double* Y, int rz, const int* lz, double* Z, int op, int agg,
                  double alpha) {
    or_shape s;
    if (build_shape(&s, n_labels, bounds, rx, lx, ry, ly, rz, lz)) return -1;
    if (agg == OR_AGG_NONE && s.n_c != 0) return -1;
    int64_t n_out = 1;
    for (int i = 0; i < rz; ++i) n_out *= bounds[lz[i]];
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t o = 0; o < n_out; ++o) {
        int64_t idx[OR_MAX_LABELS];
        memset(idx, 0, sizeof(idx));
        decode_out(&s, o, idx);
        Z[o] = eval_one(&s, idx, X, Y, op, agg, alpha);
    }
    return 0;
}

/* Selected outputs only: out_lin[p] is a row-major position in the dense output. */
int oracle_einsum_points(int n_labels, const int64_t* bounds, int rx, const int* lx, const double* X, int ry,
                         const int* ly, const double* Y, int rz, const int* lz, int64_t n_points,
                         const int64_t* out_lin, double* vals, int op, int agg, double alpha) {
    or_shape s;
    if (build_shape(&s, n_labels, bounds, rx, lx, ry, ly, rz, lz)) return -1;
    if (agg == OR_AGG_NONE && s.n_c != 0) return -1;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t p = 0; p < n_points; ++p) {
        int64_t idx[OR_MAX_LABELS];
        memset(idx, 0, sizeof(idx));
        decode_out(&s, out_lin[p], idx);
        vals[p] = eval_one(&s, idx, X, Y, op, agg, alpha);
    }
    return 0;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads for the OpenMP loops above (n >= 1); no effect without OpenMP. */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    extern void omp_set_num_threads(int);
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
