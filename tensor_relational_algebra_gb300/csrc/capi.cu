// extern "C" entry points of libtra.so (declared and documented in include/tra.h).
#include <cstring>
#include <numeric>

#include "plan.h"

using namespace tra;

namespace {

int cuda_fail(cudaError_t e, const char* what) {
    return fail(TRA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Vector loads only where the plan-time scan proved every 4-wide address aligned and
// contiguous, and the base pointer is 16-byte (fp32) / 8-byte (bf16) aligned.
void set_load_modes(SemiringParams& sp, int bf16, const int flags[5]) {
    const size_t a = bf16 ? 8 : 16;
    const bool xa = (uintptr_t)sp.x % a == 0, ya = (uintptr_t)sp.y % a == 0;
    sp.x_mode = xa && flags[0] ? 1 : (xa && flags[1] ? 2 : 0);
    sp.y_mode = ya && flags[2] ? 2 : (ya && flags[3] ? 1 : 0);
    sp.z_vec4 = flags[4] && (uintptr_t)sp.z % (sp.out_bf16 ? 8 : 16) == 0;
    // single-label contracted composite: the kernel divides by the block extent with a
    // multiply-high instead of walking the role map
    auto simple = [&](const RoleMap& m) { return m.n == 1 && m.t[0].div == 1 && m.t[0].ext == sp.K; };
    sp.xk_simple = simple(sp.xk);
    sp.yk_simple = simple(sp.yk);
    if (sp.xk_simple) {
        sp.xk_sub = FastDiv(sp.xk.t[0].sub);
        sp.xk_ks = sp.xk.t[0].key_stride;
        sp.xk_ls = sp.xk.t[0].loc_stride;
    }
    if (sp.yk_simple) {
        sp.yk_sub = FastDiv(sp.yk.t[0].sub);
        sp.yk_ks = sp.yk.t[0].key_stride;
        sp.yk_ls = sp.yk.t[0].loc_stride;
    }
}

// Elementwise joins whose fp32 X has Z's labels in Z's order share Z's relation layout, so
// element e of Z reads X at e; Y either has that layout too (or is absent) or is Z without
// its innermost label, unsplit, and then is read at e / extent.  Chunks of 8 elements need
// the sizes and the buffers' alignment below.
int flat_mode(const Plan& p, const void* x, const void* y, const void* z) {
    if (p.in_bf16 || p.X.rank != p.Z.rank) return 0;
    for (int i = 0; i < p.Z.rank; ++i)
        if (p.X.label[i] != p.Z.label[i]) return 0;
    if (p.Z.total % 8 || ((uintptr_t)x | (uintptr_t)z) % 16) return 0;
    if (p.unary) return 1;
    bool same = p.Y.rank == p.Z.rank, minus_last = p.Y.rank == p.Z.rank - 1;
    for (int i = 0; i < p.Y.rank; ++i) {
        same = same && p.Y.label[i] == p.Z.label[i];
        minus_last = minus_last && p.Y.label[i] == p.Z.label[i];
    }
    if (same) return (uintptr_t)y % 16 ? 0 : 1;
    const int last = p.Z.rank - 1;
    if (minus_last && p.Z.d[last] == 1 && p.Z.shape[last] % 8 == 0) return 2;
    return 0;
}

SemiringParams semiring_params(const Plan& p, const void* x, const void* y, void* z) {
    SemiringParams sp;
    memset(&sp, 0, sizeof(sp));
    sp.x = x;
    sp.y = y;
    sp.z = z;
    sp.xb = role_map(p, p.X, kBatch);
    sp.xm = role_map(p, p.X, kM);
    sp.xk = role_map(p, p.X, kK);
    sp.yb = role_map(p, p.Y, kBatch);
    sp.yn = role_map(p, p.Y, kN);
    sp.yk = role_map(p, p.Y, kK);
    sp.zb = role_map(p, p.Z, kBatch);
    sp.zm = role_map(p, p.Z, kM);
    sp.zn = role_map(p, p.Z, kN);
    sp.nb = (uint32_t)p.ext[kBatch];
    sp.M = (uint32_t)p.ext[kM];
    sp.N = (uint32_t)p.ext[kN];
    sp.K = (uint32_t)p.ext[kK];
    sp.op = p.op;
    sp.agg = p.agg;
    sp.alpha = (float)p.alpha;
    sp.in_bf16 = p.in_bf16;
    sp.out_bf16 = p.out_bf16;
    sp.x_kcontig = affine_stride(sp.xk) == 1;
    sp.x_mcontig = affine_stride(sp.xm) == 1;
    sp.y_ncontig = affine_stride(sp.yn) == 1;
    sp.y_kcontig = affine_stride(sp.yk) == 1;
    set_load_modes(sp, p.in_bf16, p.vec_flags);
    sp.x_elems = (uint64_t)p.X.total;
    sp.y_elems = p.unary ? 0 : (uint64_t)p.Y.total;
    sp.z_elems = (uint64_t)p.Z.total;
    cudaPointerAttributes pa;
    sp.z_device = z && cudaPointerGetAttributes(&pa, z) == cudaSuccess && pa.type == cudaMemoryTypeDevice;
    (void)cudaGetLastError();
    return sp;
}

// Literal TRA execution (section 2.2 read literally): every join tuple produces its
// own partial sub-tensor (the contracted labels run over one block only), then the
// partials of each output key are combined in canonical order.
int execute_literal(const Plan& p, const void* x, const void* y, void* z, void* ws, cudaStream_t s) {
    SemiringParams sp = semiring_params(p, x, y, ws);
    const uint32_t nb0 = sp.nb;
    // contracted composite restricted to one block: extents b_l, key part zero
    RoleMap* kmaps[2] = {&sp.xk, &sp.yk};
    const Operand* ops[2] = {&p.X, &p.Y};
    for (int a = 0; a < 2; ++a) {
        RoleMap& m = *kmaps[a];
        memset(&m, 0, sizeof(m));
        uint64_t div = 1;
        for (int l : p.comp[kK]) {
            const int i = ops[a]->pos_of(l);
            const uint32_t b = (uint32_t)(p.B[l] / p.D[l]);
            if (i >= 0) {
                Term& t = m.t[m.n++];
                t.div = (uint32_t)div;
                t.ext = b;
                t.sub = b;
                t.key_stride = 0;
                t.loc_stride = ops[a]->loc_stride[i];
            }
            div *= b;
        }
    }
    sp.K = 1;
    for (int l : p.comp[kK]) sp.K *= (uint32_t)(p.B[l] / p.D[l]);
    // batch composite extended by the contracted key components
    uint64_t div = nb0;
    const uint64_t zsub = (uint64_t)p.Z.sub;
    for (RoleMap* zm : {&sp.zb, &sp.zm, &sp.zn})
        for (int i = 0; i < zm->n; ++i) zm->t[i].key_stride *= (int64_t)p.n_agg;
    for (int l : p.comp[kK]) {
        const uint32_t D = (uint32_t)p.D[l];
        for (int a = 0; a < 2; ++a) {
            const int i = ops[a]->pos_of(l);
            if (i < 0) continue;
            RoleMap& bm = a == 0 ? sp.xb : sp.yb;
            Term& t = bm.t[bm.n++];
            t.div = (uint32_t)div;
            t.ext = D;
            t.sub = 1;
            t.key_stride = ops[a]->key_stride[i];
            t.loc_stride = 0;
        }
        // the partial's slot: contracted key linearised row-major in first-appearance order
        int64_t cstride = 1;
        bool after = false;
        for (int c : p.contracted) {
            if (after) cstride *= p.D[c];
            if (c == l) after = true;
        }
        Term& t = sp.zb.t[sp.zb.n++];
        t.div = (uint32_t)div;
        t.ext = D;
        t.sub = 1;
        t.key_stride = cstride * (int64_t)zsub;
        t.loc_stride = 0;
        div *= D;
    }
    sp.nb = (uint32_t)div;
    sp.alpha = 1.f;
    sp.out_bf16 = 0;
    sp.z_elems = p.n_tasks * zsub;  // one partial sub-tensor per join tuple
    sp.x_kcontig = affine_stride(sp.xk) == 1;
    sp.y_kcontig = affine_stride(sp.yk) == 1;
    int flags[5];
    scan_vec_flags(sp.xb, sp.xm, sp.xk, sp.yb, sp.yn, sp.yk, sp.zb, sp.zm, sp.zn, sp.nb, sp.M, sp.N, sp.K, flags);
    set_load_modes(sp, p.in_bf16, flags);
    cudaError_t e = launch_semiring(sp, s);
    if (e != cudaSuccess) return cuda_fail(e, "literal join");
    CombineParams cp;
    cp.partials = reinterpret_cast<const float*>(ws);
    cp.z = z;
    cp.n_groups = p.n_groups;
    cp.n_agg = p.n_agg;
    cp.z_sub = zsub;
    cp.agg = p.agg;
    cp.alpha = (float)p.alpha;
    cp.out_bf16 = p.out_bf16;
    e = launch_combine(cp, s);
    if (e != cudaSuccess) return cuda_fail(e, "literal combine");
    return TRA_OK;
}

int execute_plan(const Plan& p, const void* x, const void* y, void* z, void* ws, cudaStream_t s) {
    cudaError_t e = cudaSuccess;
    switch (p.kernel) {
        case TRA_KERNEL_SEMIRING_F32: {
            SemiringParams sp = semiring_params(p, x, y, z);
            if (p.op == kSqdiff && p.sqdiff_expand) {
                float* xn = reinterpret_cast<float*>(ws);
                float* yn = reinterpret_cast<float*>((char*)ws + align256((uint64_t)sp.nb * sp.M * 4));
                LsePrepParams lp;
                memset(&lp, 0, sizeof(lp));
                lp.mode = 1;
                lp.in_bf16 = 0;
                lp.nb = sp.nb;
                lp.K = sp.K;
                lp.src = x, lp.rmax = xn, lp.b = sp.xb, lp.r = sp.xm, lp.k = sp.xk, lp.R = sp.M;
                lp.src_elems = sp.x_elems;
                if ((e = launch_lse_prep(lp, s)) != cudaSuccess) return cuda_fail(e, "norms of X");
                lp.src = y, lp.rmax = yn, lp.b = sp.yb, lp.r = sp.yn, lp.k = sp.yk, lp.R = sp.N;
                lp.src_elems = sp.y_elems;
                if ((e = launch_lse_prep(lp, s)) != cudaSuccess) return cuda_fail(e, "norms of Y");
                sp.op = kMul;
                sp.xnorm = xn;
                sp.ynorm = yn;
                sp.sq_tau = sqdist_guard_tau(sp.K, kSqGuardFp32);
                sp.tile_mark = reinterpret_cast<uint32_t*>((char*)ws + align256((uint64_t)sp.nb * sp.M * 4) +
                                                           align256((uint64_t)sp.nb * sp.N * 4));
                sp.gate_tag = next_gate_tag();
                set_load_modes(sp, 0, p.vec_flags);
            }
            e = launch_semiring(sp, s);
            break;
        }
        case TRA_KERNEL_LSE_FACTORED: {
            SemiringParams sp = semiring_params(p, x, y, z);
            char* w = reinterpret_cast<char*>(ws);
            float* ex = reinterpret_cast<float*>(w);
            w += align256((uint64_t)p.X.total * 4);
            float* ey = reinterpret_cast<float*>(w);
            w += align256((uint64_t)p.Y.total * 4);
            float* rmax = reinterpret_cast<float*>(w);
            w += align256((uint64_t)sp.nb * sp.M * 4);
            float* cmax = reinterpret_cast<float*>(w);
            LsePrepParams lp;
            memset(&lp, 0, sizeof(lp));
            lp.mode = 0;
            lp.in_bf16 = p.in_bf16;
            lp.nb = sp.nb;
            lp.K = sp.K;
            lp.src = x, lp.dst = ex, lp.rmax = rmax, lp.b = sp.xb, lp.r = sp.xm, lp.k = sp.xk, lp.R = sp.M;
            lp.src_elems = sp.x_elems;
            if ((e = launch_lse_prep(lp, s)) != cudaSuccess) return cuda_fail(e, "max-shift of X");
            lp.src = y, lp.dst = ey, lp.rmax = cmax, lp.b = sp.yb, lp.r = sp.yn, lp.k = sp.yk, lp.R = sp.N;
            lp.src_elems = sp.y_elems;
            if ((e = launch_lse_prep(lp, s)) != cudaSuccess) return cuda_fail(e, "max-shift of Y");
            sp.x_raw = x;
            sp.y_raw = y;
            sp.x = ex;
            sp.y = ey;
            set_load_modes(sp, 0, p.vec_flags);
            sp.rowmax = rmax;
            sp.colmax = cmax;
            sp.op = kMul;
            sp.agg = kSum;
            e = launch_semiring(sp, s);
            break;
        }
        case TRA_KERNEL_ROW_REDUCE: {
            RowReduceParams rp;
            memset(&rp, 0, sizeof(rp));
            rp.x = x;
            rp.z = z;
            rp.xr = role_map(p, p.X, kM);
            rp.xk = role_map(p, p.X, kK);
            rp.zr = role_map(p, p.Z, kM);
            rp.R = (uint32_t)p.ext[kM];
            rp.K = (uint32_t)p.ext[kK];
            rp.agg = p.agg;
            rp.alpha = (float)p.alpha;
            rp.in_bf16 = p.in_bf16;
            rp.out_bf16 = p.out_bf16;
            rp.k_affine = rp.xk.n == 1 && rp.xk.t[0].loc_stride == 1 && rp.xk.t[0].sub == rp.xk.t[0].ext;
            rp.x_elems = (uint64_t)p.X.total;
            rp.z_elems = (uint64_t)p.Z.total;
            e = launch_row_reduce(rp, s);
            break;
        }
        case TRA_KERNEL_ELEMENTWISE: {
            ElementwiseParams ep;
            memset(&ep, 0, sizeof(ep));
            ep.x = x;
            ep.y = p.unary ? nullptr : y;
            ep.z = z;
            ep.rank = p.Z.rank;
            ep.op = p.unary ? kId : p.op;
            ep.alpha = (float)p.alpha;
            ep.in_bf16 = p.in_bf16;
            ep.out_bf16 = p.out_bf16;
            ep.sub_total = FastDiv((uint32_t)p.Z.sub);
            for (int i = 0; i < p.Z.rank; ++i) {
                const int l = p.Z.label[i];
                ep.grid[i] = FastDiv((uint32_t)p.Z.d[i]);
                ep.sub[i] = FastDiv((uint32_t)(p.Z.shape[i] / p.Z.d[i]));
                const int xi = p.X.pos_of(l);
                if (xi >= 0) ep.x_ks[i] = p.X.key_stride[xi], ep.x_ls[i] = p.X.loc_stride[xi];
                const int yi = p.unary ? -1 : p.Y.pos_of(l);
                if (yi >= 0) ep.y_ks[i] = p.Y.key_stride[yi], ep.y_ls[i] = p.Y.loc_stride[yi];
            }
            ep.I = (uint32_t)(p.Z.shape[p.Z.rank - 1] / p.Z.d[p.Z.rank - 1]);
            ep.n_runs = (uint64_t)p.Z.total / ep.I;
            ep.total = (uint64_t)p.Z.total;
            ep.flat = flat_mode(p, x, y, z);
            ep.y_div = (uint32_t)p.Z.shape[p.Z.rank - 1];
            ep.x_elems = (uint64_t)p.X.total;
            ep.y_elems = p.unary ? 0 : (uint64_t)p.Y.total;
            e = launch_elementwise(ep, s);
            break;
        }
        case TRA_KERNEL_EMPTY:
            return TRA_OK;  // no output element
        case TRA_KERNEL_FILL: {
            // each output aggregates the empty set: agg's identity, then alpha, then one rounding
            const double id = p.agg == kSum ? 0.0 : (p.agg == kMin ? HUGE_VAL : -HUGE_VAL);
            e = launch_fill(z, (uint64_t)p.Z.total, (float)(p.alpha * id), p.out_bf16 != 0, s);
            break;
        }
        case TRA_KERNEL_TC_BF16:
        case TRA_KERNEL_TC_BF16_PAIR:
            return tc_execute(p, x, y, z, s, nullptr, ws);
        case TRA_KERNEL_TC_SPLIT3: {
            // norms (squared distance) or row / column maxima (logsumexp) of the fp32 operands,
            // the hi / lo split into the GEMM's operands, the GEMM with the rank-one epilogue
            // writing Z in its relation layout, and for logsumexp the underflow fix-up
            SemiringParams sp = semiring_params(p, x, y, z);
            const bool lse = p.op == kAdd;
            const uint64_t nb = sp.nb, M = sp.M, N = sp.N, K = sp.K;
            const uint64_t Mp = split3_pad(M, 128), Np = split3_pad(N, 64), K3p = split3_pad(3 * K, 64);
            char* w = reinterpret_cast<char*>(ws);
            __nv_bfloat16* a3 = reinterpret_cast<__nv_bfloat16*>(w);
            w += align256(nb * Mp * K3p * 2);
            __nv_bfloat16* b3 = reinterpret_cast<__nv_bfloat16*>(w);
            w += align256(nb * Np * K3p * 2);
            float* rt = reinterpret_cast<float*>(w);
            w += align256(nb * M * 4);
            float* ct = reinterpret_cast<float*>(w);
            w += align256(nb * N * 4);
            int* marks = reinterpret_cast<int*>(w);
            w += 256;
            uint32_t* fix = nullptr;  // squared distance: guard words, one per 128 x 128 output tile
            if (!lse) {
                fix = reinterpret_cast<uint32_t*>(w);
                w += align256(sqdist_guard_bytes(nb, M, N));
            }
            float* parts = reinterpret_cast<float*>(w);
            Split3StatsParams st;
            memset(&st, 0, sizeof(st));
            st.mode = lse ? 0 : 1;
            st.nb = sp.nb;
            st.K = sp.K;
            st.partials = parts;
            st.src = reinterpret_cast<const float*>(x), st.out = rt, st.b = sp.xb, st.r = sp.xm, st.k = sp.xk, st.R = sp.M;
            st.src_elems = sp.x_elems;
            st.kc = split3_stats_chunks(nb * M, K);
            if ((e = launch_split3_stats(st, s)) != cudaSuccess) return cuda_fail(e, "row terms of X");
            st.src = reinterpret_cast<const float*>(y), st.out = ct, st.b = sp.yb, st.r = sp.yn, st.k = sp.yk, st.R = sp.N;
            st.src_elems = sp.y_elems;
            st.kc = split3_stats_chunks(nb * N, K);
            if ((e = launch_split3_stats(st, s)) != cudaSuccess) return cuda_fail(e, "column terms of Y");
            Split3Params s3;
            memset(&s3, 0, sizeof(s3));
            s3.src = reinterpret_cast<const float*>(x), s3.dst = a3, s3.shift = lse ? rt : nullptr;
            s3.b = sp.xb, s3.r = sp.xm, s3.k = sp.xk, s3.nb = sp.nb, s3.R = sp.M, s3.K = sp.K, s3.is_y = 0;
            s3.Rp = (uint32_t)Mp, s3.K3p = (uint32_t)K3p;
            s3.src_elems = sp.x_elems;
            if ((e = launch_split3(s3, s)) != cudaSuccess) return cuda_fail(e, "split of X");
            s3.src = reinterpret_cast<const float*>(y), s3.dst = b3, s3.shift = lse ? ct : nullptr;
            s3.b = sp.yb, s3.r = sp.yn, s3.k = sp.yk, s3.R = sp.N, s3.is_y = 1, s3.Rp = (uint32_t)Np;
            s3.src_elems = sp.y_elems;
            if ((e = launch_split3(s3, s)) != cudaSuccess) return cuda_fail(e, "split of Y");
            TcExtra ex;
            ex.epi = lse ? 2 : 1;
            ex.row_term = rt;
            ex.col_term = ct;
            ex.alpha = (float)p.alpha;
            ex.z_override = !p.split3_direct;
            ex.zb = sp.zb;
            ex.zm = sp.zm;
            ex.zn = sp.zn;
            ex.M = sp.M;
            ex.N = sp.N;
            ex.z_elems = sp.z_elems;
            if (lse) {
                ex.mark_count = marks;
                if ((e = cudaMemsetAsync(marks, 0, sizeof(int), s)) != cudaSuccess) return cuda_fail(e, "mark count");
            } else {
                ex.sq_tau = sqdist_guard_tau(K, kSqGuardSplit3);
                ex.fix_flags = fix;
                ex.fix_tiles_m = (uint32_t)((M + 127) / 128);
                ex.fix_tiles_n = (uint32_t)((N + 127) / 128);
                ex.fix_tag_index = semiring_tiles(nb, M, N);  // the word set to 1 when anything is marked
                if ((e = cudaMemsetAsync(fix, 0, sqdist_guard_bytes(nb, M, N), s)) != cudaSuccess)
                    return cuda_fail(e, "guard words");
            }
            const int rc = tc_execute(*p.inner, a3, b3, z, s, &ex);
            if (rc != TRA_OK) return rc;
            if (!lse) {
                // the outputs whose expansion cancelled too far: their tiles in the direct form
                sp.tile_gate = fix;
                sp.gate_tag = 1;
                if ((e = launch_sqdist_fixup(sp, s)) != cudaSuccess) return cuda_fail(e, "guard pass");
                return TRA_OK;
            }
            sp.x_raw = x;
            sp.y_raw = y;
            sp.mark_count = marks;
            e = launch_lse_fixup(sp, s);
            break;
        }
        case TRA_KERNEL_LITERAL:
            return execute_literal(p, x, y, z, ws, s);
        default:
            return fail(TRA_ERR_UNSUPPORTED, "no kernel for this plan");
    }
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    return TRA_OK;
}

int check_partition(int rank, const int64_t* shape, const int32_t* d, const char* what) {
    for (int i = 0; i < rank; ++i) {
        if (shape[i] < 0 || shape[i] > 0x7fffffffLL)
            return fail(TRA_ERR_ARG, "%s: extent %lld out of range", what, (long long)shape[i]);
        if (d[i] < 1 || shape[i] % d[i])
            return fail(TRA_ERR_DIVISIBILITY, "%s: D=%d does not divide B=%lld in dimension %d", what, d[i],
                        (long long)shape[i], i);
    }
    return TRA_OK;
}

}  // namespace

extern "C" {

int ein_plan(const char* spec, const int64_t* bounds, int n_bounds, const int32_t* d, int n_d, tra_plan_t* out) {
    clear_error();
    if (!out) return fail(TRA_ERR_ARG, "out is NULL");
    *out = nullptr;
    Plan* p = new Plan();
    const int rc = build_plan(spec, bounds, n_bounds, d, n_d, p);
    if (rc != TRA_OK) {
        delete p;
        return rc;
    }
    *out = reinterpret_cast<tra_plan_t>(p);
    return TRA_OK;
}

int ein_plan_info(tra_plan_t plan, tra_plan_info* o) {
    clear_error();
    if (!plan || !o) return fail(TRA_ERR_ARG, "NULL argument");
    const Plan& p = *reinterpret_cast<const Plan*>(plan);
    memset(o, 0, sizeof(*o));
    o->n_labels = p.n_labels;
    for (int l = 0; l < p.n_labels; ++l) {
        o->labels[l] = p.name[l];
        o->bound[l] = p.B[l];
        o->part[l] = p.D[l];
        o->sub_extent[l] = p.B[l] / p.D[l];
        o->role[l] = p.role[l];
    }
    o->rank_x = p.X.rank;
    o->rank_y = p.unary ? 0 : p.Y.rank;
    o->rank_z = p.Z.rank;
    for (int i = 0; i < p.X.rank; ++i) o->key_grid_x[i] = p.X.d[i];
    if (!p.unary)
        for (int i = 0; i < p.Y.rank; ++i) o->key_grid_y[i] = p.Y.d[i];
    for (int i = 0; i < p.Z.rank; ++i) o->key_grid_z[i] = p.Z.d[i];
    o->n_tasks = p.n_tasks;
    o->n_groups = p.n_groups;
    o->n_agg = p.n_agg;
    o->x_sub = (uint64_t)p.X.sub;
    o->y_sub = p.unary ? 0 : (uint64_t)p.Y.sub;
    o->z_sub = (uint64_t)p.Z.sub;
    o->cost_join = p.cost_join;
    o->cost_agg = p.cost_agg;
    o->workspace_bytes = p.ws_bytes;
    o->in_dtype = p.in_bf16;
    o->out_dtype = p.out_bf16;
    o->kernel = p.kernel;
    o->msg_join = p.msg_join;
    o->msg_agg = p.msg_agg;
    o->mem_elems = p.mem_elems;
    return TRA_OK;
}

int ein_plan_keys(tra_plan_t plan, int32_t* xyz_keys, int64_t capacity) {
    clear_error();
    if (!plan || !xyz_keys) return fail(TRA_ERR_ARG, "NULL argument");
    const Plan& p = *reinterpret_cast<const Plan*>(plan);
    const uint64_t need = p.n_tasks * (uint64_t)(p.X.rank + (p.unary ? 0 : p.Y.rank) + p.Z.rank);
    if (capacity < 0 || (uint64_t)capacity < need)
        return fail(TRA_ERR_ARG, "key buffer holds %lld int32, %llu needed", (long long)capacity,
                    (unsigned long long)need);
    fill_keys(p, xyz_keys);
    return TRA_OK;
}

int ein_execute(tra_plan_t plan, const void* in0, const void* in1, void* out, void* workspace, size_t ws_bytes,
                tra_stream_t stream) {
    clear_error();
    if (!plan) return fail(TRA_ERR_ARG, "NULL plan");
    const Plan& p = *reinterpret_cast<const Plan*>(plan);
    if (p.kernel == TRA_KERNEL_EMPTY) return TRA_OK;  // an output of no elements: nothing to read or write
    if (!out) return fail(TRA_ERR_ARG, "NULL output");
    if (p.kernel != TRA_KERNEL_FILL) {  // a fill reads no input
        if (!in0) return fail(TRA_ERR_ARG, "NULL input");
        if (!p.unary && !in1) return fail(TRA_ERR_ARG, "binary EinSum needs in1");
    }
    if (p.ws_bytes && (!workspace || ws_bytes < p.ws_bytes))
        return fail(TRA_ERR_WORKSPACE, "workspace of %llu bytes needed, %llu given",
                    (unsigned long long)p.ws_bytes, (unsigned long long)(workspace ? ws_bytes : 0));
    return execute_plan(p, in0, in1, out, workspace, reinterpret_cast<cudaStream_t>(stream));
}

int ein_repartition(int rank, const int64_t* shape, const int32_t* src_d, const int32_t* dst_d, int elem_bytes,
                    const void* src, void* dst, tra_stream_t stream) {
    clear_error();
    if (rank < 1 || rank > TRA_MAX_RANK) return fail(TRA_ERR_RANK, "rank %d outside 1..%d", rank, TRA_MAX_RANK);
    if (!shape || !src_d || !dst_d) return fail(TRA_ERR_ARG, "NULL argument");
    if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4 && elem_bytes != 8)
        return fail(TRA_ERR_ARG, "element size %d not in {1,2,4,8}", elem_bytes);
    int rc = check_partition(rank, shape, src_d, "source");
    if (rc == TRA_OK) rc = check_partition(rank, shape, dst_d, "destination");
    if (rc != TRA_OK) return rc;
    for (int i = 0; i < rank; ++i)
        if (shape[i] == 0) return TRA_OK;  // an extent of 0: nothing to copy
    int64_t total = 1;
    for (int i = 0; i < rank; ++i) total = total >= 0x7fffffffLL ? total : total * shape[i];
    if (total >= 0x7fffffffLL) return fail(TRA_ERR_UNSUPPORTED, "tensors above 2^31-1 elements are not supported");
    if (!src || !dst) return fail(TRA_ERR_ARG, "NULL buffer");
    if (((uintptr_t)src | (uintptr_t)dst) % elem_bytes) return fail(TRA_ERR_ARG, "misaligned buffer");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (total == 0) return TRA_OK;
    if (memcmp(src_d, dst_d, sizeof(int32_t) * rank) == 0) {
        cudaError_t e = cudaMemcpyAsync(dst, src, (size_t)total * elem_bytes, cudaMemcpyDeviceToDevice, s);
        return e == cudaSuccess ? TRA_OK : cuda_fail(e, "copy");
    }
    {
        const cudaError_t et = launch_repartition_tma(rank, shape, src_d, dst_d, elem_bytes, src, dst, s);
        if (et == cudaSuccess) return TRA_OK;
        if (et != cudaErrorNotSupported) return cuda_fail(et, "repartition launch");
    }
    RepartParams rp;
    memset(&rp, 0, sizeof(rp));
    rp.src = src;
    rp.dst = dst;
    rp.rank = rank;
    rp.elem_bytes = elem_bytes;
    int64_t ssub[TRA_MAX_RANK], dsub[TRA_MAX_RANK];
    int64_t ssub_total = 1, dsub_total = 1;
    for (int i = 0; i < rank; ++i) {
        ssub[i] = shape[i] / src_d[i];
        dsub[i] = shape[i] / dst_d[i];
        ssub_total *= ssub[i];
        dsub_total *= dsub[i];
    }
    int64_t ls = 1, ks = ssub_total;
    for (int i = rank - 1; i >= 0; --i) {
        rp.src_loc_stride[i] = ls;
        rp.src_key_stride[i] = ks;
        ls *= ssub[i];
        ks *= src_d[i];
        rp.dst_grid[i] = FastDiv((uint32_t)dst_d[i]);
        rp.dst_sub[i] = FastDiv((uint32_t)dsub[i]);
        rp.src_sub[i] = FastDiv((uint32_t)ssub[i]);
    }
    rp.dst_sub_total = FastDiv((uint32_t)dsub_total);
    const int64_t run = std::gcd(ssub[rank - 1], dsub[rank - 1]);
    int vb = 16;
    while (vb > elem_bytes && (((run * elem_bytes) % vb) || (((uintptr_t)src | (uintptr_t)dst) % vb))) vb >>= 1;
    rp.vec_bytes = vb;
    rp.vec_elems = vb / elem_bytes;
    rp.n_vec = (uint64_t)total / rp.vec_elems;
    const int64_t run_vec = run / rp.vec_elems;  // vectors over which both layouts stay contiguous
    rp.group = run_vec % 4 == 0 ? 4 : (run_vec % 2 == 0 ? 2 : 1);
    cudaError_t e = launch_repartition(rp, s);
    return e == cudaSuccess ? TRA_OK : cuda_fail(e, "repartition launch");
}

int ein_repartition_cost(int rank, const int64_t* shape, const int32_t* src_d, const int32_t* dst_d,
                         uint64_t* cost) {
    clear_error();
    if (rank < 1 || rank > TRA_MAX_RANK) return fail(TRA_ERR_RANK, "rank %d outside 1..%d", rank, TRA_MAX_RANK);
    if (!shape || !src_d || !dst_d || !cost) return fail(TRA_ERR_ARG, "NULL argument");
    for (int i = 0; i < rank; ++i) {
        if (shape[i] < 1) return fail(TRA_ERR_ARG, "extent < 1");
        if (src_d[i] < 1 || dst_d[i] < 1 || shape[i] % src_d[i] || shape[i] % dst_d[i])
            return fail(TRA_ERR_DIVISIBILITY, "partition count does not divide extent %lld", (long long)shape[i]);
    }
    *cost = repartition_cost_elems(rank, shape, src_d, dst_d);
    return TRA_OK;
}

int ein_repartition_messages(int rank, const int64_t* shape, const int32_t* src_d, const int32_t* dst_d,
                             uint64_t* messages) {
    clear_error();
    if (rank < 1 || rank > TRA_MAX_RANK) return fail(TRA_ERR_RANK, "rank %d outside 1..%d", rank, TRA_MAX_RANK);
    if (!shape || !src_d || !dst_d || !messages) return fail(TRA_ERR_ARG, "NULL argument");
    for (int i = 0; i < rank; ++i) {
        if (shape[i] < 1) return fail(TRA_ERR_ARG, "extent < 1");
        if (src_d[i] < 1 || dst_d[i] < 1 || shape[i] % src_d[i] || shape[i] % dst_d[i])
            return fail(TRA_ERR_DIVISIBILITY, "partition count does not divide extent %lld", (long long)shape[i]);
    }
    *messages = repartition_messages(rank, shape, src_d, dst_d);
    return TRA_OK;
}

int ein_status(tra_stream_t stream) {
    clear_error();
    int v = 0, va = 0, vr = 0;
    cudaError_t e = read_and_clear_status(&v, reinterpret_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) e = read_and_clear_attn_status(&va, reinterpret_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) e = read_and_clear_rp_status(&vr, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "status read");
    if (!v) v = va ? va : vr;
    if (v) return fail(v, "a bounded device wait gave up (status %d)", v);
    // check builds: the first out-of-range access site of each kernel unit (0 = none)
    int c[3] = {0, 0, 0};
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    e = read_and_clear_check_semiring(&c[0], st);
    if (e == cudaSuccess) e = read_and_clear_check_misc(&c[1], st);
    if (e == cudaSuccess) e = read_and_clear_check_tc(&c[2], st);
    if (e != cudaSuccess) return cuda_fail(e, "check word read");
    for (int i = 0; i < 3; ++i)
        if (c[i]) return fail(TRA_ERR_BOUNDS, "an index outside its buffer was skipped at check site %d", c[i]);
    return TRA_OK;
}

int ein_selftest_wait_timeout(uint64_t timeout_ns, tra_stream_t stream) {
    clear_error();
    cudaError_t e = launch_wait_timeout_probe(timeout_ns, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TRA_OK : cuda_fail(e, "wait probe launch");
}

void ein_plan_destroy(tra_plan_t plan) { delete reinterpret_cast<Plan*>(plan); }

int ein_build_flags(void) { return kCheckBuild ? TRA_BUILD_CHECK : 0; }

const char* ein_last_error(void) { return last_error(); }

}  // extern "C"
